// zc_encode.cu -- the encoder: bf16 -> ZC1 main stream + escape stream in one launch.
//
// [ZipCCL §2.B] split, remap to 3-bit codes, escapes to a separate array;
// [ZipCCL §2.C] three 1-bit code arrays in column-major order, 128-byte
// aligned blocks, asynchronous global->shared staging with double buffering.
//
// Design on sm_103a: a persistent, cooperatively launched grid, one CTA of 12
// warps per SM.  The work unit of a warp is a whole tile (4 blocks, 4096
// values, one 8 KB TMA bulk copy into one of its two shared-memory stages): a
// unit's fixed work (stage wait and refill, counts, offset-table entry, queue)
// is spread over twice the values of a half-tile unit, and the registers an
// 11-warp CTA may use (up to 168 a thread) hold four blocks' bookkeeping.  A
// CTA works through groups of 11 consecutive tiles (group G, G + C, ... for C
// CTAs); encoding warp w takes tile w of each group.  The group is the unit
// of the escape scan: the warps' escape counts meet in shared memory, the
// last encoding warp to finish a group publishes the group's count at once,
// the 12th "scan" warp finds the group's escape offset and posts the group's
// offsets in shared memory.
//
// CTAs drift apart by several rounds (the order in which HBM serves their
// loads), and a group's offset is known only once every group before it is
// encoded, so an encoding warp never waits for its offsets while it has
// work: it keeps each unit's escapes in a per-warp shared-memory ring, with
// a queue of up to 16 rounds in flight, and writes a round's offset-table
// entry, header parts and escapes to global memory whenever it finds that
// round's offsets posted.  It blocks only when the ring or the queue is full,
// and at the end.  A stage is refilled as soon as its data is encoded; a unit
// with more escapes than a ring share waits for its offsets and writes them
// from the stage itself.  The scan warp knows the inclusive offset of its own
// previous group, so it needs only the counts of the C - 1 groups in between,
// which their encoders publish without waiting on anyone; it adds them up
// while its own CTA is still encoding the group.  The cooperative launch
// guarantees every group owner is resident, which the waits rely on.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

// Shape of the encoder (measured on 2^26 values, the batched MoE payload and
// the batched Llama-3-8B bucket: whole-tile units on 11 warps beat half-tile
// units on 20 warps by 2-4%, with identical streams).
#ifndef ZC_ENC_UNIT_BLOCKS
#define ZC_ENC_UNIT_BLOCKS 4  // blocks per warp unit: 4 (a tile) or 2 (half a tile)
#endif
#ifndef ZC_ENC_WARPS
#define ZC_ENC_WARPS 11  // encoding warps (units per escape-scan group)
#endif
#ifndef ZC_ENC_RING
#define ZC_ENC_RING 1024  // per-warp escape ring, bytes
#endif
constexpr int kEncWarps = ZC_ENC_WARPS;         // encoding warps; the next warp is the scan warp
constexpr int kEncThreads = (kEncWarps + 1) * 32;
constexpr int kEncStages = 2;
constexpr uint32_t kUnitBlocks = ZC_ENC_UNIT_BLOCKS;  // blocks per warp unit
constexpr uint32_t kUnitElems = kUnitBlocks * kBlock;
constexpr uint32_t kUnitsPerTile = kTile / kUnitElems;
constexpr uint32_t kGroupUnits = kEncWarps;     // units per scan group (one per encoding warp)
constexpr uint32_t kGroupTiles = kGroupUnits / kUnitsPerTile;
constexpr uint32_t kEncStageBytes = kUnitElems * 2;  // 4096
constexpr int kEncSlots = 16;                   // rounds in flight per warp (round slot = round mod 16)
constexpr uint32_t kEncRing = ZC_ENC_RING;      // per-warp escape ring (bytes, a power of two)
constexpr uint32_t kEncRingUnitMax = kEncRing / 2;  // a unit with more escapes bypasses the ring
constexpr uint32_t kEncQEntry = 16;             // bytes per queued round
// After 1 KB alignment: per-warp LUTs (1 KB each, 1 KB aligned), per-warp stage
// barriers, CTA round bookkeeping, per-warp round queues, per-warp escape
// rings, per-warp stages.
constexpr uint32_t kEncLutOff = 0;
constexpr uint32_t kEncBarOff = kEncWarps * 1024;
constexpr uint32_t kEncGrpOff = kEncBarOff + 512;
constexpr uint32_t kEncGrpBytes = 4352;
constexpr uint32_t kEncQueueOff = kEncGrpOff + kEncGrpBytes;
constexpr uint32_t kEncRingOff = kEncQueueOff + kEncWarps * kEncSlots * kEncQEntry;
constexpr uint32_t kEncStageOff = kEncRingOff + kEncWarps * kEncRing;
constexpr uint32_t kEncSmem = 1024 + kEncStageOff + kEncWarps * kEncStages * kEncStageBytes;
static_assert(kGroupUnits % kUnitsPerTile == 0, "a group holds whole tiles");

template <int MAXB>
struct EncParams {
  EncTensor t[MAXB];
  uint32_t group_start[MAXB + 1];  // first global group of each tensor; [count] = total
  int count;
  uint32_t total_groups;
  WsHeader* ws;
  Flag* flags;  // one per group
  int32_t* status;
  int adaptive;  // the raw bypass runs at the end; an escape overflow is reported by it
};

// Tensor of global group G.  Every caller visits groups in increasing order,
// so it keeps a running index (`ti`, starting at 0) and only moves it forward.
template <int MAXB>
__device__ __forceinline__ uint32_t locate_group(const EncParams<MAXB>& p, uint32_t G, uint32_t& ti) {
  if (MAXB > 1)
    while (static_cast<int>(ti) + 1 < p.count && G >= p.group_start[ti + 1]) ti++;
  return MAXB > 1 ? ti : 0u;
}

// CTA bookkeeping of the rounds in flight (slot = round mod 16).  A warp
// finishes round j (after waiting for its offsets) before it starts round
// j + 16, so a slot is reused only after every warp is done with round j: the
// counts and the arrival word after the scan warp consumed them (it posts
// round j's offsets only after that), the offsets after every warp has
// arrived with its round j + 16 count.
struct RoundShared {
  uint32_t agg[kEncSlots];                           // arrivals << 16 | escape count so far (the last warp publishes)
  uint32_t cnt[kEncSlots][kEncWarps];                // escape count of each encoding warp's unit
  unsigned long long uprefix[kEncSlots][kEncWarps];  // exclusive escape offset of each warp's unit
  uint64_t cnt_bar[kEncSlots];                       // kEncWarps arrivals: all counts of the round are in
  uint64_t pre_bar[kEncSlots];                       // 1 arrival: the scan warp has posted the offsets
};
static_assert(sizeof(RoundShared) <= kEncGrpBytes, "round bookkeeping too large");

// A round queued by an encoding warp until its offsets are known.  The
// unit's escapes sit in the warp's ring at byte start % kEncRing (start is a
// running byte count; an allocation never wraps around the ring's end).
struct QEntry {
  uint32_t lt;     // local tile of the unit
  uint32_t start;  // ring position of its escapes
  uint16_t ti;     // tensor
  uint16_t cnt;    // escapes
  uint32_t has;    // the warp had a unit this round
};
static_assert(sizeof(QEntry) == kEncQEntry, "queue entry size");
static_assert(kEncRingUnitMax <= kEncRing, "a ring share fits the ring");
static_assert((kEncRing & (kEncRing - 1)) == 0, "ring positions stay contiguous across 32-bit wrap-around");

// ---------------------------------------------------------------- raw bypass
// [CCCL §3.3] leaves tensors uncompressed when compressing them does not pay;
// [CCCL §5.2] falls back to the uncompressed data when the ratio is near or
// above 1.  With ZC1's fixed-size main stream the comparison is exact: both
// forms send the same main stream, the coded form n_esc escape bytes, the RAW
// form max(0, 2n - 5632 ntiles) spill bytes; RAW is chosen exactly when n_esc
// exceeds the spill (and the spill fits the escape buffer).

// Tensor T goes RAW; a tensor whose codebook repeats an entry was not encoded
// (reported) and stays as it is.  *overflow: the coded form stays and its
// escapes did not fit.
__device__ __forceinline__ bool goes_raw(const EncTensor& T, bool* overflow) {
  *overflow = false;
  bool dup = false;
  for (int a = 0; a < 7; a++)
    for (int b = a + 1; b < 7; b++) dup |= __ldg(T.cb + a) == __ldg(T.cb + b);
  if (dup) return false;
  const uint64_t n_esc = __ldcg(reinterpret_cast<const unsigned long long*>(T.main + 24));
  const uint64_t spill = raw_spill(T.n);
  if (n_esc > spill && spill <= T.esc_cap) return true;
  *overflow = n_esc > T.esc_cap;
  return false;
}

// Rewrites T as a RAW stream, 16-byte pieces over the threads of the grid: the
// offset table zeroed, the tile region and the spill filled from the input
// (zero past 2n).  The header is written afterwards by the last CTA.
__device__ __forceinline__ void raw_rewrite(const EncTensor& T, uint64_t tid, uint64_t nthreads) {
  constexpr int kUnroll = 4;  // 16-byte copies in flight per thread
  const uint64_t ntiles = num_tiles(T.n);
  const uint64_t tbl = table_bytes(ntiles);  // a multiple of 128
  const uint64_t region = static_cast<uint64_t>(kTileBytes) * ntiles;
  const uint64_t spill = raw_spill(T.n), two_n = 2 * T.n;
  uint8_t* tiles = T.main + kHeader + tbl;
  const uint64_t table_chunks = tbl / 16;
  const uint64_t image_chunks = (region + spill + 15) / 16;
  auto load = [&](uint64_t b) -> uint4 {
    if (b + 16 <= two_n) return __ldg(reinterpret_cast<const uint4*>(T.in + b / 2));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (uint32_t j = 0; b + 2 * j < two_n; j++)
      w[j >> 1] |= static_cast<uint32_t>(__ldg(T.in + b / 2 + j)) << (16 * (j & 1));
    return make_uint4(w[0], w[1], w[2], w[3]);
  };
  auto store = [&](uint64_t b, uint4 v) {
    if (b < region) {
      *reinterpret_cast<uint4*>(tiles + b) = v;  // zero past 2n: the tile region's tail
      return;
    }
    uint8_t* dst = T.esc + (b - region);
    const uint64_t left = spill - (b - region);  // spill bytes from here, even
    if (left >= 16) {
      *reinterpret_cast<uint4*>(dst) = v;
    } else {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      for (uint32_t j = 0; 2 * j < left; j++)
        reinterpret_cast<uint16_t*>(dst)[j] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
    }
  };
  for (uint64_t c = tid; c < table_chunks; c += nthreads)
    *reinterpret_cast<uint4*>(T.main + kHeader + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
  for (uint64_t c0 = tid; c0 < image_chunks; c0 += kUnroll * nthreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const uint64_t c = c0 + u * nthreads;
      v[u] = c < image_chunks ? load(16 * c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const uint64_t c = c0 + u * nthreads;
      if (c < image_chunks) store(16 * c, v[u]);
    }
  }
}

// The raw bypass of an adaptive launch, run by every thread once its CTA's
// encoding is done.  The CTAs meet at a grid barrier (the launch is
// cooperative), so every tensor's n_esc is final; each CTA reads the counts
// and reaches the same decision.  In the usual case nothing goes RAW and that
// is all: no further launch, no counter.  Otherwise every thread of the grid
// rewrites the RAW tensors, and the last CTA to finish -- after every CTA has
// read the counts -- writes their RAW headers (flags and n_esc).  A CTA whose
// barrier wait runs out (ZC_ERR_TIMEOUT, after an earlier wait of the launch
// ran out) skips the bypass; as after any device error, the workspace is
// zeroed again before it is reused.
template <int MAXB>
__device__ __forceinline__ void raw_bypass(const EncParams<MAXB>& p) {
  static_assert(MAXB <= 32, "one mask bit per tensor");
  __shared__ uint32_t raw_mask;
  __shared__ int raw_ok;
  __syncthreads();  // this CTA's streams, headers included, are written
  if (threadIdx.x == 0) {
    raw_mask = 0;
    raw_ok = grid_barrier(&p.ws->raw_arrived, &p.ws->raw_gen, p.status);
  }
  __syncthreads();
  if (raw_ok) {
    for (int i = threadIdx.x; i < p.count; i += blockDim.x) {
      bool overflow;
      if (goes_raw(p.t[i], &overflow)) atomicOr(&raw_mask, 1u << i);
      if (overflow && blockIdx.x == 0) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
    }
  }
  __syncthreads();
  const uint32_t mask = raw_mask;
  if (mask == 0) return;  // every CTA reached the same decision
  const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t nthreads = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (int i = 0; i < p.count; i++)
    if ((mask >> i) & 1u) raw_rewrite(p.t[i], tid, nthreads);
  __syncthreads();
  if (threadIdx.x == 0 && atom_add_acq_rel_gpu(&p.ws->raw_done, 1u) == gridDim.x - 1) {
    for (int i = 0; i < p.count; i++) {
      if (!((mask >> i) & 1u)) continue;
      uint8_t* m = p.t[i].main;
      *reinterpret_cast<uint32_t*>(m + 4) = ZC_VERSION | (kFlagRaw << 16);
      *reinterpret_cast<unsigned long long*>(m + 24) = raw_spill(p.t[i].n);
    }
    p.ws->raw_done = 0;
  }
}

template <int MAXB>
__global__ void __launch_bounds__(kEncThreads, 1) encode_kernel(const __grid_constant__ EncParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;  // 1 KB aligned shared address
  uint8_t* gbase = smem + (sbase - smem_u32(smem));           // its generic pointer
  RoundShared* rs = reinterpret_cast<RoundShared*>(gbase + kEncGrpOff);
  pdl_allow_dependents();  // (the wait for the previous grid comes after the shared-memory setup)
  const uint32_t step = gridDim.x;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int r = 0; r < kEncSlots; r++) {
      mbar_init(&rs->cnt_bar[r], kEncWarps);
      mbar_init(&rs->pre_bar[r], 1);
      rs->agg[r] = 0;
    }
  }
  const uint32_t w = warp < kEncWarps ? warp : 0;  // per-warp regions (the scan warp uses none)
  uint32_t* lut = reinterpret_cast<uint32_t*>(gbase + kEncLutOff + w * 1024);
  const uint32_t lut_s = sbase + kEncLutOff + w * 1024;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gbase + kEncBarOff + w * 16);
  QEntry* queue = reinterpret_cast<QEntry*>(gbase + kEncQueueOff + w * kEncSlots * kEncQEntry);
  uint8_t* ring = gbase + kEncRingOff + w * kEncRing;
  uint8_t* wstage = gbase + kEncStageOff + w * kEncStages * kEncStageBytes;
  const uint32_t wstage_s = sbase + kEncStageOff + w * kEncStages * kEncStageBytes;
  if (warp < kEncWarps && lane == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; s++) mbar_init(&bar[s], 1);
    fence_mbar_init();  // (thread 0's round barriers above included)
  }
  pdl_wait();
  auto stage_ptr = [&](int s) { return reinterpret_cast<uint16_t*>(wstage + s * kEncStageBytes); };
  const uint32_t half = warp % kUnitsPerTile;  // this warp's half of each tile of a group
  uint32_t issue_ti = 0;  // running tensor index of issue()
  // issue()'s view of its current tensor, kept while the tensor lasts
  int issue_cur = -1;
  uint64_t issue_n = 0;
  const uint16_t* issue_in = nullptr;
  uint32_t issue_ntiles = 0, issue_g0 = 0;
  auto issue = [&](int s, uint32_t G) {
    if (G >= p.total_groups) return;
    const uint32_t ti = locate_group(p, G, issue_ti);
    if (static_cast<int>(ti) != issue_cur) {
      issue_cur = static_cast<int>(ti);
      issue_n = p.t[ti].n;
      issue_in = p.t[ti].in;
      issue_ntiles = static_cast<uint32_t>(num_tiles(issue_n));
      issue_g0 = p.group_start[ti];
    }
    const uint32_t lt = (G - issue_g0) * kGroupTiles + warp / kUnitsPerTile;
    if (lt >= issue_ntiles) return;
    if (lane == 0) {
      const uint64_t start = static_cast<uint64_t>(lt) * kTile + half * kUnitElems;
      if (issue_n >= start + kUnitElems) {
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[s], kEncStageBytes);
        tma_load_1d(stage_ptr(s), issue_in + start, kEncStageBytes, &bar[s]);
      } else {
        mbar_arrive(&bar[s]);  // ragged end of the tensor: filled by plain loads when consumed
      }
    }
  };
  // Each encoding warp starts its first two loads before anything reads global
  // memory (the epoch, the test hook, codebooks), so HBM is busy from the start.
  if (warp < kEncWarps) {
    __syncwarp();
#pragma unroll
    for (int s = 0; s < kEncStages; s++) issue(s, blockIdx.x + s * step);
  }
  // (thread 0's round barriers were initialised before its fence above; no
  // fence after the copies: a release fence would wait for them)
  // the launch's epoch and test hook, read by every thread before the barrier
  // that precedes the scan warp's count (scan_arrive)
  const uint32_t epoch = launch_epoch(p.ws);
  const uint32_t hold = launch_hold(p.ws);
  __syncthreads();

  // Tensors without tiles still get a header.
  if (blockIdx.x == 0 && warp == 0) {
    for (int i = 0; i < p.count; i++) {
      if (p.t[i].n != 0) continue;
      if (build_enc_lut(lut, p.t[i].cb)) {
        write_header_words(p.t[i].main, 0, p.t[i].cb);
        write_header_tail(p.t[i].main, 0, 0);
      } else if (lane == 0) {
        set_status(p.status, ZC_ERR_DUP_CODEBOOK);
      }
      __syncwarp();
    }
  }

  if (warp == kEncWarps) {
    // ---------------- scan warp: the escape offsets of each group
    const uint32_t arrival = lane == 0 ? scan_arrive(p.ws, epoch) : kNoArrival;
    int cur_ti = -1;
    const uint8_t* cur_cb = nullptr;
    bool cb_ok = true;
    uint32_t run_ti = 0;
    int64_t prev_G = -1;     // this CTA's previous group ...
    uint64_t prev_incl = 0;  // ... and its inclusive escape offset
    uint32_t j = 0;
    for (uint32_t G = blockIdx.x; G < p.total_groups; G += step, j++) {
      const int r = static_cast<int>(j % kEncSlots);  // round slot
      const uint32_t ph = (j / kEncSlots) & 1u;       // its barrier phase
      const uint32_t ti = locate_group(p, G, run_ti);
      if (static_cast<int>(ti) != cur_ti) {
        cur_ti = static_cast<int>(ti);
        const uint8_t* cb = p.t[ti].cb;
        if (cb != cur_cb) {  // tensors that share a codebook share the decision
          cur_cb = cb;
          cb_ok = true;
#pragma unroll
          for (int a = 0; a < 7; a++)
#pragma unroll
            for (int b = a + 1; b < 7; b++) cb_ok &= __ldg(cb + a) != __ldg(cb + b);
        }
      }
      // the groups between this CTA's previous group and G: their counts are
      // published by their encoders, so this overlaps the CTA's own encoding
      const uint32_t g0 = p.group_start[ti];
      const bool own = prev_G >= static_cast<int64_t>(g0);  // previous group of this CTA, same tensor
      uint64_t prefix = 0;
      if (cb_ok) {
        bool timed_out;
        prefix = (own ? prev_incl : 0) +
                 window_sum(p.flags, own ? static_cast<uint32_t>(prev_G) + 1 : g0, G, epoch, p.status, &timed_out);
      }
      mbar_wait_bounded(&rs->cnt_bar[r], ph, p.status);
      if (lane == 0) rs->agg[r] = 0;  // every warp has added to it; ready for round j + kEncSlots
      const uint32_t c = lane < kGroupUnits ? rs->cnt[r][lane] : 0u;
      const uint32_t inc = warp_inclusive_scan(c);
      prev_G = G;
      prev_incl = prefix + __shfl_sync(kFull, inc, 31);
      if (lane < kGroupUnits) rs->uprefix[r][lane] = prefix + (inc - c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs->pre_bar[r]);  // release: the offsets are visible to waiters
    }
    scan_exit(p.ws, p.flags, epoch, p.total_groups, arrival);
  } else {
    // ---------------- encoding warps: unit `warp` of every group
    // Second half of round k, once its offsets are posted (slot k mod 16):
    // the offset-table entry and header parts of unit (ti, lt); returns the
    // unit's escape offset.
    auto write_meta = [&](uint32_t k, uint32_t ti, uint32_t lt, uint32_t cnt) -> uint64_t {
      const EncTensor& T = p.t[ti];
      const uint64_t ntiles = num_tiles(T.n);
      const uint64_t prefix = rs->uprefix[k % kEncSlots][warp];
      if (half == 0) {
        if (lane == 0) *reinterpret_cast<uint32_t*>(T.main + kHeader + 4ull * lt) = static_cast<uint32_t>(prefix);
        if (lt == 0) write_header_words(T.main, T.n, T.cb);
      }
      if (half == kUnitsPerTile - 1 && lt + 1 == ntiles) {
        const uint64_t n_esc = prefix + cnt;
        write_header_tail(T.main, ntiles, n_esc);
        if (lane == 0 && n_esc > T.esc_cap && !p.adaptive) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
      }
      return prefix;
    };
    // Finishes queued round k: waits for its offsets, then writes its meta
    // data and moves its escapes from the ring to the escape stream.
    auto finish = [&](uint32_t k) {
      mbar_wait_bounded(&rs->pre_bar[k % kEncSlots], (k / kEncSlots) & 1u, p.status);
      const QEntry e = queue[k % kEncSlots];
      if (e.has) {
        const uint64_t prefix = write_meta(k, e.ti, e.lt, e.cnt);
        const EncTensor& T = p.t[e.ti];
        const uint8_t* src = ring + e.start % kEncRing;
        uint8_t* dst = T.esc + prefix;
        if (prefix + e.cnt <= T.esc_cap) {
          for (uint32_t i = lane; i < e.cnt; i += 32) dst[i] = src[i];
        } else {
          for (uint32_t i = lane; i < e.cnt; i += 32)
            if (prefix + i < T.esc_cap) dst[i] = src[i];
        }
      }
      __syncwarp();
    };

    uint32_t phase = 0;
    int cur_ti = -1;
    const uint8_t* cur_cb = nullptr;
    uint64_t cur_n = 0;            // the current tensor's size ...
    uint32_t cur_ntiles = 0;       // ... tiles ...
    uint8_t* cur_tiles = nullptr;  // ... first tile ...
    uint32_t cur_g0 = 0;           // ... and first group
    bool cb_ok = true;
    uint32_t run_ti = 0;
    uint32_t fin = 0;   // oldest round not finished; rounds fin .. j - 1 are queued
    uint32_t head = 0;  // ring bytes allocated so far (running count)
    uint32_t j = 0;
    for (uint32_t G = blockIdx.x; G < p.total_groups; G += step, j++) {
      const int r = static_cast<int>(j % kEncSlots);
      const int s = static_cast<int>(j & 1u);
      if (j - fin == kEncSlots) finish(fin++);  // slot r is still held by round j - 16
      const uint32_t ti = locate_group(p, G, run_ti);
      const EncTensor& T = p.t[ti];
      if (static_cast<int>(ti) != cur_ti) {  // per-tensor values, kept while the tensor lasts
        cur_ti = static_cast<int>(ti);
        cur_n = T.n;
        cur_ntiles = static_cast<uint32_t>(num_tiles(cur_n));
        cur_tiles = T.main + kHeader + table_bytes(cur_ntiles);
        cur_g0 = p.group_start[ti];
        if (T.cb != cur_cb) {  // tensors that share a codebook (same pointer) share the table
          cb_ok = build_enc_lut(lut, T.cb);  // every warp of the group reaches the same decision
          cur_cb = T.cb;
          if (!cb_ok && lane == 0) set_status(p.status, ZC_ERR_DUP_CODEBOOK);
        }
      }
      const uint32_t lt = (G - cur_g0) * kGroupTiles + warp / kUnitsPerTile;
      bool has = lt < cur_ntiles;
      EscBook<kUnitBlocks> te;
      te.total = 0;
      const uint32_t tb_s = wstage_s + s * kEncStageBytes;
      if (has) {
        const uint64_t start = static_cast<uint64_t>(lt) * kTile + half * kUnitElems;
        const uint32_t nv =
            cur_n <= start ? 0u : (cur_n - start >= kUnitElems ? kUnitElems : static_cast<uint32_t>(cur_n - start));
        const uint64_t rem = cur_n - static_cast<uint64_t>(lt) * kTile;
        const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
        mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        if (nv < kUnitElems) {
          uint16_t* tb = stage_ptr(s);
          const uint16_t* src = T.in + static_cast<uint64_t>(lt) * kTile + half * kUnitElems;
          for (uint32_t i = lane; i < kUnitElems; i += 32) tb[i] = i < nv ? src[i] : static_cast<uint16_t>(0);
          __syncwarp();
        }
        if (cb_ok)
          encode_blocks<kUnitBlocks>(tb_s, half * kUnitBlocks, n_tile, lut_s,
                                     cur_tiles + static_cast<uint64_t>(lt) * kTileBytes + half * kUnitBlocks * kBlockBytes,
                                     te);
        else
          has = false;
      }
      const uint32_t cnt = te.total;
      if (lane == 0) {
        rs->cnt[r][warp] = cnt;
        // the last warp of the group publishes the group's escape count right away
        const uint32_t old = atomicAdd(&rs->agg[r], (1u << 16) | cnt);
        if ((old >> 16) == kEncWarps - 1 && cb_ok && hold != G + 1) {
          const uint32_t agg = (old & 0xFFFFu) + cnt;
          const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
          st_relaxed(&p.flags[G].agg, tag | agg);
        }
        mbar_arrive(&rs->cnt_bar[r]);  // release: the count is visible to the scan warp
      }
      __syncwarp();
      if (cnt <= kEncRingUnitMax) {
        // a contiguous ring share: skip the ring's tail if the share would
        // cross its end; finish old rounds until the share is free
        uint32_t pos;
        for (;;) {
          pos = head;
          if (pos % kEncRing + cnt > kEncRing) pos += kEncRing - pos % kEncRing;
          const uint32_t tail = fin == j ? pos : queue[fin % kEncSlots].start;
          if (pos + cnt - tail <= kEncRing) break;
          finish(fin++);
        }
        if (cnt != 0) stage_escapes_smem<kUnitBlocks>(tb_s, te, ring + pos % kEncRing);
        head = pos + cnt;
        if (lane == 0) {
          QEntry e;
          e.lt = lt;
          e.start = pos;
          e.ti = static_cast<uint16_t>(ti);
          e.cnt = static_cast<uint16_t>(cnt);
          e.has = has;
          queue[r] = e;
        }
        __syncwarp();
        issue(s, G + kEncStages * step);  // refill now; the escapes are in the ring
      } else {
        // too many escapes for the ring: finish everything before, wait for
        // this round's offsets and write the escapes from the stage, a block
        // at a time through the ring (empty now)
        while (fin < j) finish(fin++);
        mbar_wait_bounded(&rs->pre_bar[r], (j / kEncSlots) & 1u, p.status);
        const uint64_t prefix = write_meta(j, ti, lt, cnt);
        write_escapes_coalesced<kUnitBlocks>(tb_s, te, prefix, T.esc, T.esc_cap, ring);
        __syncwarp();
        fin = j + 1;
        issue(s, G + kEncStages * step);
      }
      // finish whatever rounds already have their offsets
      while (fin <= j && mbar_test_wait(&rs->pre_bar[fin % kEncSlots], (fin / kEncSlots) & 1u)) finish(fin++);
    }
    while (fin < j) finish(fin++);  // drain
  }
  if (p.adaptive) raw_bypass(p);
}

template <int MAXB>
static cudaError_t launch_encode_t(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                                   cudaStream_t stream, const DeviceInfo& dev, bool adaptive) {
  EncParams<MAXB> p;
  p.adaptive = adaptive ? 1 : 0;
  uint32_t groups = 0;
  for (int i = 0; i < count; i++) {
    p.t[i] = ts[i];
    p.group_start[i] = groups;
    const uint32_t nt = static_cast<uint32_t>(num_tiles(ts[i].n));
    groups += (nt + kGroupTiles - 1) / kGroupTiles;
  }
  p.group_start[count] = groups;
  p.count = count;
  p.total_groups = groups;
  p.ws = ws;
  p.flags = flags;
  p.status = status;
  static_assert(sizeof(EncParams<MAXB>) < 4000, "encode parameters too large");
  static_assert(kEncSmem + 1024 <= 232448, "shared memory budget");
  static KernelPrep prep;
  int per_sm = 0;
  cudaError_t err =
      prepare_kernel(prep, reinterpret_cast<const void*>(encode_kernel<MAXB>), kEncThreads, kEncSmem, dev, &per_sm);
  if (err != cudaSuccess) return err;
  uint32_t ctas = groups;
  const uint32_t cap = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&p};
  return launch_kernel(reinterpret_cast<const void*>(encode_kernel<MAXB>), dim3(ctas), dim3(kEncThreads), kEncSmem,
                       stream, args, true);
}

cudaError_t launch_encode(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                          cudaStream_t stream, const DeviceInfo& dev, bool adaptive) {
  if (count == 1) return launch_encode_t<1>(ts, count, ws, flags, status, stream, dev, adaptive);
  return launch_encode_t<kMaxBatch>(ts, count, ws, flags, status, stream, dev, adaptive);
}

}  // namespace zc
