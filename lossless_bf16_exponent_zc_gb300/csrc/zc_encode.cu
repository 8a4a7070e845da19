// zc_encode.cu -- the encoder: bf16 -> ZC1 main stream + escape stream in one launch.
//
// [ZipCCL §2.B] split, remap to 3-bit codes, escapes to a separate array;
// [ZipCCL §2.C] three 1-bit code arrays in column-major order, 128-byte
// aligned blocks, asynchronous global->shared staging with double (here
// triple) buffering.
//
// Design on sm_103a: a persistent, cooperatively launched grid of 12-warp
// CTAs, one CTA per SM.  A CTA works through groups of 12 consecutive tiles
// (group G, G + C, G + 2C, ... for C CTAs); warp w encodes tile w of each
// group from shared memory, where one TMA bulk copy per tile has staged it
// (2 stages per warp, 192 KB per SM).  The group is the unit of the escape
// scan: the warps' escape counts meet in shared memory, a 13th "scan" warp
// publishes the group's count and finds the group's escape offset with a
// single-pass decoupled look-back over preceding groups, and the encoding
// warps, one round later, write their tiles' escapes at their final global
// positions (no second pass).  Escapes wait in a small per-warp buffer so the
// tile's stage is refilled at once; the look-back gets a whole round of slack.
// One look-back participant per SM instead of one per warp keeps the
// resolved front ahead of the tiles; the cooperative launch guarantees every
// group owner is resident, which the look-back's waits rely on.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kEncWarps = 12;                   // encoding warps; warp 12 is the scan warp
constexpr int kEncThreads = (kEncWarps + 1) * 32;
constexpr int kEncStages = 2;
constexpr uint32_t kGroupTiles = kEncWarps;     // tiles per look-back group (one per encoding warp)
constexpr uint32_t kEncStageBytes = kTile * 2;  // 8192
constexpr uint32_t kEncEscBuf = 512;            // staged escapes per tile; more falls back to the tile itself
// After 1 KB alignment: per-warp LUTs (1 KB each, 1 KB aligned), per-warp stage
// barriers, CTA round bookkeeping, per-warp escape buffers, per-warp stages.
constexpr uint32_t kEncLutOff = 0;
constexpr uint32_t kEncBarOff = kEncWarps * 1024;
constexpr uint32_t kEncGrpOff = kEncBarOff + 256;
constexpr uint32_t kEncEbufOff = kEncGrpOff + 512;
constexpr uint32_t kEncStageOff = kEncEbufOff + kEncWarps * kEncStages * kEncEscBuf;
constexpr uint32_t kEncSmem = 1024 + kEncStageOff + kEncWarps * kEncStages * kEncStageBytes;

template <int MAXB>
struct EncParams {
  EncTensor t[MAXB];
  uint32_t group_start[MAXB + 1];  // first global group of each tensor; [count] = total
  int count;
  uint32_t total_groups;
  WsHeader* ws;
  Flag* flags;  // one per group
  int32_t* status;
};

template <int MAXB>
__device__ __forceinline__ uint32_t locate_group(const EncParams<MAXB>& p, uint32_t G) {
  uint32_t ti = 0;
  if (MAXB > 1)
    while (static_cast<int>(ti) + 1 < p.count && G >= p.group_start[ti + 1]) ti++;
  return ti;
}

// CTA bookkeeping of the two rounds in flight (index = round parity).  A slot
// of round j + 2 is written only after every warp is done with round j: the
// counts after the scan warp consumed them (it posts round j's prefixes before
// any warp can finish round j + 1), the prefixes after every warp has arrived
// with its round j + 2 count (which it does after finishing round j).
struct RoundShared {
  uint32_t cnt[kEncStages][16];                // escape count of each encoding warp's tile
  unsigned long long tprefix[kEncStages][16];  // exclusive escape offset of each warp's tile
  uint64_t cnt_bar[kEncStages];                // 12 arrivals: all counts of the round are in
  uint64_t pre_bar[kEncStages];                // 1 arrival: the scan warp has posted the prefixes
};

// What an encoding warp remembers about its tile of a round until the
// round's prefix is known.
struct Pending {
  bool has;       // the warp had a tile this round
  bool spilled;   // more escapes than the staging buffer: written from the tile itself
  uint32_t ti, lt;
  TileEsc te;
};

template <int MAXB>
__global__ void __launch_bounds__(kEncThreads, 1) encode_kernel(const __grid_constant__ EncParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;  // 1 KB aligned shared address
  uint8_t* gbase = smem + (sbase - smem_u32(smem));           // its generic pointer
  RoundShared* rs = reinterpret_cast<RoundShared*>(gbase + kEncGrpOff);
  const uint32_t epoch = launch_epoch(p.ws);
  const uint32_t hold = launch_hold(p.ws);
  const uint32_t step = gridDim.x;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; s++) {
      mbar_init(&rs->cnt_bar[s], kEncWarps);
      mbar_init(&rs->pre_bar[s], 1);
    }
  }
  const uint32_t w = warp < kEncWarps ? warp : 0;  // per-warp regions (the scan warp uses none)
  uint32_t* lut = reinterpret_cast<uint32_t*>(gbase + kEncLutOff + w * 1024);
  const uint32_t lut_s = sbase + kEncLutOff + w * 1024;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gbase + kEncBarOff + w * 16);
  uint8_t* ebuf = gbase + kEncEbufOff + w * kEncStages * kEncEscBuf;
  uint8_t* wstage = gbase + kEncStageOff + w * kEncStages * kEncStageBytes;
  const uint32_t wstage_s = sbase + kEncStageOff + w * kEncStages * kEncStageBytes;
  if (warp < kEncWarps && lane == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; s++) mbar_init(&bar[s], 1);
  }
  if (lane == 0) fence_mbar_init();
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
    // ---------------- scan warp: one decoupled look-back per group
    int cur_ti = -1;
    bool cb_ok = true;
    uint32_t j = 0;
    for (uint32_t G = blockIdx.x; G < p.total_groups; G += step, j++) {
      const int s = static_cast<int>(j & 1u);
      const uint32_t ti = locate_group(p, G);
      if (static_cast<int>(ti) != cur_ti) {
        cur_ti = static_cast<int>(ti);
        const uint8_t* cb = p.t[ti].cb;
        cb_ok = true;
#pragma unroll
        for (int a = 0; a < 7; a++)
#pragma unroll
          for (int b = a + 1; b < 7; b++) cb_ok &= __ldg(cb + a) != __ldg(cb + b);
      }
      mbar_wait_bounded(&rs->cnt_bar[s], (j >> 1) & 1u, p.status);
      const uint32_t gl = G - p.group_start[ti];
      uint64_t prefix = 0;
      if (cb_ok && hold != G + 1) {
        const uint32_t agg = warp_sum(lane < kGroupTiles ? rs->cnt[s][lane] : 0u);
        const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
        if (gl == 0) {
          if (lane == 0) st_relaxed(&p.flags[G].incl, tag | agg);
        } else {
          if (lane == 0) st_relaxed(&p.flags[G].agg, tag | agg);
          bool timed_out;
          prefix = lookback(p.flags, G, G - gl, epoch, p.status, &timed_out);
          if (lane == 0) st_relaxed(&p.flags[G].incl, tag | static_cast<uint32_t>(prefix + agg));
        }
      }
      // per-tile offsets: the group's prefix plus the counts of the tiles before
      const uint32_t c = lane < kGroupTiles ? rs->cnt[s][lane] : 0u;
      const uint32_t inc = warp_inclusive_scan(c);
      if (lane < kGroupTiles) rs->tprefix[s][lane] = prefix + (inc - c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs->pre_bar[s]);  // release: the prefixes are visible to waiters
    }
  } else {
    // ---------------- encoding warps
    auto stage_ptr = [&](int s) { return reinterpret_cast<uint16_t*>(wstage + s * kEncStageBytes); };
    auto my_tile = [&](uint32_t G, uint32_t& ti, uint32_t& lt) {
      ti = locate_group(p, G);
      lt = (G - p.group_start[ti]) * kGroupTiles + warp;
      return static_cast<uint64_t>(lt) < num_tiles(p.t[ti].n);
    };
    auto issue = [&](int s, uint32_t G) {
      if (G >= p.total_groups) return;
      uint32_t ti, lt;
      if (!my_tile(G, ti, lt)) return;
      const uint64_t rem = p.t[ti].n - static_cast<uint64_t>(lt) * kTile;
      if (lane == 0) {
        if (rem >= kTile) {
          fence_proxy_async();
          mbar_arrive_expect_tx(&bar[s], kEncStageBytes);
          tma_load_1d(stage_ptr(s), p.t[ti].in + static_cast<uint64_t>(lt) * kTile, kEncStageBytes, &bar[s]);
        } else {
          mbar_arrive(&bar[s]);  // ragged last tile: filled by plain loads when consumed
        }
      }
    };
    // Second half of round j (stage s): the group's prefix has been posted;
    // write the offset-table entry, this tile's header parts and escapes.
    auto finish = [&](uint32_t j, int s, uint32_t G, const Pending& pd) {
      mbar_wait_bounded(&rs->pre_bar[s], (j >> 1) & 1u, p.status);
      if (pd.has) {
        const EncTensor& T = p.t[pd.ti];
        const uint64_t ntiles = num_tiles(T.n);
        const uint64_t prefix = rs->tprefix[s][warp];
        if (lane == 0) *reinterpret_cast<uint32_t*>(T.main + kHeader + 4ull * pd.lt) = static_cast<uint32_t>(prefix);
        if (pd.lt == 0) write_header_words(T.main, T.n, T.cb);
        if (pd.lt + 1 == ntiles) {
          const uint64_t n_esc = prefix + pd.te.total;
          write_header_tail(T.main, ntiles, n_esc);
          if (lane == 0 && n_esc > T.esc_cap) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
        }
        if (pd.spilled) {
          write_escapes(wstage_s + s * kEncStageBytes, pd.te, prefix, T.esc, T.esc_cap);
        } else {
          const uint8_t* src = ebuf + s * kEncEscBuf;
          const uint64_t cap = T.esc_cap;
          for (uint32_t i = lane; i < pd.te.total; i += 32)
            if (prefix + i < cap) T.esc[prefix + i] = src[i];
        }
      }
      __syncwarp();
      if (pd.spilled) issue(s, G + kEncStages * step);  // the stage was held for the escapes
    };

#pragma unroll
    for (int s = 0; s < kEncStages; s++) issue(s, blockIdx.x + s * step);

    uint32_t phase = 0;
    int cur_ti = -1;
    bool cb_ok = true;
    Pending prev;
    prev.has = false;
    prev.spilled = false;
    uint32_t j = 0;
    for (uint32_t G = blockIdx.x; G < p.total_groups; G += step, j++) {
      const int s = static_cast<int>(j & 1u);
      Pending cur;
      cur.has = my_tile(G, cur.ti, cur.lt);
      cur.spilled = false;
      cur.te.total = 0;
      const EncTensor& T = p.t[cur.ti];
      if (static_cast<int>(cur.ti) != cur_ti) {
        cb_ok = build_enc_lut(lut, T.cb);  // every warp of the group reaches the same verdict
        cur_ti = static_cast<int>(cur.ti);
        if (!cb_ok && lane == 0) set_status(p.status, ZC_ERR_DUP_CODEBOOK);
      }
      if (cur.has) {
        const uint32_t tb_s = wstage_s + s * kEncStageBytes;
        const uint64_t rem = T.n - static_cast<uint64_t>(cur.lt) * kTile;
        const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
        mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        if (n_tile < kTile) {
          uint16_t* tb = stage_ptr(s);
          const uint16_t* src = T.in + static_cast<uint64_t>(cur.lt) * kTile;
          for (uint32_t i = lane; i < kTile; i += 32) tb[i] = i < n_tile ? src[i] : static_cast<uint16_t>(0);
          __syncwarp();
        }
        if (cb_ok) {
          encode_tile(tb_s, n_tile, lut_s, tile_ptr(T.main, num_tiles(T.n), cur.lt), cur.te);
          cur.spilled = cur.te.total > kEncEscBuf;
          if (!cur.spilled) stage_tile_escapes(tb_s, cur.te, ebuf + s * kEncEscBuf);
        } else {
          cur.has = false;
        }
      }
      if (lane == 0) {
        rs->cnt[s][warp] = cur.te.total;
        mbar_arrive(&rs->cnt_bar[s]);  // release: the count is visible to the scan warp
      }
      __syncwarp();
      if (!cur.spilled) issue(s, G + kEncStages * step);  // refill now; escapes are staged
      if (j > 0) finish(j - 1, s ^ 1, G - step, prev);
      prev = cur;
    }
    if (j > 0) finish(j - 1, static_cast<int>((j - 1) & 1u), blockIdx.x + (j - 1) * step, prev);
  }
  cta_exit(p.ws, p.flags, epoch, p.total_groups);
}

template <int MAXB>
static cudaError_t launch_encode_t(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                                   cudaStream_t stream, const DeviceInfo& dev) {
  EncParams<MAXB> p;
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
  static_assert(sizeof(RoundShared) <= 512, "round bookkeeping too large");
  cudaError_t err = cudaFuncSetAttribute(encode_kernel<MAXB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEncSmem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kernel<MAXB>, kEncThreads, kEncSmem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  uint32_t ctas = groups;
  const uint32_t cap = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&p};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(encode_kernel<MAXB>), dim3(ctas),
                                     dim3(kEncThreads), args, kEncSmem, stream);
}

cudaError_t launch_encode(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                          cudaStream_t stream, const DeviceInfo& dev) {
  if (count == 1) return launch_encode_t<1>(ts, count, ws, flags, status, stream, dev);
  return launch_encode_t<kMaxBatch>(ts, count, ws, flags, status, stream, dev);
}

}  // namespace zc
