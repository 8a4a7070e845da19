// zc_encode.cu -- the encoder: bf16 -> ZC1 main stream + escape stream in one launch.
//
// [ZipCCL §2.B] split, remap to 3-bit codes, escapes to a separate array;
// [ZipCCL §2.C] three 1-bit code arrays in column-major order, 128-byte
// aligned blocks, asynchronous global->shared staging with double buffering.
//
// Design on sm_103a: a persistent, cooperatively launched grid, one CTA of 21
// warps per SM.  The work unit of a warp is half a tile (2 blocks, 2048
// values, one 4 KB TMA bulk copy into one of its two shared-memory stages).  A
// CTA works through groups of 10 consecutive tiles (group G, G + C, ... for C
// CTAs); encoding warp w takes half-tile w of each group.  The group is the
// unit of the escape scan: the warps' escape counts meet in shared memory,
// the last encoding warp to finish a group publishes the group's count at
// once, the 21st "scan" warp finds the group's escape offset with a single-pass
// decoupled look-back, and the encoding warps write their
// escapes at the final global positions two rounds later.  Meanwhile the
// escapes wait in a small per-warp buffer, so a stage is refilled as soon as
// its data is encoded.  The scan warp knows the inclusive offset of its own
// previous group, so a look-back needs only the aggregates of the C - 1 groups
// in between, which are published without waiting on anyone.  The cooperative
// launch guarantees every group owner is resident, which the waits rely on.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kEncWarps = 20;                   // encoding warps; warp 20 is the scan warp
constexpr int kEncThreads = (kEncWarps + 1) * 32;
constexpr int kEncStages = 2;
constexpr uint32_t kUnitBlocks = 2;             // blocks per warp unit (half a tile)
constexpr uint32_t kUnitElems = kUnitBlocks * kBlock;
constexpr uint32_t kUnitsPerTile = kTile / kUnitElems;
constexpr uint32_t kGroupUnits = kEncWarps;     // units per look-back group (one per encoding warp)
constexpr uint32_t kGroupTiles = kGroupUnits / kUnitsPerTile;
constexpr uint32_t kEncStageBytes = kUnitElems * 2;  // 4096
constexpr uint32_t kEncEscBuf = 512;            // staged escapes per unit; more falls back to the stage itself
constexpr int kEncSlots = 3;                    // rounds in flight: a round's escapes are written two rounds later
// After 1 KB alignment: per-warp LUTs (1 KB each, 1 KB aligned), per-warp stage
// barriers, CTA round bookkeeping, per-warp escape buffers, per-warp stages.
constexpr uint32_t kEncLutOff = 0;
constexpr uint32_t kEncBarOff = kEncWarps * 1024;
constexpr uint32_t kEncGrpOff = kEncBarOff + 512;
constexpr uint32_t kEncEbufOff = kEncGrpOff + 1280;
constexpr uint32_t kEncStageOff = kEncEbufOff + kEncWarps * kEncSlots * kEncEscBuf;
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
};

template <int MAXB>
__device__ __forceinline__ uint32_t locate_group(const EncParams<MAXB>& p, uint32_t G) {
  uint32_t ti = 0;
  if (MAXB > 1)
    while (static_cast<int>(ti) + 1 < p.count && G >= p.group_start[ti + 1]) ti++;
  return ti;
}

// CTA bookkeeping of the rounds in flight (slot = round mod 3).  Round j's
// escapes are written in round j + 2, so a slot is reused by round j + 3 only
// after every warp is done with round j: the counts after the scan warp
// consumed them (it posts round j's offsets before any warp can finish round
// j, which happens before that warp writes round j + 3's count), the offsets
// after every warp has arrived with its round j + 3 count.
struct RoundShared {
  uint32_t agg[kEncSlots];                    // arrivals << 16 | escape count so far (the last warp publishes)
  uint32_t cnt[kEncSlots][32];                // escape count of each encoding warp's unit
  unsigned long long uprefix[kEncSlots][32];  // exclusive escape offset of each warp's unit
  uint64_t cnt_bar[kEncSlots];                // kEncWarps arrivals: all counts of the round are in
  uint64_t pre_bar[kEncSlots];                // 1 arrival: the scan warp has posted the offsets
};

// What an encoding warp remembers about its unit of a round until the
// round's offsets are known.
struct Pending {
  bool has;      // the warp had a unit this round
  bool spilled;  // more escapes than the staging buffer: written from the stage itself
  bool done;     // already finished (a spilled unit finishes early to free its stage)
  uint32_t ti, lt;
  EscBook<kUnitBlocks> te;
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
  uint8_t* ebuf = gbase + kEncEbufOff + w * kEncSlots * kEncEscBuf;
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
    int64_t prev_G = -1;     // this CTA's previous group ...
    uint64_t prev_incl = 0;  // ... and its inclusive escape offset
    uint32_t j = 0;
    for (uint32_t G = blockIdx.x; G < p.total_groups; G += step, j++) {
      const int r = static_cast<int>(j % kEncSlots);  // round slot
      const uint32_t ph = (j / kEncSlots) & 1u;       // its barrier phase
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
      mbar_wait_bounded(&rs->cnt_bar[r], ph, p.status);
      if (lane == 0) rs->agg[r] = 0;  // every warp has added to it; ready for round j + 3
      const uint32_t gl = G - p.group_start[ti];
      const uint32_t c = lane < kGroupUnits ? rs->cnt[r][lane] : 0u;
      const uint32_t inc = warp_inclusive_scan(c);
      const uint32_t agg = __shfl_sync(kFull, inc, 31);
      uint64_t prefix = 0;
      if (cb_ok && hold != G + 1) {
        const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
        if (gl != 0) {  // (the group's count is already published by its last encoding warp)
          bool timed_out;
          const uint32_t g0 = G - gl;
          const bool own = prev_G >= static_cast<int64_t>(g0);  // previous group of this CTA, same tensor
          prefix = lookback(p.flags, G, g0, epoch, p.status, &timed_out, own ? prev_G : -1, own ? prev_incl : 0);
          if (lane == 0) st_relaxed(&p.flags[G].incl, tag | static_cast<uint32_t>(prefix + agg));
        }
        prev_G = G;
        prev_incl = prefix + agg;
      }
      if (lane < kGroupUnits) rs->uprefix[r][lane] = prefix + (inc - c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs->pre_bar[r]);  // release: the offsets are visible to waiters
    }
  } else {
    // ---------------- encoding warps: unit `warp` of every group
    auto stage_ptr = [&](int s) { return reinterpret_cast<uint16_t*>(wstage + s * kEncStageBytes); };
    // This warp's unit of group G: tensor ti, local tile lt, half (warp & 1);
    // false if the group (the last of its tensor) has fewer tiles.
    auto my_unit = [&](uint32_t G, uint32_t& ti, uint32_t& lt) {
      ti = locate_group(p, G);
      lt = (G - p.group_start[ti]) * kGroupTiles + warp / kUnitsPerTile;
      return static_cast<uint64_t>(lt) < num_tiles(p.t[ti].n);
    };
    const uint32_t half = warp % kUnitsPerTile;
    // valid elements of this warp's unit in tile lt
    auto unit_valid = [&](const EncTensor& T, uint32_t lt) -> uint32_t {
      const uint64_t start = static_cast<uint64_t>(lt) * kTile + half * kUnitElems;
      return T.n <= start ? 0u : (T.n - start >= kUnitElems ? kUnitElems : static_cast<uint32_t>(T.n - start));
    };
    auto issue = [&](int s, uint32_t G) {
      if (G >= p.total_groups) return;
      uint32_t ti, lt;
      if (!my_unit(G, ti, lt)) return;
      const EncTensor& T = p.t[ti];
      if (lane == 0) {
        if (unit_valid(T, lt) == kUnitElems) {
          fence_proxy_async();
          mbar_arrive_expect_tx(&bar[s], kEncStageBytes);
          tma_load_1d(stage_ptr(s), T.in + static_cast<uint64_t>(lt) * kTile + half * kUnitElems, kEncStageBytes,
                      &bar[s]);
        } else {
          mbar_arrive(&bar[s]);  // ragged end of the tensor: filled by plain loads when consumed
        }
      }
    };
    // Second half of round j: the group's offsets have been posted (slot r);
    // write the offset-table entry, this unit's header parts and escapes.  A
    // spilled unit's escapes come from its stage, which is refilled afterwards.
    auto finish = [&](uint32_t j, uint32_t G, const Pending& pd) {
      const int r = static_cast<int>(j % kEncSlots);
      const int s = static_cast<int>(j & 1u);
      mbar_wait_bounded(&rs->pre_bar[r], (j / kEncSlots) & 1u, p.status);
      if (pd.has) {
        const EncTensor& T = p.t[pd.ti];
        const uint64_t ntiles = num_tiles(T.n);
        const uint64_t prefix = rs->uprefix[r][warp];
        if (half == 0) {
          if (lane == 0) *reinterpret_cast<uint32_t*>(T.main + kHeader + 4ull * pd.lt) = static_cast<uint32_t>(prefix);
          if (pd.lt == 0) write_header_words(T.main, T.n, T.cb);
        }
        if (half == kUnitsPerTile - 1 && pd.lt + 1 == ntiles) {
          const uint64_t n_esc = prefix + pd.te.total;
          write_header_tail(T.main, ntiles, n_esc);
          if (lane == 0 && n_esc > T.esc_cap) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
        }
        if (pd.spilled) {
          write_escapes<kUnitBlocks>(wstage_s + s * kEncStageBytes, pd.te, prefix, T.esc, T.esc_cap);
        } else {
          const uint8_t* src = ebuf + r * kEncEscBuf;
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
    Pending pend[kEncStages];  // rounds j - 2 and j - 1, indexed by round parity (= stage)
#pragma unroll
    for (int s = 0; s < kEncStages; s++) {
      pend[s].has = pend[s].spilled = false;
      pend[s].done = true;
    }
    uint32_t j = 0;
    bool more = true;
    while (more) {
#pragma unroll
      for (int s = 0; s < kEncStages; s++) {  // rounds of stage 0, then stage 1
        const uint32_t G = blockIdx.x + j * step;
        if (G >= p.total_groups) {
          more = false;
          break;
        }
        const int r = static_cast<int>(j % kEncSlots);
        // round j - 2 used this stage; if it spilled, finish it now to free the stage
        if (!pend[s].done && pend[s].spilled) {
          finish(j - 2, G - 2 * step, pend[s]);
          pend[s].done = true;
        }
        Pending cur;
        cur.has = my_unit(G, cur.ti, cur.lt);
        cur.spilled = false;
        cur.done = false;
        cur.te.total = 0;
        const EncTensor& T = p.t[cur.ti];
        if (static_cast<int>(cur.ti) != cur_ti) {
          cb_ok = build_enc_lut(lut, T.cb);  // every warp of the group reaches the same verdict
          cur_ti = static_cast<int>(cur.ti);
          if (!cb_ok && lane == 0) set_status(p.status, ZC_ERR_DUP_CODEBOOK);
        }
        if (cur.has) {
          const uint32_t tb_s = wstage_s + s * kEncStageBytes;
          const uint32_t nv = unit_valid(T, cur.lt);
          const uint64_t rem = T.n - static_cast<uint64_t>(cur.lt) * kTile;
          const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
          mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
          phase ^= 1u << s;
          if (nv < kUnitElems) {
            uint16_t* tb = stage_ptr(s);
            const uint16_t* src = T.in + static_cast<uint64_t>(cur.lt) * kTile + half * kUnitElems;
            for (uint32_t i = lane; i < kUnitElems; i += 32) tb[i] = i < nv ? src[i] : static_cast<uint16_t>(0);
            __syncwarp();
          }
          if (cb_ok) {
            encode_blocks<kUnitBlocks>(tb_s, half * kUnitBlocks, n_tile, lut_s,
                                       tile_ptr(T.main, num_tiles(T.n), cur.lt) + half * kUnitBlocks * kBlockBytes,
                                       cur.te);
            cur.spilled = cur.te.total > kEncEscBuf;
            if (!cur.spilled) stage_escapes_smem<kUnitBlocks>(tb_s, cur.te, ebuf + r * kEncEscBuf);
          } else {
            cur.has = false;
          }
        }
        if (lane == 0) {
          rs->cnt[r][warp] = cur.te.total;
          // the last warp of the group publishes the group's escape count right away
          const uint32_t old = atomicAdd(&rs->agg[r], (1u << 16) | cur.te.total);
          if ((old >> 16) == kEncWarps - 1 && cb_ok && hold != G + 1) {
            const uint32_t agg = (old & 0xFFFFu) + cur.te.total;
            const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
            if (G == p.group_start[cur.ti])
              st_relaxed(&p.flags[G].incl, tag | agg);  // first group of its tensor: nothing before it
            else
              st_relaxed(&p.flags[G].agg, tag | agg);
          }
          mbar_arrive(&rs->cnt_bar[r]);  // release: the count is visible to the scan warp
        }
        __syncwarp();
        if (!cur.spilled) issue(s, G + kEncStages * step);  // refill now; escapes are staged
        if (!pend[s].done) finish(j - 2, G - 2 * step, pend[s]);  // round j - 2, oldest first
        pend[s] = cur;
        j++;
      }
    }
    // drain the last two rounds, oldest first
    auto drain = [&](uint32_t k, Pending& pd) {
      if (!pd.done) finish(k, blockIdx.x + k * step, pd);
    };
    if (j >= 2) {
      if (((j - 2) & 1u) == 0) {
        drain(j - 2, pend[0]);
        drain(j - 1, pend[1]);
      } else {
        drain(j - 2, pend[1]);
        drain(j - 1, pend[0]);
      }
    } else if (j == 1) {
      drain(0, pend[0]);
    }
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
  static_assert(sizeof(RoundShared) <= 1280, "round bookkeeping too large");
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
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(encode_kernel<MAXB>), dim3(ctas),
                                     dim3(kEncThreads), args, kEncSmem, stream);
}

cudaError_t launch_encode(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                          cudaStream_t stream, const DeviceInfo& dev) {
  if (count == 1) return launch_encode_t<1>(ts, count, ws, flags, status, stream, dev);
  return launch_encode_t<kMaxBatch>(ts, count, ws, flags, status, stream, dev);
}

}  // namespace zc
