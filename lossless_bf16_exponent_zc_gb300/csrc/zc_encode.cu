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
// scan: the warps' escape counts meet in shared memory, warp 0 publishes the
// group's count and finds the group's escape offset with a single-pass
// decoupled look-back over preceding groups, and each warp then writes its
// tile's escapes at their final global positions, read back from the tile
// still in shared memory (no second pass).  One look-back participant per SM
// instead of one per warp keeps the resolved front ahead of the tiles; the
// cooperative launch guarantees every group owner is resident, which the
// look-back's waits rely on.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kEncWarps = 12;
constexpr int kEncStages = 2;
constexpr uint32_t kGroupTiles = kEncWarps;     // tiles per look-back group (one per warp)
constexpr uint32_t kEncStageBytes = kTile * 2;  // 8192
// After 1 KB alignment: per-warp LUTs (1 KB each, 1 KB aligned), barriers,
// group bookkeeping (counts and prefixes, double-buffered), stages.
constexpr uint32_t kEncLutOff = 0;
constexpr uint32_t kEncBarOff = kEncWarps * 1024;
constexpr uint32_t kEncGrpOff = kEncBarOff + 256;
constexpr uint32_t kEncStageOff = kEncGrpOff + 256;
constexpr uint32_t kEncSmem = 1024 + kEncStageOff + kEncWarps * kEncStages * kEncStageBytes;

template <int MAXB>
struct EncParams {
  EncTensor t[MAXB];
  uint32_t group_start[MAXB + 1];  // first global group of each tensor; [count] = total
  int count;
  uint32_t total_groups;
  uint32_t total_tiles;
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

// Shared group bookkeeping of one round: escape count of each warp's tile and
// the group's exclusive escape prefix.
struct GroupShared {
  uint32_t cnt[kEncStages][16];
  unsigned long long prefix[kEncStages];
};

template <int MAXB>
__global__ void __launch_bounds__(kEncWarps * 32, 1) encode_kernel(const __grid_constant__ EncParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;  // 1 KB aligned shared address
  uint8_t* gbase = smem + (sbase - smem_u32(smem));           // its generic pointer
  uint32_t* lut = reinterpret_cast<uint32_t*>(gbase + kEncLutOff + warp * 1024);
  const uint32_t lut_s = sbase + kEncLutOff + warp * 1024;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gbase + kEncBarOff + warp * 16);
  GroupShared* grp = reinterpret_cast<GroupShared*>(gbase + kEncGrpOff);
  uint8_t* wstage = gbase + kEncStageOff + warp * kEncStages * kEncStageBytes;
  const uint32_t wstage_s = sbase + kEncStageOff + warp * kEncStages * kEncStageBytes;
  const uint32_t epoch = launch_epoch(p.ws);
  const uint32_t hold = launch_hold(p.ws);

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; s++) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

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

  auto stage_ptr = [&](int s) { return reinterpret_cast<uint16_t*>(wstage + s * kEncStageBytes); };
  // This warp's tile of group G: tensor ti, local tile lt; false if the group
  // (the last of its tensor) has fewer tiles than warps.
  auto my_tile = [&](uint32_t G, uint32_t& ti, uint32_t& lt) {
    ti = locate_group(p, G);
    lt = (G - p.group_start[ti]) * kGroupTiles + warp;
    return static_cast<uint64_t>(lt) < num_tiles(p.t[ti].n);
  };
  auto issue = [&](int s, uint32_t G) -> bool {
    if (G >= p.total_groups) return false;
    uint32_t ti, lt;
    if (!my_tile(G, ti, lt)) return false;
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
    return true;
  };

  const uint32_t step = gridDim.x;
  bool issued[kEncStages];
#pragma unroll
  for (int s = 0; s < kEncStages; s++) issued[s] = issue(s, blockIdx.x + s * step);

  uint32_t phase = 0;
  int cur_ti = -1;
  bool cb_ok = true;
  for (uint32_t G0 = blockIdx.x; G0 < p.total_groups; G0 += kEncStages * step) {
#pragma unroll
    for (int s = 0; s < kEncStages; s++) {
      const uint32_t G = G0 + s * step;  // the same in every warp of the CTA
      if (G >= p.total_groups) break;
      uint32_t ti, lt;
      my_tile(G, ti, lt);
      const EncTensor& T = p.t[ti];
      const uint32_t gl = G - p.group_start[ti];
      const uint64_t ntiles = num_tiles(T.n);
      const uint32_t tb_s = wstage_s + s * kEncStageBytes;
      if (static_cast<int>(ti) != cur_ti) {
        cb_ok = build_enc_lut(lut, T.cb);  // every warp of the group reaches the same verdict
        cur_ti = static_cast<int>(ti);
        if (!cb_ok && lane == 0) set_status(p.status, ZC_ERR_DUP_CODEBOOK);
      }
      TileEsc te;
      te.total = 0;
      uint32_t n_tile = 0;
      if (issued[s]) {
        const uint64_t rem = T.n - static_cast<uint64_t>(lt) * kTile;
        n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
        mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        if (n_tile < kTile) {
          uint16_t* tb = stage_ptr(s);
          const uint16_t* src = T.in + static_cast<uint64_t>(lt) * kTile;
          for (uint32_t i = lane; i < kTile; i += 32) tb[i] = i < n_tile ? src[i] : static_cast<uint16_t>(0);
          __syncwarp();
        }
        if (cb_ok) encode_tile(tb_s, n_tile, lut_s, tile_ptr(T.main, ntiles, lt), te);
      }
      if (lane == 0) grp->cnt[s][warp] = te.total;
      __syncthreads();
      // warp 0: publish the group's escape count and find its offset (one look-back per group)
      if (warp == 0 && cb_ok && hold != G + 1) {
        const uint32_t agg = warp_sum(lane < kGroupTiles ? grp->cnt[s][lane] : 0u);
        const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
        uint64_t prefix = 0;
        if (gl == 0) {
          if (lane == 0) st_relaxed(&p.flags[G].incl, tag | agg);
        } else {
          if (lane == 0) st_relaxed(&p.flags[G].agg, tag | agg);
          bool timed_out;
          prefix = lookback(p.flags, G, G - gl, epoch, p.status, &timed_out);
          if (lane == 0) st_relaxed(&p.flags[G].incl, tag | static_cast<uint32_t>(prefix + agg));
        }
        if (lane == 0) grp->prefix[s] = prefix;
      }
      __syncthreads();
      if (issued[s] && cb_ok && hold != G + 1) {
        uint64_t prefix = grp->prefix[s];
        for (uint32_t w = 0; w < warp; w++) prefix += grp->cnt[s][w];
        if (lane == 0) *reinterpret_cast<uint32_t*>(T.main + kHeader + 4ull * lt) = static_cast<uint32_t>(prefix);
        if (lt == 0) write_header_words(T.main, T.n, T.cb);
        if (lt + 1 == ntiles) {
          const uint64_t n_esc = prefix + te.total;
          write_header_tail(T.main, ntiles, n_esc);
          if (lane == 0 && n_esc > T.esc_cap) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
        }
        write_escapes(tb_s, te, prefix, T.esc, T.esc_cap);
      }
      __syncwarp();
      issued[s] = issue(s, G + kEncStages * step);
    }
  }
  cta_exit(p.ws, p.flags, epoch, p.total_groups);
}

template <int MAXB>
static cudaError_t launch_encode_t(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                                   cudaStream_t stream, const DeviceInfo& dev) {
  EncParams<MAXB> p;
  uint32_t groups = 0, tiles = 0;
  for (int i = 0; i < count; i++) {
    p.t[i] = ts[i];
    p.group_start[i] = groups;
    const uint32_t nt = static_cast<uint32_t>(num_tiles(ts[i].n));
    tiles += nt;
    groups += (nt + kGroupTiles - 1) / kGroupTiles;
  }
  p.group_start[count] = groups;
  p.count = count;
  p.total_groups = groups;
  p.total_tiles = tiles;
  p.ws = ws;
  p.flags = flags;
  p.status = status;
  static_assert(sizeof(EncParams<MAXB>) < 4000, "encode parameters too large");
  static_assert(sizeof(GroupShared) <= 256, "group bookkeeping too large");
  cudaError_t err = cudaFuncSetAttribute(encode_kernel<MAXB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEncSmem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kernel<MAXB>, kEncWarps * 32, kEncSmem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  uint32_t ctas = groups;
  const uint32_t cap = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&p};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(encode_kernel<MAXB>), dim3(ctas),
                                     dim3(kEncWarps * 32), args, kEncSmem, stream);
}

cudaError_t launch_encode(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                          cudaStream_t stream, const DeviceInfo& dev) {
  if (count == 1) return launch_encode_t<1>(ts, count, ws, flags, status, stream, dev);
  return launch_encode_t<kMaxBatch>(ts, count, ws, flags, status, stream, dev);
}

}  // namespace zc
