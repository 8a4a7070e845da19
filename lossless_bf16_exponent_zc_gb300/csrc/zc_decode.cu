// zc_decode.cu -- the decoder: ZC1 main stream + escape stream -> bf16, bit for bit.
//
// The inverse of [ZipCCL §2.B]: code 001..111 -> codebook exponent, code 000
// -> next byte of the escape ("zero-point") array; the exponent is joined with
// the sign-mantissa byte.
//
// Design on sm_103a: a persistent grid of 16-warp CTAs, one per SM.  Warp w owns tiles
// w, w + W, w + 2W, ... (W = warps in the grid); no tile waits on another.
// Per tile, one TMA bulk copy stages the 5632-byte tile into shared memory and
// 16-byte cp.async copies stage the tile's escape bytes (up to 512 of them;
// any excess is read straight from global memory), all completing on one
// mbarrier; two stages are in flight per warp.  Code -> exponent goes
// through byte permutes on an 8-byte table held in registers, with a spread
// table in shared memory (16 lane copies, so data-dependent lookups put at
// most two lanes on a bank) turning the three plane bytes into a permute
// selector.  Output is written with 16-byte vector stores.  A RAW stream
// (the raw bypass: the values' own bytes) skips the staging: each warp
// copies its tiles' 8192 bytes with 16-byte loads and stores.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kDecWarps = 16;
constexpr int kDecStages = 2;
constexpr uint32_t kDecEscCap = 512;  // escape bytes staged per tile (multiple of 16)
constexpr uint32_t kDecStageBytes = kTileBytes + kDecEscCap;
constexpr int kDecSpreadCopies = 16;  // lane copies of the spread table (at most two lanes per bank)
// (after 1 KB alignment) spread table 16 KB, per-warp scratch 1 KB, barriers, stages
constexpr uint32_t kDecScratchOff = 1024 * kDecSpreadCopies;
constexpr uint32_t kDecBarOff = kDecScratchOff + kDecWarps * 1024;
constexpr uint32_t kDecStageOff = kDecBarOff + kDecWarps * 16;
constexpr uint32_t kDecSmem = 1024 + kDecStageOff + kDecWarps * kDecStages * kDecStageBytes;

template <int MAXB>
struct DecParams {
  DecTensor t[MAXB];
  uint32_t tile_start[MAXB + 1];
  int count;
  uint32_t total_tiles;
  int32_t* status;
};

// Header of one tensor as seen by a warp: validity, escape count, code table.
struct HdrInfo {
  int ti;
  bool ok;
  bool raw;  // RAW stream
  uint64_t n_esc;
  DecTable dt;
};

// Reads and validates a ZC1 header (one thread; it records a bad header in
// *status).
__device__ __forceinline__ HdrInfo read_header(const DecTensor& T, int ti, int32_t* status) {
  HdrInfo h;
  h.ti = ti;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(T.main);
  const uint32_t magic = __ldg(w + 0), vf = __ldg(w + 1), tile_elems = __ldg(w + 4), ntiles = __ldg(w + 5);
  const uint64_t n = static_cast<uint64_t>(__ldg(w + 2)) | (static_cast<uint64_t>(__ldg(w + 3)) << 32);
  h.n_esc = static_cast<uint64_t>(__ldg(w + 6)) | (static_cast<uint64_t>(__ldg(w + 7)) << 32);
  const uint32_t c0 = __ldg(w + 8), c1 = __ldg(w + 9);
  uint8_t cb[7];
#pragma unroll
  for (int k = 0; k < 4; k++) cb[k] = static_cast<uint8_t>(c0 >> (8 * k));
#pragma unroll
  for (int k = 0; k < 3; k++) cb[4 + k] = static_cast<uint8_t>(c1 >> (8 * k));
  bool dup = false;
#pragma unroll
  for (int a = 0; a < 7; a++)
#pragma unroll
    for (int b = a + 1; b < 7; b++) dup |= cb[a] == cb[b];
  int err = 0;
  h.raw = vf == (ZC_VERSION | (kFlagRaw << 16));
  if (magic != ZC_MAGIC || (vf != ZC_VERSION && !h.raw) || tile_elems != kTile || ntiles != num_tiles(T.n) ||
      dup || h.n_esc > T.esc_bytes || h.n_esc > T.n || (h.raw && h.n_esc != raw_spill(T.n)))
    err = ZC_ERR_BAD_HEADER;
  if (n != T.n) err = ZC_ERR_SIZE_MISMATCH;
  h.ok = err == 0;
  if (!h.ok) set_status(status, err);
  h.dt = make_dec_table(cb);
  return h;
}

// Tensor of global tile g.  Every caller visits tiles in increasing order, so
// it keeps a running index (`ti`, starting at 0) and only moves it forward.
template <int MAXB>
__device__ __forceinline__ uint32_t dec_locate(const DecParams<MAXB>& p, uint32_t g, uint32_t& ti) {
  if (MAXB > 1)
    while (static_cast<int>(ti) + 1 < p.count && g >= p.tile_start[ti + 1]) ti++;
  return MAXB > 1 ? ti : 0u;
}

// Escape range [a, b) of local tile lt, or ok = false when the table is corrupt.
__device__ __forceinline__ void tile_escape_range(const DecTensor& T, const HdrInfo& h, uint32_t lt, uint32_t& a,
                                                  uint32_t& cnt, bool& ok) {
  const uint32_t* tbl = reinterpret_cast<const uint32_t*>(T.main + kHeader);
  const uint64_t ntiles = num_tiles(T.n);
  const uint64_t aa = __ldg(tbl + lt);
  const uint64_t bb = (lt + 1 < ntiles) ? static_cast<uint64_t>(__ldg(tbl + lt + 1)) : h.n_esc;
  ok = h.ok && aa <= bb && bb <= h.n_esc && bb - aa <= kTile;
  a = ok ? static_cast<uint32_t>(aa) : 0;
  cnt = ok ? static_cast<uint32_t>(bb - aa) : 0;
}

// Stages the escape bytes [a, a + cnt) into `dst` starting at dst + (a & 15),
// at most kDecEscCap - (a & 15) of them; returns how many were staged.  Every
// lane then arrives on `bar` when its copies land.
__device__ __forceinline__ uint32_t stage_escapes(uint8_t* dst, const uint8_t* esc, uint32_t a, uint32_t cnt,
                                                  uint64_t* bar) {
  const uint32_t lane = lane_id();
  const uint32_t head = a & 15u;
  const uint32_t c0 = a - head;
  uint32_t region = head + cnt;  // bytes from c0 to the end of the range
  if (region > kDecEscCap) region = kDecEscCap;
  const uint32_t staged = cnt == 0 ? 0 : region - head;
  if (cnt != 0) {
    for (uint32_t c = lane; c * 16 < region; c += 32) {
      const uint32_t left = region - c * 16;
      cp_async_16(dst + c * 16, esc + c0 + c * 16, left < 16 ? left : 16);
    }
  }
  cp_async_arrive_noinc(bar);
  return staged;
}

template <int MAXB>
__global__ void __launch_bounds__(kDecWarps * 32, 1) decode_kernel(const __grid_constant__ DecParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_allow_dependents();
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;
  uint8_t* gbase = smem + (sbase - smem_u32(smem));
  uint32_t* spread = reinterpret_cast<uint32_t*>(gbase);
  const uint32_t spread_lb = sbase + 4 * (lane % kDecSpreadCopies);
  uint8_t* scratch = gbase + kDecScratchOff + warp * 1024;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gbase + kDecBarOff + warp * 16);
  uint8_t* wstage = gbase + kDecStageOff + warp * kDecStages * kDecStageBytes;
  const uint32_t wstage_s = sbase + kDecStageOff + warp * kDecStages * kDecStageBytes;

  // every tensor's header, read once per CTA (a warp's tiles cross many tensors)
  __shared__ HdrInfo hdr_cache[MAXB];
  // shared-memory setup first: it overlaps the end of the previous kernel
  build_spread_replicated<kDecSpreadCopies>(spread);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kDecStages; s++) mbar_init(&bar[s], 33);  // 1 TMA arrival + 32 cp.async arrivals
    fence_mbar_init();
  }
  pdl_wait();
  const uint32_t total_warps = gridDim.x * kDecWarps;
  const uint32_t gw = blockIdx.x * kDecWarps + warp;
  // The first stages' offset-table entries are loaded with the headers (the end
  // of a tensor's last tile is its header's escape count, read directly), so
  // the escape ranges are known once the headers are.
  uint64_t pre_a[kDecStages], pre_b[kDecStages];
  {
    uint32_t ti0 = 0;
#pragma unroll
    for (int s = 0; s < kDecStages; s++) {
      const uint32_t g = gw + s * total_warps;
      pre_a[s] = pre_b[s] = 0;
      if (g < p.total_tiles) {
        const uint32_t ti = dec_locate(p, g, ti0);
        const DecTensor& T = p.t[ti];
        const uint32_t lt = g - p.tile_start[ti];
        const uint64_t ntiles = num_tiles(T.n);
        const uint32_t* hw = reinterpret_cast<const uint32_t*>(T.main);
        const uint32_t* tbl = reinterpret_cast<const uint32_t*>(T.main + kHeader);
        pre_a[s] = __ldg(tbl + lt);
        pre_b[s] = (lt + 1 < ntiles) ? static_cast<uint64_t>(__ldg(tbl + lt + 1))
                                     : static_cast<uint64_t>(__ldg(hw + 6)) | (static_cast<uint64_t>(__ldg(hw + 7)) << 32);
      }
    }
  }
  for (int i = threadIdx.x; i < p.count; i += blockDim.x) hdr_cache[i] = read_header(p.t[i], i, p.status);
  __syncthreads();
  auto stage_ptr = [&](int s) { return wstage + s * kDecStageBytes; };

  HdrInfo issue_hdr;
  issue_hdr.ti = -1;
  uint32_t st_a[kDecStages], st_cnt[kDecStages], st_staged[kDecStages];
  bool st_ok[kDecStages], st_raw[kDecStages];
  DecTable st_dt[kDecStages];  // code table of the staged tile's tensor (read when it was issued)
  uint32_t issue_ti = 0;  // running tensor index of issue()
  auto issue = [&](int s, uint32_t g, bool first) {
    const uint32_t ti = dec_locate(p, g, issue_ti);
    const DecTensor& T = p.t[ti];
    if (issue_hdr.ti != static_cast<int>(ti)) issue_hdr = hdr_cache[ti];
    const uint32_t lt = g - p.tile_start[ti];
    uint32_t a = 0, cnt = 0;
    bool ok = issue_hdr.ok;
    st_raw[s] = issue_hdr.raw;
    if (!issue_hdr.raw) {
      if (first) {
        const uint64_t aa = pre_a[s], bb = pre_b[s];
        ok = ok && aa <= bb && bb <= issue_hdr.n_esc && bb - aa <= kTile;
        a = ok ? static_cast<uint32_t>(aa) : 0;
        cnt = ok ? static_cast<uint32_t>(bb - aa) : 0;
      } else {
        tile_escape_range(T, issue_hdr, lt, a, cnt, ok);
      }
      if (!ok && issue_hdr.ok && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
    }
    uint8_t* sp = stage_ptr(s);
    st_dt[s] = issue_hdr.dt;
    st_a[s] = a;
    st_cnt[s] = cnt;
    st_ok[s] = ok;
    st_staged[s] = stage_escapes(sp + kTileBytes, T.esc, a, ok ? cnt : 0, &bar[s]);
    if (lane == 0) {
      if (issue_hdr.raw) {
        mbar_arrive(&bar[s]);  // nothing to stage: the tile is copied from global memory
      } else {
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[s], kTileBytes);
        tma_load_1d(sp, tile_ptr(T.main, num_tiles(T.n), lt), kTileBytes, &bar[s]);
      }
    }
  };

#pragma unroll
  for (int s = 0; s < kDecStages; s++) {
    const uint32_t g = gw + s * total_warps;
    if (g < p.total_tiles) issue(s, g, true);
  }

  uint32_t run_ti = 0;
  uint32_t phase = 0;
  for (uint32_t g0 = gw; g0 < p.total_tiles; g0 += kDecStages * total_warps) {
#pragma unroll
    for (int s = 0; s < kDecStages; s++) {
      const uint32_t g = g0 + s * total_warps;
      if (g >= p.total_tiles) break;
      const uint32_t ti = dec_locate(p, g, run_ti);
      const DecTensor& T = p.t[ti];
      const uint32_t lt = g - p.tile_start[ti];
      const uint64_t rem = T.n - static_cast<uint64_t>(lt) * kTile;
      const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
      const uint8_t* tile = stage_ptr(s);
      const uint32_t tile_s = wstage_s + s * kDecStageBytes;

      mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
      phase ^= 1u << s;
      if (st_ok[s] && st_raw[s]) {
        // RAW: bytes [8192 lt, 8192 lt + 2 n_tile) of the image, 16 per lane and step
        const uint64_t ntiles = num_tiles(T.n);
        const uint8_t* tiles = tile_ptr(T.main, ntiles, 0);
        const uint64_t region = static_cast<uint64_t>(kTileBytes) * ntiles;
        uint16_t* out = T.out + static_cast<uint64_t>(lt) * kTile;
#pragma unroll 1
        for (uint32_t q = 0; q < 4; q++) {
          uint4 v[4];
#pragma unroll
          for (uint32_t k = 0; k < 4; k++)
            v[k] = raw_load16(tiles, T.esc, region, 2 * T.n,
                              2 * (static_cast<uint64_t>(lt) * kTile + q * kBlock + k * 256 + lane * 8));
#pragma unroll
          for (uint32_t k = 0; k < 4; k++) store8_guarded(out, q * kBlock + k * 256 + lane * 8, rem, v[k]);
        }
      } else if (st_ok[s]) {
        EscSource es;
        es.smem = tile + kTileBytes + (st_a[s] & 15u);
        es.glob = T.esc + st_a[s];
        es.staged = st_staged[s];
        es.count = st_cnt[s];
        uint32_t run = 0;
        uint16_t* out = T.out + static_cast<uint64_t>(lt) * kTile;
        const uint64_t n_left = rem;
#pragma unroll 1
        for (uint32_t blk = 0; blk < 4; blk++) {
          uint4 v[4];
          decode_block<kDecSpreadCopies>(tile_s, blk, n_tile, spread_lb, st_dt[s], es, run, scratch, v);
#pragma unroll
          for (uint32_t k = 0; k < 4; k++) store8_guarded(out, blk * kBlock + k * 256 + lane * 8, n_left, v[k]);
        }
        if (run != st_cnt[s] && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
      }
      __syncwarp();
      const uint32_t gn = g + kDecStages * total_warps;
      if (gn < p.total_tiles) issue(s, gn, false);
    }
  }
}

template <int MAXB>
static cudaError_t launch_decode_t(const DecTensor* ts, int count, int32_t* status, cudaStream_t stream,
                                   const DeviceInfo& dev) {
  DecParams<MAXB> p;
  uint32_t total = 0;
  for (int i = 0; i < count; i++) {
    p.t[i] = ts[i];
    p.tile_start[i] = total;
    total += static_cast<uint32_t>(num_tiles(ts[i].n));
  }
  p.tile_start[count] = total;
  p.count = count;
  p.total_tiles = total;
  p.status = status;
  if (total == 0) return cudaSuccess;
  static KernelPrep prep;
  int per_sm = 0;
  cudaError_t err =
      prepare_kernel(prep, reinterpret_cast<const void*>(decode_kernel<MAXB>), kDecWarps * 32, kDecSmem, dev, &per_sm);
  if (err != cudaSuccess) return err;
  uint32_t ctas = (total + kDecWarps - 1) / kDecWarps;
  if (ctas > static_cast<uint32_t>(dev.sm_count)) ctas = dev.sm_count;
  void* args[] = {&p};
  return launch_kernel(reinterpret_cast<const void*>(decode_kernel<MAXB>), dim3(ctas), dim3(kDecWarps * 32),
                       kDecSmem, stream, args, false);
}

cudaError_t launch_decode(const DecTensor* ts, int count, int32_t* status, cudaStream_t stream,
                          const DeviceInfo& dev) {
  if (count == 1) return launch_decode_t<1>(ts, count, status, stream, dev);
  return launch_decode_t<kMaxBatch>(ts, count, status, stream, dev);
}

}  // namespace zc
