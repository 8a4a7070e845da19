// zc_reduce.cu -- fused local stage of a zipped reduce-scatter [ZipCCL §2.D]:
// decode P compressed shards, add them in fp32 in rank order 0..P-1, round to
// bfloat16 (nearest even), optionally re-encode the result -- one launch, no
// decoded intermediate ever touches global memory.
//
// Design on sm_103a: 8 warps per CTA, one CTA per SM.  A warp owns one output
// tile at a time and keeps its 4096 fp32 partial sums in registers (128 per
// lane).  Its pipeline streams the P compressed copies of that tile (TMA for
// the 5632-byte tile, cp.async for its escape bytes, two stages in flight);
// each copy is decoded from shared memory straight into the accumulators.
// With re-encoding, the rounded tile goes to shared memory and through the
// same encoder and look-back as zc_compress (cooperative launch: every tile
// owner is resident).  Warp w owns tiles w, w + W, w + 2W, ...
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kRedWarps = 8;
constexpr int kRedStages = 2;
constexpr uint32_t kRedEscCap = 512;
constexpr uint32_t kRedStageBytes = kTileBytes + kRedEscCap;  // 6144
// After 1 KB alignment: spread tables (3 KB), per-warp encoder LUTs (1 KB each,
// 1 KB aligned), shard tables, a flag, then per warp: stages, y tile (8 KB),
// exponent scratch (1 KB), barriers.
constexpr uint32_t kRedLutOff = 3 * 1024;
constexpr uint32_t kRedShardOff = kRedLutOff + kRedWarps * 1024;
constexpr uint32_t kRedFlagOff = kRedShardOff + ZC_MAX_SHARDS * 16;
constexpr uint32_t kRedWarpOff = kRedFlagOff + 16;
constexpr uint32_t kRedWarpSmem = kRedStages * kRedStageBytes + 8192 + 1024 + 64;
constexpr uint32_t kRedSmem = 1024 + kRedWarpOff + kRedWarps * kRedWarpSmem;

struct RedParams {
  Shard s[ZC_MAX_SHARDS];
  int P;
  uint64_t n;
  uint32_t ntiles;
  uint16_t* out;
  const uint8_t* out_cb;
  uint8_t* out_main;
  uint8_t* out_esc;
  uint64_t out_cap;
  WsHeader* ws;
  Flag* flags;
  int32_t* status;
};

struct ShardInfo {
  uint32_t t0, t1;  // code -> exponent permute table
  unsigned long long n_esc;
};

// Offsets [a, b) of the current tile for shard `lane` (a0, b0) and `lane + 32` (a1, b1).
struct TileOffs {
  uint32_t a0, b0, a1, b1;
};

__device__ __forceinline__ TileOffs load_offs(const RedParams& p, const ShardInfo* si, uint32_t g) {
  TileOffs o{0, 0, 0, 0};
  if (g >= p.ntiles) return o;
  const uint32_t lane = lane_id();
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int r = static_cast<int>(lane) + 32 * h;
    if (r < p.P) {
      const uint32_t* tbl = reinterpret_cast<const uint32_t*>(p.s[r].main + kHeader);
      const uint32_t a = __ldg(tbl + g);
      const uint64_t b = (g + 1 < p.ntiles) ? static_cast<uint64_t>(__ldg(tbl + g + 1)) : si[r].n_esc;
      const uint32_t bb = b > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(b);
      if (h == 0) {
        o.a0 = a;
        o.b0 = bb;
      } else {
        o.a1 = a;
        o.b1 = bb;
      }
    }
  }
  return o;
}

__device__ __forceinline__ void accumulate(float (&acc)[8], uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(w[i] << 16));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(w[i] & 0xFFFF0000u));
  }
}

__device__ __forceinline__ uint4 round_pack(const float (&acc)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; i++) w[i] = f32_to_bf16_rne(acc[2 * i]) | (f32_to_bf16_rne(acc[2 * i + 1]) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool REENC>
__global__ void __launch_bounds__(kRedWarps * 32, 1) reduce_kernel(const __grid_constant__ RedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;
  uint8_t* gbase = smem + (sbase - smem_u32(smem));
  uint32_t* spread = reinterpret_cast<uint32_t*>(gbase);
  uint32_t* lut = reinterpret_cast<uint32_t*>(gbase + kRedLutOff + warp * 1024);
  const uint32_t lut_s = sbase + kRedLutOff + warp * 1024;
  ShardInfo* si = reinterpret_cast<ShardInfo*>(gbase + kRedShardOff);
  int* bad = reinterpret_cast<int*>(gbase + kRedFlagOff);
  uint8_t* wbase = gbase + kRedWarpOff + warp * kRedWarpSmem;
  const uint32_t wbase_s = sbase + kRedWarpOff + warp * kRedWarpSmem;
  uint16_t* ytile = reinterpret_cast<uint16_t*>(wbase + kRedStages * kRedStageBytes);
  const uint32_t ytile_s = wbase_s + kRedStages * kRedStageBytes;
  uint8_t* scratch = wbase + kRedStages * kRedStageBytes + 8192;
  uint64_t* bar = reinterpret_cast<uint64_t*>(scratch + 1024);

  build_spread_tables(spread);
  if (threadIdx.x == 0) *bad = 0;
  __syncthreads();
  // validate every shard header (each CTA reaches the same verdict)
  for (int r = threadIdx.x; r < p.P; r += blockDim.x) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p.s[r].main);
    const uint64_t n = static_cast<uint64_t>(__ldg(w + 2)) | (static_cast<uint64_t>(__ldg(w + 3)) << 32);
    const uint64_t n_esc = static_cast<uint64_t>(__ldg(w + 6)) | (static_cast<uint64_t>(__ldg(w + 7)) << 32);
    const uint32_t c0 = __ldg(w + 8), c1 = __ldg(w + 9);
    uint8_t cb[7];
    for (int k = 0; k < 4; k++) cb[k] = static_cast<uint8_t>(c0 >> (8 * k));
    for (int k = 0; k < 3; k++) cb[4 + k] = static_cast<uint8_t>(c1 >> (8 * k));
    bool dup = false;
    for (int a = 0; a < 7; a++)
      for (int b = a + 1; b < 7; b++) dup |= cb[a] == cb[b];
    int err = 0;
    if (__ldg(w) != ZC_MAGIC || __ldg(w + 1) != ZC_VERSION || __ldg(w + 4) != kTile ||
        __ldg(w + 5) != p.ntiles || dup || n_esc > p.s[r].esc_bytes || n_esc > p.n)
      err = ZC_ERR_BAD_HEADER;
    if (n != p.n) err = ZC_ERR_SIZE_MISMATCH;
    if (err) {
      atomicExch(bad, 1);
      set_status(p.status, err);
    }
    const DecTable dt = make_dec_table(cb);
    si[r].t0 = dt.t0;
    si[r].t1 = dt.t1;
    si[r].n_esc = n_esc;
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kRedStages; s++) mbar_init(&bar[s], 33);
    fence_mbar_init();
  }
  bool ok_out = true;
  if (REENC) {
    ok_out = build_enc_lut(lut, p.out_cb);
    if (!ok_out && lane == 0) set_status(p.status, ZC_ERR_DUP_CODEBOOK);
  }
  __syncthreads();
  const uint32_t epoch = REENC ? launch_epoch(p.ws) : 0u;
  const uint32_t hold = REENC ? launch_hold(p.ws) : 0u;
  const uint32_t total_warps = gridDim.x * kRedWarps;
  const bool skip = (*bad != 0) || !ok_out;
  if (REENC && !skip && p.ntiles == 0 && blockIdx.x == 0 && warp == 0) {
    write_header_words(p.out_main, 0, p.out_cb);
    write_header_tail(p.out_main, 0, 0);
  }

  // ---- tile sequence: warp w owns tiles w, w + W, w + 2W, ...
  uint32_t static_next = blockIdx.x * kRedWarps + warp;
  auto next_tile = [&]() -> uint32_t {
    if (skip) return 0xFFFFFFFFu;
    const uint32_t g = static_next;
    static_next += total_warps;
    return g;
  };

  // ---- producer state
  uint32_t pg = next_tile();
  TileOffs po = load_offs(p, si, pg);
  uint32_t qg = next_tile();
  TileOffs qo = load_offs(p, si, qg);
  int pr = 0;

  uint32_t st_g[kRedStages], st_r[kRedStages], st_a[kRedStages], st_cnt[kRedStages], st_staged[kRedStages];
  bool st_ok[kRedStages];
  auto stage_ptr = [&](int s) { return wbase + s * kRedStageBytes; };
  auto issue_item = [&](int s) {
    st_g[s] = pg;
    if (pg >= p.ntiles) return;
    const int r = pr;
    const uint32_t src = static_cast<uint32_t>(r & 31);
    const uint32_t a = __shfl_sync(kFull, r < 32 ? po.a0 : po.a1, src);
    const uint32_t b = __shfl_sync(kFull, r < 32 ? po.b0 : po.b1, src);
    const bool ok = a <= b && b <= si[r].n_esc && b - a <= kTile;
    if (!ok && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
    st_r[s] = static_cast<uint32_t>(r);
    st_a[s] = ok ? a : 0;
    st_cnt[s] = ok ? b - a : 0;
    st_ok[s] = ok;
    uint8_t* sp = stage_ptr(s);
    // escape bytes (cp.async) -- same staging rule as the decoder
    {
      const uint32_t cnt = st_cnt[s], aa = st_a[s];
      const uint32_t head = aa & 15u;
      uint32_t region = head + cnt;
      if (region > kRedEscCap) region = kRedEscCap;
      st_staged[s] = cnt == 0 ? 0 : region - head;
      if (cnt != 0)
        for (uint32_t c = lane; c * 16 < region; c += 32) {
          const uint32_t left = region - c * 16;
          cp_async_16(sp + kTileBytes + c * 16, p.s[r].esc + (aa - head) + c * 16, left < 16 ? left : 16);
        }
      cp_async_arrive_noinc(&bar[s]);
    }
    if (lane == 0) {
      fence_proxy_async();
      mbar_arrive_expect_tx(&bar[s], kTileBytes);
      tma_load_1d(sp, tile_ptr(p.s[r].main, p.ntiles, pg), kTileBytes, &bar[s]);
    }
    if (++pr == p.P) {
      pr = 0;
      pg = qg;
      po = qo;
      qg = next_tile();
      qo = load_offs(p, si, qg);
    }
  };

#pragma unroll
  for (int s = 0; s < kRedStages; s++) issue_item(s);

  float acc[4][4][8];
  uint32_t phase = 0;
  bool done = false;
  while (!done) {
#pragma unroll
    for (int s = 0; s < kRedStages; s++) {
      const uint32_t g = st_g[s];
      if (g >= p.ntiles) {
        done = true;
        break;
      }
      const uint32_t r = st_r[s];
      const uint64_t rem = p.n - static_cast<uint64_t>(g) * kTile;
      const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
      if (r == 0) {
#pragma unroll
        for (int b = 0; b < 4; b++)
#pragma unroll
          for (int k = 0; k < 4; k++)
#pragma unroll
            for (int j = 0; j < 8; j++) acc[b][k][j] = -0.0f;  // -0 + x == x for every x
      }
      const uint8_t* tile = stage_ptr(s);
      const uint32_t tile_s = wbase_s + s * kRedStageBytes;
      mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
      phase ^= 1u << s;
      {
        DecTable dt;
        dt.t0 = si[r].t0;
        dt.t1 = si[r].t1;
        EscSource es;
        es.smem = tile + kTileBytes + (st_a[s] & 15u);
        es.glob = p.s[r].esc + st_a[s];
        es.staged = st_staged[s];
        es.count = st_cnt[s];
        uint32_t run = 0;
#pragma unroll
        for (uint32_t blk = 0; blk < 4; blk++) {
          uint4 v[4];
          decode_block(tile_s, blk, n_tile, sbase, dt, es, run, scratch, v);
#pragma unroll
          for (int k = 0; k < 4; k++) accumulate(acc[blk][k], v[k]);
        }
        if (st_ok[s] && run != st_cnt[s] && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
      }
      if (r + 1 == static_cast<uint32_t>(p.P)) {
        // finished tile g: round, store, re-encode
#pragma unroll
        for (uint32_t blk = 0; blk < 4; blk++) {
#pragma unroll
          for (uint32_t k = 0; k < 4; k++) {
            const uint32_t idx = blk * kBlock + k * 256 + lane * 8;
            uint4 v = round_pack(acc[blk][k]);
            if (n_tile < kTile) {
              uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (uint32_t j = 0; j < 8; j++)
                if (idx + j >= n_tile) w[j >> 1] &= (j & 1) ? 0x0000FFFFu : 0xFFFF0000u;
              v = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (p.out) store8_guarded(p.out + static_cast<uint64_t>(g) * kTile, idx, rem, v);
            if (REENC) *reinterpret_cast<uint4*>(ytile + idx) = v;
          }
        }
        if (REENC) {
          __syncwarp();
          TileEsc te;
          encode_tile(ytile_s, n_tile, lut_s, tile_ptr(p.out_main, p.ntiles, g), te);
          publish_tile(p.flags, g, g, epoch, te, ytile_s, p.out_main, p.n, p.out_cb, p.out_esc, p.out_cap, p.status,
                       hold);
        }
      }
      __syncwarp();
      issue_item(s);
    }
  }
  if (REENC) cta_exit(p.ws, p.flags, epoch, p.ntiles);
}

cudaError_t launch_reduce(const Shard* shards, int P, uint64_t n, uint16_t* out, const uint8_t* out_cb,
                          uint8_t* out_main, uint8_t* out_esc, uint64_t out_cap, WsHeader* ws, Flag* flags,
                          int32_t* status, cudaStream_t stream, const DeviceInfo& dev) {
  RedParams p;
  for (int r = 0; r < P; r++) p.s[r] = shards[r];
  p.P = P;
  p.n = n;
  p.ntiles = static_cast<uint32_t>(num_tiles(n));
  p.out = out;
  p.out_cb = out_cb;
  p.out_main = out_main;
  p.out_esc = out_esc;
  p.out_cap = out_cap;
  p.ws = ws;
  p.flags = flags;
  p.status = status;
  uint32_t ctas = (p.ntiles + kRedWarps - 1) / kRedWarps;
  if (ctas > static_cast<uint32_t>(dev.sm_count)) ctas = dev.sm_count;
  if (ctas == 0) ctas = 1;
  cudaError_t err;
  if (out_cb) {
    err = cudaFuncSetAttribute(reduce_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRedSmem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reduce_kernel<true>, kRedWarps * 32, kRedSmem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    void* args[] = {&p};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(reduce_kernel<true>), dim3(ctas),
                                       dim3(kRedWarps * 32), args, kRedSmem, stream);
  }
  if (p.ntiles == 0) return cudaSuccess;
  err = cudaFuncSetAttribute(reduce_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRedSmem);
  if (err != cudaSuccess) return err;
  reduce_kernel<false><<<ctas, kRedWarps * 32, kRedSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace zc
