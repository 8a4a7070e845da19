// zc_encode.cu -- the encoder: bf16 -> ZC1 main stream + escape stream in one launch.
//
// [ZipCCL §2.B] split, remap to 3-bit codes, escapes to a separate array;
// [ZipCCL §2.C] three 1-bit code arrays in column-major order, 128-byte
// aligned blocks, asynchronous global->shared staging with double (here
// triple) buffering.
//
// Design on sm_103a: a persistent grid of 12-warp CTAs, one CTA per SM.  Each
// warp is its own producer/consumer pipeline: it draws tile tickets from an
// atomic counter, stages each 8 KB input tile into shared memory with one TMA
// bulk copy (2 stages per warp, 192 KB per SM), encodes the tile from shared
// memory, publishes the tile's escape count, and finds its escape offset with
// a decoupled look-back over the preceding tiles' flags.  The tile stays in
// shared memory until its escapes are written at their final global
// positions, so the escape stream needs no second pass.  The next ticket is
// drawn before the tile is encoded, hiding the atomic's round trip.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kEncWarps = 12;
constexpr int kEncStages = 2;
constexpr uint32_t kEncStageBytes = kTile * 2;  // 8192
// 1 KB alignment slack, per-warp LUTs (1 KB each, 1 KB aligned), barriers, stages
constexpr uint32_t kEncLutOff = 0;
constexpr uint32_t kEncBarOff = kEncWarps * 1024;
constexpr uint32_t kEncStageOff = kEncBarOff + 256;
constexpr uint32_t kEncSmem = 1024 + kEncStageOff + kEncWarps * kEncStages * kEncStageBytes;

template <int MAXB>
struct EncParams {
  EncTensor t[MAXB];
  uint32_t tile_start[MAXB + 1];  // first global tile of each tensor; [count] = total
  int count;
  uint32_t total_tiles;
  WsHeader* ws;
  Flag* flags;
  int32_t* status;
};

template <int MAXB>
__device__ __forceinline__ uint32_t locate(const EncParams<MAXB>& p, uint32_t g) {
  uint32_t ti = 0;
  if (MAXB > 1)
    while (static_cast<int>(ti) + 1 < p.count && g >= p.tile_start[ti + 1]) ti++;
  return ti;
}

template <int MAXB>
__global__ void __launch_bounds__(kEncWarps * 32, 1) encode_kernel(const __grid_constant__ EncParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;  // 1 KB aligned shared address
  uint8_t* gbase = smem + (sbase - smem_u32(smem));           // its generic pointer
  uint32_t* lut = reinterpret_cast<uint32_t*>(gbase + kEncLutOff + warp * 1024);
  const uint32_t lut_s = sbase + kEncLutOff + warp * 1024;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gbase + kEncBarOff + warp * 16);
  uint8_t* wstage = gbase + kEncStageOff + warp * kEncStages * kEncStageBytes;
  const uint32_t wstage_s = sbase + kEncStageOff + warp * kEncStages * kEncStageBytes;
  const uint32_t epoch = launch_epoch(p.ws);
  const uint32_t total_warps = gridDim.x * kEncWarps;

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
  auto issue = [&](int s, uint32_t g) {
    const uint32_t ti = locate(p, g);
    const uint32_t lt = g - p.tile_start[ti];
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

  uint32_t tk[kEncStages];
#pragma unroll
  for (int s = 0; s < kEncStages; s++) {
    tk[s] = draw_ticket(p.ws);
    if (tk[s] < p.total_tiles) issue(s, tk[s]);
  }

  uint32_t phase = 0;
  int cur_ti = -1;
  bool cb_ok = true;
  bool done = false;
  while (!done) {
#pragma unroll
    for (int s = 0; s < kEncStages; s++) {
      const uint32_t g = tk[s];
      if (g >= p.total_tiles) {
        done = true;
        break;
      }
      const uint32_t ti = locate(p, g);
      const EncTensor& T = p.t[ti];
      const uint32_t lt = g - p.tile_start[ti];
      const uint64_t ntiles = num_tiles(T.n);
      const uint64_t rem = T.n - static_cast<uint64_t>(lt) * kTile;
      const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
      uint16_t* tb = stage_ptr(s);
      const uint32_t tb_s = wstage_s + s * kEncStageBytes;
      // draw the ticket that refills this stage now; the atomic completes while the tile is encoded
      uint32_t next_raw = 0;
      if (lane == 0) next_raw = atomicAdd(&p.ws->ticket, 1u);

      mbar_wait_bounded(&bar[s], (phase >> s) & 1u, p.status);
      phase ^= 1u << s;
      if (n_tile < kTile) {
        const uint16_t* src = T.in + static_cast<uint64_t>(lt) * kTile;
        for (uint32_t i = lane; i < kTile; i += 32) tb[i] = i < n_tile ? src[i] : static_cast<uint16_t>(0);
        __syncwarp();
      }
      if (static_cast<int>(ti) != cur_ti) {
        cb_ok = build_enc_lut(lut, T.cb);
        cur_ti = static_cast<int>(ti);
        if (!cb_ok && lane == 0) set_status(p.status, ZC_ERR_DUP_CODEBOOK);
      }
      if (cb_ok) {
        TileEsc te;
        encode_tile(tb_s, n_tile, lut_s, tile_ptr(T.main, ntiles, lt), te);
        publish_tile(p.flags, g, lt, epoch, te, tb_s, T.main, T.n, T.cb, T.esc, T.esc_cap, p.status);
      }
      __syncwarp();
      tk[s] = __shfl_sync(kFull, next_raw, 0);
      if (tk[s] < p.total_tiles) issue(s, tk[s]);
    }
  }
  ticket_exit(p.ws, p.flags, epoch, p.total_tiles, total_warps);
}

template <int MAXB>
static cudaError_t launch_encode_t(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                                   cudaStream_t stream, const DeviceInfo& dev) {
  EncParams<MAXB> p;
  uint32_t total = 0;
  for (int i = 0; i < count; i++) {
    p.t[i] = ts[i];
    p.tile_start[i] = total;
    total += static_cast<uint32_t>(num_tiles(ts[i].n));
  }
  p.tile_start[count] = total;
  p.count = count;
  p.total_tiles = total;
  p.ws = ws;
  p.flags = flags;
  p.status = status;
  static_assert(sizeof(EncParams<MAXB>) < 4000, "encode parameters too large");
  cudaError_t err = cudaFuncSetAttribute(encode_kernel<MAXB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEncSmem);
  if (err != cudaSuccess) return err;
  uint32_t ctas = (total + kEncWarps - 1) / kEncWarps;
  if (ctas > static_cast<uint32_t>(dev.sm_count)) ctas = dev.sm_count;
  if (ctas == 0) ctas = 1;
  encode_kernel<MAXB><<<ctas, kEncWarps * 32, kEncSmem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_encode(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                          cudaStream_t stream, const DeviceInfo& dev) {
  if (count == 1) return launch_encode_t<1>(ts, count, ws, flags, status, stream, dev);
  return launch_encode_t<kMaxBatch>(ts, count, ws, flags, status, stream, dev);
}

}  // namespace zc
