// zc_hist.cu -- exact exponent histogram and its top 7, in one launch.
//
// [ZipCCL §2.A] avoids this online histogram by predicting the top-7
// exponents from sigma; the histogram path is kept for tensors whose sigma is
// unknown or whose values are not Gaussian, and it is what the closed form is
// checked against.  Orders (count desc, exponent asc) like the oracle.
//
// Design on sm_103a: a persistent grid, one CTA of 16 warps per SM.  Each
// warp streams 4 KB chunks of the input (chunk c = its global warp index +
// i * all warps) through two shared-memory stages with TMA bulk copies, so
// HBM stays busy while the warp counts.  Counting goes into a shared-memory
// histogram with 32 copies of each bin, one per lane, laid out bin-major so
// lane l always hits bank l (no bank conflicts within a warp whatever the
// data).  The ragged tail (fewer than 2048 values) is counted with plain
// loads by CTA 0.  CTAs add their totals into 256 global bins in the
// workspace; the last CTA to finish ranks the bins, writes the codebook (and
// the counts), and clears the global bins for the next call.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kHistWarps = 16;
constexpr int kHistThreads = kHistWarps * 32;
constexpr int kHistStages = 2;
constexpr uint32_t kHistChunk = 4096;                 // bytes per stage
constexpr uint32_t kHistChunkElems = kHistChunk / 2;  // 2048 values
// dynamic shared memory after 128-byte alignment: bins, stage barriers, stages
constexpr uint32_t kHistBinOff = 0;                            // 256 x 32 u32
constexpr uint32_t kHistBarOff = kHistBinOff + 256 * 32 * 4;   // per-warp stage barriers
constexpr uint32_t kHistStageOff = kHistBarOff + kHistWarps * kHistStages * 8;
constexpr uint32_t kHistSmem = 128 + kHistStageOff + kHistWarps * kHistStages * kHistChunk;
static_assert(kHistStageOff % 128 == 0, "stage alignment");

__device__ __forceinline__ void count_word(uint32_t* h, uint32_t w, uint32_t lane) {
  atomicAdd(&h[((w >> 7) & 0xFFu) * 32 + lane], 1u);
  atomicAdd(&h[((w >> 23) & 0xFFu) * 32 + lane], 1u);
}

__global__ void __launch_bounds__(kHistThreads, 1) hist_kernel(const uint16_t* __restrict__ in, uint64_t n,
                                                               WsHeader* ws, uint8_t* cb_out, uint32_t* hist_out,
                                                               int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  pdl_begin();
  uint8_t* smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127u)) & 127u);
  uint32_t* h = reinterpret_cast<uint32_t*>(smem + kHistBinOff);
  __shared__ uint32_t cnt[256];
  __shared__ int last;
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kHistBarOff) + warp * kHistStages;
  uint8_t* stage = smem + kHistStageOff + warp * kHistStages * kHistChunk;
  for (uint32_t i = threadIdx.x; i < 256 * 32; i += blockDim.x) h[i] = 0;
  if (lane == 0) {
    for (int s = 0; s < kHistStages; s++) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t nchunks = n / kHistChunkElems;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * kHistWarps + warp;
  const uint64_t nw = static_cast<uint64_t>(gridDim.x) * kHistWarps;
  auto issue = [&](int s, uint64_t c) {
    if (c < nchunks && lane == 0) {
      fence_proxy_async();
      mbar_arrive_expect_tx(&bar[s], kHistChunk);
      tma_load_1d(stage + s * kHistChunk, in + c * kHistChunkElems, kHistChunk, &bar[s]);
    }
  };
#pragma unroll
  for (int s = 0; s < kHistStages; s++) issue(s, gw + s * nw);
  uint32_t phase = 0;
  const uint32_t stage_s = smem_u32(stage);
  for (uint64_t k = 0;; k++) {
    const uint64_t c = gw + k * nw;
    if (c >= nchunks) break;
    const int s = static_cast<int>(k % kHistStages);
    mbar_wait_bounded(&bar[s], (phase >> s) & 1u, status);
    phase ^= 1u << s;
    uint4 x[kHistChunk / 512];
#pragma unroll
    for (uint32_t q = 0; q < kHistChunk / 512; q++) x[q] = lds128(stage_s + s * kHistChunk + (q * 32 + lane) * 16);
    __syncwarp();
    issue(s, c + kHistStages * nw);  // the stage is free again: its data is in registers
#pragma unroll
    for (uint32_t q = 0; q < kHistChunk / 512; q++) {
      count_word(h, x[q].x, lane);
      count_word(h, x[q].y, lane);
      count_word(h, x[q].z, lane);
      count_word(h, x[q].w, lane);
    }
  }
  if (blockIdx.x == 0)
    for (uint64_t j = nchunks * kHistChunkElems + threadIdx.x; j < n; j += blockDim.x)
      atomicAdd(&h[((in[j] >> 7) & 0xFFu) * 32 + lane], 1u);
  __syncthreads();
  for (uint32_t e = threadIdx.x; e < 256; e += blockDim.x) {
    uint32_t s = 0;
    for (uint32_t l = 0; l < 32; l++) s += h[e * 32 + ((l + e) & 31)];
    if (s) atomicAdd(&ws->hist[e], s);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&ws->hist_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (uint32_t e = threadIdx.x; e < 256; e += blockDim.x)
    cnt[e] = atomicAdd(&ws->hist[e], 0u);  // coherent read of the final totals
  __syncthreads();
  for (uint32_t e = threadIdx.x; e < 256; e += blockDim.x) {
    const uint32_t c = cnt[e];
    uint32_t rank = 0;
    for (uint32_t f = 0; f < 256; f++) {
      const uint32_t d = cnt[f];
      rank += (d > c) || (d == c && f < e);
    }
    if (rank < 7) cb_out[rank] = static_cast<uint8_t>(e);
    if (hist_out) hist_out[e] = c;
    ws->hist[e] = 0;
  }
  if (threadIdx.x == 0) ws->hist_done = 0;
}

cudaError_t launch_histogram(const uint16_t* in, uint64_t n, uint8_t* cb_out, uint32_t* hist_out, WsHeader* ws,
                             int32_t* status, cudaStream_t stream, const DeviceInfo& dev) {
  static KernelPrep prep;
  int per_sm = 0;
  cudaError_t err =
      prepare_kernel(prep, reinterpret_cast<const void*>(hist_kernel), kHistThreads, kHistSmem, dev, &per_sm);
  if (err != cudaSuccess) return err;
  const uint64_t nchunks = n / kHistChunkElems;
  uint64_t ctas = (nchunks + kHistWarps - 1) / kHistWarps;
  const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * static_cast<uint64_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&in, &n, &ws, &cb_out, &hist_out, &status};
  return launch_kernel(reinterpret_cast<const void*>(hist_kernel), dim3(static_cast<unsigned>(ctas)),
                       dim3(kHistThreads), kHistSmem, stream, args, false);
}

}  // namespace zc
