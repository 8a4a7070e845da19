// zc_hist.cu -- exact exponent histogram and its top 7, in one launch.
//
// [ZipCCL §2.A] avoids this online histogram by predicting the top-7
// exponents from sigma; the histogram path is kept for tensors whose sigma is
// unknown or whose values are not Gaussian, and it is what the closed form is
// checked against.  Orders (count desc, exponent asc) like the oracle.
//
// Design on sm_103a: every CTA counts into a shared-memory histogram with 32
// copies of each bin, one per lane, laid out bin-major so lane l always hits
// bank l (no bank conflicts within a warp whatever the data); 16-byte loads,
// four in flight per thread.  CTAs add their totals into 256 global bins in
// the workspace; the last CTA to finish ranks the bins, writes the codebook
// (and the counts), and clears the global bins for the next call.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kHistThreads = 512;
constexpr int kHistUnroll = 4;

__device__ __forceinline__ void count_word(uint32_t* h, uint32_t w, uint32_t lane) {
  atomicAdd(&h[((w >> 7) & 0xFFu) * 32 + lane], 1u);
  atomicAdd(&h[((w >> 23) & 0xFFu) * 32 + lane], 1u);
}

__global__ void __launch_bounds__(kHistThreads) hist_kernel(const uint16_t* __restrict__ in, uint64_t n,
                                                            WsHeader* ws, uint8_t* cb_out, uint32_t* hist_out) {
  __shared__ uint32_t h[256 * 32];
  __shared__ uint32_t cnt[256];
  __shared__ int last;
  const uint32_t lane = lane_id();
  for (uint32_t i = threadIdx.x; i < 256 * 32; i += blockDim.x) h[i] = 0;
  __syncthreads();

  const uint4* v = reinterpret_cast<const uint4*>(in);
  const uint64_t nvec = n / 8;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kHistUnroll - 1) * stride < nvec; i += kHistUnroll * stride) {
    uint4 x[kHistUnroll];
#pragma unroll
    for (int u = 0; u < kHistUnroll; u++) x[u] = __ldg(v + i + u * stride);
#pragma unroll
    for (int u = 0; u < kHistUnroll; u++) {
      count_word(h, x[u].x, lane);
      count_word(h, x[u].y, lane);
      count_word(h, x[u].z, lane);
      count_word(h, x[u].w, lane);
    }
  }
  for (; i < nvec; i += stride) {
    const uint4 x = __ldg(v + i);
    count_word(h, x.x, lane);
    count_word(h, x.y, lane);
    count_word(h, x.z, lane);
    count_word(h, x.w, lane);
  }
  if (blockIdx.x == 0)
    for (uint64_t j = nvec * 8 + threadIdx.x; j < n; j += blockDim.x)
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
                             cudaStream_t stream, const DeviceInfo& dev) {
  const uint64_t nvec = n / 8;
  uint64_t ctas = (nvec + kHistThreads * kHistUnroll - 1) / (kHistThreads * kHistUnroll);
  const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * 4;
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  hist_kernel<<<static_cast<unsigned>(ctas), kHistThreads, 0, stream>>>(in, n, ws, cb_out, hist_out);
  return cudaGetLastError();
}

}  // namespace zc
