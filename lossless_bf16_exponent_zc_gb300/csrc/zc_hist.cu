// zc_hist.cu -- exact exponent histogram and its top 7, in one launch.
//
// [ZipCCL §2.A] avoids this online histogram by predicting the top-7
// exponents from sigma; the histogram path is kept for tensors whose sigma is
// unknown or whose values are not Gaussian, and it is what the closed form is
// checked against.  Orders (count desc, exponent asc) like the oracle.
//
// Design on sm_103a: a persistent grid, one CTA per SM, streaming the input
// in 32 KB chunks (chunk c = CTA + i * CTAs, so the machine reads the tensor
// front to back) through four shared-memory stages.  One producer warp issues
// one TMA bulk copy per chunk as soon as its stage is free; 16 counting warps
// take 2 KB of each stage apiece, free the stage as soon as their values are
// in registers, and count into a shared-memory histogram with 32 copies of
// each bin, one per lane, laid out bin-major so lane l always hits bank l (no
// bank conflicts within a warp whatever the data).  Copies of 4 KB per warp
// kept HBM less busy than these larger ones.  The last values (fewer than 8)
// are counted with plain loads by CTA 0.  CTAs add their totals into 256
// global bins in the workspace (relaxed reductions, then one acquire-release
// count of finished CTAs, so no full fences); the last CTA to finish ranks
// the bins that hold a count, writes the codebook (and the counts), and
// clears the global bins for the next call.  Streaming alone takes ~21 us for
// 2^26 values, counting adds ~1 us (the last chunk's), and the hand-over to the
// last CTA with its ranking ~2.5 us (three dependent L2 round trips).
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kHistCounters = 16;                      // counting warps
constexpr int kHistThreads = (kHistCounters + 1) * 32;  // + the producer warp
constexpr int kHistStages = 4;
constexpr uint32_t kHistChunk = 32768;                            // bytes per stage
constexpr uint32_t kHistUnits = kHistChunk / 16;                     // 16-byte pieces per stage
constexpr uint32_t kHistWarpUnits = kHistUnits / kHistCounters;      // 128 per counting warp
// dynamic shared memory after 128-byte alignment: bins, stage barriers, stages
constexpr uint32_t kHistBinOff = 0;                           // 256 x 32 u32
constexpr uint32_t kHistBarOff = kHistBinOff + 256 * 32 * 4;  // full[4], empty[4]
constexpr uint32_t kHistStageOff = kHistBarOff + 128;
constexpr uint32_t kHistSmem = 128 + kHistStageOff + kHistStages * kHistChunk;
static_assert(kHistStageOff % 128 == 0, "stage alignment");
static_assert(kHistWarpUnits % 32 == 0, "whole pieces per lane");

__device__ __forceinline__ void count_word(uint32_t* h, uint32_t w, uint32_t lane) {
  atomicAdd(&h[((w >> 7) & 0xFFu) * 32 + lane], 1u);
  atomicAdd(&h[((w >> 23) & 0xFFu) * 32 + lane], 1u);
}

__global__ void __launch_bounds__(kHistThreads, 1) hist_kernel(const uint16_t* __restrict__ in, uint64_t n,
                                                               WsHeader* ws, uint8_t* cb_out, uint32_t* hist_out,
                                                               int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  pdl_allow_dependents();  // (the wait for the previous grid comes after the shared-memory setup)
  uint8_t* smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127u)) & 127u);
  uint32_t* h = reinterpret_cast<uint32_t*>(smem + kHistBinOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kHistBarOff);
  uint64_t* empty = full + kHistStages;
  uint8_t* stage = smem + kHistStageOff;
  __shared__ uint32_t cnt[256];
  __shared__ uint32_t rank_hi[256];
  __shared__ uint32_t nz_bin[256];
  __shared__ uint32_t nz_warp[8];
  __shared__ uint32_t nz_total;
  __shared__ int last;
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  // the input as 16-byte pieces; chunk c holds pieces [c * kHistUnits, ...)
  const uint64_t units = n / 8;
  const uint64_t nchunks = (units + kHistUnits - 1) / kHistUnits;
  const uint64_t step = gridDim.x;
  const bool producer = warp == kHistCounters && lane == 0;
  // Barriers and cleared bins first (shared memory only: this overlaps the end
  // of the previous kernel), then the producer starts the first copies.
  if (producer) {
    for (int s = 0; s < kHistStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kHistCounters);
    }
    fence_mbar_init();
  }
  for (uint32_t i = threadIdx.x; i < 256 * 32; i += blockDim.x) h[i] = 0;
  pdl_wait();
  auto issue = [&](int s, uint64_t c) {
    const uint64_t u0 = c * kHistUnits;
    const uint32_t bytes = static_cast<uint32_t>(units - u0 < kHistUnits ? units - u0 : kHistUnits) * 16u;
    mbar_arrive_expect_tx(&full[s], bytes);
    tma_load_1d(stage + s * kHistChunk, in + u0 * 8, bytes, &full[s]);
  };
  if (producer)
    for (int s = 0; s < kHistStages; s++)
      if (blockIdx.x + s * step < nchunks) issue(s, blockIdx.x + s * step);
  __syncthreads();

  if (warp == kHistCounters) {
    // ---------------- producer: one bulk copy per chunk into the next free stage
    if (producer) {
      uint32_t k = kHistStages;
      for (uint64_t c = blockIdx.x + kHistStages * step; c < nchunks; c += step, k++) {
        const int s = static_cast<int>(k % kHistStages);
        if (!mbar_wait_bounded(&empty[s], ((k / kHistStages) - 1) & 1u, status)) break;
        issue(s, c);
      }
    }
  } else {
    // ---------------- counting warps: 2 KB of every chunk each
    const uint32_t stage_s = smem_u32(stage);
    uint32_t k = 0;
    for (uint64_t c = blockIdx.x; c < nchunks; c += step, k++) {
      const int s = static_cast<int>(k % kHistStages);
      if (!mbar_wait_bounded(&full[s], (k / kHistStages) & 1u, status)) break;
      const uint64_t left = units - c * kHistUnits;  // pieces in this chunk: min(left, kHistUnits)
      constexpr uint32_t kPer = kHistWarpUnits / 32;
      uint4 x[kPer];
#pragma unroll
      for (uint32_t q = 0; q < kPer; q++)
        x[q] = lds128(stage_s + s * kHistChunk + (warp * kHistWarpUnits + q * 32 + lane) * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled: this warp's data is in registers
      if (left >= kHistUnits) {
#pragma unroll
        for (uint32_t q = 0; q < kPer; q++) {
          count_word(h, x[q].x, lane);
          count_word(h, x[q].y, lane);
          count_word(h, x[q].z, lane);
          count_word(h, x[q].w, lane);
        }
      } else {
#pragma unroll
        for (uint32_t q = 0; q < kPer; q++) {
          if (warp * kHistWarpUnits + q * 32 + lane < left) {
            count_word(h, x[q].x, lane);
            count_word(h, x[q].y, lane);
            count_word(h, x[q].z, lane);
            count_word(h, x[q].w, lane);
          }
        }
      }
    }
    if (blockIdx.x == 0 && warp == 0)
      for (uint64_t j = units * 8 + lane; j < n; j += 32) atomicAdd(&h[((in[j] >> 7) & 0xFFu) * 32 + lane], 1u);
  }
  __syncthreads();
  // This CTA's counts go into the global bins; the barrier then orders every
  // thread's additions before thread 0's release of the completion count, and
  // the CTA whose increment completes the count acquires all of them.
  for (uint32_t e = threadIdx.x; e < 256; e += blockDim.x) {
    uint32_t s = 0;
#pragma unroll 8
    for (uint32_t l = 0; l < 32; l++) s += h[e * 32 + ((l + e) & 31)];
    if (s) red_add_relaxed_gpu(&ws->hist[e], s);
  }
  __syncthreads();
  if (threadIdx.x == 0) last = atom_add_acq_rel_gpu(&ws->hist_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  for (uint32_t e = threadIdx.x; e < 256; e += blockDim.x) cnt[e] = ld_relaxed_gpu(&ws->hist[e]);
  __syncthreads();
  // Rank of bin e (count desc, exponent asc).  Bins with a count are ranked
  // among themselves (two threads per bin, each comparing it with half of
  // them); the m empty bins follow all of them in exponent order.  Gaussian
  // data fills ~20 bins, so the comparisons are few.
  const uint32_t e = threadIdx.x & 255u, half = (threadIdx.x >> 8) & 1u;
  const bool ranker = threadIdx.x < 512;
  uint32_t c = 0, before = 0;  // before: bins with a count below index e
  if (threadIdx.x < 256) {
    c = cnt[e];
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, c != 0);
    before = __popc(b & ((1u << lane) - 1u));
    if (lane == 0) nz_warp[warp] = __popc(b);
  }
  __syncthreads();
  uint32_t m = 0;
  if (threadIdx.x < 256) {
#pragma unroll
    for (uint32_t w = 0; w < 8; w++) {
      before += w < warp ? nz_warp[w] : 0u;
      m += nz_warp[w];
    }
    if (c) nz_bin[before] = e;
  }
  if (threadIdx.x == 0) {
    uint32_t t = 0;
#pragma unroll
    for (uint32_t w = 0; w < 8; w++) t += nz_warp[w];
    nz_total = t;
  }
  __syncthreads();
  m = nz_total;
  uint32_t rank = 0;
  if (ranker) {
    c = cnt[e];
    if (c) {
      const uint32_t j0 = half * (m / 2), j1 = half ? m : m / 2;
      for (uint32_t j = j0; j < j1; j++) {
        const uint32_t f = nz_bin[j], d = cnt[f];
        rank += (d > c) || (d == c && f < e);
      }
    }
    if (half) rank_hi[e] = rank;
  }
  __syncthreads();
  if (ranker && !half) {
    rank = c ? rank + rank_hi[e] : m + (e - before);
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
  const uint64_t nchunks = (n / 8 + kHistUnits - 1) / kHistUnits;
  uint64_t ctas = nchunks;
  const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * static_cast<uint64_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&in, &n, &ws, &cb_out, &hist_out, &status};
  return launch_kernel(reinterpret_cast<const void*>(hist_kernel), dim3(static_cast<unsigned>(ctas)),
                       dim3(kHistThreads), kHistSmem, stream, args, false);
}

}  // namespace zc
