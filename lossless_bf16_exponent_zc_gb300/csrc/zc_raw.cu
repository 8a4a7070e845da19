// zc_raw.cu -- the raw bypass: after an adaptive encode, store a tensor as a
// RAW stream (its own little-endian bytes) when coding does not shrink it.
//
// [CCCL §3.3] leaves tensors uncompressed when compressing them does not pay
// (tiny tensors); [CCCL §5.2] falls back to the uncompressed data when the
// ratio is near or above 1.  With ZC1's fixed-size main stream the comparison
// is exact: both forms send the same main stream, the coded form n_esc escape
// bytes, the RAW form max(0, 2n - 5632 ntiles) spill bytes; RAW is chosen
// exactly when n_esc exceeds the spill.
//
// Design on sm_103a: one launch right after the encoder on the same stream,
// so the decision reads the header's n_esc on the device and the host never
// waits.  It is a programmatic dependent launch: the encoder releases it as
// soon as it starts, its small CTAs settle beside the encoder's and wait in
// griddepcontrol.wait, and they read the headers the moment the encoder's
// writes are visible -- no launch gap.  Every CTA reads the escape counts and
// reaches the same verdict; when nothing goes RAW it leaves at once.  The RAW
// tensors are rewritten by a grid-stride loop of 16-byte copies (offset table
// zeroed, tile region and spill filled from the input); the last CTA to
// finish -- after every CTA has read the counts -- writes the RAW headers
// (flags and n_esc) and resets its counter in the workspace.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

// 256 threads at <= 40 registers (6 CTAs per SM) fit in what an encoder CTA
// leaves free of an SM (21 warps at 80 registers), so the dependent launch can
// be resident before the encoder ends.
constexpr int kRawThreads = 256;
constexpr int kRawUnroll = 4;     // 16-byte copies in flight per thread

template <int MAXB>
struct RawParams {
  EncTensor t[MAXB];
  int count;
  WsHeader* ws;
  int32_t* status;
};

// Tensor i is rewritten as RAW: its coded form has more escapes than the
// spill and the spill fits its escape capacity.  A tensor whose codebook has
// repeated entries was not encoded (the encoder reported it) and stays as is.
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

template <int MAXB>
__global__ void __launch_bounds__(kRawThreads, 6) raw_switch_kernel(const __grid_constant__ RawParams<MAXB> p) {
  static_assert(MAXB <= 32, "one mask bit per tensor");
  __shared__ uint32_t raw_mask;
  if (threadIdx.x == 0) raw_mask = 0;
  pdl_begin();  // the encoder has finished and its writes are visible
  __syncthreads();
  for (int i = threadIdx.x; i < p.count; i += blockDim.x) {
    bool overflow;
    if (goes_raw(p.t[i], &overflow)) atomicOr(&raw_mask, 1u << i);
    if (overflow && blockIdx.x == 0) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
  }
  __syncthreads();
  const uint32_t mask = raw_mask;
  if (mask == 0) return;  // every CTA reached the same verdict: nothing to rewrite, no counter to touch
  const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t nthreads = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (int i = 0; i < p.count; i++) {
    if (!((mask >> i) & 1u)) continue;
    const EncTensor& T = p.t[i];
    const uint64_t ntiles = num_tiles(T.n);
    const uint64_t tbl = table_bytes(ntiles);  // a multiple of 128
    const uint64_t region = static_cast<uint64_t>(kTileBytes) * ntiles;
    const uint64_t spill = raw_spill(T.n), two_n = 2 * T.n;
    uint8_t* tiles = T.main + kHeader + tbl;
    const uint64_t table_chunks = tbl / 16;
    const uint64_t chunks = table_chunks + (region + spill + 15) / 16;
    // 16 bytes of the RAW image at byte b (a multiple of 16), zero past 2n
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
    const uint64_t image_chunks = chunks - table_chunks;
    for (uint64_t c0 = tid; c0 < image_chunks; c0 += kRawUnroll * nthreads) {
      uint4 v[kRawUnroll];
#pragma unroll
      for (int u = 0; u < kRawUnroll; u++) {
        const uint64_t c = c0 + u * nthreads;
        v[u] = c < image_chunks ? load(16 * c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kRawUnroll; u++) {
        const uint64_t c = c0 + u * nthreads;
        if (c < image_chunks) store(16 * c, v[u]);
      }
    }
  }
  // The last CTA writes the RAW headers once every CTA has read the counts
  // (the barrier, then thread 0's acquire-release count of finished CTAs).
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
static cudaError_t launch_raw_switch_t(const EncTensor* ts, int count, WsHeader* ws, int32_t* status,
                                       cudaStream_t stream, const DeviceInfo& dev) {
  RawParams<MAXB> p;
  uint64_t chunks = 0;  // 16-byte copies if every tensor went RAW
  for (int i = 0; i < count; i++) {
    p.t[i] = ts[i];
    const uint64_t nt = num_tiles(ts[i].n);
    chunks += (table_bytes(nt) + static_cast<uint64_t>(kTileBytes) * nt + raw_spill(ts[i].n) + 15) / 16;
  }
  p.count = count;
  p.ws = ws;
  p.status = status;
  uint64_t ctas = (chunks + kRawThreads * kRawUnroll - 1) / (kRawThreads * kRawUnroll);
  const uint64_t cap = 6ull * static_cast<uint64_t>(dev.sm_count);  // a full SM of them keeps ~96 KB of copies in flight
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  // it may start while the encoder runs and waits for it in pdl_begin()
  void* args[] = {&p};
  return launch_kernel(reinterpret_cast<const void*>(raw_switch_kernel<MAXB>), dim3(static_cast<unsigned>(ctas)),
                       dim3(kRawThreads), 0, stream, args, false);
}

cudaError_t launch_raw_switch(const EncTensor* ts, int count, WsHeader* ws, int32_t* status, cudaStream_t stream,
                              const DeviceInfo& dev) {
  if (count == 1) return launch_raw_switch_t<1>(ts, count, ws, status, stream, dev);
  return launch_raw_switch_t<kMaxBatch>(ts, count, ws, status, stream, dev);
}

}  // namespace zc
