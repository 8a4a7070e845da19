// zc_noalloc.cu -- zc_compress for callers that cannot allocate device memory.
//
// Some callers have no way to provide a workspace: hooks invoked by a
// communication or training framework that hands over only the tensors to
// send, and latency-critical paths that must never call cudaMalloc (it can
// synchronise the whole device).  For them this file keeps the encoder's
// scratch in a fixed device array that is part of the library itself.
//
// The array is a file-scope static __device__ object, so every GPU that loads
// libzc holds it (about 1 MiB) until the process exits.  Host code cannot use
// its name as an address: on the host the name denotes a host-side stand-in.
// The real device address is looked up with cudaGetSymbolAddress once per
// device, with that device current, and passed to the kernel like any other
// workspace pointer.
#include <mutex>

#include "zc_device.cuh"
#include "zc_internal.h"

#ifndef ZC_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace {

// Largest tensor this entry point encodes: 2^28 values (512 MiB of bf16).
constexpr uint64_t kNoAllocMaxElems = 1ull << 28;
constexpr uint64_t kNoAllocScratchBytes =
    ZC_WORKSPACE_HEADER_BYTES + ZC_WORKSPACE_BYTES_PER_TILE * ((kNoAllocMaxElems + ZC_TILE_ELEMS - 1) / ZC_TILE_ELEMS);

// Zero-initialised when the module is loaded on a device, which is the state
// the encoder's workspace protocol starts from.
static __device__ __align__(256) uint8_t zc_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; the first call
// per device looks it up (this must not happen during stream capture).
zc_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, zc_noalloc_scratch) != cudaSuccess || !ptr) return ZC_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return ZC_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The call's NVTX range (as for the other entry points that enqueue work).
struct NoAllocRange {
#ifndef ZC_NO_NVTX
  NoAllocRange() { nvtxRangePushA("zc_compress_noalloc"); }
  ~NoAllocRange() { nvtxRangePop(); }
#endif
};

}  // namespace

extern "C" zc_status zc_compress_noalloc(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                                         uint64_t esc_capacity, int32_t* d_status, void* stream) {
  const NoAllocRange range_;
  if (!d_status || !d_main || !d_cb || (!d_in && n) || (!d_esc && esc_capacity)) return ZC_ERR_INVALID_ARG;
  if (n > kNoAllocMaxElems) return ZC_ERR_WORKSPACE;  // the fixed scratch covers at most 2^28 values
  if (!aligned16(d_in) || !aligned16(d_main) || !aligned16(d_esc) || (reinterpret_cast<uintptr_t>(d_status) & 3u))
    return ZC_ERR_ALIGNMENT;
  void* scratch = nullptr;
  if (zc_status s = scratch_for_current_device(&scratch)) return s;
  zc::DeviceInfo dev;
  if (zc::device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The scratch keeps whatever the previous call left.  The escape-scan flags
  // are tagged with a launch epoch kept in the scratch itself, so stale flags
  // never match; the two counters that must start at zero (the test hook and
  // the exit count) are cleared here.  A call that overlaps another on the GPU
  // shares the same scratch and races with it.
  if (cudaMemsetAsync(scratch, 0, 8, st) != cudaSuccess) return ZC_ERR_CUDA;
  zc::EncTensor t{static_cast<const uint16_t*>(d_in), static_cast<uint8_t*>(d_main), static_cast<uint8_t*>(d_esc),
                  d_cb, n, esc_capacity};
  zc::WsHeader* ws = static_cast<zc::WsHeader*>(scratch);
  zc::Flag* flags = reinterpret_cast<zc::Flag*>(static_cast<uint8_t*>(scratch) + ZC_WORKSPACE_HEADER_BYTES);
  return zc::launch_encode(&t, 1, ws, flags, d_status, st, dev) == cudaSuccess ? ZC_OK : ZC_ERR_CUDA;
}
