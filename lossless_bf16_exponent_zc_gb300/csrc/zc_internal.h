// zc_internal.h -- launch interface between the C ABI (zc_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "zc.h"

namespace zc {

struct WsHeader;
struct Flag;

// Largest number of tensors one batched launch carries in its parameters;
// larger batches are split into several launches by the host.
constexpr int kMaxBatch = 32;

struct EncTensor {
  const uint16_t* in;
  uint8_t* main;
  uint8_t* esc;
  const uint8_t* cb;
  uint64_t n;
  uint64_t esc_cap;
};

struct DecTensor {
  const uint8_t* main;
  const uint8_t* esc;
  uint16_t* out;
  uint64_t n;
  uint64_t esc_bytes;
};

struct Shard {
  const uint8_t* main;
  const uint8_t* esc;
  uint64_t esc_bytes;
};

// Devices whose properties and kernel set-up are cached by the library.
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int device;
  int sm_count;
};

// The current device and its SM count (looked up once per device).
cudaError_t device_info(DeviceInfo* info);

// Launch preparation of one kernel, done once per device: raise its dynamic
// shared-memory limit and find how many CTAs fit on an SM.  Later calls on the
// same device return the cached count without calling the runtime, so a
// launch costs no extra driver calls.  Zero-initialised as a static object.
struct KernelPrep {
  std::atomic<int> per_sm[kMaxDevices];
};
cudaError_t prepare_kernel(KernelPrep& kp, const void* fn, int threads, int smem_bytes, const DeviceInfo& dev,
                           int* per_sm);

// Launches kernel `fn` (args: pointers to its parameters) on `stream` as a
// programmatic dependent of the work before it (the kernel begins with
// pdl_begin()), and cooperatively -- every CTA resident at once -- if asked.
cudaError_t launch_kernel(const void* fn, dim3 grid, dim3 block, int smem_bytes, cudaStream_t stream, void** args,
                          bool cooperative);

// count <= kMaxBatch; flags = workspace flag array (one per tile of the launch).
// adaptive: the raw bypass in the same launch -- each tensor whose coded form
// has more escapes than its RAW spill (and whose spill fits its escape
// capacity) is rewritten as a RAW stream, the escape overflow of the others is
// reported.
cudaError_t launch_encode(const EncTensor* ts, int count, WsHeader* ws, Flag* flags, int32_t* status,
                          cudaStream_t stream, const DeviceInfo& dev, bool adaptive = false);

cudaError_t launch_decode(const DecTensor* ts, int count, int32_t* status, cudaStream_t stream,
                          const DeviceInfo& dev);

// Zipped transfer pipeline of n values in chunks of c (a multiple of 8):
// compress on sc, link on sl, decompress on sd; ws holds
// pipeline_workspace_bytes(c) bytes (zero-filled before first use).
uint64_t pipeline_workspace_bytes(uint64_t c);
cudaError_t launch_pipeline(const uint16_t* in, uint64_t n, const uint8_t* cb, uint16_t* out, uint64_t c,
                            uint8_t* ws, int32_t* status, cudaStream_t sc, cudaStream_t sl, cudaStream_t sd,
                            const DeviceInfo& dev);

// The same launch sequence captured into an instantiated CUDA graph, from
// three private streams (overlap) or one; *exec = nullptr when n == 0.
cudaError_t capture_pipeline(const uint16_t* in, uint64_t n, const uint8_t* cb, uint16_t* out, uint64_t c,
                             uint8_t* ws, int32_t* status, bool overlap, const DeviceInfo& dev,
                             cudaGraphExec_t* exec);

cudaError_t launch_reduce(const Shard* shards, int P, uint64_t n, uint16_t* out, const uint8_t* out_cb,
                          uint8_t* out_main, uint8_t* out_esc, uint64_t out_cap, WsHeader* ws, Flag* flags,
                          int32_t* status, cudaStream_t stream, const DeviceInfo& dev);

// QLC (zq.cu): widths and sym validated by the caller.
uint64_t zq_stream_max_bytes(uint64_t n);
cudaError_t launch_zq_encode(const uint8_t* in, uint64_t n, const uint8_t width[8], const uint8_t sym[256],
                             uint8_t* out, uint64_t out_bytes, WsHeader* ws, Flag* flags, int32_t* status,
                             cudaStream_t stream, const DeviceInfo& dev);
cudaError_t launch_zq_decode(const uint8_t* in, uint64_t in_bytes, uint64_t n, uint8_t* out, int32_t* status,
                             cudaStream_t stream, const DeviceInfo& dev);

cudaError_t launch_histogram(const uint16_t* in, uint64_t n, uint8_t* cb_out, uint32_t* hist_out, WsHeader* ws,
                             int32_t* status, cudaStream_t stream, const DeviceInfo& dev);

}  // namespace zc
