// zc_api.cu -- the C ABI of libzc (declared and documented in include/zc.h).
//
// Host work only: argument validation, workspace layout, the sigma closed form
// of [ZipCCL §2.A], and kernel launches on the caller's stream.  Nothing here
// allocates device memory, synchronises, or keeps per-call state; a pipeline
// plan is an object the caller owns (a host struct and an instantiated CUDA
// graph).
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "zc_device.cuh"
#include "zc_internal.h"

#ifndef ZC_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

using namespace zc;

namespace {
// An NVTX range named after the entry point around each call that enqueues
// device work, so a profiler attributes kernels to the library call that
// launched them (a pointer check per push and pop when no tool is attached).
struct ApiRange {
#ifndef ZC_NO_NVTX
  explicit ApiRange(const char* name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
#else
  explicit ApiRange(const char*) {}
#endif
};
}  // namespace

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr uint64_t kMaxN = 0xFFFFFFFFull;  // n < 2^32

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

zc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ZC_OK : ZC_ERR_CUDA; }

// Workspace bytes for a launch covering `tiles` tiles.
uint64_t ws_bytes_for_tiles(uint64_t tiles) {
  return ZC_WORKSPACE_HEADER_BYTES + static_cast<uint64_t>(ZC_WORKSPACE_BYTES_PER_TILE) * tiles;
}

zc_status check_ws(const void* d_ws, uint64_t ws_bytes, uint64_t tiles) {
  if (!d_ws) return ZC_ERR_INVALID_ARG;
  if (!aligned(d_ws, 16)) return ZC_ERR_ALIGNMENT;
  if (ws_bytes < ws_bytes_for_tiles(tiles)) return ZC_ERR_WORKSPACE;
  return ZC_OK;
}

WsHeader* ws_header(void* d_ws) { return static_cast<WsHeader*>(d_ws); }
Flag* ws_flags(void* d_ws) {
  return reinterpret_cast<Flag*>(static_cast<uint8_t*>(d_ws) + ZC_WORKSPACE_HEADER_BYTES);
}

// ---- sigma closed form ------------------------------------------------------
// Edges of the set of reals that round (to nearest even) to a bfloat16 whose
// exponent field is e: the binade [2^(e-127), 2^(e-126)) shifted down by half
// an ulp (2^-9 relative), with the subnormal spacing below 2^-126 and
// overflow to infinity above 2^128 (1 - 2^-9).
void rounded_binade(int e, double* lo, double* hi) {
  const double shrink = 1.0 - std::ldexp(1.0, -9);
  const double min_normal_edge = std::ldexp(1.0 - std::ldexp(1.0, -8), -126);
  if (e == 0) {
    *lo = 0.0;
    *hi = min_normal_edge;
  } else if (e == 255) {
    *lo = std::ldexp(shrink, 128);
    *hi = INFINITY;
  } else {
    *lo = e == 1 ? min_normal_edge : std::ldexp(shrink, e - 127);
    *hi = std::ldexp(shrink, e - 126);
  }
}

// P(lo <= |X| < hi) for X ~ N(0, sigma^2); erfc in the upper tail keeps
// small probabilities accurate.
double binade_mass(int e, double sigma) {
  double lo, hi;
  rounded_binade(e, &lo, &hi);
  const double scale = 1.0 / (sigma * std::sqrt(2.0));
  const double a = lo * scale;
  if (a >= 1.0) return std::erfc(a) - (std::isinf(hi) ? 0.0 : std::erfc(hi * scale));
  return (std::isinf(hi) ? 1.0 : std::erf(hi * scale)) - std::erf(a);
}

}  // namespace

namespace zc {
namespace {
std::atomic<int> g_sm_count[kMaxDevices];
}

cudaError_t device_info(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  info->device = dev;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    info->sm_count = g_sm_count[dev].load(std::memory_order_relaxed);
    if (info->sm_count > 0) return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(&info->sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && cached) g_sm_count[dev].store(info->sm_count, std::memory_order_relaxed);
  return e;
}

cudaError_t prepare_kernel(KernelPrep& kp, const void* fn, int threads, int smem_bytes, const DeviceInfo& dev,
                           int* per_sm) {
  const bool cached = dev.device >= 0 && dev.device < kMaxDevices;
  if (cached) {
    *per_sm = kp.per_sm[dev.device].load(std::memory_order_acquire);
    if (*per_sm > 0) return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, fn, threads, static_cast<size_t>(smem_bytes));
  if (e != cudaSuccess) return e;
  if (*per_sm < 1) return cudaErrorInvalidConfiguration;
  if (cached) kp.per_sm[dev.device].store(*per_sm, std::memory_order_release);
  return cudaSuccess;
}

cudaError_t launch_kernel(const void* fn, dim3 grid, dim3 block, int smem_bytes, cudaStream_t stream, void** args,
                          bool cooperative) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 2u : 1u;
  return cudaLaunchKernelExC(&cfg, fn, args);
}
}  // namespace zc

extern "C" {

const char* zc_status_string(int status) {
  switch (status) {
    case ZC_OK: return "ZC_OK";
    case ZC_ERR_INVALID_ARG: return "ZC_ERR_INVALID_ARG";
    case ZC_ERR_ALIGNMENT: return "ZC_ERR_ALIGNMENT";
    case ZC_ERR_TOO_LARGE: return "ZC_ERR_TOO_LARGE";
    case ZC_ERR_WORKSPACE: return "ZC_ERR_WORKSPACE";
    case ZC_ERR_CODEBOOK: return "ZC_ERR_CODEBOOK";
    case ZC_ERR_CUDA: return "ZC_ERR_CUDA";
    case ZC_ERR_ESCAPE_OVERFLOW: return "ZC_ERR_ESCAPE_OVERFLOW";
    case ZC_ERR_BAD_HEADER: return "ZC_ERR_BAD_HEADER";
    case ZC_ERR_CORRUPT_STREAM: return "ZC_ERR_CORRUPT_STREAM";
    case ZC_ERR_SIZE_MISMATCH: return "ZC_ERR_SIZE_MISMATCH";
    case ZC_ERR_TIMEOUT: return "ZC_ERR_TIMEOUT";
    case ZC_ERR_DUP_CODEBOOK: return "ZC_ERR_DUP_CODEBOOK";
    case ZC_ERR_OUT_OF_ROOM: return "ZC_ERR_OUT_OF_ROOM";
    default: return "ZC_ERR_UNKNOWN";
  }
}

const char* zc_version(void) { return "libzc 1.0 ZC1"; }

zc_status zc_codebook_from_sigma(double sigma, uint8_t cb_out[7]) {
  if (!cb_out || !(sigma > 0.0) || !std::isfinite(sigma)) return ZC_ERR_INVALID_ARG;
  double p[256];
  for (int e = 0; e < 256; e++) p[e] = binade_mass(e, sigma);
  bool used[256] = {false};
  for (int k = 0; k < 7; k++) {
    int best = -1;
    for (int e = 0; e < 256; e++)
      if (!used[e] && (best < 0 || p[e] > p[best])) best = e;  // ties keep the smaller exponent
    used[best] = true;
    cb_out[k] = static_cast<uint8_t>(best);
  }
  return ZC_OK;
}

zc_status zc_compressed_size(uint64_t n, uint64_t* main_bytes_out, uint64_t* max_escape_bytes) {
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (main_bytes_out) *main_bytes_out = main_bytes(n);
  if (max_escape_bytes) *max_escape_bytes = n;
  return ZC_OK;
}

zc_status zc_workspace_size(const uint64_t* h_ns, int count, uint64_t* bytes) {
  if (!h_ns || count < 1 || !bytes) return ZC_ERR_INVALID_ARG;
  uint64_t tiles = 0;
  for (int i = 0; i < count; i++) {
    if (h_ns[i] > kMaxN) return ZC_ERR_TOO_LARGE;
    tiles += num_tiles(h_ns[i]);
  }
  *bytes = ws_bytes_for_tiles(tiles);
  return ZC_OK;
}

zc_status zc_histogram_topk(const void* d_in, uint64_t n, uint8_t* d_cb_out, uint32_t* d_hist_out, void* d_ws,
                            uint64_t ws_bytes, int32_t* d_status, void* stream) {
  const ApiRange range_("zc_histogram_topk");
  if ((!d_in && n) || !d_cb_out || !d_status) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(d_in, 16) || !aligned(d_status, 4) || (d_hist_out && !aligned(d_hist_out, 4)))
    return ZC_ERR_ALIGNMENT;
  if (zc_status s = check_ws(d_ws, ws_bytes, 0)) return s;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  return cuda_status(launch_histogram(static_cast<const uint16_t*>(d_in), n, d_cb_out, d_hist_out, ws_header(d_ws),
                                      d_status, as_stream(stream), dev));
}

static zc_status validate_encode_tensor(const void* in, uint64_t n, const uint8_t* cb, const void* main,
                                        const void* esc, uint64_t esc_cap) {
  if (!main || !cb || (!in && n) || (!esc && esc_cap)) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(in, 16) || !aligned(main, 16) || !aligned(esc, 16)) return ZC_ERR_ALIGNMENT;
  return ZC_OK;
}

static zc_status compress_one(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                              uint64_t esc_capacity, void* d_ws, uint64_t ws_bytes, int32_t* d_status, void* stream,
                              bool adaptive) {
  if (!d_status) return ZC_ERR_INVALID_ARG;
  if (!aligned(d_status, 4)) return ZC_ERR_ALIGNMENT;
  if (zc_status s = validate_encode_tensor(d_in, n, d_cb, d_main, d_esc, esc_capacity)) return s;
  if (zc_status s = check_ws(d_ws, ws_bytes, num_tiles(n))) return s;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  EncTensor t{static_cast<const uint16_t*>(d_in), static_cast<uint8_t*>(d_main), static_cast<uint8_t*>(d_esc),
              d_cb, n, esc_capacity};
  return cuda_status(launch_encode(&t, 1, ws_header(d_ws), ws_flags(d_ws), d_status, as_stream(stream), dev,
                                   adaptive));
}
zc_status zc_compress(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                      uint64_t esc_capacity, void* d_ws, uint64_t ws_bytes, int32_t* d_status, void* stream) {
  const ApiRange range_("zc_compress");
  return compress_one(d_in, n, d_cb, d_main, d_esc, esc_capacity, d_ws, ws_bytes, d_status, stream, false);
}
zc_status zc_compress_adaptive(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                               uint64_t esc_capacity, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                               void* stream) {
  const ApiRange range_("zc_compress_adaptive");
  return compress_one(d_in, n, d_cb, d_main, d_esc, esc_capacity, d_ws, ws_bytes, d_status, stream, true);
}
zc_status zc_raw_spill(uint64_t n, uint64_t* bytes) {
  if (!bytes) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  *bytes = raw_spill(n);
  return ZC_OK;
}

static zc_status validate_decode_tensor(const void* main, const void* esc, uint64_t esc_bytes, uint64_t n,
                                        const void* out) {
  if (!main || (!out && n) || (!esc && esc_bytes)) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(main, 16) || !aligned(esc, 16) || !aligned(out, 16)) return ZC_ERR_ALIGNMENT;
  return ZC_OK;
}

zc_status zc_decompress(const void* d_main, const void* d_esc, uint64_t esc_bytes, uint64_t n, void* d_out,
                        int32_t* d_status, void* stream) {
  const ApiRange range_("zc_decompress");
  if (!d_status) return ZC_ERR_INVALID_ARG;
  if (!aligned(d_status, 4)) return ZC_ERR_ALIGNMENT;
  if (zc_status s = validate_decode_tensor(d_main, d_esc, esc_bytes, n, d_out)) return s;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  DecTensor t{static_cast<const uint8_t*>(d_main), static_cast<const uint8_t*>(d_esc), static_cast<uint16_t*>(d_out),
              n, esc_bytes};
  return cuda_status(launch_decode(&t, 1, d_status, as_stream(stream), dev));
}

zc_status zc_decompress_reduce(int P, const void* const* h_mains, const void* const* h_escs,
                               const uint64_t* h_esc_bytes, uint64_t n, void* d_out, const uint8_t* d_out_cb,
                               void* d_out_main, void* d_out_esc, uint64_t out_esc_capacity, void* d_ws,
                               uint64_t ws_bytes, int32_t* d_status, void* stream) {
  const ApiRange range_("zc_decompress_reduce");
  if (P < 1 || P > ZC_MAX_SHARDS || !h_mains || !h_escs || !h_esc_bytes || !d_status) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(d_status, 4) || !aligned(d_out, 16)) return ZC_ERR_ALIGNMENT;
  if (!d_out && !d_out_cb) return ZC_ERR_INVALID_ARG;
  Shard shards[ZC_MAX_SHARDS];
  for (int r = 0; r < P; r++) {
    if (!h_mains[r] || (!h_escs[r] && h_esc_bytes[r])) return ZC_ERR_INVALID_ARG;
    if (!aligned(h_mains[r], 16) || !aligned(h_escs[r], 16)) return ZC_ERR_ALIGNMENT;
    shards[r] = Shard{static_cast<const uint8_t*>(h_mains[r]), static_cast<const uint8_t*>(h_escs[r]),
                      h_esc_bytes[r]};
  }
  WsHeader* ws = nullptr;
  Flag* flags = nullptr;
  if (d_out_cb) {
    if (zc_status s = validate_encode_tensor(d_out ? d_out : d_out_main, n, d_out_cb, d_out_main, d_out_esc,
                                             out_esc_capacity))
      return s;
    if (zc_status s = check_ws(d_ws, ws_bytes, num_tiles(n))) return s;
    ws = ws_header(d_ws);
    flags = ws_flags(d_ws);
  }
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  return cuda_status(launch_reduce(shards, P, n, static_cast<uint16_t*>(d_out), d_out_cb,
                                   static_cast<uint8_t*>(d_out_main), static_cast<uint8_t*>(d_out_esc),
                                   out_esc_capacity, ws, flags, d_status, as_stream(stream), dev));
}

static zc_status compress_batched(int count, const zc_tensor* h_tensors, void* d_ws, uint64_t ws_bytes,
                                  int32_t* d_status, void* stream, bool adaptive) {
  if (count < 1 || !h_tensors || !d_status) return ZC_ERR_INVALID_ARG;
  if (!aligned(d_status, 4)) return ZC_ERR_ALIGNMENT;
  uint64_t tiles = 0;
  for (int i = 0; i < count; i++) {
    const zc_tensor& t = h_tensors[i];
    if (zc_status s = validate_encode_tensor(t.bf16, t.n, t.cb, t.main, t.esc, t.esc_bytes)) return s;
    tiles += num_tiles(t.n);
  }
  if (zc_status s = check_ws(d_ws, ws_bytes, tiles)) return s;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  // Launches of up to kMaxBatch tensors each, ordered on the stream; each
  // launch uses the flags from offset 0 (an epoch separates the launches).
  EncTensor ts[kMaxBatch];
  for (int base = 0; base < count; base += kMaxBatch) {
    const int m = count - base < kMaxBatch ? count - base : kMaxBatch;
    for (int i = 0; i < m; i++) {
      const zc_tensor& t = h_tensors[base + i];
      ts[i] = EncTensor{static_cast<const uint16_t*>(t.bf16), static_cast<uint8_t*>(t.main),
                        static_cast<uint8_t*>(t.esc), t.cb, t.n, t.esc_bytes};
    }
    cudaError_t e = launch_encode(ts, m, ws_header(d_ws), ws_flags(d_ws), d_status, as_stream(stream), dev, adaptive);
    if (e != cudaSuccess) return ZC_ERR_CUDA;
  }
  return ZC_OK;
}
zc_status zc_compress_batched(int count, const zc_tensor* h_tensors, void* d_ws, uint64_t ws_bytes,
                              int32_t* d_status, void* stream) {
  const ApiRange range_("zc_compress_batched");
  return compress_batched(count, h_tensors, d_ws, ws_bytes, d_status, stream, false);
}
zc_status zc_compress_batched_adaptive(int count, const zc_tensor* h_tensors, void* d_ws, uint64_t ws_bytes,
                                       int32_t* d_status, void* stream) {
  const ApiRange range_("zc_compress_batched_adaptive");
  return compress_batched(count, h_tensors, d_ws, ws_bytes, d_status, stream, true);
}

struct zc_pipeline_plan_s {
  cudaGraphExec_t exec;
  int device;
};
static zc_status pipeline_args_ok(const void* d_in, uint64_t n, const uint8_t* d_cb, const void* d_out,
                                  uint64_t chunk_elems, const void* d_ws, uint64_t ws_bytes, const int32_t* d_status) {
  if (!d_status || !d_cb || !d_ws || ((!d_in || !d_out) && n) || chunk_elems == 0 || chunk_elems % 8 != 0)
    return ZC_ERR_INVALID_ARG;
  if (chunk_elems > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(d_in, 16) || !aligned(d_out, 16) || !aligned(d_ws, 256) || !aligned(d_status, 4))
    return ZC_ERR_ALIGNMENT;
  if (ws_bytes < pipeline_workspace_bytes(chunk_elems)) return ZC_ERR_WORKSPACE;
  return ZC_OK;
}
zc_status zc_pipeline_plan_create(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_out,
                                  uint64_t chunk_elems, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                  int overlap, zc_pipeline_plan* plan) {
  const ApiRange range_("zc_pipeline_plan_create");
  if (!plan) return ZC_ERR_INVALID_ARG;
  *plan = nullptr;
  const zc_status a = pipeline_args_ok(d_in, n, d_cb, d_out, chunk_elems, d_ws, ws_bytes, d_status);
  if (a != ZC_OK) return a;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (capture_pipeline(static_cast<const uint16_t*>(d_in), n, d_cb, static_cast<uint16_t*>(d_out), chunk_elems,
                       static_cast<uint8_t*>(d_ws), d_status, overlap != 0, dev, &exec) != cudaSuccess)
    return ZC_ERR_CUDA;
  zc_pipeline_plan p = new (std::nothrow) zc_pipeline_plan_s{exec, dev.device};
  if (!p) {
    if (exec) cudaGraphExecDestroy(exec);
    return ZC_ERR_CUDA;
  }
  *plan = p;
  return ZC_OK;
}
zc_status zc_pipeline_plan_launch(zc_pipeline_plan plan, void* stream) {
  const ApiRange range_("zc_pipeline_plan_launch");
  if (!plan) return ZC_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  if (dev != plan->device) return ZC_ERR_INVALID_ARG;
  if (!plan->exec) return ZC_OK;  // n == 0
  return cuda_status(cudaGraphLaunch(plan->exec, as_stream(stream)));
}
zc_status zc_pipeline_plan_destroy(zc_pipeline_plan plan) {
  if (!plan) return ZC_OK;
  const cudaError_t e = plan->exec ? cudaGraphExecDestroy(plan->exec) : cudaSuccess;
  delete plan;
  return cuda_status(e);
}
zc_status zc_pipeline_workspace_size(uint64_t chunk_elems, uint64_t* bytes) {
  if (!bytes || chunk_elems == 0 || chunk_elems % 8 != 0) return ZC_ERR_INVALID_ARG;
  if (chunk_elems > kMaxN) return ZC_ERR_TOO_LARGE;
  *bytes = pipeline_workspace_bytes(chunk_elems);
  return ZC_OK;
}
zc_status zc_pipelined_transfer(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_out,
                                uint64_t chunk_elems, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                void* stream_compress, void* stream_link, void* stream_decompress) {
  const ApiRange range_("zc_pipelined_transfer");
  const zc_status a = pipeline_args_ok(d_in, n, d_cb, d_out, chunk_elems, d_ws, ws_bytes, d_status);
  if (a != ZC_OK) return a;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  return cuda_status(launch_pipeline(static_cast<const uint16_t*>(d_in), n, d_cb, static_cast<uint16_t*>(d_out),
                                     chunk_elems, static_cast<uint8_t*>(d_ws), d_status, as_stream(stream_compress),
                                     as_stream(stream_link), as_stream(stream_decompress), dev));
}
static bool models_valid(const zc_link_model* link, const zc_codec_model* codec) {
  return link && codec && link->bandwidth_gbps > 0 && link->latency_us >= 0 && codec->compress_gbps > 0 &&
         codec->decompress_gbps > 0 && codec->ratio > 0 && std::isfinite(link->bandwidth_gbps) &&
         std::isfinite(link->latency_us) && std::isfinite(codec->compress_gbps) &&
         std::isfinite(codec->decompress_gbps) && std::isfinite(codec->ratio);
}
// microseconds to move `bytes` at `gbps` (1 GB/s = 1e3 bytes per microsecond)
static double us_at(double bytes, double gbps) { return bytes / (gbps * 1e3); }
zc_status zc_transfer_pays(uint64_t bytes, const zc_link_model* link, const zc_codec_model* codec, int* pays,
                           double* t_raw_us, double* t_zipped_us) {
  if (!models_valid(link, codec)) return ZC_ERR_INVALID_ARG;
  const double b = static_cast<double>(bytes);
  const double raw = link->latency_us + us_at(b, link->bandwidth_gbps);
  const double zipped = us_at(b, codec->compress_gbps) + link->latency_us +
                        us_at(b / codec->ratio, link->bandwidth_gbps) + us_at(b, codec->decompress_gbps);
  if (pays) *pays = zipped < raw ? 1 : 0;
  if (t_raw_us) *t_raw_us = raw;
  if (t_zipped_us) *t_zipped_us = zipped;
  return ZC_OK;
}
zc_status zc_reduce_scatter_choose(uint64_t bytes, int P, const zc_link_model* link, const zc_codec_model* codec,
                                   int* use_zipped, double* t_native_us, double* t_zipped_us) {
  if (!models_valid(link, codec) || P < 1) return ZC_ERR_INVALID_ARG;
  const double b = static_cast<double>(bytes), p = static_cast<double>(P);
  const double native = (p - 1.0) * (link->latency_us + us_at(b / p, link->bandwidth_gbps));
  const double exchange = P > 1 ? link->latency_us + us_at((p - 1.0) / p * b / codec->ratio, link->bandwidth_gbps) : 0.0;
  const double zipped = us_at(b, codec->compress_gbps) + exchange + us_at(b, codec->decompress_gbps);
  if (use_zipped) *use_zipped = zipped < native ? 1 : 0;
  if (t_native_us) *t_native_us = native;
  if (t_zipped_us) *t_zipped_us = zipped;
  return ZC_OK;
}
static const uint8_t kZqDefaultWidths[8] = {3, 3, 3, 3, 3, 4, 5, 8};
static bool zq_widths_valid(const uint8_t* w) {
  uint32_t cap = 0;
  for (int r = 0; r < 8; r++) {
    if (w[r] > 8) return false;
    cap += 1u << w[r];
  }
  return cap >= 256;
}
static bool zq_table_valid(const zq_table* t) {
  if (!zq_widths_valid(t->width)) return false;
  bool seen[256] = {false};
  for (int k = 0; k < 256; k++) {
    if (seen[t->sym[k]]) return false;
    seen[t->sym[k]] = true;
  }
  return true;
}
zc_status zq_default_widths(uint8_t widths[8]) {
  if (!widths) return ZC_ERR_INVALID_ARG;
  std::memcpy(widths, kZqDefaultWidths, 8);
  return ZC_OK;
}
zc_status zq_table_from_histogram(const uint64_t* h_hist, const uint8_t* widths, zq_table* out) {
  if (!h_hist || !out) return ZC_ERR_INVALID_ARG;
  const uint8_t* w = widths ? widths : kZqDefaultWidths;
  if (!zq_widths_valid(w)) return ZC_ERR_CODEBOOK;
  std::memcpy(out->width, w, 8);
  bool taken[256] = {false};
  for (int k = 0; k < 256; k++) {
    int best = -1;
    for (int s = 0; s < 256; s++)
      if (!taken[s] && (best < 0 || h_hist[s] > h_hist[best])) best = s;  // ties keep the smaller byte
    taken[best] = true;
    out->sym[k] = static_cast<uint8_t>(best);
  }
  return ZC_OK;
}
zc_status zq_max_bytes(uint64_t n, uint64_t* bytes) {
  if (!bytes) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  *bytes = zq_stream_max_bytes(n);
  return ZC_OK;
}
zc_status zq_compress(const void* d_in, uint64_t n, const zq_table* h_table, void* d_out, uint64_t out_capacity,
                      void* d_ws, uint64_t ws_bytes, int32_t* d_status, void* stream) {
  const ApiRange range_("zq_compress");
  if (!d_status || !h_table || !d_out || (!d_in && n)) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(d_in, 16) || !aligned(d_out, 16) || !aligned(d_status, 4)) return ZC_ERR_ALIGNMENT;
  if (!zq_table_valid(h_table)) return ZC_ERR_CODEBOOK;
  if (out_capacity < ZQ_HEADER_BYTES + (4 * ((n + ZQ_BLOCK_SYMBOLS - 1) / ZQ_BLOCK_SYMBOLS) + 127) / 128 * 128)
    return ZC_ERR_INVALID_ARG;  // not even the header and offset table fit
  if (zc_status s = check_ws(d_ws, ws_bytes, num_tiles(n))) return s;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  return cuda_status(launch_zq_encode(static_cast<const uint8_t*>(d_in), n, h_table->width, h_table->sym,
                                      static_cast<uint8_t*>(d_out), out_capacity, ws_header(d_ws), ws_flags(d_ws),
                                      d_status, as_stream(stream), dev));
}
zc_status zq_decompress(const void* d_in, uint64_t in_bytes, uint64_t n, void* d_out, int32_t* d_status,
                        void* stream) {
  const ApiRange range_("zq_decompress");
  if (!d_status || !d_in || (!d_out && n)) return ZC_ERR_INVALID_ARG;
  if (n > kMaxN) return ZC_ERR_TOO_LARGE;
  if (!aligned(d_in, 16) || !aligned(d_out, 16) || !aligned(d_status, 4)) return ZC_ERR_ALIGNMENT;
  if (in_bytes < ZQ_HEADER_BYTES) return ZC_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  return cuda_status(launch_zq_decode(static_cast<const uint8_t*>(d_in), in_bytes, n, static_cast<uint8_t*>(d_out),
                                      d_status, as_stream(stream), dev));
}
zc_status zc_decompress_batched(int count, const zc_tensor* h_tensors, int32_t* d_status, void* stream) {
  const ApiRange range_("zc_decompress_batched");
  if (count < 1 || !h_tensors || !d_status) return ZC_ERR_INVALID_ARG;
  if (!aligned(d_status, 4)) return ZC_ERR_ALIGNMENT;
  for (int i = 0; i < count; i++) {
    const zc_tensor& t = h_tensors[i];
    if (zc_status s = validate_decode_tensor(t.main, t.esc, t.esc_bytes, t.n, t.bf16)) return s;
  }
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  DecTensor ts[kMaxBatch];
  for (int base = 0; base < count; base += kMaxBatch) {
    const int m = count - base < kMaxBatch ? count - base : kMaxBatch;
    for (int i = 0; i < m; i++) {
      const zc_tensor& t = h_tensors[base + i];
      ts[i] = DecTensor{static_cast<const uint8_t*>(t.main), static_cast<const uint8_t*>(t.esc),
                        static_cast<uint16_t*>(t.bf16), t.n, t.esc_bytes};
    }
    cudaError_t e = launch_decode(ts, m, d_status, as_stream(stream), dev);
    if (e != cudaSuccess) return ZC_ERR_CUDA;
  }
  return ZC_OK;
}

}  // extern "C"
