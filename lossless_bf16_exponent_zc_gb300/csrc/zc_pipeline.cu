// zc_pipeline.cu -- the zipped transfer pipeline: compress, link and decompress
// overlapped chunk by chunk on three streams.
//
// [CCCL §3.2] cuts a tensor into chunks and runs three stages concurrently on
// separate streams: compress chunk k, transfer chunk k - 1, decompress chunk
// k - 2, with double-buffered send and receive buffers.  [ZipCCL §2.D] sends
// each compressed tensor in two parts: a fixed-size part first (here the main
// stream, whose size depends on n alone) and a variable-size part after it
// (the escape stream, n_esc bytes).
//
// On one GPU the link is a device-to-device copy into receive slots that stand
// in for the peer's buffers, done by one kernel per chunk: the static part (the
// main stream, whose size the host knows) and the dynamic part (exactly n_esc
// escape bytes, n_esc read on the device from the sender's header, as a sender
// sizes its second message) -- the host never waits for a count.  Chunks are
// compressed adaptively, so an incompressible chunk travels RAW and an escape
// slot of 5/8 of the chunk's values never overflows.
//
// Each chunk costs three launches and up to seven event operations, which the host
// submits more slowly than the GPU runs them once chunks are small.  A
// pipeline plan captures the whole launch sequence once into a CUDA graph
// (from three private streams, so the graph keeps the three-stage overlap) and
// replays it with one launch.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kLinkThreads = 256;

// The link of one chunk: the main stream (main_bytes, a multiple of 16) and
// then n_esc escape bytes, n_esc read from the sender's header (clamped to the
// slot's capacity; a bad count is then caught by the decoder's header check).
// One index space of 16-byte pieces covers both parts; all four buffers are
// 16-byte aligned.
__global__ void __launch_bounds__(kLinkThreads) link_kernel(const uint8_t* __restrict__ send_main,
                                                            uint8_t* __restrict__ recv_main, uint64_t main_bytes,
                                                            const uint8_t* __restrict__ send_esc,
                                                            uint8_t* __restrict__ recv_esc, uint64_t cap) {
  pdl_begin();
  uint64_t n_esc = __ldcg(reinterpret_cast<const unsigned long long*>(send_main + 24));
  if (n_esc > cap) n_esc = cap;
  const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t nthreads = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  const uint64_t main_vecs = main_bytes / 16;
  const uint64_t vecs = main_vecs + n_esc / 16;
  for (uint64_t i = tid; i < vecs; i += nthreads) {
    if (i < main_vecs)
      reinterpret_cast<uint4*>(recv_main)[i] = __ldcg(reinterpret_cast<const uint4*>(send_main) + i);
    else
      reinterpret_cast<uint4*>(recv_esc)[i - main_vecs] =
          __ldcg(reinterpret_cast<const uint4*>(send_esc) + (i - main_vecs));
  }
  for (uint64_t i = 16 * (n_esc / 16) + tid; i < n_esc; i += nthreads) recv_esc[i] = send_esc[i];
}

// Workspace of a pipeline with chunks of c values: the encoder's workspace,
// then two send and two receive slots of (main stream, escape buffer).
struct PipeLayout {
  uint64_t enc_bytes, main_bytes, esc_bytes, slot_bytes, total;
};

static uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

static PipeLayout pipeline_layout(uint64_t c) {
  PipeLayout L;
  L.enc_bytes = round_up(ZC_WORKSPACE_HEADER_BYTES + ZC_WORKSPACE_BYTES_PER_TILE * num_tiles(c), 256);
  L.main_bytes = round_up(main_bytes(c), 256);
  // 5m/8 bounds the RAW spill of every chunk of m <= c values (the last one
  // may be shorter and spill more than a full chunk would when c is not a
  // multiple of 4096), so an adaptive chunk never overflows its slot
  L.esc_bytes = round_up((5 * c + 7) / 8 + 16, 256);
  L.slot_bytes = L.main_bytes + L.esc_bytes;
  L.total = L.enc_bytes + 4 * L.slot_bytes;
  return L;
}

uint64_t pipeline_workspace_bytes(uint64_t c) { return pipeline_layout(c).total; }

namespace {

// Events of one call, destroyed (after their last use is enqueued) on return.
struct Events {
  cudaEvent_t fork = nullptr, comp[2] = {nullptr, nullptr}, link[2] = {nullptr, nullptr},
              dec[2] = {nullptr, nullptr};
  cudaError_t create() {
    cudaError_t e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    for (int s = 0; s < 2 && e == cudaSuccess; s++) {
      e = cudaEventCreateWithFlags(&comp[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&link[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dec[s], cudaEventDisableTiming);
    }
    return e;
  }
  ~Events() {
    for (cudaEvent_t ev : {fork, comp[0], comp[1], link[0], link[1], dec[0], dec[1]})
      if (ev) cudaEventDestroy(ev);
  }
};

#define ZC_TRY(x)                              \
  do {                                         \
    cudaError_t e_ = (x);                      \
    if (e_ != cudaSuccess) return e_;          \
  } while (0)

// Enqueues the whole pipeline on sc / sl / sd, using the caller's events.
cudaError_t enqueue_pipeline(const uint16_t* in, uint64_t n, const uint8_t* cb, uint16_t* out, uint64_t c,
                             uint8_t* ws, int32_t* status, cudaStream_t sc, cudaStream_t sl, cudaStream_t sd,
                             const DeviceInfo& dev, Events& ev) {
  const PipeLayout L = pipeline_layout(c);
  WsHeader* enc_ws = reinterpret_cast<WsHeader*>(ws);
  Flag* enc_flags = reinterpret_cast<Flag*>(ws + ZC_WORKSPACE_HEADER_BYTES);
  uint8_t* slots = ws + L.enc_bytes;
  auto send_main = [&](int s) { return slots + s * L.slot_bytes; };
  auto send_esc = [&](int s) { return slots + s * L.slot_bytes + L.main_bytes; };
  auto recv_main = [&](int s) { return slots + (2 + s) * L.slot_bytes; };
  auto recv_esc = [&](int s) { return slots + (2 + s) * L.slot_bytes + L.main_bytes; };
  const uint64_t esc_cap = L.esc_bytes;

  // On three distinct streams the compress and decompress stages get disjoint
  // shares of the SMs: both kernels are persistent and ask for a whole SM's
  // shared memory per CTA, so with full grids one stage would wait for the
  // other to leave the GPU and the stages would not overlap.  (The encoder's
  // cooperative grid then stays within its share.)  Compress is the longer
  // stage; on chunks of at most 8 tiles per SM it gets two thirds of the SMs
  // (16 chunks of 2^22 values: 231 us against 252-260 us with halves), on
  // larger chunks half (4 chunks of 2^24: 173 against 179 us).  On one
  // stream the stages run one after the other and keep the whole GPU.
  DeviceInfo enc_part = dev, dec_part = dev;
  if (sc != sd && dev.sm_count >= 3) {
    const bool small = num_tiles(c) <= 8ull * static_cast<uint64_t>(dev.sm_count);
    enc_part.sm_count = small ? dev.sm_count * 2 / 3 : dev.sm_count / 2;
    dec_part.sm_count = dev.sm_count - enc_part.sm_count;
  }

  // the other two streams start after everything already enqueued on the compress stream
  ZC_TRY(cudaEventRecord(ev.fork, sc));
  ZC_TRY(cudaStreamWaitEvent(sl, ev.fork, 0));
  ZC_TRY(cudaStreamWaitEvent(sd, ev.fork, 0));
  const uint64_t chunks = (n + c - 1) / c;
  int last = 0;
  for (uint64_t k = 0; k < chunks; k++) {
    const int s = static_cast<int>(k & 1u);
    last = s;
    const uint64_t m = n - k * c < c ? n - k * c : c;
    // compress chunk k into send slot s once the link has taken chunk k - 2 out of it
    if (k >= 2) ZC_TRY(cudaStreamWaitEvent(sc, ev.link[s], 0));
    EncTensor t{in + k * c, send_main(s), send_esc(s), cb, m, esc_cap};
    ZC_TRY(launch_encode(&t, 1, enc_ws, enc_flags, status, sc, enc_part, true));
    ZC_TRY(cudaEventRecord(ev.comp[s], sc));
    // link: the static part (fixed-size main stream) and the dynamic part
    // (n_esc escape bytes, counted on the device), once receive slot s is free
    ZC_TRY(cudaStreamWaitEvent(sl, ev.comp[s], 0));
    if (k >= 2) ZC_TRY(cudaStreamWaitEvent(sl, ev.dec[s], 0));
    {
      const uint64_t mb = main_bytes(m);
      uint64_t blocks = (mb + raw_spill(m) + kLinkThreads * 16 - 1) / (kLinkThreads * 16);
      const uint64_t cap = 4ull * static_cast<uint64_t>(dev.sm_count);
      if (blocks > cap) blocks = cap;
      if (blocks == 0) blocks = 1;
      const uint8_t* sm_ = send_main(s);
      uint8_t* rm = recv_main(s);
      const uint8_t* se = send_esc(s);
      uint8_t* re = recv_esc(s);
      uint64_t lc = esc_cap;
      uint64_t lmb = mb;
      void* args[] = {&sm_, &rm, &lmb, &se, &re, &lc};
      ZC_TRY(launch_kernel(reinterpret_cast<const void*>(link_kernel), dim3(static_cast<unsigned>(blocks)),
                           dim3(kLinkThreads), 0, sl, args, false));
    }
    ZC_TRY(cudaEventRecord(ev.link[s], sl));
    // decompress chunk k from receive slot s
    ZC_TRY(cudaStreamWaitEvent(sd, ev.link[s], 0));
    DecTensor d{recv_main(s), recv_esc(s), out + k * c, m, esc_cap};
    ZC_TRY(launch_decode(&d, 1, status, sd, dec_part));
    ZC_TRY(cudaEventRecord(ev.dec[s], sd));
  }
  // join: the compress and link streams continue after the last chunk is decoded
  ZC_TRY(cudaStreamWaitEvent(sc, ev.dec[last], 0));
  ZC_TRY(cudaStreamWaitEvent(sl, ev.dec[last], 0));
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_pipeline(const uint16_t* in, uint64_t n, const uint8_t* cb, uint16_t* out, uint64_t c,
                            uint8_t* ws, int32_t* status, cudaStream_t sc, cudaStream_t sl, cudaStream_t sd,
                            const DeviceInfo& dev) {
  if (n == 0) return cudaSuccess;
  Events ev;
  ZC_TRY(ev.create());
  return enqueue_pipeline(in, n, cb, out, c, ws, status, sc, sl, sd, dev, ev);
}

cudaError_t capture_pipeline(const uint16_t* in, uint64_t n, const uint8_t* cb, uint16_t* out, uint64_t c,
                             uint8_t* ws, int32_t* status, bool overlap, const DeviceInfo& dev,
                             cudaGraphExec_t* exec) {
  *exec = nullptr;
  if (n == 0) return cudaSuccess;
  // private streams: the capture depends on nothing the caller has enqueued
  cudaStream_t st[3] = {nullptr, nullptr, nullptr};
  const int ns = overlap ? 3 : 1;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < ns && e == cudaSuccess; i++) e = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking);
  if (e == cudaSuccess) {
    Events ev;  // outlives the capture
    e = ev.create();
    if (e == cudaSuccess) e = cudaStreamBeginCapture(st[0], cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      cudaStream_t sl = overlap ? st[1] : st[0], sd = overlap ? st[2] : st[0];
      cudaError_t ee = enqueue_pipeline(in, n, cb, out, c, ws, status, st[0], sl, sd, dev, ev);
      cudaGraph_t g = nullptr;
      e = cudaStreamEndCapture(st[0], &g);  // always ends the capture, also after a failed enqueue
      if (ee != cudaSuccess) e = ee;
      if (e == cudaSuccess) e = cudaGraphInstantiateWithFlags(exec, g, 0);
      if (g) cudaGraphDestroy(g);
    }
  }
  for (int i = 0; i < ns; i++)
    if (st[i]) cudaStreamDestroy(st[i]);
  return e;
}

}  // namespace zc
