// zc_device.cuh -- device building blocks shared by the libzc kernels (sm_103a).
//
// Format constants, the per-warp TMA/mbarrier pipeline primitives, the
// bounded window sum that gives every scan unit its escape offset, and the
// per-block encode and decode routines of ZC1 (layout in include/zc.h).
// Method: [ZipCCL §2.B] field split, 3-bit codes, escape array; [ZipCCL §2.C]
// three 1-bit code arrays, column-major, 128-byte blocks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zc.h"

namespace zc {

constexpr uint32_t kTile = ZC_TILE_ELEMS;          // 4096 elements
constexpr uint32_t kBlock = ZC_BLOCK_ELEMS;        // 1024 elements
constexpr uint32_t kTileBytes = ZC_TILE_BYTES;     // 5632
constexpr uint32_t kBlockBytes = ZC_BLOCK_BYTES;   // 1408
constexpr uint32_t kHeader = ZC_HEADER_BYTES;      // 128
constexpr uint32_t kFull = 0xFFFFFFFFu;
// Upper bound on any inter-block wait (escape scan, TMA completion).  Normal
// waits last microseconds; after this the kernel records ZC_ERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------- workspace
// The caller zero-fills the workspace once.  Every kernel returns it to a
// reusable state: the exit counter is reset by the CTA that completes it, escape
// scan flags are tagged with a per-launch epoch so stale flags of earlier
// launches never match, and histogram bins are cleared by the last CTA.
struct WsHeader {
  uint32_t hold_tile;  // test hook for the bounded waits: if non-zero, scan unit hold_tile - 1
                       // publishes no count, so the scans that need it must time out; reset
                       // to 0 by the launch (scan_exit)
  uint32_t exited;     // CTAs of the running encoding launch counted in once they have read the
                       // epoch (after their scan, in the decode-reduce's long launches; as they
                       // leave, in the launch whose epoch wraps)
  uint32_t epoch;      // epoch tag of the last finished encoding launch
  uint32_t max_tiles;  // largest flag range ever used (cleared when the epoch wraps)
  uint32_t hist_done;  // CTAs of the running histogram launch that have finished
  uint32_t raw_done;   // CTAs of the running adaptive encoding launch done with a RAW rewrite
  uint32_t raw_arrived;  // CTAs of the running adaptive encoding launch at its grid barrier
  uint32_t raw_gen;      // generation of that barrier: bumped by the last CTA to arrive
  uint32_t pad[24];
  uint32_t hist[256];  // global exponent bins, all zero between calls
};
static_assert(sizeof(WsHeader) <= ZC_WORKSPACE_HEADER_BYTES, "workspace header too large");

// Look-back flag of one tile: {epoch << 32 | escape count of the tile,
// epoch << 32 | inclusive escape prefix}.  Each half is written once per
// launch with a single 64-bit store, so a reader sees it whole or stale.
struct __align__(16) Flag {
  unsigned long long agg;
  unsigned long long incl;
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ void set_status(int32_t* status, int code) {
  atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory loads by 32-bit shared address.  volatile keeps them after
// the mbarrier waits that publish TMA data (those carry a memory clobber).
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---------------------------------------------------------------- mbarrier + TMA
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Non-blocking probe: true if phase `parity` of `bar` has completed (acquire).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete is suspended by
// the hardware until it completes or about `hint_ns` pass, instead of coming
// back at once: a waiting warp then issues almost nothing.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may be scheduled while the kernel before it on the stream is still
// running, and every kernel lets the launch after it be scheduled as soon as
// all its CTAs have started (pdl_allow_dependents, first thing).  pdl_wait()
// waits until every grid this one depends on has completed and its memory
// operations are visible; every thread calls it before it touches global
// memory, so stream order holds for all data.  What overlaps is the launch
// itself, the placement of CTAs on SMs that the previous grid has left, and
// whatever setup a kernel does in shared memory alone before its wait
// (mbarriers, lookup tables, cleared bins).  Without the launch attribute the
// wait returns at once.  pdl_begin() is both, for kernels with no such setup.
__device__ __forceinline__ void pdl_allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
  pdl_allow_dependents();
  pdl_wait();
}

// Wait for phase `parity` of `bar` to complete, at most kWaitLimitNs.  Returns
// false (and records ZC_ERR_TIMEOUT) if the limit is reached.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity, 100000u)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      set_status(status, ZC_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// One-dimensional TMA bulk copy global -> shared, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous copy that reads only `src_bytes` (0..16) and zero-fills
// the rest; src and dst 16-byte aligned.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies land; the
// arrival counts toward the barrier's expected count.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------- warp scans
__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(kFull, v, d);
    if (lane >= static_cast<uint32_t>(d)) v += u;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
  return v;
}

// ---------------------------------------------------------------- format helpers
__host__ __device__ __forceinline__ uint64_t num_tiles(uint64_t n) { return (n + kTile - 1) / kTile; }
__host__ __device__ __forceinline__ uint64_t table_bytes(uint64_t ntiles) { return (4 * ntiles + 127) / 128 * 128; }
__host__ __device__ __forceinline__ uint64_t main_bytes(uint64_t n) {
  return kHeader + table_bytes(num_tiles(n)) + static_cast<uint64_t>(kTileBytes) * num_tiles(n);
}
__device__ __forceinline__ uint8_t* tile_ptr(uint8_t* main, uint64_t ntiles, uint64_t t) {
  return main + kHeader + table_bytes(ntiles) + static_cast<uint64_t>(kTileBytes) * t;
}
__device__ __forceinline__ const uint8_t* tile_ptr(const uint8_t* main, uint64_t ntiles, uint64_t t) {
  return main + kHeader + table_bytes(ntiles) + static_cast<uint64_t>(kTileBytes) * t;
}

// ---------------------------------------------------------------- RAW streams
// Header flags bit 0 marks a RAW stream: the values' 2n little-endian bytes
// fill the tile region (5632 ntiles bytes) and the rest, the spill, is the
// escape stream.
constexpr uint32_t kFlagRaw = ZC_FLAG_RAW;
__host__ __device__ __forceinline__ uint64_t raw_spill(uint64_t n) {
  const uint64_t region = static_cast<uint64_t>(kTileBytes) * num_tiles(n);
  return 2 * n > region ? 2 * n - region : 0;
}

// 16 bytes of a RAW image at byte offset `b` (a multiple of 16): from the
// tile region below `region`, from the escape stream above it; bytes at or
// past `two_n` read as zero and are never loaded.  Both sources are
// 16-byte aligned and `region` is a multiple of 16, so a 16-byte piece never
// straddles the two.
__device__ __forceinline__ uint4 raw_load16(const uint8_t* tiles, const uint8_t* esc, uint64_t region,
                                            uint64_t two_n, uint64_t b) {
  if (b >= two_n) return make_uint4(0u, 0u, 0u, 0u);
  const uint8_t* src = b < region ? tiles + b : esc + (b - region);
  if (b + 16 <= two_n) return __ldg(reinterpret_cast<const uint4*>(src));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  const uint16_t* h = reinterpret_cast<const uint16_t*>(src);
  for (uint32_t j = 0; b + 2 * j < two_n; j++) w[j >> 1] |= static_cast<uint32_t>(__ldg(h + j)) << (16 * (j & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Valid-element mask of this lane in block `blk` of a tile holding `n_tile`
// valid elements: bit 8k + j <-> block element 256k + 8*lane + j.
__device__ __forceinline__ uint32_t lane_valid_mask(uint32_t blk, uint32_t n_tile, uint32_t lane) {
  if (n_tile >= kTile) return kFull;
  uint32_t v = 0;
#pragma unroll
  for (uint32_t k = 0; k < 4; k++) {
    const int start = static_cast<int>(blk * kBlock + k * 256 + lane * 8);
    int c = static_cast<int>(n_tile) - start;
    c = c < 0 ? 0 : (c > 8 ? 8 : c);
    v |= ((1u << c) - 1u) << (8 * k);
  }
  return v;
}

// ---------------------------------------------------------------- encode side
// Encoder lookup table, one u32 per exponent e: bit 0 / 8 / 16 = bits 0 / 1 / 2
// of e's code, bit 24 = "escape".  Shifting an entry left by j (0..7) and
// adding moves element j's bits into bit j of four byte lanes at once.
__device__ __forceinline__ uint32_t enc_lut_entry(uint32_t code) {
  return code ? ((code & 1u) | (((code >> 1) & 1u) << 8) | (((code >> 2) & 1u) << 16)) : (1u << 24);
}

// Builds the per-warp encoder table from a device codebook; returns false if
// the codebook repeats an exponent.  Ends with __syncwarp().
__device__ __forceinline__ bool build_enc_lut(uint32_t* lut, const uint8_t* cb_dev) {
  const uint32_t lane = lane_id();
  uint32_t cb[7];
#pragma unroll
  for (int k = 0; k < 7; k++) cb[k] = __ldg(cb_dev + k);
  bool dup = false;
#pragma unroll
  for (int a = 0; a < 7; a++)
#pragma unroll
    for (int b = a + 1; b < 7; b++) dup |= (cb[a] == cb[b]);
  for (uint32_t e = lane; e < 256; e += 32) {
    uint32_t code = 0;
#pragma unroll
    for (int k = 0; k < 7; k++) code = (cb[k] == e) ? static_cast<uint32_t>(k + 1) : code;
    lut[e] = enc_lut_entry(code);
  }
  __syncwarp();
  return !dup;
}

// Table entries of the low / high value of a 32-bit word holding two bf16.
// `lut` is the table's shared address, 1 KB aligned, so the byte offset
// (exponent * 4) can be OR-ed in.
__device__ __forceinline__ uint32_t lut_lo(uint32_t w, uint32_t lut) { return lds32(((w >> 5) & 0x3FCu) | lut); }
__device__ __forceinline__ uint32_t lut_hi(uint32_t w, uint32_t lut) { return lds32(((w >> 21) & 0x3FCu) | lut); }

// Per-lane escape bookkeeping of NB encoded blocks (a tile: NB = 4).
template <int NB>
struct EscBook {
  uint32_t mask[NB];  // bit 8k + j: block element 256k + 8*lane + j is an escape
  uint32_t base[NB];  // rank of this lane's first escape in each block, from the first block on
  uint32_t total;     // escapes in the NB blocks (same in every lane)
};

// Encodes NB consecutive blocks held in shared memory (shared address `tb`:
// NB * 1024 bf16 bit patterns, zero beyond the valid ones) into their 1408-byte
// ZC1 blocks at `out` (global).  `blk0` is the index of the first block in its
// tile and `n_tile` the tile's valid elements (positions past it get code 0 and
// are not escapes).  One warp.  Lane l of group k handles block elements
// 256k + 8l .. 256k + 8l + 7 (one 16-byte vector); its 4 groups' code bits form
// one plane word per plane, which is exactly the column-major plane layout
// (byte 4l + k).  Escape ranks come from one packed warp scan over all blocks.
template <int NB>
__device__ __forceinline__ void encode_blocks(uint32_t tb, uint32_t blk0, uint32_t n_tile, uint32_t lut, uint8_t* out,
                                              EscBook<NB>& te) {
  const uint32_t lane = lane_id();
  uint32_t cnt[NB];
#pragma unroll
  for (uint32_t blk = 0; blk < NB; blk++) {
    uint32_t acc[4];
    uint2 smv[4];
#pragma unroll
    for (uint32_t k = 0; k < 4; k++) {
      const uint4 v = lds128(tb + 2 * (blk * kBlock + k * 256 + lane * 8));
      const uint32_t e0 = lut_lo(v.x, lut), e1 = lut_hi(v.x, lut), e2 = lut_lo(v.y, lut), e3 = lut_hi(v.y, lut);
      const uint32_t e4 = lut_lo(v.z, lut), e5 = lut_hi(v.z, lut), e6 = lut_lo(v.w, lut), e7 = lut_hi(v.w, lut);
      acc[k] = (e0 + (e1 << 1)) + ((e2 << 2) + (e3 << 3)) + ((e4 << 4) + (e5 << 5)) + ((e6 << 6) + (e7 << 7));
      // sign-mantissa bytes: low byte of each value holds 7 mantissa bits,
      // high byte holds the sign in bit 7
      const uint32_t lo01 = __byte_perm(v.x, v.y, 0x6420), hi01 = __byte_perm(v.x, v.y, 0x7531);
      const uint32_t lo23 = __byte_perm(v.z, v.w, 0x6420), hi23 = __byte_perm(v.z, v.w, 0x7531);
      smv[k] = make_uint2((lo01 & 0x7F7F7F7Fu) | (hi01 & 0x80808080u), (lo23 & 0x7F7F7F7Fu) | (hi23 & 0x80808080u));
    }
    uint8_t* ob = out + blk * kBlockBytes;
#pragma unroll
    for (uint32_t k = 0; k < 4; k++) *reinterpret_cast<uint2*>(ob + k * 256 + lane * 8) = smv[k];
    // transpose: byte k of plane word b = byte b of acc[k]
    const uint32_t t01 = __byte_perm(acc[0], acc[1], 0x5140), t23 = __byte_perm(acc[2], acc[3], 0x5140);
    const uint32_t u01 = __byte_perm(acc[0], acc[1], 0x7362), u23 = __byte_perm(acc[2], acc[3], 0x7362);
    uint32_t w0 = __byte_perm(t01, t23, 0x5410);
    uint32_t w1 = __byte_perm(t01, t23, 0x7632);
    uint32_t w2 = __byte_perm(u01, u23, 0x5410);
    uint32_t x = __byte_perm(u01, u23, 0x7632);
    if (n_tile < kTile) {
      const uint32_t valid = lane_valid_mask(blk0 + blk, n_tile, lane);
      w0 &= valid;
      w1 &= valid;
      w2 &= valid;
      x &= valid;
    }
    *reinterpret_cast<uint32_t*>(ob + 1024 + lane * 4) = w0;
    *reinterpret_cast<uint32_t*>(ob + 1152 + lane * 4) = w1;
    *reinterpret_cast<uint32_t*>(ob + 1280 + lane * 4) = w2;
    te.mask[blk] = x;
    cnt[blk] = __popc(x);
  }
  // packed scan: two blocks per 32-bit word, 16-bit fields (a block's total is at most 1024)
  uint32_t run = 0;
#pragma unroll
  for (int b = 0; b < NB; b += 2) {
    const uint32_t packed = cnt[b] | ((b + 1 < NB ? cnt[b + 1] : 0u) << 16);
    const uint32_t inc = warp_inclusive_scan(packed);
    const uint32_t tot = __shfl_sync(kFull, inc, 31);
    const uint32_t exc = inc - packed;
    te.base[b] = run + (exc & 0xFFFFu);
    run += tot & 0xFFFFu;
    if (b + 1 < NB) {
      te.base[b + 1] = run + (exc >> 16);
      run += tot >> 16;
    }
  }
  te.total = run;
}


// Writes the escapes of NB blocks (their 8-bit exponents, read back from the
// blocks in shared memory at shared address `tb`) at global positions prefix +
// rank, skipping positions at or beyond `cap`.  Escapes of a lane are
// consecutive, in bit order.
template <int NB>
__device__ __forceinline__ void write_escapes(uint32_t tb, const EscBook<NB>& te, uint64_t prefix, uint8_t* esc,
                                              uint64_t cap) {
  const uint32_t lane = lane_id();
  const bool fits = prefix + te.total <= cap;
  const uint32_t lane_off = tb + 16 * lane;
#pragma unroll
  for (uint32_t blk = 0; blk < NB; blk++) {
    uint32_t m = te.mask[blk];
    uint8_t* dst = esc + prefix + te.base[blk];
    const uint32_t src = lane_off + 2 * blk * kBlock;
    if (fits) {
      while (m) {
        const uint32_t p = __ffs(m) - 1;
        m &= m - 1;
        *dst++ = static_cast<uint8_t>(lds_u16(src + 512 * (p >> 3) + 2 * (p & 7)) >> 7);
      }
    } else {
      uint64_t pos = prefix + te.base[blk];
      while (m) {
        const uint32_t p = __ffs(m) - 1;
        m &= m - 1;
        if (pos < cap) esc[pos] = static_cast<uint8_t>(lds_u16(src + 512 * (p >> 3) + 2 * (p & 7)) >> 7);
        pos++;
      }
    }
  }
}

// write_escapes for a warp that has a free 1 KB shared buffer `buf`: one
// block at a time, the block's escapes (at most 1024) are gathered in `buf`
// and then stored with consecutive lanes on consecutive bytes, so each store
// instruction fills one 32-byte sector instead of touching 32 of them.
template <int NB>
__device__ __forceinline__ void write_escapes_coalesced(uint32_t tb, const EscBook<NB>& te, uint64_t prefix,
                                                        uint8_t* esc, uint64_t cap, uint8_t* buf) {
  const uint32_t lane = lane_id();
  const uint32_t lane_off = tb + 16 * lane;
#pragma unroll
  for (uint32_t blk = 0; blk < NB; blk++) {
    const uint32_t first = __shfl_sync(kFull, te.base[blk], 0);  // escapes before this block
    const uint32_t end = blk + 1 < NB ? __shfl_sync(kFull, te.base[blk + 1], 0) : te.total;
    uint32_t m = te.mask[blk];
    uint8_t* dst = buf + (te.base[blk] - first);
    const uint32_t src = lane_off + 2 * blk * kBlock;
    while (m) {
      const uint32_t p = __ffs(m) - 1;
      m &= m - 1;
      *dst++ = static_cast<uint8_t>(lds_u16(src + 512 * (p >> 3) + 2 * (p & 7)) >> 7);
    }
    __syncwarp();
    const uint64_t g0 = prefix + first;
    for (uint32_t i = lane; i < end - first; i += 32)
      if (g0 + i < cap) esc[g0 + i] = buf[i];
    __syncwarp();
  }
}

// Moves the escapes of NB blocks (8-bit exponents read back from the blocks at
// shared address `tb`) into a shared staging buffer `buf` in escape order; the
// caller guarantees te.total fits.  Escapes of a lane are consecutive.  Up to
// four escapes per iteration, so their shared loads overlap.
template <int NB>
__device__ __forceinline__ void stage_escapes_smem(uint32_t tb, const EscBook<NB>& te, uint8_t* buf) {
  const uint32_t lane = lane_id();
  const uint32_t lane_off = tb + 16 * lane;
#pragma unroll
  for (uint32_t blk = 0; blk < NB; blk++) {
    uint32_t m = te.mask[blk];
    uint8_t* dst = buf + te.base[blk];
    const uint32_t src = lane_off + 2 * blk * kBlock;
    while (m) {
      uint32_t p[4], v[4];
      int k = 0;
#pragma unroll
      for (int u = 0; u < 4; u++) {
        p[u] = m ? static_cast<uint32_t>(__ffs(m) - 1) : 0u;
        k += m != 0;
        m &= m - 1;
      }
#pragma unroll
      for (int u = 0; u < 4; u++) v[u] = lds_u16(src + 512 * (p[u] >> 3) + 2 * (p[u] & 7));
#pragma unroll
      for (int u = 0; u < 4; u++)
        if (u < k) dst[u] = static_cast<uint8_t>(v[u] >> 7);
      dst += k;
    }
  }
}

// Escape scan across scan units (a group of tiles; one flag per unit).  The
// owner of a unit publishes the unit's escape count ("aggregate", tagged with
// the launch epoch) in flags[u].agg as soon as the unit is encoded, without
// waiting on anyone.  Each CTA visits its units in increasing order, so the
// exclusive offset of its unit G is the inclusive offset of its previous unit
// P of the same tensor plus the aggregates of the units in between (or, for
// its first unit of a tensor, the aggregates from the tensor's first unit):
// window_sum() adds the aggregates of units [lo, hi) with one warp.  This is
// a decoupled look-back whose window is fixed in advance, so it never waits
// for another unit's scan, only for aggregates.  Each pass reads up to 160
// flags (5 per lane) and re-reads only those not yet published.  The wait is
// bounded (ZC_ERR_TIMEOUT; the sum is then meaningless).  All lanes return
// the sum.
constexpr int kWindowPerLane = 5;

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t window_sum(const Flag* flags, uint32_t lo, uint32_t hi, uint32_t epoch,
                                               int32_t* status, bool* timed_out) {
  const uint32_t lane = lane_id();
  uint64_t sum = 0;
  *timed_out = false;
  for (uint32_t base = lo; base < hi; base += 32 * kWindowPerLane) {
    uint32_t pending = 0;  // bit q: unit base + lane + 32q not yet counted
#pragma unroll
    for (int q = 0; q < kWindowPerLane; q++)
      if (base + lane + 32u * q < hi) pending |= 1u << q;
    unsigned long long t0 = 0;
    while (true) {
      unsigned long long f[kWindowPerLane];
#pragma unroll
      for (int q = 0; q < kWindowPerLane; q++)
        f[q] = (pending >> q) & 1u ? ld_relaxed_u64(&flags[base + lane + 32u * q].agg) : 0ull;
#pragma unroll
      for (int q = 0; q < kWindowPerLane; q++) {
        if (((pending >> q) & 1u) && static_cast<uint32_t>(f[q] >> 32) == epoch) {
          sum += static_cast<uint32_t>(f[q]);
          pending &= ~(1u << q);
        }
      }
      if (!__any_sync(kFull, pending != 0)) break;
      unsigned long long now = 0;
      if (lane == 0) now = global_ns();
      now = __shfl_sync(kFull, now, 0);
      if (t0 == 0) t0 = now;
      if (now - t0 > kWaitLimitNs) {
        if (lane == 0) set_status(status, ZC_ERR_TIMEOUT);
        *timed_out = true;
        break;
      }
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(kFull, sum, d);
  return sum;
}

// ---------------------------------------------------------------- decode side
// One spread table S(v) (bit j of byte v at bit 4j) held in NC lane copies,
// interleaved: word v * NC + c holds S(v), and lane l reads copy l % NC.  A
// lookup by 32 lanes with data-dependent bytes then touches bank (v * NC +
// l % NC) mod 32, so NC = 32 puts every lane in its own bank (no conflicts,
// 32 KB) and NC = 16 leaves at most two lanes per bank.  The three planes
// share the table: the selector is S(p0) + 2 S(p1) + 4 S(p2), the bits being
// disjoint.
template <int NC>
__device__ __forceinline__ void build_spread_replicated(uint32_t* tab) {
  for (uint32_t i = threadIdx.x; i < 256u * NC; i += blockDim.x) {
    const uint32_t v = i / NC;
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) s |= ((v >> j) & 1u) << (4 * j);
    tab[i] = s;
  }
}

// Permute selector of group k of a lane's plane words (nibble j = the 3-bit
// code of element 8 lane + 256 k + j); `lb` = the table's shared address plus
// 4 (lane % NC).
template <int NC>
__device__ __forceinline__ uint32_t spread_sel(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t k, uint32_t lb) {
  const uint32_t s0 = lds32(lb + __byte_perm(w0, 0u, 0x4440u + k) * (4u * NC));
  const uint32_t s1 = lds32(lb + __byte_perm(w1, 0u, 0x4440u + k) * (4u * NC));
  const uint32_t s2 = lds32(lb + __byte_perm(w2, 0u, 0x4440u + k) * (4u * NC));
  return s0 + 2u * s1 + 4u * s2;
}

// An exponent rotated right by one bit: (e & 1) << 7 | e >> 1.  In this form
// the exponent's low bit sits where a bf16's low byte wants it (bit 7) and its
// other seven bits where the high byte wants them (bits 0..6), so a bf16 is
// a bit-select between its sign-mantissa byte and this byte (see bf16_quad).
__device__ __forceinline__ uint32_t rot_exp(uint32_t e) { return ((e >> 1) | (e << 7)) & 0xFFu; }

// Code -> rotated exponent table as two words for __byte_perm: byte c of
// (t0, t1) is rot_exp of the exponent of code c (byte 0, code 0 = escape, is
// a placeholder 0).
struct DecTable {
  uint32_t t0, t1;
};

__device__ __forceinline__ DecTable make_dec_table(const uint8_t cb[7]) {
  DecTable d;
  d.t0 = (rot_exp(cb[0]) << 8) | (rot_exp(cb[1]) << 16) | (rot_exp(cb[2]) << 24);
  d.t1 = rot_exp(cb[3]) | (rot_exp(cb[4]) << 8) | (rot_exp(cb[5]) << 16) | (rot_exp(cb[6]) << 24);
  return d;
}

// The four bf16 values of a group of four elements, as two packed pairs
// (p0 = elements 0, 1; p1 = elements 2, 3), from the group's sign-mantissa
// word `sm` (byte i = s << 7 | m of element i) and its rotated-exponent word
// `rx` (byte i = rot_exp(e) of element i): two bit-selects give all four low
// bytes ((e & 1) << 7 | m) and all four high bytes (s << 7 | e >> 1), two byte
// permutes interleave them.
__device__ __forceinline__ void bf16_quad(uint32_t sm, uint32_t rx, uint32_t& p0, uint32_t& p1) {
  const uint32_t lo = (sm & 0x7F7F7F7Fu) | (rx & 0x80808080u);
  const uint32_t hi = (rx & 0x7F7F7F7Fu) | (sm & 0x80808080u);
  p0 = __byte_perm(lo, hi, 0x5140);
  p1 = __byte_perm(lo, hi, 0x7362);
}

// Source of escape bytes for one (tile, stream): the first `staged` ranks sit
// in shared memory at `smem`, the rest are read from global at `glob`; ranks at
// or beyond `count` are invalid (corrupt stream) and read as 0.
struct EscSource {
  const uint8_t* smem;
  const uint8_t* glob;
  uint32_t staged;
  uint32_t count;
};

__device__ __forceinline__ uint32_t esc_byte(const EscSource& s, uint32_t rank) {
  if (rank < s.staged) return s.smem[rank];
  if (rank < s.count) return __ldg(s.glob + rank);
  return 0;
}

// Decodes block `blk` of a ZC1 tile held in shared memory (shared address
// `tile`: 5632 B) for this lane: out[k] (k = 0..3) receives 4 words = 8 bf16
// values of block elements 256k + 8*lane + 0..7.  `spread_lb` is the lane's
// base address in a spread table of NC lane copies (build_spread_replicated);
// `scratch` is this warp's 1 KB exponent scratch.  `run` is the tile-local
// rank of the block's first escape and is advanced past the block.  Returns
// the number of code-0 positions (escapes).
template <int NC>
__device__ __forceinline__ uint32_t decode_block(uint32_t tile, uint32_t blk, uint32_t n_tile, uint32_t spread_lb,
                                                 DecTable dt, const EscSource& es, uint32_t& run, uint8_t* scratch,
                                                 uint4 out[4]) {
  const uint32_t lane = lane_id();
  const uint32_t b = tile + blk * kBlockBytes;
  const uint32_t w0 = lds32(b + 1024 + lane * 4);
  const uint32_t w1 = lds32(b + 1152 + lane * 4);
  const uint32_t w2 = lds32(b + 1280 + lane * 4);
  uint32_t z = ~(w0 | w1 | w2);
  if (n_tile < kTile) z &= lane_valid_mask(blk, n_tile, lane);
  const uint32_t c = __popc(z);
  const uint32_t inc = warp_inclusive_scan(c);
  uint32_t rank = run + inc - c;
  run += __shfl_sync(kFull, inc, 31);
  const uint32_t run_end = run;  // the tile-local rank just past the block's escapes

  // rotated exponents of the 32 elements, 4 per word: word 2k = elements 0..3 of group k,
  // word 2k + 1 = elements 4..7 (exa holds words 0..3, exb words 4..7)
  uint4 exa, exb;  // ex words 0..3 and 4..7 (16-byte vectors: stored and reloaded without moves)
  {
    uint32_t sel[4];
#pragma unroll
    for (uint32_t k = 0; k < 4; k++) sel[k] = spread_sel<NC>(w0, w1, w2, k, spread_lb);
    exa.x = __byte_perm(dt.t0, dt.t1, sel[0]);
    exa.y = __byte_perm(dt.t0, dt.t1, sel[0] >> 16);
    exa.z = __byte_perm(dt.t0, dt.t1, sel[1]);
    exa.w = __byte_perm(dt.t0, dt.t1, sel[1] >> 16);
    exb.x = __byte_perm(dt.t0, dt.t1, sel[2]);
    exb.y = __byte_perm(dt.t0, dt.t1, sel[2] >> 16);
    exb.z = __byte_perm(dt.t0, dt.t1, sel[3]);
    exb.w = __byte_perm(dt.t0, dt.t1, sel[3] >> 16);
  }
  if (z) {
    // patch escapes through shared memory (bit p of z <-> byte p of ex)
    // bytes 0..15 of the lane at scratch[16 lane], bytes 16..31 at scratch[512 + 16 lane]:
    // each 16-byte access of the warp then touches every bank once per quarter
    uint4* sp = reinterpret_cast<uint4*>(scratch + lane * 16);
    sp[0] = exa;
    sp[32] = exb;
    uint32_t m = z;
    uint8_t* dst = scratch + lane * 16;  // byte q at dst[(q & 15) + 32 (q & 16)]
    if (run_end <= es.staged) {  // (warp-uniform) every escape of the block is staged
      const uint8_t* src = es.smem + rank;
      do {
        const uint32_t p = __ffs(m) - 1;
        m &= m - 1;
        dst[(p & 15u) + 32u * (p & 16u)] = static_cast<uint8_t>(rot_exp(*src++));
      } while (m);
    } else {
      while (m) {
        const uint32_t p = __ffs(m) - 1;
        m &= m - 1;
        dst[(p & 15u) + 32u * (p & 16u)] = static_cast<uint8_t>(rot_exp(esc_byte(es, rank)));
        rank++;
      }
    }
    exa = sp[0];
    exb = sp[32];
  }
#pragma unroll
  for (uint32_t k = 0; k < 4; k++) {
    const uint2 sm = lds64(b + k * 256 + lane * 8);
    const uint32_t r0 = k == 0 ? exa.x : k == 1 ? exa.z : k == 2 ? exb.x : exb.z;
    const uint32_t r1 = k == 0 ? exa.y : k == 1 ? exa.w : k == 2 ? exb.y : exb.w;
    bf16_quad(sm.x, r0, out[k].x, out[k].y);
    bf16_quad(sm.y, r1, out[k].z, out[k].w);
  }
  return c;
}

// acc[i] += bf16 value i of the 8 packed in v: each add takes the bf16 operand
// as it is (mixed-precision add, exact widening), IEEE round-to-nearest,
// subnormals kept.
__device__ __forceinline__ void accumulate8(float (&acc)[8], uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++)
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\t"
        "add.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
        : "r"(w[i]));
}

// Stores 8 bf16 values (one 16-byte vector) at element index `idx` of a tensor
// of n elements, element by element past the end.
__device__ __forceinline__ void store8_guarded(uint16_t* out, uint64_t idx, uint64_t n, uint4 v) {
  if (idx + 8 <= n) {
    *reinterpret_cast<uint4*>(out + idx) = v;
  } else if (idx < n) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    for (uint32_t j = 0; idx + j < n; j++) out[idx + j] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
  }
}

// Writes the 128-byte ZC1 header words of a tensor except n_esc (bytes 24..31).
// Lane i writes word i.
__device__ __forceinline__ void write_header_words(uint8_t* main, uint64_t n, const uint8_t* cb_dev) {
  const uint32_t lane = lane_id();
  const uint64_t nt = num_tiles(n);
  uint32_t w = 0;
  switch (lane) {
    case 0: w = ZC_MAGIC; break;
    case 1: w = ZC_VERSION; break;  // flags 0 in the high half
    case 2: w = static_cast<uint32_t>(n); break;
    case 3: w = static_cast<uint32_t>(n >> 32); break;
    case 4: w = kTile; break;
    case 5: w = static_cast<uint32_t>(nt); break;
    case 8:
      w = static_cast<uint32_t>(__ldg(cb_dev)) | (static_cast<uint32_t>(__ldg(cb_dev + 1)) << 8) |
          (static_cast<uint32_t>(__ldg(cb_dev + 2)) << 16) | (static_cast<uint32_t>(__ldg(cb_dev + 3)) << 24);
      break;
    case 9:
      w = static_cast<uint32_t>(__ldg(cb_dev + 4)) | (static_cast<uint32_t>(__ldg(cb_dev + 5)) << 8) |
          (static_cast<uint32_t>(__ldg(cb_dev + 6)) << 16);
      break;
    default: w = 0;
  }
  if (lane != 6 && lane != 7) reinterpret_cast<uint32_t*>(main)[lane] = w;
}

// Writes n_esc into the header and zeroes the offset table's padding.  Warp.
__device__ __forceinline__ void write_header_tail(uint8_t* main, uint64_t ntiles, uint64_t n_esc) {
  const uint32_t lane = lane_id();
  if (lane == 0) *reinterpret_cast<unsigned long long*>(main + 24) = n_esc;
  const uint64_t first = kHeader + 4 * ntiles, last = kHeader + table_bytes(ntiles);
  for (uint64_t o = first + 4 * lane; o < last; o += 128) *reinterpret_cast<uint32_t*>(main + o) = 0;
}

// The epoch tag used by a launch: one more than the last finished launch's,
// never 0 (the value of a zero-filled workspace).
__device__ __forceinline__ uint32_t launch_hold(const WsHeader* ws) {
  return *reinterpret_cast<const volatile uint32_t*>(&ws->hold_tile);
}

__device__ __forceinline__ uint32_t launch_epoch(const WsHeader* ws) {
  const uint32_t e = *reinterpret_cast<const volatile uint32_t*>(&ws->epoch) + 1u;
  return e == 0 ? 1u : e;
}

// Completion counts without full fences: relaxed reductions before a
// __syncthreads, then one thread's acquire-release increment of a counter.
// The barrier puts every thread's earlier accesses before the release, and
// the increment that completes the count acquires those of every CTA.
__device__ __forceinline__ void red_add_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier of every CTA of a grid whose CTAs are all resident (a cooperative
// launch), run by thread 0 of each CTA between two __syncthreads.  The count
// of arrivals is reset by the CTA that completes it, which then bumps the
// generation word the others wait on (read before arriving), so the barrier
// is ready for the next launch with no further round trip.  Bounded: after
// kWaitLimitNs it records ZC_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool grid_barrier(uint32_t* arrived, uint32_t* gen, int32_t* status) {
  const uint32_t g = ld_relaxed_gpu(gen);
  if (atom_add_acq_rel_gpu(arrived, 1u) == gridDim.x - 1) {
    *arrived = 0;
    st_release_gpu(gen, g + 1u);
    return true;
  }
  if (ld_acquire_gpu(gen) != g) return true;
  const unsigned long long t0 = global_ns();
  while (ld_acquire_gpu(gen) == g) {
    if (global_ns() - t0 > kWaitLimitNs) {
      set_status(status, ZC_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Entry and exit of a launch that uses escape-scan flags.  Every thread that
// needs the epoch or the test hook reads them from the workspace before a
// barrier of its CTA, and after that barrier lane 0 of the CTA's scan warp
// counts the CTA in with one release increment of the exit counter
// (scan_arrive): the encoders at once, with the result needed only at the
// end, so that the count's round trip to L2 overlaps the CTA's work; the
// decode-reduce at the end of its scan, since there an increment at the start
// delays the scan warp's first look-back.  The CTA that completes the count
// knows that every thread of the launch has read both words (the barrier puts
// the CTA's reads before its increment), so at the end of its own scan it
// publishes the epoch for the next launch and resets the counter and the hook
// (scan_exit) without waiting for any other CTA.  The launch whose epoch
// wraps (tag 2^32 - 1) clears every flag, so a flag written 2^32 launches
// earlier can never pass for a current one; that has to wait until no CTA
// reads or writes a flag, so that launch counts CTAs when they leave instead,
// and the last to leave clears the flags.
constexpr uint32_t kNoArrival = 0xFFFFFFFFu;

// The increment is release-only (it orders the CTA's reads before it); the
// CTA that completes the count acquires the other CTAs' increments with a
// fence in scan_exit.
__device__ __forceinline__ uint32_t scan_arrive(WsHeader* ws, uint32_t epoch) {
  if (epoch == 0xFFFFFFFFu) return kNoArrival;
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(&ws->exited) : "memory");
  return old;
}

// Run by the whole scan warp once the CTA's last escape offsets are posted
// (the CTA's units' counts were published before they reached this warp, and
// the rest of the CTA may still be writing escapes); `arrival` is lane 0's
// scan_arrive result.
__device__ __forceinline__ void scan_exit(WsHeader* ws, Flag* flags, uint32_t epoch, uint32_t total_units,
                                          uint32_t arrival) {
  const uint32_t lane = lane_id();
  if (epoch != 0xFFFFFFFFu) {
    if (__shfl_sync(kFull, arrival, 0) != gridDim.x - 1) return;
    if (lane == 0) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");  // (acquires every CTA's increment and reads)
      ws->max_tiles = max(*reinterpret_cast<volatile uint32_t*>(&ws->max_tiles), total_units);
      ws->exited = 0;
      ws->hold_tile = 0;
      ws->epoch = epoch;
    }
    return;
  }
  // the wrap: the last CTA to leave clears the flags, then publishes epoch 0
  // (lane 0's acquire-release increment orders the CTA's flag accesses before
  // the count, and the CTA completing it acquires those of every CTA)
  int last = 0;
  if (lane == 0) last = atom_add_acq_rel_gpu(&ws->exited, 1u) == gridDim.x - 1;
  if (!__shfl_sync(kFull, last, 0)) return;
  __syncwarp();
  const uint32_t maxt = max(*reinterpret_cast<volatile uint32_t*>(&ws->max_tiles), total_units);
  for (uint32_t i = lane; i < maxt; i += 32) flags[i] = Flag{0ull, 0ull};
  __threadfence();
  __syncwarp();
  if (lane == 0) {
    ws->max_tiles = maxt;
    ws->exited = 0;
    ws->hold_tile = 0;
    ws->epoch = 0u;
  }
}

// bfloat16 bits of f, rounded to nearest even (IEEE-754 definition: add half
// an ulp minus one plus the kept lowest bit, then truncate); NaN -> 0x7FC0.
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  const uint32_t a = __float_as_uint(f);
  if ((a & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  return (a + 0x7FFFu + ((a >> 16) & 1u)) >> 16;
}

}  // namespace zc
