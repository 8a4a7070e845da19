// zq.cu -- Quad Length Codes (QLC) for FP8 e4m3 bytes: encoder and decoder.
//
// [QLC §3.1-§3.3]: a 3-bit prefix picks one of 8 regions of the
// frequency-ranked symbol space and fixes how many bits follow (code lengths
// 6/7/8/11 in the static table); [QLC §4.1-§4.2]: one table lookup per symbol
// each way.  The stream layout "ZQ1" is defined in include/zc.h.
//
// Design on sm_103a (the article's design is a hardware pipeline of one
// symbol per cycle; here a warp codes one 4096-symbol block):
//   * A block is 256 runs of 16 symbols; lane l owns runs l, l + 32, ...,
//     l + 224, so every global read and write of symbols is a warp-wide
//     512-byte run of 16-byte accesses.
//   * Encoder: one table lookup per symbol gives (code, length); codes are
//     packed most-significant-bit first into a 64-bit accumulator and leave
//     as 32-bit words into the lane's shared-memory buffer.  The warp packs
//     its 32 lanes' words behind the 8 words of lane counts and stores the
//     block with consecutive lanes on consecutive words.  Block offsets come
//     from the same single-pass scan as the bf16 encoder: a CTA's 8 warps form
//     a group, the group's size is published at once, and the CTA's offset is
//     its previous group's end plus the sizes published in between
//     (cooperative launch, bounded waits, launch epochs in the workspace).
//   * Decoder: the block's words are copied to shared memory with coalesced
//     loads; each lane decodes its runs with a 64-bit bit buffer and a
//     2048-entry table indexed by the next 11 bits, which gives the symbol
//     and its code length in one shared load.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr uint32_t kQBlock = ZQ_BLOCK_SYMBOLS;  // 4096
constexpr uint32_t kQHeader = ZQ_HEADER_BYTES;  // 384
constexpr uint32_t kQMagic = 0x3142515Au;      // "ZQB1"
constexpr uint32_t kQLaneWordsMax = 44;         // 128 symbols x 11 bits
constexpr uint32_t kQBlockWordsMax = 8 + 32 * kQLaneWordsMax;  // 1416
constexpr uint32_t kQLaneStride = 45;           // words per lane buffer (odd: no bank conflicts)
constexpr int kQEncWarps = 8;
constexpr int kQDecWarps = 8;

__host__ __device__ __forceinline__ uint64_t zq_blocks(uint64_t n) { return (n + kQBlock - 1) / kQBlock; }
__host__ __device__ __forceinline__ uint64_t zq_table_bytes(uint64_t nb) { return (4 * nb + 127) / 128 * 128; }

// Symbol i of lane `lane`'s run j (0..7), position t (0..15) within the block.
__device__ __forceinline__ uint32_t zq_run_offset(uint32_t lane, uint32_t j) { return 16u * (lane + 32u * j); }

struct QEncParams {
  const uint8_t* in;
  uint64_t n;
  uint8_t* out;
  uint64_t out_words;  // payload words available after the header and offset table
  uint8_t width[8];
  uint8_t sym[256];
  uint32_t code[256];  // symbol -> (length << 16) | code, built on the host from the table
  WsHeader* ws;
  Flag* flags;
  int32_t* status;
};

// Shared memory of the encoder, per CTA.
struct QEncShared {
  uint32_t lut[256];
  uint32_t total[kQEncWarps];   // words of each warp's block this round
  uint64_t offset[kQEncWarps];  // payload word offset of each warp's block this round
  uint32_t lanebuf[kQEncWarps][32 * kQLaneStride];
  uint32_t packed[kQEncWarps][kQBlockWordsMax];
};

__global__ void __launch_bounds__(kQEncWarps * 32, 1) zq_encode_kernel(const __grid_constant__ QEncParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  QEncShared& S = *reinterpret_cast<QEncShared*>(smem_raw);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) S.lut[i] = p.code[i];
  const uint64_t nb = zq_blocks(p.n);
  const uint64_t tbl = zq_table_bytes(nb);
  uint8_t* payload = p.out + kQHeader + tbl;
  // fixed header fields and the table (payload words come with the last block)
  if (blockIdx.x == 0 && warp == 0) {
    uint32_t* h = reinterpret_cast<uint32_t*>(p.out);
    for (uint32_t i = lane; i < kQHeader / 4; i += 32) {
      uint32_t v = 0;
      if (i == 0) v = kQMagic;
      else if (i == 1) v = 1u;  // version 1, flags 0
      else if (i == 2) v = static_cast<uint32_t>(p.n);
      else if (i == 3) v = static_cast<uint32_t>(p.n >> 32);
      else if (i == 4) v = kQBlock;
      else if (i == 5) v = static_cast<uint32_t>(nb);
      else if (i == 6 || i == 7) continue;  // payload words
      else if (i == 16 || i == 17) {
        const uint32_t b = 4 * (i - 16);
        v = p.width[b] | (p.width[b + 1] << 8) | (p.width[b + 2] << 16) | (uint32_t(p.width[b + 3]) << 24);
      } else if (i >= 32) {
        const uint32_t b = 4 * (i - 32);
        v = p.sym[b] | (p.sym[b + 1] << 8) | (p.sym[b + 2] << 16) | (uint32_t(p.sym[b + 3]) << 24);
      }
      h[i] = v;
    }
    if (nb == 0 && lane == 0) *reinterpret_cast<unsigned long long*>(p.out + 24) = 0ull;
  }
  __syncthreads();
  const uint32_t epoch = launch_epoch(p.ws);
  const uint32_t ngroups = static_cast<uint32_t>((nb + kQEncWarps - 1) / kQEncWarps);
  uint32_t* lb = &S.lanebuf[warp][lane * kQLaneStride];
  uint32_t* packed = S.packed[warp];
  int64_t prev_G = -1;
  uint64_t prev_incl = 0;
  for (uint32_t G = blockIdx.x; G < ngroups; G += gridDim.x) {
    const uint64_t b = static_cast<uint64_t>(G) * kQEncWarps + warp;
    uint32_t T = 0;
    if (b < nb) {
      // ---- load this lane's 8 runs and code them
      const uint64_t base = b * kQBlock;
      uint4 v[8];
#pragma unroll
      for (uint32_t j = 0; j < 8; j++) {
        const uint64_t i0 = base + zq_run_offset(lane, j);
        if (i0 + 16 <= p.n) {
          v[j] = __ldg(reinterpret_cast<const uint4*>(p.in + i0));
        } else {
          uint32_t w[4] = {0u, 0u, 0u, 0u};
          for (uint32_t t = 0; i0 + t < p.n && t < 16; t++) w[t >> 2] |= uint32_t(__ldg(p.in + i0 + t)) << (8 * (t & 3));
          v[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      unsigned long long acc = 0;
      uint32_t nacc = 0, wc = 0;
#pragma unroll
      for (uint32_t j = 0; j < 8; j++) {
        const uint64_t i0 = base + zq_run_offset(lane, j);
        const uint32_t valid = i0 >= p.n ? 0u : (p.n - i0 >= 16 ? 16u : static_cast<uint32_t>(p.n - i0));
        const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (uint32_t t = 0; t < 16; t++) {
          if (t < valid) {
            const uint32_t e = S.lut[(w4[t >> 2] >> (8 * (t & 3))) & 0xFFu];
            const uint32_t len = e >> 16;
            acc |= static_cast<unsigned long long>(e & 0xFFFFu) << (64 - nacc - len);
            nacc += len;
            if (nacc >= 32) {
              lb[wc++] = static_cast<uint32_t>(acc >> 32);
              acc <<= 32;
              nacc -= 32;
            }
          }
        }
      }
      if (nacc > 0) lb[wc++] = static_cast<uint32_t>(acc >> 32);
      // ---- pack: lane counts, then the lanes' words in lane order
      const uint32_t inc = warp_inclusive_scan(wc);
      const uint32_t pre = inc - wc;
      T = 8 + __shfl_sync(kFull, inc, 31);
      reinterpret_cast<uint8_t*>(packed)[lane] = static_cast<uint8_t>(wc);
      for (uint32_t k = 0; k < wc; k++) packed[8 + pre + k] = lb[k];
    }
    if (lane == 0) S.total[warp] = T;
    __syncthreads();
    // ---- the group's offset: warp 0 publishes the group's size and adds the
    // sizes published since this CTA's previous group
    if (warp == 0) {
      const uint32_t t = lane < kQEncWarps ? S.total[lane] : 0u;
      const uint32_t tinc = warp_inclusive_scan(t);
      const uint32_t gsum = __shfl_sync(kFull, tinc, 31);
      if (lane == 0) {
        const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
        st_relaxed(&p.flags[G].agg, tag | gsum);
      }
      bool timed_out;
      const uint64_t prefix = prev_incl + window_sum(p.flags, static_cast<uint32_t>(prev_G + 1), G, epoch, p.status,
                                                     &timed_out);
      if (lane < kQEncWarps) S.offset[lane] = prefix + (tinc - t);
      prev_G = G;
      prev_incl = prefix + gsum;
    }
    __syncthreads();
    if (b < nb) {
      const uint64_t off = S.offset[warp];
      if (lane == 0) *reinterpret_cast<uint32_t*>(p.out + kQHeader + 4 * b) = static_cast<uint32_t>(off);
      if (off + T <= p.out_words) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(payload) + off;
        for (uint32_t k = lane; k < T; k += 32) dst[k] = packed[k];
      } else if (lane == 0) {
        set_status(p.status, ZC_ERR_OUT_OF_ROOM);
      }
      if (b + 1 == nb) {
        // the last block: total payload words and the offset table's padding
        if (lane == 0) *reinterpret_cast<unsigned long long*>(p.out + 24) = off + T;
        for (uint64_t o = kQHeader + 4 * nb + 4 * lane; o < kQHeader + tbl; o += 128)
          *reinterpret_cast<uint32_t*>(p.out + o) = 0u;
      }
    }
  }
  if (warp == 0) scan_exit(p.ws, p.flags, epoch, ngroups);
}

// ---------------------------------------------------------------- decoder
struct QDecParams {
  const uint8_t* in;
  uint64_t in_bytes;
  uint64_t n;
  uint8_t* out;
  int32_t* status;
};

struct QDecShared {
  uint16_t lut[2048];  // next 11 bits -> (code length << 8) | symbol; 0 = no valid code
  int bad;
  uint32_t words[kQDecWarps][kQBlockWordsMax];
};

__global__ void __launch_bounds__(kQDecWarps * 32) zq_decode_kernel(const __grid_constant__ QDecParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  QDecShared& S = *reinterpret_cast<QDecShared*>(smem_raw);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint64_t nb = zq_blocks(p.n);
  const uint64_t tbl = zq_table_bytes(nb);
  // header checks (every CTA reaches the same verdict) and the 11-bit table
  if (threadIdx.x == 0) {
    const uint32_t* h = reinterpret_cast<const uint32_t*>(p.in);
    int err = 0;
    if (p.in_bytes < kQHeader + tbl || __ldg(h) != kQMagic || __ldg(h + 1) != 1u || __ldg(h + 4) != kQBlock ||
        __ldg(h + 5) != nb)
      err = ZC_ERR_BAD_HEADER;
    else if ((static_cast<uint64_t>(__ldg(h + 2)) | (static_cast<uint64_t>(__ldg(h + 3)) << 32)) != p.n)
      err = ZC_ERR_SIZE_MISMATCH;
    if (!err) {
      const uint64_t words = static_cast<uint64_t>(__ldg(h + 6)) | (static_cast<uint64_t>(__ldg(h + 7)) << 32);
      uint32_t cap = 0, seen[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      for (int r = 0; r < 8; r++) {
        const uint32_t w = __ldg(p.in + 64 + r);
        if (w > 8) err = ZC_ERR_BAD_HEADER;
        else cap += 1u << w;
      }
      for (int k = 0; k < 256; k++) {
        const uint32_t s = __ldg(p.in + 128 + k);
        if (seen[s >> 5] & (1u << (s & 31))) err = ZC_ERR_BAD_HEADER;
        seen[s >> 5] |= 1u << (s & 31);
      }
      if (cap < 256 || kQHeader + tbl + 4 * words > p.in_bytes) err = ZC_ERR_BAD_HEADER;
    }
    S.bad = err;
    if (err) set_status(p.status, err);
  }
  __syncthreads();
  if (S.bad) return;
  for (uint32_t q = threadIdx.x; q < 2048; q += blockDim.x) {
    const uint32_t r = q >> 8;
    uint32_t start = 0;
    for (uint32_t i = 0; i < r; i++) start += 1u << __ldg(p.in + 64 + i);
    const uint32_t w = __ldg(p.in + 64 + r);
    const uint32_t rank = start + (w == 0 ? 0u : ((q & 0xFFu) >> (8 - w)));
    S.lut[q] = rank > 255 ? uint16_t(0) : static_cast<uint16_t>(((3 + w) << 8) | __ldg(p.in + 128 + rank));
  }
  __syncthreads();
  const uint64_t words = static_cast<uint64_t>(reinterpret_cast<const uint32_t*>(p.in)[6]) |
                         (static_cast<uint64_t>(reinterpret_cast<const uint32_t*>(p.in)[7]) << 32);
  const uint32_t* table = reinterpret_cast<const uint32_t*>(p.in + kQHeader);
  const uint32_t* payload = reinterpret_cast<const uint32_t*>(p.in + kQHeader + tbl);
  uint32_t* wbuf = S.words[warp];
  const uint64_t total_warps = static_cast<uint64_t>(gridDim.x) * kQDecWarps;
  for (uint64_t b = static_cast<uint64_t>(blockIdx.x) * kQDecWarps + warp; b < nb; b += total_warps) {
    const uint64_t off = __ldg(table + b);
    const uint64_t end = b + 1 < nb ? static_cast<uint64_t>(__ldg(table + b + 1)) : words;
    if (off + 8 > end || end > words || end - off > kQBlockWordsMax) {
      if (lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
      continue;
    }
    const uint32_t T = static_cast<uint32_t>(end - off);
    for (uint32_t k = lane; k < T; k += 32) wbuf[k] = __ldg(payload + off + k);
    __syncwarp();
    const uint32_t wc = reinterpret_cast<const uint8_t*>(wbuf)[lane];
    const uint32_t inc = warp_inclusive_scan(wc);
    const uint32_t first = 8 + inc - wc;
    bool ok = 8 + __shfl_sync(kFull, inc, 31) == T;
    const uint32_t limit = ok ? first + wc : first;  // this lane's words are [first, limit)
    uint32_t next = first;
    unsigned long long buf = 0;
    uint32_t nbits = 0;
    auto refill = [&]() {
      while (nbits <= 32) {
        const uint32_t w = next < limit ? wbuf[next] : 0u;
        buf |= static_cast<unsigned long long>(w) << (32 - nbits);
        nbits += 32;
        next++;
      }
    };
    refill();
    uint64_t bits_used = 0;
    const uint64_t base = b * kQBlock;
#pragma unroll 1
    for (uint32_t j = 0; j < 8; j++) {
      const uint64_t i0 = base + zq_run_offset(lane, j);
      const uint32_t valid = i0 >= p.n ? 0u : (p.n - i0 >= 16 ? 16u : static_cast<uint32_t>(p.n - i0));
      uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (uint32_t t = 0; t < 16; t++) {
        if (t < valid) {
          const uint32_t e = S.lut[buf >> 53];
          const uint32_t len = e >> 8;
          ok &= len != 0;
          const uint32_t use = len != 0 ? len : 11u;
          o[t >> 2] |= (e & 0xFFu) << (8 * (t & 3));
          buf <<= use;
          nbits -= use;
          bits_used += use;
          if (nbits <= 32) refill();
        }
      }
      if (valid == 16) {
        *reinterpret_cast<uint4*>(p.out + i0) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        for (uint32_t t = 0; t < valid; t++) p.out[i0 + t] = static_cast<uint8_t>(o[t >> 2] >> (8 * (t & 3)));
      }
    }
    ok &= (bits_used + 31) / 32 == wc;
    if (!__all_sync(kFull, ok) && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
    __syncwarp();
  }
}

// ---------------------------------------------------------------- launches
uint64_t zq_stream_max_bytes(uint64_t n) {
  const uint64_t nb = zq_blocks(n);
  return kQHeader + zq_table_bytes(nb) + nb * static_cast<uint64_t>(kQBlockWordsMax) * 4;
}

cudaError_t launch_zq_encode(const uint8_t* in, uint64_t n, const uint8_t width[8], const uint8_t sym[256],
                             uint8_t* out, uint64_t out_bytes, WsHeader* ws, Flag* flags, int32_t* status,
                             cudaStream_t stream, const DeviceInfo& dev) {
  QEncParams p;
  p.in = in;
  p.n = n;
  p.out = out;
  const uint64_t nb = zq_blocks(n);
  const uint64_t fixed = kQHeader + zq_table_bytes(nb);
  p.out_words = out_bytes > fixed ? (out_bytes - fixed) / 4 : 0;
  uint32_t start[9] = {0};
  for (int r = 0; r < 8; r++) {
    p.width[r] = width[r];
    start[r + 1] = start[r] + (1u << width[r]);
  }
  for (int k = 0; k < 256; k++) p.sym[k] = sym[k];
  for (uint32_t k = 0; k < 256; k++) {
    int r = 0;
    while (k >= start[r + 1]) r++;
    const uint32_t code = (static_cast<uint32_t>(r) << width[r]) | (k - start[r]);
    p.code[sym[k]] = ((3u + width[r]) << 16) | code;
  }
  p.ws = ws;
  p.flags = flags;
  p.status = status;
  static_assert(sizeof(QEncParams) < 4000, "encode parameters too large");
  static KernelPrep prep;
  int per_sm = 0;
  const int smem = static_cast<int>(sizeof(QEncShared));
  cudaError_t err = prepare_kernel(prep, reinterpret_cast<const void*>(zq_encode_kernel), kQEncWarps * 32, smem, dev,
                                   &per_sm);
  if (err != cudaSuccess) return err;
  const uint32_t groups = static_cast<uint32_t>((nb + kQEncWarps - 1) / kQEncWarps);
  uint32_t ctas = groups;
  const uint32_t cap = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&p};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(zq_encode_kernel), dim3(ctas),
                                     dim3(kQEncWarps * 32), args, smem, stream);
}

cudaError_t launch_zq_decode(const uint8_t* in, uint64_t in_bytes, uint64_t n, uint8_t* out, int32_t* status,
                             cudaStream_t stream, const DeviceInfo& dev) {
  QDecParams p{in, in_bytes, n, out, status};
  static KernelPrep prep;
  int per_sm = 0;
  const int smem = static_cast<int>(sizeof(QDecShared));
  cudaError_t err = prepare_kernel(prep, reinterpret_cast<const void*>(zq_decode_kernel), kQDecWarps * 32, smem, dev,
                                   &per_sm);
  if (err != cudaSuccess) return err;
  const uint64_t nb = zq_blocks(n);
  uint64_t ctas = (nb + kQDecWarps - 1) / kQDecWarps;
  const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * static_cast<uint64_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  zq_decode_kernel<<<static_cast<unsigned>(ctas), kQDecWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace zc
