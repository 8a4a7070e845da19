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
//     block with consecutive lanes on consecutive words.  Every symbol is
//     coded once: a CTA codes a group of 16 blocks per round (one per warp)
//     and keeps them on chip while its scan warp finds the group's offset
//     from the totals other CTAs publish (the escape scan's window sums and
//     epoch protocol, cooperative launch); a block is stored one round later.
//   * Decoder: the block's words arrive in shared memory with one TMA bulk
//     copy per block (the block offsets are read one block ahead); each lane
//     decodes its runs with a 32-bit funnel-shift window over two words and a
//     2048-entry table indexed by the next 11 bits, which gives the symbol and
//     its code length in one shared load; two symbols are decoded per window
//     refill (a code is at most 11 bits, so the second one still lies within
//     the next two words).
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr uint32_t kQBlock = ZQ_BLOCK_SYMBOLS;  // 4096
constexpr uint32_t kQHeader = ZQ_HEADER_BYTES;  // 384
constexpr uint32_t kQMagic = 0x3142515Au;      // "ZQB1"
constexpr uint32_t kQLaneWordsMax = 44;         // 128 symbols x 11 bits
constexpr uint32_t kQBlockWordsMax = 8 + 32 * kQLaneWordsMax;  // 1416
constexpr uint32_t kQLaneStride = 45;           // words per lane buffer (odd: no bank conflicts)
constexpr int kQEncWarps = 16;                 // coding warps; a group is 16 blocks
constexpr int kQEncThreads = (kQEncWarps + 1) * 32;  // + the scan warp
constexpr int kQDecWarps = 12;                 // 3 CTAs per SM: 36 decoding warps

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
  uint32_t lanebuf[kQEncWarps][32 * kQLaneStride];  // a lane's words of the block being coded
  uint32_t packed[kQEncWarps][kQBlockWordsMax];     // a warp's block, packed, until its offset is known
  uint32_t words[2][kQEncWarps];                    // block sizes of a round (slot = round mod 2)
  uint32_t offs[2][kQEncWarps];                     // block word offsets of a round
};

// Run j of lane `lane` in block b (zero past n); *valid = its symbols below n.
__device__ __forceinline__ uint4 zq_load_run(const uint8_t* in, uint64_t n, uint64_t b, uint32_t lane, uint32_t j,
                                            uint32_t* valid) {
  const uint64_t i0 = b * kQBlock + zq_run_offset(lane, j);
  *valid = i0 >= n ? 0u : (n - i0 >= 16 ? 16u : static_cast<uint32_t>(n - i0));
  if (*valid == 16) return __ldg(reinterpret_cast<const uint4*>(in + i0));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (uint32_t t = 0; t < *valid; t++) w[t >> 2] |= uint32_t(__ldg(in + i0 + t)) << (8 * (t & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The 16 table entries of a run (0 past the valid symbols).
__device__ __forceinline__ void zq_lookup_run(const uint32_t* lut, uint4 v, uint32_t valid, uint32_t (&e)[16]) {
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (uint32_t t = 0; t < 16; t++) e[t] = t < valid ? lut[(w4[t >> 2] >> (8 * (t & 3))) & 0xFFu] : 0u;
}

// Design of the launch: one CTA of 16 coding warps and 1 scan warp per SM.
// Round r of CTA c codes group G = c + r C (C CTAs): blocks 16 G .. 16 G + 15,
// one per coding warp.  A warp codes its block once, into its lane buffers
// (its runs' 32-bit words) and their word counts; the scan warp adds the
// group's 16 block sizes, publishes the group's total at once and finds the
// group's first word offset as the offset after its CTA's previous group plus
// the totals of the C - 1 groups in between (published by the CTAs that own
// them, which never wait for this one).  Stores lag one round: after the
// round's barrier a warp stores the block it packed in the previous round (at
// the offset the scan warp posted meanwhile) and packs this round's block, so
// the scan's wait overlaps the next round's coding.  The wait is bounded
// (ZC_ERR_TIMEOUT); the launch is cooperative, so every group's owner is
// resident.
__global__ void __launch_bounds__(kQEncThreads, 1) zq_encode_kernel(const __grid_constant__ QEncParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_begin();
  QEncShared& S = *reinterpret_cast<QEncShared*>(smem_raw);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) S.lut[i] = p.code[i];
  const uint64_t nb = zq_blocks(p.n);
  const uint64_t tbl = zq_table_bytes(nb);
  uint32_t* table = reinterpret_cast<uint32_t*>(p.out + kQHeader);
  uint8_t* payload = p.out + kQHeader + tbl;
  // fixed header fields and the rank table (payload words come with the last group)
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
  const uint32_t epoch = launch_epoch(p.ws);  // (both before the barrier that precedes scan_arrive)
  const uint32_t hold = launch_hold(p.ws);    // test hook: group hold - 1 publishes no size
  __syncthreads();
  const uint64_t groups = (nb + kQEncWarps - 1) / kQEncWarps;
  const uint32_t R = blockIdx.x < groups
                         ? static_cast<uint32_t>((groups - blockIdx.x + gridDim.x - 1) / gridDim.x)
                         : 0u;  // rounds of this CTA
  auto group_of = [&](uint32_t r) { return static_cast<uint64_t>(blockIdx.x) + static_cast<uint64_t>(r) * gridDim.x; };

  if (warp < kQEncWarps) {
    // ---------------- coding warps: block 16 G + warp of each group G
    auto block_of = [&](uint32_t k) { return group_of(k >> 3) * kQEncWarps + warp; };  // run k's block
    const uint32_t nruns = 8 * R;
    auto load_k = [&](uint32_t k, uint32_t* valid) -> uint4 {
      if (k >= nruns) {
        *valid = 0;
        return make_uint4(0u, 0u, 0u, 0u);
      }
      return zq_load_run(p.in, p.n, block_of(k), lane, k & 7u, valid);  // no symbols past n
    };
    uint32_t* lb = &S.lanebuf[warp][lane * kQLaneStride];
    uint32_t* packed = S.packed[warp];
    // Four runs are loaded ahead (64 bytes per lane in flight), across rounds.
    uint32_t v0, v1, v2, v3;
    uint4 q0 = load_k(0, &v0), q1 = load_k(1, &v1), q2 = load_k(2, &v2), q3 = load_k(3, &v3);
    bool prev_has = false;  // the block packed in the previous round, waiting for its offset ...
    uint32_t prev_T = 0;    // ... and its words
#pragma unroll 1
    for (uint32_t r = 0; r <= R; r++) {
      const bool has = r < R && block_of(8 * r) < nb;
      uint32_t wc = 0, T = 0;
      if (r < R) {
        unsigned long long acc = 0;  // codes most significant bit first; nacc bits used
        uint32_t nacc = 0;
#pragma unroll 1
        for (uint32_t j = 0; j < 8; j++) {
          // the run's 16 lookups first, all in flight at once (the word stores
          // below would otherwise keep each lookup behind the previous store)
          uint32_t e[16];
          zq_lookup_run(S.lut, q0, v0, e);
          q0 = q1, v0 = v1, q1 = q2, v1 = v2, q2 = q3, v2 = v3;
          q3 = load_k(8 * r + j + 4, &v3);
          // two codes at a time (at most 22 bits): one insertion and at most
          // one full word per pair
#pragma unroll
          for (uint32_t t = 0; t < 16; t += 2) {
            const uint32_t l1 = e[t + 1] >> 16;  // 0 past n
            const uint32_t len = (e[t] >> 16) + l1;
            const uint32_t code = ((e[t] & 0xFFFFu) << l1) | (e[t + 1] & 0xFFFFu);
            acc |= static_cast<unsigned long long>(code) << ((64 - nacc - len) & 63);
            nacc += len;
            if (nacc >= 32) {
              lb[wc++] = static_cast<uint32_t>(acc >> 32);
              acc <<= 32;
              nacc -= 32;
            }
          }
        }
        if (nacc > 0) lb[wc++] = static_cast<uint32_t>(acc >> 32);
        T = has ? 8 + warp_sum(wc) : 0u;
        if (lane == 0) S.words[r & 1][warp] = T;
      }
      __syncthreads();  // round r's sizes are in; round r - 1's offsets are posted
      if (prev_has) {
        const uint64_t off = S.offs[(r - 1) & 1][warp];
        if (off + prev_T <= p.out_words) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(payload) + off;
          for (uint32_t i = lane; i < prev_T; i += 32) dst[i] = packed[i];
        } else if (lane == 0) {
          set_status(p.status, ZC_ERR_OUT_OF_ROOM);
        }
      }
      __syncwarp();
      if (has) {  // pack: lane counts, then the lanes' words in lane order
        const uint32_t inc = warp_inclusive_scan(wc);
        const uint32_t pre = inc - wc;
        reinterpret_cast<uint8_t*>(packed)[lane] = static_cast<uint8_t>(wc);
        for (uint32_t i = 0; i < wc; i++) packed[8 + pre + i] = lb[i];
      }
      __syncwarp();
      prev_has = has;
      prev_T = T;
    }
  } else {
    // ---------------- scan warp: each group's first word offset
    const uint32_t arrival = lane == 0 ? scan_arrive(p.ws, epoch) : kNoArrival;
    uint64_t prev_incl = 0;  // offset after this CTA's previous group
#pragma unroll 1
    for (uint32_t r = 0; r <= R; r++) {
      __syncthreads();  // round r's sizes are in
      if (r == R) break;
      const uint64_t G = group_of(r);
      const uint32_t w = lane < kQEncWarps ? S.words[r & 1][lane] : 0u;
      const uint32_t inc = warp_inclusive_scan(w);
      const uint32_t total = __shfl_sync(kFull, inc, 31);
      if (lane == 0 && static_cast<uint64_t>(hold) != G + 1)
        st_relaxed(&p.flags[G].agg, (static_cast<unsigned long long>(epoch) << 32) | total);
      bool timed_out;
      const uint32_t lo = r > 0 ? static_cast<uint32_t>(group_of(r - 1)) + 1u : 0u;
      const uint64_t prefix = (r > 0 ? prev_incl : 0) +
                              window_sum(p.flags, lo, static_cast<uint32_t>(G), epoch, p.status, &timed_out);
      if (lane < kQEncWarps) {
        const uint64_t off = prefix + inc - w;
        S.offs[r & 1][lane] = static_cast<uint32_t>(off);
        if (G * kQEncWarps + lane < nb) table[G * kQEncWarps + lane] = static_cast<uint32_t>(off);
      }
      prev_incl = prefix + total;
      if (G + 1 == groups) {  // the last group: payload words and the offset table's padding
        if (lane == 0) *reinterpret_cast<unsigned long long*>(p.out + 24) = prev_incl;
        for (uint64_t o = kQHeader + 4 * nb + 4 * lane; o < kQHeader + tbl; o += 128)
          *reinterpret_cast<uint32_t*>(p.out + o) = 0u;
      }
      __syncwarp();
    }
    scan_exit(p.ws, p.flags, epoch, static_cast<uint32_t>(groups), arrival);
  }
}

// ---------------------------------------------------------------- decoder
struct QDecParams {
  const uint8_t* in;
  uint64_t in_bytes;
  uint64_t n;
  uint8_t* out;
  int32_t* status;
};

// A warp's block buffer: the block lands at word (offset mod 4) of its row (a
// bulk copy starts on a 16-byte boundary).  + 52 words: up to 3 words of that
// shift, and a lane's window start advances at most 44 times (1408 bits) plus
// 2 words of look-ahead, from at most word 1416.
constexpr uint32_t kQDecRowWords = kQBlockWordsMax + 52;  // 1468: rows of 5872 bytes, 16-byte aligned

struct QDecShared {
  uint32_t words[kQDecWarps][kQDecRowWords];
  uint64_t bar[kQDecWarps];  // one mbarrier per warp: its block's bulk copy
  uint16_t lut[2048];  // next 11 bits -> (symbol << 8) | code length; bit 7 set: no valid code
  uint32_t seen[8];    // byte values met in the rank table
  uint32_t start[9];   // first rank of each region
  int bad;
};
// A table entry's low byte is the code length (bits 0-3) with the "no valid
// code" flag in bit 7, so whole entries can be added to a bit position: bits
// 0-5 of the sum stay exact while positions plus lengths stay below 64.
constexpr uint16_t kQBadCode = 0x80u | 11u;
constexpr uint32_t kQBadFlag = 0x80u;

__global__ void __launch_bounds__(kQDecWarps * 32) zq_decode_kernel(const __grid_constant__ QDecParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_begin();
  QDecShared& S = *reinterpret_cast<QDecShared*>(smem_raw);
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint64_t nb = zq_blocks(p.n);
  const uint64_t tbl = zq_table_bytes(nb);
  // header checks (every CTA reaches the same decision) and the 11-bit table
  if (threadIdx.x < 8) S.seen[threadIdx.x] = 0u;
  if (lane == 0) {
    mbar_init(&S.bar[warp], 1);
    fence_mbar_init();
  }
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
      uint32_t cap = 0;
      S.start[0] = 0;
      for (int r = 0; r < 8; r++) {
        const uint32_t w = __ldg(p.in + 64 + r);
        if (w > 8) err = ZC_ERR_BAD_HEADER;
        cap += 1u << (w & 15u);
        S.start[r + 1] = cap;
      }
      if (cap < 256 || kQHeader + tbl + 4 * words > p.in_bytes) err = ZC_ERR_BAD_HEADER;
    }
    S.bad = err;
  }
  __syncthreads();
  if (S.bad == 0 && threadIdx.x < 256) {  // the rank table is a permutation: every byte value once
    const uint32_t v = __ldg(p.in + 128 + threadIdx.x);
    atomicOr(&S.seen[v >> 5], 1u << (v & 31u));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (S.bad == 0)
      for (int i = 0; i < 8; i++)
        if (S.seen[i] != 0xFFFFFFFFu) S.bad = ZC_ERR_BAD_HEADER;
    if (S.bad) set_status(p.status, S.bad);
  }
  __syncthreads();
  if (S.bad) return;
  for (uint32_t q = threadIdx.x; q < 2048; q += blockDim.x) {
    const uint32_t r = q >> 8;
    const uint32_t w = __ldg(p.in + 64 + r);
    const uint32_t rank = S.start[r] + (w == 0 ? 0u : ((q & 0xFFu) >> (8 - w)));
    S.lut[q] = rank > 255 ? kQBadCode : static_cast<uint16_t>((uint32_t(__ldg(p.in + 128 + rank)) << 8) | (3 + w));
  }
  __syncthreads();
  const uint64_t words = static_cast<uint64_t>(reinterpret_cast<const uint32_t*>(p.in)[6]) |
                         (static_cast<uint64_t>(reinterpret_cast<const uint32_t*>(p.in)[7]) << 32);
  const uint32_t* table = reinterpret_cast<const uint32_t*>(p.in + kQHeader);
  const uint32_t* payload = reinterpret_cast<const uint32_t*>(p.in + kQHeader + tbl);
  uint32_t* const row = S.words[warp];
  // The payload starts on 16 bytes (the stream does, and the header and the
  // offset table are whole 16-byte units); a block whose copy, rounded up to
  // 16 bytes, would reach past the stream's end is loaded with plain loads.
  const uint8_t* in_end = p.in + p.in_bytes;
  const uint64_t total_warps = static_cast<uint64_t>(gridDim.x) * kQDecWarps;
  uint64_t next_off = 0, next_end = 0;  // offsets of the warp's next block, loaded one block ahead
  auto load_offsets = [&](uint64_t bb) {
    next_off = __ldg(table + bb);
    next_end = bb + 1 < nb ? static_cast<uint64_t>(__ldg(table + bb + 1)) : words;
  };
  const uint64_t b_first = static_cast<uint64_t>(blockIdx.x) * kQDecWarps + warp;
  if (b_first < nb) load_offsets(b_first);
  uint32_t phase = 0;
  for (uint64_t b = b_first; b < nb; b += total_warps) {
    const uint64_t off = next_off, end = next_end;
    if (b + total_warps < nb) load_offsets(b + total_warps);
    if (off + 8 > end || end > words || end - off > kQBlockWordsMax) {
      if (lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
      continue;
    }
    const uint32_t T = static_cast<uint32_t>(end - off);
    const uint64_t c0 = off & ~3ull, c1 = (end + 3) & ~3ull;  // the copy: whole 16-byte units
    const uint32_t* wbuf = row;
    if (reinterpret_cast<const uint8_t*>(payload + c1) <= in_end) {
      wbuf = row + (off & 3u);
      if (lane == 0) {
        fence_proxy_async();  // the previous block's reads of the row come first
        const uint32_t bytes = static_cast<uint32_t>(4 * (c1 - c0));
        mbar_arrive_expect_tx(&S.bar[warp], bytes);
        tma_load_1d(row, payload + c0, bytes, &S.bar[warp]);
      }
      mbar_wait_bounded(&S.bar[warp], phase, p.status);
      phase ^= 1u;
    } else {
      for (uint32_t k0 = 0; k0 < T; k0 += 8 * 32) {  // 8 independent loads in flight per lane
        uint32_t t[8];
#pragma unroll
        for (uint32_t u = 0; u < 8; u++) {
          const uint32_t k = k0 + 32 * u + lane;
          t[u] = k < T ? __ldg(payload + off + k) : 0u;
        }
#pragma unroll
        for (uint32_t u = 0; u < 8; u++) {
          const uint32_t k = k0 + 32 * u + lane;
          if (k < T) row[k] = t[u];
        }
      }
    }
    __syncwarp();
    const uint32_t wc = reinterpret_cast<const uint8_t*>(wbuf)[lane];
    const uint32_t inc = warp_inclusive_scan(wc);
    bool ok = 8 + __shfl_sync(kFull, inc, 31) == T;
    const uint32_t first = ok ? 8 + inc - wc : 8u;  // lane counts that do not add up: read anything in range
    // window: bits [pos, pos + 32) of the lane's stream are the funnel shift
    // of (w0, w1); w2 is the word after them, loaded ahead.  The window may run
    // past the lane's words into the next lane's (or the slack words): those
    // bits only ever fill the unused tail of the last peek.
    uint32_t idx = first + 2;
    uint32_t w0 = wbuf[first], w1 = wbuf[first + 1], w2 = wbuf[idx];
    uint32_t pos = 0, badcode = 0;
    const uint64_t base = b * kQBlock;
    auto decode_one = [&]() -> uint32_t {  // returns the lookup entry, advances the window
      const uint32_t e = S.lut[__funnelshift_l(w1, w0, pos) >> 21];
      badcode |= e;
      pos += e & 15u;
      const bool adv = pos >= 32;
      pos &= 31u;
      w0 = adv ? w1 : w0;
      w1 = adv ? w2 : w1;
      idx += adv ? 1u : 0u;
      w2 = wbuf[idx];
      return e;
    };
    // Two symbols per refill: a code is at most 11 bits, so after the first
    // symbol the second starts at most 42 bits into (w0, w1, w2) and ends
    // inside w1; one advance (at most one word) follows the pair.
    // Positions add whole entries (pos + two lengths <= 53 < 64); the funnel
    // shifts take the shift amount modulo 32.
    auto decode_two = [&](uint32_t& ea, uint32_t& eb) {
      ea = S.lut[__funnelshift_l(w1, w0, pos) >> 21];
      const uint32_t p2 = pos + ea;
      const bool hi = (p2 & 32u) != 0;
      eb = S.lut[__funnelshift_l(hi ? w2 : w1, hi ? w1 : w0, p2) >> 21];
      badcode |= ea | eb;
      const uint32_t p3 = p2 + eb;
      const bool adv = (p3 & 32u) != 0;
      pos = p3 & 31u;
      w0 = adv ? w1 : w0;
      w1 = adv ? w2 : w1;
      idx += adv ? 1u : 0u;
      if (adv) w2 = wbuf[idx];
    };
#pragma unroll 1
    for (uint32_t j = 0; j < 8; j++) {
      const uint64_t i0 = base + zq_run_offset(lane, j);
      const uint32_t valid = i0 >= p.n ? 0u : (p.n - i0 >= 16 ? 16u : static_cast<uint32_t>(p.n - i0));
      if (valid == 16) {
        uint32_t o[4];
#pragma unroll
        for (uint32_t q = 0; q < 4; q++) {
          uint32_t e0, e1, e2, e3;
          decode_two(e0, e1);
          decode_two(e2, e3);
          o[q] = __byte_perm(__byte_perm(e0, e1, 0x0051), __byte_perm(e2, e3, 0x0051), 0x5410);
        }
        *reinterpret_cast<uint4*>(p.out + i0) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        for (uint32_t t = 0; t < valid; t++) p.out[i0 + t] = static_cast<uint8_t>(decode_one() >> 8);
      }
    }
    // words consumed: the window started at word `first`, advanced idx - first - 2 times
    const uint32_t bits_used = 32u * (idx - first - 2u) + pos;
    ok &= (badcode & kQBadFlag) == 0;
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
  cudaError_t err =
      prepare_kernel(prep, reinterpret_cast<const void*>(zq_encode_kernel), kQEncThreads, smem, dev, &per_sm);
  if (err != cudaSuccess) return err;
  const uint32_t groups = static_cast<uint32_t>((nb + kQEncWarps - 1) / kQEncWarps);
  uint32_t ctas = groups;  // one group per CTA and round, at most all resident CTAs
  const uint32_t cap = static_cast<uint32_t>(dev.sm_count) * static_cast<uint32_t>(per_sm);
  if (ctas > cap) ctas = cap;
  if (ctas == 0) ctas = 1;
  void* args[] = {&p};
  return launch_kernel(reinterpret_cast<const void*>(zq_encode_kernel), dim3(ctas), dim3(kQEncThreads), smem,
                       stream, args, true);
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
  void* args[] = {&p};
  return launch_kernel(reinterpret_cast<const void*>(zq_decode_kernel), dim3(static_cast<unsigned>(ctas)),
                       dim3(kQDecWarps * 32), smem, stream, args, false);
}

}  // namespace zc
