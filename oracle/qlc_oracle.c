/*
 * qlc_oracle.c -- plain, slow, single-threaded CPU oracle for Quad Length
 * Codes (QLC) on FP8 (e4m3) bytes.
 *
 * TEST INFRASTRUCTURE ONLY, like zc_oracle.c: only the test-suite, the smoke
 * check and the benchmark's CPU legs load it (through oracle/__init__.py); it
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Source, cited as [QLC §x]: the ijyty.com article on Quad Length Codes
 * (QLC) for lossless compression of e4m3 tensors in LLM training --
 *   §3.1  a 3-bit prefix splits the 256-symbol space into 8 regions, each
 *         coded on its own; only four code lengths (6, 7, 8 and 11 bits); a
 *         256-entry lookup table instead of a code tree;
 *   §3.2  the static table for FFN1 activations: symbols ranked by frequency,
 *         the prefix says how many bits follow (3, 4, 5 or 8), the last
 *         region covers the rarest ranks up to 255;
 *   §3.3  dynamic variants: a region of 2 symbols with 4-bit codes for the
 *         most frequent ones, wider middle regions, one table per layer;
 *   §4.1  encoder: symbols sorted by frequency beforehand, one table lookup
 *         per symbol at run time;
 *   §4.2  decoder: read the 3-bit prefix, take that region's number of bits,
 *         map the rank back through the table;
 *   §6.1  NaN / Inf need room in the code space.
 *
 * Readings taken where the article is silent or garbled (each one is listed
 * again, with the reason, in the design notes):
 *   Q1  table = 8 region widths w[r] (bits after the prefix) and a rank ->
 *       symbol permutation sym[256]; region r holds ranks [s_r, s_r + 2^w[r]),
 *       s_0 = 0, s_(r+1) = s_r + 2^w[r]; valid when sum 2^w[r] >= 256 and
 *       every w[r] <= 8.  Rank k in region r is coded as r (3 bits) followed by
 *       k - s_r (w[r] bits), most significant bit first.
 *   Q2  default widths {3,3,3,3,3,4,5,8}: five regions of 8 ranks (6-bit
 *       codes), one of 16 (7-bit), one of 32 (8-bit), the rest, ranks 88-255,
 *       11-bit -- the four code lengths of the static table; symbols ranked
 *       by (count desc, symbol asc).  Every byte value, NaN and Inf
 *       included, is an ordinary symbol with a code (section 6.1's room).
 *   Q3  stream "ZQ1": 384-byte header (magic "ZQB1", version 1, n, 4096,
 *       nblocks, payload words, widths at 64, the 256-byte rank table at
 *       128); u32 word offset of each block in the payload (zero-padded to a
 *       multiple of 128 bytes); the payload.  Block b (symbols 4096 b ...)
 *       is 8 words of lane word counts (byte l = words of lane l) followed
 *       by the words of lanes 0..31.  The block's 4096 symbols form 256 runs
 *       of 16; lane l codes runs l, l + 32, ..., l + 224 in that order (the
 *       symbols below n) into little-endian u32 words, first code at bit 31 of
 *       its first word, the last word zero-padded.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define Q_BLOCK 4096u
#define Q_LANES 32u
#define Q_HEADER 384u

enum { Q_OK = 0, Q_ERR_ARG = 1, Q_ERR_TABLE = 2, Q_ERR_HEADER = 3, Q_ERR_CORRUPT = 4, Q_ERR_SIZE = 5, Q_ERR_ROOM = 6 };

static void q_put_u32(uint8_t *p, uint32_t v) {
  for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static void q_put_u64(uint8_t *p, uint64_t v) {
  for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t q_get_u32(const uint8_t *p) {
  uint32_t v = 0;
  for (int i = 3; i >= 0; i--) v = (v << 8) | p[i];
  return v;
}
static uint64_t q_get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; i--) v = (v << 8) | p[i];
  return v;
}

uint64_t zqo_num_blocks(uint64_t n) { return (n + Q_BLOCK - 1) / Q_BLOCK; }

/* the j-th symbol (0..127) of lane l within its block: run l + 32 (j / 16), position j % 16 */
static uint64_t q_lane_symbol(unsigned l, unsigned j) { return 16u * (l + 32u * (j / 16u)) + j % 16u; }
static uint64_t q_table_bytes(uint64_t nblocks) { return (4 * nblocks + 127) / 128 * 128; }

/* ---- the table, readings Q1 and Q2 --------------------------------------- */
int zqo_table_is_valid(const uint8_t w[8], const uint8_t sym[256]) {
  uint32_t cap = 0;
  for (int r = 0; r < 8; r++) {
    if (w[r] > 8) return 0;
    cap += 1u << w[r];
  }
  if (cap < 256) return 0;
  int seen[256] = {0};
  for (int k = 0; k < 256; k++) {
    if (seen[sym[k]]) return 0;
    seen[sym[k]] = 1;
  }
  return 1;
}

/* rank -> symbol ordered by (count desc, symbol asc) */
void zqo_table_from_histogram(const uint64_t hist[256], uint8_t sym[256]) {
  int taken[256] = {0};
  for (int k = 0; k < 256; k++) {
    int best = -1;
    for (int s = 0; s < 256; s++)
      if (!taken[s] && (best < 0 || hist[s] > hist[best])) best = s;
    taken[best] = 1;
    sym[k] = (uint8_t)best;
  }
}

/* region of a rank and its start */
static int q_region(const uint8_t w[8], unsigned rank, unsigned *start) {
  unsigned s = 0;
  for (int r = 0; r < 8; r++) {
    unsigned cap = 1u << w[r];
    if (rank < s + cap) {
      *start = s;
      return r;
    }
    s += cap;
  }
  return -1; /* cannot happen for a valid table */
}

/* code length in bits of symbol `symbol` */
int zqo_code_length(const uint8_t w[8], const uint8_t sym[256], unsigned symbol) {
  for (unsigned k = 0; k < 256; k++)
    if (sym[k] == symbol) {
      unsigned start = 0;
      int r = q_region(w, k, &start);
      return 3 + w[r];
    }
  return -1;
}

/* ---- a most-significant-bit-first bit writer over u32 words --------------- */
typedef struct {
  uint32_t *words;
  uint64_t cap;  /* words available */
  uint64_t nbits;
} BitWriter;

static int bw_put(BitWriter *bw, uint32_t value, unsigned bits) {
  for (int i = (int)bits - 1; i >= 0; i--) {
    uint64_t word = bw->nbits / 32;
    if (word >= bw->cap) return 0;
    if (bw->nbits % 32 == 0) bw->words[word] = 0;
    if ((value >> i) & 1u) bw->words[word] |= 1u << (31 - bw->nbits % 32);
    bw->nbits++;
  }
  return 1;
}

/* ---- encode, reading Q3 ---------------------------------------------------- */
uint64_t zqo_max_bytes(uint64_t n) {
  uint64_t nb = zqo_num_blocks(n);
  return Q_HEADER + q_table_bytes(nb) + nb * (uint64_t)(8 + 32 * 44) * 4;
}

int zqo_compress(const uint8_t *x, uint64_t n, const uint8_t w[8], const uint8_t sym[256], uint8_t *out,
                 uint64_t out_cap, uint64_t *out_bytes) {
  if (n >= ((uint64_t)1 << 32)) return Q_ERR_ARG;
  if (!zqo_table_is_valid(w, sym)) return Q_ERR_TABLE;
  uint64_t nb = zqo_num_blocks(n), tb = q_table_bytes(nb);
  if (out_cap < Q_HEADER + tb) return Q_ERR_ROOM;
  memset(out, 0, Q_HEADER + tb);
  unsigned rank_of[256];
  for (unsigned k = 0; k < 256; k++) rank_of[sym[k]] = k;
  uint8_t *payload = out + Q_HEADER + tb;
  uint64_t room_words = (out_cap - Q_HEADER - tb) / 4;
  uint64_t off = 0; /* words so far */
  uint32_t lane_words[Q_LANES][44];
  for (uint64_t b = 0; b < nb; b++) {
    q_put_u32(out + Q_HEADER + 4 * b, (uint32_t)off);
    uint32_t count[Q_LANES];
    for (unsigned l = 0; l < Q_LANES; l++) {
      BitWriter bw = {lane_words[l], 44, 0};
      for (unsigned j = 0; j < Q_BLOCK / Q_LANES; j++) {
        uint64_t i = b * Q_BLOCK + q_lane_symbol(l, j);
        if (i >= n) break;
        unsigned k = rank_of[x[i]], start = 0;
        int r = q_region(w, k, &start);
        if (!bw_put(&bw, (uint32_t)r, 3) || !bw_put(&bw, k - start, w[r])) return Q_ERR_ARG;
      }
      count[l] = (uint32_t)((bw.nbits + 31) / 32);
    }
    uint64_t total = 8;
    for (unsigned l = 0; l < Q_LANES; l++) total += count[l];
    if (off + total > room_words) return Q_ERR_ROOM;
    uint8_t *blk = payload + 4 * off;
    for (unsigned l = 0; l < Q_LANES; l++) blk[l] = (uint8_t)count[l];
    uint64_t pos = 8;
    for (unsigned l = 0; l < Q_LANES; l++)
      for (uint32_t i = 0; i < count[l]; i++, pos++) q_put_u32(blk + 4 * pos, lane_words[l][i]);
    off += total;
  }
  q_put_u32(out + 0, 0x3142515Au); /* bytes 'Z','Q','B','1' */
  out[4] = 1;                       /* version (u16), flags 0 */
  q_put_u64(out + 8, n);
  q_put_u32(out + 16, Q_BLOCK);
  q_put_u32(out + 20, (uint32_t)nb);
  q_put_u64(out + 24, off);
  memcpy(out + 64, w, 8);
  memcpy(out + 128, sym, 256);
  *out_bytes = Q_HEADER + tb + 4 * off;
  return Q_OK;
}

/* ---- decode: the inverse, bit for bit -------------------------------------- */
int zqo_decompress(const uint8_t *in, uint64_t in_bytes, uint64_t n, uint8_t *x) {
  if (in_bytes < Q_HEADER || q_get_u32(in) != 0x3142515Au || in[4] != 1 || in[5] != 0 || in[6] != 0 ||
      in[7] != 0 || q_get_u32(in + 16) != Q_BLOCK)
    return Q_ERR_HEADER;
  if (q_get_u64(in + 8) != n) return Q_ERR_SIZE;
  uint64_t nb = zqo_num_blocks(n), tb = q_table_bytes(nb);
  if (q_get_u32(in + 20) != nb) return Q_ERR_HEADER;
  const uint8_t *w = in + 64, *sym = in + 128;
  if (!zqo_table_is_valid(w, sym)) return Q_ERR_HEADER;
  uint64_t words = q_get_u64(in + 24);
  if (Q_HEADER + tb + 4 * words > in_bytes) return Q_ERR_HEADER;
  const uint8_t *payload = in + Q_HEADER + tb;
  unsigned start_of[8], s = 0;
  for (int r = 0; r < 8; r++) {
    start_of[r] = s;
    s += 1u << w[r];
  }
  for (uint64_t b = 0; b < nb; b++) {
    uint64_t off = q_get_u32(in + Q_HEADER + 4 * b);
    uint64_t end = b + 1 < nb ? q_get_u32(in + Q_HEADER + 4 * (b + 1)) : words;
    if (off + 8 > end || end > words) return Q_ERR_CORRUPT;
    const uint8_t *blk = payload + 4 * off;
    uint64_t pos = 8;
    for (unsigned l = 0; l < Q_LANES; l++) {
      uint64_t first = pos, limit = pos + blk[l];
      if (limit > end - off) return Q_ERR_CORRUPT;
      uint64_t bit = 0; /* bits read from this lane's words */
      for (unsigned j = 0; j < Q_BLOCK / Q_LANES; j++) {
        uint64_t i = b * Q_BLOCK + q_lane_symbol(l, j);
        if (i >= n) break;
        uint32_t v[2] = {0, 0};
        unsigned need[2] = {3, 0};
        for (int part = 0; part < 2; part++) {
          if (part == 1) need[1] = w[v[0]];
          for (unsigned t = 0; t < need[part]; t++, bit++) {
            uint64_t word = first + bit / 32;
            if (word >= limit) return Q_ERR_CORRUPT;
            uint32_t wv = q_get_u32(blk + 4 * word);
            v[part] = (v[part] << 1) | ((wv >> (31 - bit % 32)) & 1u);
          }
        }
        unsigned rank = start_of[v[0]] + v[1];
        if (rank > 255) return Q_ERR_CORRUPT;
        x[i] = sym[rank];
      }
      if ((bit + 31) / 32 != blk[l]) return Q_ERR_CORRUPT;
      pos = limit;
    }
    if (off + pos != end) return Q_ERR_CORRUPT;
  }
  return Q_OK;
}
