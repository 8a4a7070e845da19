/*
 * zc_oracle.c -- plain, slow, single-threaded CPU oracle for lossless BF16
 * exponent coding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg load it (through oracle/__init__.py).  It shares no code,
 * header, table or constant generator with the CUDA library: every constant
 * below is written out again here from the format definition.
 *
 * Sources (cited as [ZipCCL §x] = the gist.science technical summary of
 * "ZipCCL: Efficient Lossless Data Compression of Communication Collectives
 * for Accelerating LLM Training", Lin, Pan, Fan, Shi, Chu, 2026):
 *   [ZipCCL §2.A]  Gaussian tensors; the 7 most frequent exponents cover >97%;
 *                  the remap table is derived from the layer's sigma instead
 *                  of an online histogram or sort.
 *   [ZipCCL §2.B]  split into sign-mantissa and exponent bits; an exponent in
 *                  the top 7 maps to a 3-bit code 001..111; any other exponent
 *                  gets code 000 and its full 8-bit value goes to a separate
 *                  "zero-point" (escape) array; 16 -> 11 bits per value.
 *   [ZipCCL §2.C]  the 3-bit codes are kept as three separate 1-bit arrays in
 *                  a column-major layout; blocks padded to 128-byte bounds.
 *   [ZipCCL §2.D]  reduce-scatter as zipped all-to-all + local reduction;
 *                  MoE all-to-all split into a fixed-size (static) part and a
 *                  variable-size (dynamic) part.
 *
 * Readings taken where the pages are silent (each one is listed again, with
 * the reason, in the design notes):
 *   R1  code numbering: codebook entry k (rank order, most probable first)
 *       <-> code k+1.
 *   R2  sign-mantissa byte = sign << 7 | 7-bit mantissa.
 *   R3  format "ZC1": 4096-element tiles of four 1024-element blocks; a block
 *       is [1024 sign-mantissa bytes][plane0 128 B][plane1 128 B][plane2 128 B];
 *       plane byte q, bit j holds the code bit of block element
 *       256*(q%4) + 8*(q/4) + j (a 4 x 32 byte matrix stored column-major).
 *   R4  escapes of a tile: blocks in order, inside a block in ascending
 *       plane-bit position (q, j); u32 exclusive offsets per tile.
 *   R5  sigma closed form: p_e = P(exponent field of RNE_bf16(X) == e),
 *       X ~ N(0, sigma^2), edges adjusted for round-to-nearest-even; top 7 by
 *       (p desc, e asc).
 *   R6  histogram top 7: exact count of all n exponent fields, sorted
 *       (count desc, e asc); zero-count exponents fill up, smallest first.
 *   R7  local reduction = sum (not mean), fp32, rank order 0..P-1, IEEE
 *       round-to-nearest with subnormals kept, then RNE to bf16; a NaN sum
 *       becomes 0x7FC0.
 *   R12 raw bypass ([CCCL §3.3] tiny tensors are not worth compressing;
 *       [CCCL §5.2] a ratio near or above 1 means fall back to sending the
 *       data uncompressed): header flags bit 0 marks a RAW stream.  It holds
 *       the 2n little-endian bytes of the n values in order: the first
 *       min(2n, 5632 ntiles) fill the tile region (the rest of it is zero),
 *       the remaining 2n - 5632 ntiles bytes (the "spill", if any) form the
 *       escape stream, n_esc = spill, and the offset table is zero.  The main
 *       stream keeps its size.  The adaptive encoder stores RAW exactly when
 *       the coded form's escape count exceeds the spill, i.e. when RAW is
 *       strictly smaller in total.
 *
 * Compile: plain C11, -O2 -ffp-contract=off, no -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define O_TILE 4096u
#define O_BLOCK 1024u
#define O_BLOCKS_PER_TILE 4u
#define O_BLOCK_BYTES 1408u /* 1024 + 3 * 128 */
#define O_TILE_BYTES 5632u  /* 4 * 1408 */
#define O_HEADER 128u

enum {
  O_OK = 0,
  O_ERR_ARG = 1,
  O_ERR_CODEBOOK = 2,
  O_ERR_ESCAPE_OVERFLOW = 3,
  O_ERR_HEADER = 4,
  O_ERR_CORRUPT = 5,
  O_ERR_SIZE = 6
};

/* ---- little-endian field access ---------------------------------------- */
static void put_u16(uint8_t *p, uint16_t v) {
  p[0] = (uint8_t)v;
  p[1] = (uint8_t)(v >> 8);
}
static void put_u32(uint8_t *p, uint32_t v) {
  for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t *p, uint64_t v) {
  for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t *p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; i++) v |= (uint32_t)p[i] << (8 * i);
  return v;
}
static uint64_t get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i);
  return v;
}
static uint16_t get_u16(const uint8_t *p) {
  return (uint16_t)(p[0] | (p[1] << 8));
}

/* ---- sizes (format R3) -------------------------------------------------- */
uint64_t zo_num_tiles(uint64_t n) { return (n + O_TILE - 1) / O_TILE; }

static uint64_t table_bytes(uint64_t ntiles) {
  uint64_t raw = 4 * ntiles;
  return (raw + 127) / 128 * 128;
}

uint64_t zo_main_bytes(uint64_t n) {
  uint64_t t = zo_num_tiles(n);
  return O_HEADER + table_bytes(t) + (uint64_t)O_TILE_BYTES * t;
}

/* ---- field split [ZipCCL §2.B], reading R2 ------------------------------ */
static unsigned exponent_of(uint16_t u) { return (u >> 7) & 0xFFu; }
static unsigned sign_mantissa_of(uint16_t u) {
  unsigned sign = (u >> 15) & 1u;
  unsigned mant = u & 0x7Fu;
  return (sign << 7) | mant;
}
static uint16_t join_fields(unsigned sm, unsigned e) {
  unsigned sign = (sm >> 7) & 1u;
  unsigned mant = sm & 0x7Fu;
  return (uint16_t)((sign << 15) | (e << 7) | mant);
}

/* Block-local element index held by plane byte q, bit j (reading R3). */
static unsigned element_of_plane_bit(unsigned q, unsigned j) {
  return 256u * (q % 4u) + 8u * (q / 4u) + j;
}

static int codebook_is_valid(const uint8_t cb[7]) {
  for (int a = 0; a < 7; a++)
    for (int b = a + 1; b < 7; b++)
      if (cb[a] == cb[b]) return 0;
  return 1;
}

/* Code of exponent e under codebook cb (reading R1): k+1 if cb[k]==e, else 0. */
static unsigned code_of(const uint8_t cb[7], unsigned e) {
  for (unsigned k = 0; k < 7; k++)
    if (cb[k] == e) return k + 1;
  return 0;
}

/* ---- sigma closed form [ZipCCL §2.A], reading R5 -------------------------
 * The pages derive the top-7 exponent set from the layer's sigma without
 * printing the formula.  For X ~ N(0, sigma^2), the probability that the
 * bf16 value RNE(X) has exponent field e is P(lo_e <= |X| < hi_e), where the
 * binade [2^(e-127), 2^(e-126)) is widened downward by half an ulp of the
 * binade below (values that round up into it) and loses the top half ulp of
 * its own (values that round up out of it).                                */
static void binade_edges(int e, double *lo, double *hi) {
  const double top_frac = 1.0 - ldexp(1.0, -9); /* 1 - half ulp of 8-bit significand */
  if (e == 0) {
    *lo = 0.0;
    /* the subnormal spacing is 2^-133; half of it below 2^-126 rounds up */
    *hi = ldexp(1.0 - ldexp(1.0, -8), -126);
  } else if (e == 255) {
    *lo = ldexp(top_frac, 128); /* rounds to infinity */
    *hi = INFINITY;
  } else {
    *lo = (e == 1) ? ldexp(1.0 - ldexp(1.0, -8), -126) : ldexp(top_frac, e - 127);
    *hi = ldexp(top_frac, e - 126);
  }
}

/* P(lo <= |X| < hi), X ~ N(0, sigma^2) = erf(hi/(s*sqrt2)) - erf(lo/(s*sqrt2)).
 * For arguments past 1 the complementary form keeps the tail accurate.     */
double zo_exponent_probability(int e, double sigma) {
  double lo, hi;
  binade_edges(e, &lo, &hi);
  double a = lo / (sigma * sqrt(2.0));
  double b = isinf(hi) ? INFINITY : hi / (sigma * sqrt(2.0));
  if (a >= 1.0) {
    double eb = isinf(b) ? 0.0 : erfc(b);
    return erfc(a) - eb;
  }
  double eb = isinf(b) ? 1.0 : erf(b);
  return eb - erf(a);
}

int zo_codebook_from_sigma(double sigma, uint8_t cb[7], double probs_out[256]) {
  if (!(sigma > 0.0) || isinf(sigma) || isnan(sigma)) return O_ERR_ARG;
  double p[256];
  for (int e = 0; e < 256; e++) p[e] = zo_exponent_probability(e, sigma);
  if (probs_out)
    for (int e = 0; e < 256; e++) probs_out[e] = p[e];
  int taken[256] = {0};
  for (int k = 0; k < 7; k++) { /* selection by (p desc, e asc) */
    int best = -1;
    for (int e = 0; e < 256; e++) {
      if (taken[e]) continue;
      if (best < 0 || p[e] > p[best]) best = e;
    }
    taken[best] = 1;
    cb[k] = (uint8_t)best;
  }
  return O_OK;
}

/* ---- exact histogram top 7 [ZipCCL §2.A, the avoided alternative] R6 ---- */
void zo_exponent_histogram(const uint16_t *x, uint64_t n, uint64_t hist[256]) {
  for (int e = 0; e < 256; e++) hist[e] = 0;
  for (uint64_t i = 0; i < n; i++) hist[exponent_of(x[i])]++;
}

void zo_topk_from_histogram(const uint64_t hist[256], uint8_t cb[7]) {
  int taken[256] = {0};
  for (int k = 0; k < 7; k++) { /* (count desc, e asc) */
    int best = -1;
    for (int e = 0; e < 256; e++) {
      if (taken[e]) continue;
      if (best < 0 || hist[e] > hist[best]) best = e;
    }
    taken[best] = 1;
    cb[k] = (uint8_t)best;
  }
}

/* ---- encode [ZipCCL §2.B, §2.C], readings R1-R4 -------------------------- */
int zo_compress(const uint16_t *x, uint64_t n, const uint8_t cb[7], uint8_t *main_out,
                uint8_t *esc_out, uint64_t esc_capacity, uint64_t *n_esc_out) {
  if (n >= ((uint64_t)1 << 32)) return O_ERR_ARG;
  if (!codebook_is_valid(cb)) return O_ERR_CODEBOOK;
  uint64_t ntiles = zo_num_tiles(n);
  uint64_t tbl = table_bytes(ntiles);
  uint64_t mb = zo_main_bytes(n);
  memset(main_out, 0, mb);

  uint64_t n_esc = 0;
  int overflow = 0;
  for (uint64_t t = 0; t < ntiles; t++) {
    put_u32(main_out + O_HEADER + 4 * t, (uint32_t)n_esc); /* exclusive offset */
    for (unsigned b = 0; b < O_BLOCKS_PER_TILE; b++) {
      uint8_t *blk = main_out + O_HEADER + tbl + O_TILE_BYTES * t + O_BLOCK_BYTES * b;
      uint64_t base = O_TILE * t + O_BLOCK * b;
      /* sign-mantissa plane and the three code bit planes */
      for (unsigned i = 0; i < O_BLOCK; i++) {
        uint64_t idx = base + i;
        if (idx >= n) continue; /* padding: sm 0, code 0, not an escape */
        uint16_t u = x[idx];
        blk[i] = (uint8_t)sign_mantissa_of(u);
        unsigned code = code_of(cb, exponent_of(u));
        unsigned q = 4u * ((i / 8u) % 32u) + (i / 256u);
        unsigned j = i % 8u;
        for (unsigned c = 0; c < 3; c++)
          if ((code >> c) & 1u) blk[O_BLOCK + 128u * c + q] |= (uint8_t)(1u << j);
      }
      /* escapes, in ascending plane-bit position */
      for (unsigned q = 0; q < 128; q++) {
        for (unsigned j = 0; j < 8; j++) {
          uint64_t idx = base + element_of_plane_bit(q, j);
          if (idx >= n) continue;
          unsigned e = exponent_of(x[idx]);
          if (code_of(cb, e) != 0) continue;
          if (n_esc < esc_capacity)
            esc_out[n_esc] = (uint8_t)e;
          else
            overflow = 1;
          n_esc++;
        }
      }
    }
  }
  /* header */
  put_u32(main_out + 0, 0x3142435Au); /* bytes 'Z','C','B','1' */
  put_u16(main_out + 4, 1);           /* version */
  put_u16(main_out + 6, 0);           /* flags */
  put_u64(main_out + 8, n);
  put_u32(main_out + 16, O_TILE);
  put_u32(main_out + 20, (uint32_t)ntiles);
  put_u64(main_out + 24, n_esc);
  for (int k = 0; k < 7; k++) main_out[32 + k] = cb[k];
  *n_esc_out = n_esc;
  return overflow ? O_ERR_ESCAPE_OVERFLOW : O_OK;
}

/* ---- raw bypass, reading R12 ---------------------------------------------- */
/* bytes of a RAW stream that do not fit in the tile region */
uint64_t zo_raw_spill(uint64_t n) {
  uint64_t region = (uint64_t)O_TILE_BYTES * zo_num_tiles(n);
  return 2 * n > region ? 2 * n - region : 0;
}

/* byte k of the raw little-endian image of x */
static uint8_t raw_byte(const uint16_t *x, uint64_t k) {
  uint16_t u = x[k / 2];
  return (uint8_t)(k % 2 == 0 ? u & 0xFFu : u >> 8);
}

/* Encode like zo_compress, then switch to RAW when that is strictly smaller
 * (coded escapes > spill) and the spill fits in esc_capacity.  *raw_out = 1
 * for a RAW stream.  An overflowing coded form that RAW rescues is not an
 * error; when neither fits, the coded output and ESCAPE_OVERFLOW stand. */
int zo_compress_adaptive(const uint16_t *x, uint64_t n, const uint8_t cb[7], uint8_t *main_out,
                         uint8_t *esc_out, uint64_t esc_capacity, uint64_t *n_esc_out,
                         int *raw_out) {
  *raw_out = 0;
  int rc = zo_compress(x, n, cb, main_out, esc_out, esc_capacity, n_esc_out);
  if (rc != O_OK && rc != O_ERR_ESCAPE_OVERFLOW) return rc;
  uint64_t spill = zo_raw_spill(n);
  if (*n_esc_out <= spill || spill > esc_capacity) return rc;
  uint64_t ntiles = zo_num_tiles(n);
  uint64_t tbl = table_bytes(ntiles);
  uint64_t region = (uint64_t)O_TILE_BYTES * ntiles;
  uint8_t *tiles = main_out + O_HEADER + tbl;
  memset(main_out + O_HEADER, 0, tbl + region); /* offset table and tile region */
  for (uint64_t k = 0; k < 2 * n; k++) {
    if (k < region)
      tiles[k] = raw_byte(x, k);
    else
      esc_out[k - region] = raw_byte(x, k);
  }
  put_u16(main_out + 6, 1); /* flags: RAW */
  put_u64(main_out + 24, spill);
  *n_esc_out = spill;
  *raw_out = 1;
  return O_OK;
}

/* ---- decode: the inverse of zo_compress, bit for bit --------------------- */
int zo_decompress(const uint8_t *main_in, const uint8_t *esc_in, uint64_t esc_bytes, uint64_t n,
                  uint16_t *out) {
  unsigned flags = get_u16(main_in + 6);
  if (get_u32(main_in + 0) != 0x3142435Au || get_u16(main_in + 4) != 1 || flags > 1 ||
      get_u32(main_in + 16) != O_TILE)
    return O_ERR_HEADER;
  if (get_u64(main_in + 8) != n) return O_ERR_SIZE;
  uint64_t ntiles = zo_num_tiles(n);
  if (get_u32(main_in + 20) != ntiles) return O_ERR_HEADER;
  uint64_t n_esc = get_u64(main_in + 24);
  if (n_esc > esc_bytes || n_esc > n) return O_ERR_HEADER;
  uint8_t cb[7];
  for (int k = 0; k < 7; k++) cb[k] = main_in[32 + k];
  if (!codebook_is_valid(cb)) return O_ERR_HEADER;
  uint64_t tbl = table_bytes(ntiles);

  if (flags == 1) { /* RAW, reading R12: the bytes in order, tile region then escapes */
    if (n_esc != zo_raw_spill(n)) return O_ERR_HEADER;
    uint64_t region = (uint64_t)O_TILE_BYTES * ntiles;
    const uint8_t *tiles = main_in + O_HEADER + tbl;
    for (uint64_t i = 0; i < n; i++) {
      uint64_t k = 2 * i;
      uint8_t lo = k < region ? tiles[k] : esc_in[k - region];
      uint8_t hi = k + 1 < region ? tiles[k + 1] : esc_in[k + 1 - region];
      out[i] = (uint16_t)(lo | hi << 8);
    }
    return O_OK;
  }

  for (uint64_t t = 0; t < ntiles; t++) {
    uint64_t start = get_u32(main_in + O_HEADER + 4 * t);
    uint64_t end = (t + 1 < ntiles) ? get_u32(main_in + O_HEADER + 4 * (t + 1)) : n_esc;
    if (start > end || end > n_esc) return O_ERR_CORRUPT;
    uint64_t next = start;
    for (unsigned b = 0; b < O_BLOCKS_PER_TILE; b++) {
      const uint8_t *blk = main_in + O_HEADER + tbl + O_TILE_BYTES * t + O_BLOCK_BYTES * b;
      uint64_t base = O_TILE * t + O_BLOCK * b;
      for (unsigned q = 0; q < 128; q++) {
        for (unsigned j = 0; j < 8; j++) {
          unsigned i = element_of_plane_bit(q, j);
          uint64_t idx = base + i;
          if (idx >= n) continue;
          unsigned code = 0;
          for (unsigned c = 0; c < 3; c++) code |= ((blk[O_BLOCK + 128u * c + q] >> j) & 1u) << c;
          unsigned e;
          if (code != 0) {
            e = cb[code - 1];
          } else {
            if (next >= end) return O_ERR_CORRUPT;
            e = esc_in[next++];
          }
          out[idx] = join_fields(blk[i], e);
        }
      }
    }
    if (next != end) return O_ERR_CORRUPT;
  }
  return O_OK;
}

/* ---- local reduction [ZipCCL §2.D], reading R7 --------------------------- */
static float bf16_to_float(uint16_t u) {
  uint32_t bits = (uint32_t)u << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* Round-to-nearest-even from binary32 to bfloat16, from the IEEE-754
 * definition: add half an ulp minus one plus the lowest kept bit, truncate.
 * A carry out of the significand bumps the exponent, and the largest finite
 * values round to infinity as they should.  NaN becomes the quiet 0x7FC0.  */
uint16_t zo_float_to_bf16_rne(float f) {
  if (isnan(f)) return 0x7FC0u;
  uint32_t a;
  memcpy(&a, &f, sizeof a);
  uint32_t lsb = (a >> 16) & 1u;
  return (uint16_t)((a + 0x7FFFu + lsb) >> 16);
}

void zo_reduce(int P, const uint16_t *const *xs, uint64_t n, uint16_t *y) {
  for (uint64_t i = 0; i < n; i++) {
    float acc = bf16_to_float(xs[0][i]);
    for (int r = 1; r < P; r++) acc = acc + bf16_to_float(xs[r][i]);
    y[i] = zo_float_to_bf16_rne(acc);
  }
}

/* decode every shard, reduce, and (when out_cb is given) encode the result */
int zo_decompress_reduce(int P, const uint8_t *const *mains, const uint8_t *const *escs,
                         const uint64_t *esc_bytes, uint64_t n, uint16_t *y,
                         const uint8_t *out_cb, uint8_t *out_main, uint8_t *out_esc,
                         uint64_t out_esc_capacity, uint64_t *out_n_esc) {
  if (P < 1 || P > 64) return O_ERR_ARG;
  uint16_t **dec = (uint16_t **)calloc((size_t)P, sizeof(uint16_t *));
  if (!dec) return O_ERR_ARG;
  int rc = O_OK;
  for (int r = 0; r < P && rc == O_OK; r++) {
    dec[r] = (uint16_t *)malloc((size_t)(n ? n : 1) * sizeof(uint16_t));
    if (!dec[r]) {
      rc = O_ERR_ARG;
      break;
    }
    rc = zo_decompress(mains[r], escs[r], esc_bytes[r], n, dec[r]);
  }
  if (rc == O_OK) {
    zo_reduce(P, (const uint16_t *const *)dec, n, y);
    if (out_cb) rc = zo_compress(y, n, out_cb, out_main, out_esc, out_esc_capacity, out_n_esc);
  }
  for (int r = 0; r < P; r++) free(dec[r]);
  free(dec);
  return rc;
}
