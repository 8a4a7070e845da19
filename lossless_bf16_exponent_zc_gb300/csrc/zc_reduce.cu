// zc_reduce.cu -- fused local stage of a zipped reduce-scatter [ZipCCL §2.D]:
// decode P compressed shards, add them in fp32 in rank order 0..P-1, round to
// bfloat16 (nearest even), optionally re-encode the result -- one launch, no
// decoded intermediate ever touches global memory.
//
// Design on sm_103a: a persistent grid, one CTA of 19 warps per SM.
//   * 16 consumer warps in 4 teams; team t owns tile 4G + t of each group G
//     (G, G + C, ... for C CTAs) and warp b of the team owns block b of that
//     tile, keeping its 1024 fp32 partial sums in registers (32 per lane).
//     Inputs of at most two tiles per SM give each CTA one tile per round
//     instead, and the teams share its P copies: team t decodes copies t, t + 4, ... into
//     shared memory and all 16 warps add each four, in rank order, to the sums
//     of their 256 values (one warp per block and copy would leave the SM's
//     schedulers a single warp each).
//   * 2 producer warps, each serving two teams, stream the P compressed copies
//     of a team's tile through the team's 4-stage ring: one TMA bulk copy for
//     the 5632-byte tile and one for the 16-byte-aligned span holding its
//     escape bytes, both completing on the stage's full barrier; the team's
//     4 warps release the stage on its empty barrier.  Offset-table entries
//     are prefetched a round ahead, and each round's copies are planned for
//     all shards at once (one shard per lane), so issuing a copy is short.
//   * The code planes become permute selectors through one spread table kept
//     in 32 lane copies, so the data-dependent lookups never conflict.
//   * A block's escape ranks: a warp scan inside the block, and the totals of
//     the tile's earlier blocks exchanged by the team's four warps through
//     shared memory at one named barrier per copy.
//   * Each consumer decodes its block straight into its sums (one fp32 += bf16
//     add per value, the decoded half-word as the addend), rounds, stores, and
//     -- when re-encoding -- encodes its block of the result from shared memory.
//   * A RAW shard (the raw bypass: the values' own bytes) stages nothing: the
//     producer only signals the stage, and each consumer reads its block's
//     values of that shard straight from global memory.
//   * With re-encoding, 1 scan warp runs the escape scan of the output exactly
//     like the encoder: the last warp of a group publishes the group's count,
//     the scan warp adds the counts of the groups since its own previous
//     group to that group's inclusive offset, and the consumers write their
//     escapes one round later.  The cooperative launch keeps every group owner resident.
#include "zc_device.cuh"
#include "zc_internal.h"

namespace zc {

constexpr int kRedTeams = 4;
constexpr int kRedCons = kRedTeams * 4;           // consumer warps: team t, block b = warp 4t + b
constexpr int kRedProducers = 2;                    // producer warps kRedProd + q, each serving 2 teams
constexpr int kRedProd = kRedCons;
constexpr int kRedScan = kRedProd + kRedProducers;  // scan warp (re-encoding only)
constexpr int kRedThreads = (kRedScan + 1) * 32;    // 608 (at most 5 warps per scheduler: 96 registers)
constexpr int kTeamsPerProducer = kRedTeams / kRedProducers;
constexpr int kRedStages = 4;                     // stage ring per team
constexpr uint32_t kRedEscCap = 512;              // staged input escape bytes per tile copy
constexpr uint32_t kRedStageBytes = kTileBytes + kRedEscCap;
constexpr uint32_t kRedEbuf = 512;                // staged output escapes per block and round
constexpr int kRedSlots = 2;                      // rounds in flight for the output offsets
constexpr uint32_t kGroupTilesR = kRedTeams;      // tiles per escape-scan group (1 for inputs of few tiles)
constexpr int kSpreadCopies = 32;
// Shared-memory layout after 1 KB alignment.
constexpr uint32_t kRSpread = 0;                              // spread table, 32 lane copies (32 KB)
constexpr uint32_t kRLut = kRSpread + 1024 * kSpreadCopies;  // encoder LUT of the output codebook, 1 KB aligned
constexpr uint32_t kRShard = kRLut + 1024;                    // per-shard tables, 64 x 16 B
constexpr uint32_t kRRound = kRShard + 1024;                  // round bookkeeping (<= 512 B)
constexpr uint32_t kRFlag = kRRound + 512;                    // validity flags, then the RAW shard mask (u64)
constexpr uint32_t kRBars = kRFlag + 16;                      // full / empty barriers, 2 x 4 teams x 4 stages
constexpr uint32_t kRMeta = kRBars + 2 * kRedTeams * kRedStages * 8;  // stage metadata
constexpr uint32_t kRTot = kRMeta + kRedTeams * kRedStages * 16;      // block escape totals, 2 x 4 per team
constexpr uint32_t kRScratch = (kRTot + kRedTeams * 2 * 16 + 127) / 128 * 128;  // per-consumer exponent scratch, 1 KB each
constexpr uint32_t kREbuf = kRScratch + kRedCons * 1024;
constexpr uint32_t kRYtile = kREbuf + kRedCons * kRedSlots * kRedEbuf;  // per-team rounded tile, 8 KB
constexpr uint32_t kRStage = kRYtile + kRedTeams * 8192;
constexpr uint32_t kRedSmem = 1024 + kRStage + kRedTeams * kRedStages * kRedStageBytes;
static_assert(kRedSmem + 1024 <= 232448, "shared memory budget");

struct RedParams {
  Shard s[ZC_MAX_SHARDS];
  int P;
  uint64_t n;
  uint32_t ntiles;
  uint16_t* out;
  const uint8_t* out_cb;
  uint8_t* out_main;
  uint8_t* out_esc;
  uint64_t out_cap;
  WsHeader* ws;
  Flag* flags;
  int32_t* status;
  int single;   // the RAW-capable launch runs alone and does the work whatever the shards are
  uint32_t gt;  // tiles per escape-scan group: kGroupTilesR (one per team), or 1 (team 0 alone)
};

struct ShardInfo {
  uint32_t t0, t1;  // code -> exponent permute table
  unsigned long long n_esc;
};

// What the producer tells the consumers about a staged tile copy.
struct StageMeta {
  uint32_t a;       // first escape of the tile in the shard's escape stream
  uint32_t cnt;     // escapes of the tile
  uint32_t staged;  // how many of them sit in the stage
  uint16_t shard;
  uint16_t ok;      // kMetaOk: offset table consistent; kMetaRaw: RAW shard, nothing staged
};
constexpr uint16_t kMetaOk = 1, kMetaRaw = 2;

struct RedRound {
  uint32_t agg[kRedSlots];                    // arrivals << 16 | escape count so far
  uint32_t cnt[kRedSlots][16];                // output escapes of each consumer's block
  unsigned long long uprefix[kRedSlots][16];  // exclusive output escape offset of each block
  uint64_t cnt_bar[kRedSlots];
  uint64_t pre_bar[kRedSlots];
};
static_assert(sizeof(RedRound) <= 512, "round bookkeeping too large");

// A consumer's output block of a round, kept until the round's offsets arrive.
struct RedPending {
  bool has, spilled, done;
  uint32_t g;
  EscBook<1> te;
};

// The 8 sums of a lane's 8-element run rounded to bf16 (nearest even) and
// packed.  The hardware conversion rounds exactly as the IEEE definition
// does but returns its own NaN pattern, so when a NaN may be among the sums
// (their total is NaN; an inf - inf total only costs the slow path) the
// run is rounded by the definition instead, which maps NaN to 0x7FC0.
__device__ __forceinline__ uint4 round_pack(const float (&acc)[8]) {
  uint32_t w[4];
  const float t = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  if (t != t) {
#pragma unroll
    for (int i = 0; i < 4; i++) w[i] = f32_to_bf16_rne(acc[2 * i]) | (f32_to_bf16_rne(acc[2 * i + 1]) << 16);
  } else {
#pragma unroll
    for (int i = 0; i < 4; i++) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(acc[2 * i + 1]), "f"(acc[2 * i]));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// RAW = false: the launch for all-coded inputs; it leaves at once when a shard
// is RAW.  RAW = true: the launch that follows it and does the work only when
// some shard is RAW (its shard loop tests every copy for RAW; keeping that
// test out of the all-coded kernel keeps its code as lean as before).  A grid
// of at most one CTA per SM is launch-bound: there the RAW-capable kernel
// runs alone (p.single) and does the work for any shards.  SPLIT = true: that
// kernel for inputs of at most two tiles per SM (one tile per group, gt == 1).
template <bool REENC, bool RAW, bool SPLIT>
__global__ void __launch_bounds__(kRedThreads, 1) reduce_kernel(const __grid_constant__ RedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_allow_dependents();  // (the wait for the previous grid comes after the shared-memory setup)
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t sbase = (smem_u32(smem) + 1023u) & ~1023u;
  uint8_t* gbase = smem + (sbase - smem_u32(smem));
  uint32_t* spread = reinterpret_cast<uint32_t*>(gbase + kRSpread);
  uint32_t* lut = reinterpret_cast<uint32_t*>(gbase + kRLut);
  ShardInfo* si = reinterpret_cast<ShardInfo*>(gbase + kRShard);
  RedRound* rs = reinterpret_cast<RedRound*>(gbase + kRRound);
  int* flags_s = reinterpret_cast<int*>(gbase + kRFlag);  // [0] bad input, [1] bad output codebook
  unsigned long long* raw_s = reinterpret_cast<unsigned long long*>(gbase + kRFlag + 8);  // RAW shards (bit r)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(gbase + kRBars);
  uint64_t* empty_bar = full_bar + kRedTeams * kRedStages;
  StageMeta* meta = reinterpret_cast<StageMeta*>(gbase + kRMeta);
  // A RAW-capable launch that follows the all-coded one has work only when a
  // shard is RAW, which the headers tell after the wait: it checks before any
  // setup, so that in the usual case it leaves at once.
  const bool check_first = RAW && !p.single;
  if (check_first) {
    pdl_wait();
    bool any = false;
    for (int r = threadIdx.x; r < p.P; r += blockDim.x)
      any |= __ldg(reinterpret_cast<const uint32_t*>(p.s[r].main) + 1) == (ZC_VERSION | (kFlagRaw << 16));
    if (!__syncthreads_or(any)) return;
  }
  build_spread_replicated<kSpreadCopies>(spread);
  if (threadIdx.x == 0) {
    flags_s[0] = flags_s[1] = 0;
    *raw_s = 0ull;
    for (int i = 0; i < kRedTeams * kRedStages; i++) {
      mbar_init(&full_bar[i], 1);  // the producer's arrival with the expected bytes
      mbar_init(&empty_bar[i], 4);  // the team's 4 consumer warps
    }
    for (int r = 0; r < kRedSlots; r++) {
      rs->agg[r] = 0;
      mbar_init(&rs->cnt_bar[r], kRedCons);
      mbar_init(&rs->pre_bar[r], 1);
    }
    fence_mbar_init();
  }
  if (!check_first) pdl_wait();  // after the shared-memory setup, which overlaps the previous kernel
  __syncthreads();
  // validate every shard header (each CTA reaches the same decision)
  for (int r = threadIdx.x; r < p.P; r += blockDim.x) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p.s[r].main);
    const uint64_t n = static_cast<uint64_t>(__ldg(w + 2)) | (static_cast<uint64_t>(__ldg(w + 3)) << 32);
    const uint64_t n_esc = static_cast<uint64_t>(__ldg(w + 6)) | (static_cast<uint64_t>(__ldg(w + 7)) << 32);
    const uint32_t c0 = __ldg(w + 8), c1 = __ldg(w + 9);
    uint8_t cb[7];
    for (int k = 0; k < 4; k++) cb[k] = static_cast<uint8_t>(c0 >> (8 * k));
    for (int k = 0; k < 3; k++) cb[4 + k] = static_cast<uint8_t>(c1 >> (8 * k));
    bool dup = false;
    for (int a = 0; a < 7; a++)
      for (int b = a + 1; b < 7; b++) dup |= cb[a] == cb[b];
    int err = 0;
    const uint32_t vf = __ldg(w + 1);
    const bool raw = vf == (ZC_VERSION | (kFlagRaw << 16));
    if (__ldg(w) != ZC_MAGIC || (vf != ZC_VERSION && !raw) || __ldg(w + 4) != kTile || __ldg(w + 5) != p.ntiles ||
        dup || n_esc > p.s[r].esc_bytes || n_esc > p.n || (raw && n_esc != raw_spill(p.n)))
      err = ZC_ERR_BAD_HEADER;
    if (raw) atomicOr(raw_s, 1ull << r);
    if (n != p.n) err = ZC_ERR_SIZE_MISMATCH;
    if (err) {
      atomicExch(&flags_s[0], 1);
      set_status(p.status, err);
    }
    const DecTable dt = make_dec_table(cb);
    si[r].t0 = dt.t0;
    si[r].t1 = dt.t1;
    si[r].n_esc = n_esc;
  }
  if (REENC && warp == 0) {
    if (!build_enc_lut(lut, p.out_cb)) {
      if (lane == 0) {
        flags_s[1] = 1;
        set_status(p.status, ZC_ERR_DUP_CODEBOOK);
      }
    }
  }
  // (re-encoding: the launch's epoch and test hook, read by every thread before the
  // barrier that precedes the scan warp's count, scan_arrive)
  const uint32_t epoch = REENC ? launch_epoch(p.ws) : 0u;
  const uint32_t hold = REENC ? launch_hold(p.ws) : 0u;
  // Producer warps: offsets [a, b) of the tile of team pt0 + u in a round, for
  // shard lane + 32 h.  The first round's are loaded here, so that they arrive
  // while the headers are checked; the end of a shard's last tile is the
  // header's escape count, read directly.
  const uint32_t ngroups = (p.ntiles + p.gt - 1) / p.gt;
  const uint32_t pt0 = (warp - kRedProd) * kTeamsPerProducer;
  uint32_t na[kTeamsPerProducer][2], nb[kTeamsPerProducer][2];
  auto load_offsets = [&](uint32_t G) {
#pragma unroll
    for (int u = 0; u < kTeamsPerProducer; u++)
#pragma unroll
      for (int h = 0; h < 2; h++) {
        na[u][h] = nb[u][h] = 0;
        const uint32_t g = SPLIT ? G : G * p.gt + pt0 + u;
        const uint32_t r = lane + 32u * h;
        if ((SPLIT || pt0 + u < p.gt) && G < ngroups && g < p.ntiles && r < static_cast<uint32_t>(p.P)) {
          const uint32_t* hdr = reinterpret_cast<const uint32_t*>(p.s[r].main);
          const uint32_t* tbl = reinterpret_cast<const uint32_t*>(p.s[r].main + kHeader);
          na[u][h] = __ldg(tbl + g);
          const uint64_t bb = (g + 1 < p.ntiles)
                                  ? static_cast<uint64_t>(__ldg(tbl + g + 1))
                                  : static_cast<uint64_t>(__ldg(hdr + 6)) | (static_cast<uint64_t>(__ldg(hdr + 7)) << 32);
          nb[u][h] = bb > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(bb);
        }
      }
  };
  if (warp >= kRedProd && warp < kRedScan) load_offsets(blockIdx.x);
  __syncthreads();
  if (!RAW && *raw_s != 0ull) return;  // the RAW-capable launch that follows does the work
  const bool skip = flags_s[0] != 0 || flags_s[1] != 0;
  // The scan warp counts the CTA in at once in the RAW-capable kernel, which
  // runs alone when every CTA has at most one group (there the count's round
  // trip would otherwise end the launch), and at the end of its scan in the
  // all-coded kernel of longer launches (an increment at the start delays the
  // first look-back).
  const uint32_t arrival = REENC && RAW && warp == kRedScan && lane == 0 ? scan_arrive(p.ws, epoch) : kNoArrival;
  auto exit_scan = [&]() {
    scan_exit(p.ws, p.flags, epoch, ngroups, RAW || lane != 0 ? arrival : scan_arrive(p.ws, epoch));
  };
  const uint32_t step = gridDim.x;
  // SPLIT (inputs of at most two tiles per SM, gt == 1; a RAW-capable kernel):
  // the four teams share each of the CTA's tiles, team t decoding copies t, t + 4, ...
  // into its 8 KB of the rounded-tile area, and after every four copies all 16
  // consumer warps add them, in rank order, to the sums of their 256 values of
  // the tile; team 0 then rounds and re-encodes as usual.
  static_assert(RAW || !SPLIT, "the SPLIT kernel is a RAW-capable one");
  constexpr bool split = SPLIT;
  if (REENC && !skip && p.ntiles == 0 && blockIdx.x == 0 && warp == 0) {
    write_header_words(p.out_main, 0, p.out_cb);
    write_header_tail(p.out_main, 0, 0);
  }

  if (skip) {
    // nothing to do; the exit protocol below still runs
  } else if (warp >= kRedProd && warp < kRedScan) {
    // ---------------- producer q: stage the P copies of the tiles of teams 2q, 2q + 1, in the
    // order the consumers take them.  What a copy needs (its escape range and its checks, the
    // span of escape bytes to stage) is worked out once per round for every shard at once, one
    // shard per lane, so that issuing a copy is short: lane u waits for team 2q + u's stage,
    // writes 16 bytes and starts the two bulk copies, both teams in the same instructions, and
    // the copies follow each other closely.
    const uint32_t t0 = (warp - kRedProd) * kTeamsPerProducer;
    const uint32_t P = static_cast<uint32_t>(p.P);
    uint32_t uses = 0;  // copies this lane has started for its team (lanes < kTeamsPerProducer)
    // the round's plan per team and shard: pa = the tile's first escape;
    // pk = count | staged << 13 | (span / 16) << 23 | consistent << 31
    uint32_t pa[kTeamsPerProducer][2], pk[kTeamsPerProducer][2];
    auto plan_round = [&]() {
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t r = lane + 32u * h;
        const uint64_t n_esc = r < P ? si[r].n_esc : 0ull;
        const uint64_t buf = r < P ? p.s[r].esc_bytes : 0ull;
#pragma unroll
        for (int u = 0; u < kTeamsPerProducer; u++) {
          const uint32_t a = na[u][h], b = nb[u][h];
          // (absent tiles and shards have a = b = 0; a RAW shard's offset table is
          // zero and it stages nothing, so it is not checked)
          const bool raw_r = RAW && r < P && ((*raw_s >> r) & 1ull);
          const bool ok = raw_r || (a <= b && b <= n_esc && b - a <= kTile);
          if (!ok) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
          const uint32_t aa = ok ? a : 0, cnt = ok ? b - a : 0;
          // escape bytes: the 16-byte-aligned span [aa - head, ...) that holds
          // them, at most kRedEscCap bytes and never past the end of the
          // buffer; ranks beyond it are read from global memory by consumers
          const uint32_t head = aa & 15u;
          const uint64_t base = aa - head;
          uint32_t span = cnt == 0 ? 0u : (head + cnt + 15u) & ~15u;
          if (span > kRedEscCap) span = kRedEscCap;
          if (base + span > buf) span = base >= buf ? 0u : static_cast<uint32_t>((buf - base) & ~15ull);
          const uint32_t staged = span <= head ? 0u : (span - head < cnt ? span - head : cnt);
          pa[u][h] = aa;
          pk[u][h] = cnt | (staged << 13) | ((span >> 4) << 23) | (ok ? 0x80000000u : 0u);
        }
      }
    };
    for (uint32_t G = blockIdx.x; G < ngroups; G += step) {
      plan_round();              // from this round's offsets
      load_offsets(G + step);    // the next round's, consumed once this round is issued
      for (int r = 0; r < p.P; r++) {
        const uint32_t src = static_cast<uint32_t>(r & 31);
        uint32_t ca[kTeamsPerProducer], ck[kTeamsPerProducer];
#pragma unroll
        for (int u = 0; u < kTeamsPerProducer; u++) {
          ca[u] = __shfl_sync(kFull, r < 32 ? pa[u][0] : pa[u][1], src);
          ck[u] = __shfl_sync(kFull, r < 32 ? pk[u][0] : pk[u][1], src);
        }
        if (lane < static_cast<uint32_t>(kTeamsPerProducer)) {
          // lane u serves team t0 + u: the teams' copies start in the same instructions
          uint32_t cau = ca[0], cku = ck[0];
#pragma unroll
          for (int q = 1; q < kTeamsPerProducer; q++)
            if (lane == static_cast<uint32_t>(q)) {
              cau = ca[q];
              cku = ck[q];
            }
          const uint32_t t = t0 + lane;
          const uint32_t g = split ? G : G * p.gt + t;
          if (split ? ((static_cast<uint32_t>(r) & 3u) == t && g < p.ntiles) : (t < p.gt && g < p.ntiles)) {
            const uint32_t bi = t * kRedStages + uses % kRedStages;
            if (uses >= static_cast<uint32_t>(kRedStages))
              mbar_wait_bounded(&empty_bar[bi], (uses / kRedStages - 1) & 1u, p.status);
            uses++;
            StageMeta m;
            m.shard = static_cast<uint16_t>(r);
            if (RAW && ((*raw_s >> r) & 1ull)) {  // RAW shard: the consumers read global memory
              m.a = m.cnt = m.staged = 0;
              m.ok = kMetaOk | kMetaRaw;
              meta[bi] = m;
              mbar_arrive(&full_bar[bi]);
            } else {
              const uint32_t span = ((cku >> 23) & 0x3Fu) << 4;
              m.a = cau;
              m.cnt = cku & 0x1FFFu;
              m.staged = (cku >> 13) & 0x3FFu;
              m.ok = static_cast<uint16_t>(cku >> 31);
              meta[bi] = m;
              uint8_t* stage = gbase + kRStage + bi * kRedStageBytes;
              // (the stage is only ever written by these bulk copies; the
              // consumers' reads of its previous contents completed before their
              // release of it, which the wait above observed)
              mbar_arrive_expect_tx(&full_bar[bi], kTileBytes + span);
              tma_load_1d(stage, tile_ptr(p.s[r].main, p.ntiles, g), kTileBytes, &full_bar[bi]);
              if (span != 0) tma_load_1d(stage + kTileBytes, p.s[r].esc + (cau & ~15u), span, &full_bar[bi]);
            }
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == kRedScan) {
    // ---------------- scan warp (re-encoding): the escape offsets of each group of output tiles
    if (REENC) {
      int64_t prev_G = -1;
      uint64_t prev_incl = 0;
      uint32_t j = 0;
      for (uint32_t G = blockIdx.x; G < ngroups; G += step, j++) {
        const int sl = static_cast<int>(j & 1u);
        // the groups between this CTA's previous group and G (their counts are
        // published by their consumers), added while this CTA still works on G
        bool timed_out;
        const uint64_t prefix =
            prev_incl + window_sum(p.flags, static_cast<uint32_t>(prev_G + 1), G, epoch, p.status, &timed_out);
        mbar_wait_bounded(&rs->cnt_bar[sl], (j >> 1) & 1u, p.status);
        if (lane == 0) rs->agg[sl] = 0;
        const uint32_t c = lane < kRedCons ? rs->cnt[sl][lane] : 0u;
        const uint32_t inc = warp_inclusive_scan(c);
        prev_G = G;
        prev_incl = prefix + __shfl_sync(kFull, inc, 31);
        if (lane < kRedCons) rs->uprefix[sl][lane] = prefix + (inc - c);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rs->pre_bar[sl]);
      }
      exit_scan();
    }
  } else {
    // ---------------- consumers: team t, block b
    const uint32_t t = warp >> 2, b = warp & 3u;
    uint8_t* scratch = gbase + kRScratch + warp * 1024;
    uint8_t* ebuf = gbase + kREbuf + warp * kRedSlots * kRedEbuf;
    const uint32_t ytile_s = sbase + kRYtile + t * 8192;  // shared address of the team's rounded tile
    uint16_t* ytile = reinterpret_cast<uint16_t*>(gbase + kRYtile + t * 8192);
    const uint32_t lut_s = sbase + kRLut;
    const uint32_t spread_lb = sbase + kRSpread + 4 * (lane % kSpreadCopies);
    uint32_t k_item = 0;

    // output offsets posted for round j: write the table entry, header parts, escapes
    auto finish = [&](uint32_t j, const RedPending& pd) {
      const int sl = static_cast<int>(j & 1u);
      mbar_wait_bounded(&rs->pre_bar[sl], (j >> 1) & 1u, p.status);
      if (pd.has) {
        const uint64_t prefix = rs->uprefix[sl][warp];
        if (b == 0) {
          if (lane == 0) *reinterpret_cast<uint32_t*>(p.out_main + kHeader + 4ull * pd.g) = static_cast<uint32_t>(prefix);
          if (pd.g == 0) write_header_words(p.out_main, p.n, p.out_cb);
        }
        if (b == 3 && pd.g + 1 == p.ntiles) {
          const uint64_t n_esc = prefix + pd.te.total;
          write_header_tail(p.out_main, p.ntiles, n_esc);
          if (lane == 0 && n_esc > p.out_cap) set_status(p.status, ZC_ERR_ESCAPE_OVERFLOW);
        }
        if (pd.spilled) {
          write_escapes<1>(ytile_s + b * 2048, pd.te, prefix, p.out_esc, p.out_cap);
        } else {
          const uint8_t* src = ebuf + sl * kRedEbuf;
          for (uint32_t i = lane; i < pd.te.total; i += 32)
            if (prefix + i < p.out_cap) p.out_esc[prefix + i] = src[i];
        }
      }
      __syncwarp();
    };

    RedPending prev;
    prev.has = prev.spilled = false;
    prev.done = true;
    uint32_t j = 0;
    for (uint32_t G = blockIdx.x; G < ngroups; G += step, j++) {
      const uint32_t g = split ? G : G * p.gt + t;
      const bool work = split ? g < p.ntiles : (t < p.gt && g < p.ntiles);  // this team decodes copies of tile g
      const bool has = work && (!split || t == 0);                          // ... and owns its output block b
      const uint64_t rem = work ? p.n - static_cast<uint64_t>(g) * kTile : 0;
      const uint32_t n_tile = rem >= kTile ? kTile : static_cast<uint32_t>(rem);
      float acc[4][8];
#pragma unroll
      for (int k = 0; k < 4; k++)
#pragma unroll
        for (int i = 0; i < 8; i++) acc[k][i] = -0.0f;  // -0 + x == x for every x
      if constexpr (SPLIT) {
        if (work) {
          // One staged copy of block b of tile g (the team's next stage): its 1024
          // values as bf16 go to sink(v) (quarter k: 8 values per lane in v[k]),
          // then the stage is released to the producer.  (The loop below the
          // split path takes the same steps inline: through this helper the
          // re-encoding all-coded kernel measured 1 us slower.)
          auto take_copy = [&](uint32_t g, uint32_t n_tile, auto&& sink) {
            const uint32_t s = k_item % kRedStages;
            const uint32_t bi = t * kRedStages + s;
            mbar_wait_bounded(&full_bar[bi], (k_item / kRedStages) & 1u, p.status);
            const StageMeta m = meta[bi];
            if (RAW && (m.ok & kMetaRaw)) {
              // RAW shard: this block's values, 16 bytes per lane and chunk
              const uint8_t* tiles = tile_ptr(p.s[m.shard].main, p.ntiles, 0);
              const uint64_t region = static_cast<uint64_t>(kTileBytes) * p.ntiles;
              const uint64_t b0 = 2 * (static_cast<uint64_t>(g) * kTile + b * kBlock + lane * 8);
              uint4 v[4];
#pragma unroll
              for (int k = 0; k < 4; k++) v[k] = raw_load16(tiles, p.s[m.shard].esc, region, 2 * p.n, b0 + 512 * k);
              sink(v);
            } else {
              const uint32_t tile_s = sbase + kRStage + bi * kRedStageBytes;
              const uint32_t blk_s = tile_s + b * kBlockBytes;
              const uint32_t w0 = lds32(blk_s + 1024 + lane * 4);
              const uint32_t w1 = lds32(blk_s + 1152 + lane * 4);
              const uint32_t w2 = lds32(blk_s + 1280 + lane * 4);
              uint32_t z = ~(w0 | w1 | w2);
              if (n_tile < kTile) z &= lane_valid_mask(b, n_tile, lane);
              // the block's escape ranks: a scan inside the block, and the totals of
              // the tile's earlier blocks from the team's other three warps
              const uint32_t c = __popc(z);
              const uint32_t inc = warp_inclusive_scan(c);
              const uint32_t total = __shfl_sync(kFull, inc, 31);
              const uint32_t tot_s = sbase + kRTot + (t * 2 + (k_item & 1u)) * 16;
              if (lane == 0) asm volatile("st.shared.u32 [%0], %1;" ::"r"(tot_s + 4 * b), "r"(total) : "memory");
              // code planes -> permute selectors -> rotated exponents, while the totals meet
              uint4 exa, exb;
              {
                uint32_t sel[4];
#pragma unroll
                for (uint32_t k = 0; k < 4; k++) sel[k] = spread_sel<kSpreadCopies>(w0, w1, w2, k, spread_lb);
                const uint32_t t0 = si[m.shard].t0, t1 = si[m.shard].t1;
                exa.x = __byte_perm(t0, t1, sel[0]);
                exa.y = __byte_perm(t0, t1, sel[0] >> 16);
                exa.z = __byte_perm(t0, t1, sel[1]);
                exa.w = __byte_perm(t0, t1, sel[1] >> 16);
                exb.x = __byte_perm(t0, t1, sel[2]);
                exb.y = __byte_perm(t0, t1, sel[2] >> 16);
                exb.z = __byte_perm(t0, t1, sel[3]);
                exb.w = __byte_perm(t0, t1, sel[3] >> 16);
              }
              // the team's four warps: every block total of this copy is written
              // (the two buffers alternate; a buffer is rewritten only after all
              // four warps have passed the next copy's barrier, so after their reads)
              asm volatile("bar.sync %0, 128;" ::"r"(1 + t) : "memory");
              const uint4 tt = lds128(tot_s);
              const uint32_t first = (b > 0 ? tt.x : 0u) + (b > 1 ? tt.y : 0u) + (b > 2 ? tt.z : 0u);
              if (b == 3 && m.ok && first + total != m.cnt && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
              if (z) {
                // patch escapes through the lane's 32 scratch bytes (bit q of z <-> byte q)
                EscSource es;
                es.smem = gbase + kRStage + bi * kRedStageBytes + kTileBytes + (m.a & 15u);
                es.glob = p.s[m.shard].esc + m.a;
                es.staged = m.staged;
                es.count = m.cnt;
                uint32_t rank = first + inc - c;
                // bytes 0..15 of the lane at scratch[16 lane], bytes 16..31 at scratch[512 + 16 lane]:
                // each 16-byte access of the warp then touches every bank once per quarter
                uint4* sp = reinterpret_cast<uint4*>(scratch + lane * 16);
                sp[0] = exa;
                sp[32] = exb;
                uint32_t mz = z;
                uint8_t* dst = scratch + lane * 16;  // byte q at dst[(q & 15) + 32 (q & 16)]
                if (first + total <= es.staged) {  // (warp-uniform) every escape of the block is staged
                  const uint8_t* src = es.smem + rank;
                  do {
                    const uint32_t q = __ffs(mz) - 1;
                    mz &= mz - 1;
                    dst[(q & 15u) + 32u * (q & 16u)] = static_cast<uint8_t>(rot_exp(*src++));
                  } while (mz);
                } else {
                  while (mz) {
                    const uint32_t q = __ffs(mz) - 1;
                    mz &= mz - 1;
                    dst[(q & 15u) + 32u * (q & 16u)] = static_cast<uint8_t>(rot_exp(esc_byte(es, rank)));
                    rank++;
                  }
                }
                exa = sp[0];
                exb = sp[32];
              }
              uint4 v[4];
#pragma unroll
              for (uint32_t k = 0; k < 4; k++) {
                const uint2 sm = lds64(blk_s + k * 256 + lane * 8);
                const uint32_t r0 = k == 0 ? exa.x : k == 1 ? exa.z : k == 2 ? exb.x : exb.z;
                const uint32_t r1 = k == 0 ? exa.y : k == 1 ? exa.w : k == 2 ? exb.y : exb.w;
                bf16_quad(sm.x, r0, v[k].x, v[k].y);
                bf16_quad(sm.y, r1, v[k].z, v[k].w);
              }
              sink(v);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[bi]);  // release the stage to the producer
            k_item++;
          };
          if (REENC && !prev.done && prev.spilled) {  // its escapes sit where this tile's copies go
            finish(j - 1, prev);
            prev.done = true;
          }
          // this thread's 8 values of the tile: elements 256 warp + 8 lane + i
          const uint32_t idx = warp * 256 + lane * 8;
          const uint32_t own_s = sbase + kRYtile + 2 * idx;
          uint8_t* dec = gbase + kRYtile + t * 8192 + b * 2048;  // team t's decoded block b
          const uint32_t P = static_cast<uint32_t>(p.P);
          for (uint32_t q = 0; 4 * q < P; q++) {
            if (4 * q + t < P)
              take_copy(g, n_tile, [&](const uint4 (&v)[4]) {
#pragma unroll
                for (int k = 0; k < 4; k++) *reinterpret_cast<uint4*>(dec + k * 512 + lane * 16) = v[k];
              });
            asm volatile("bar.sync 5, 512;" ::: "memory");  // the 16 consumer warps: four copies decoded
            for (uint32_t u = 0; u < 4 && 4 * q + u < P; u++) accumulate8(acc[0], lds128(own_s + u * 8192));
            asm volatile("bar.sync 5, 512;" ::: "memory");  // ... and added
          }
          uint4 v = round_pack(acc[0]);
          if (n_tile < kTile) {
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (uint32_t jj = 0; jj < 8; jj++)
              if (idx + jj >= n_tile) w[jj >> 1] &= (jj & 1) ? 0x0000FFFFu : 0xFFFF0000u;
            v = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (p.out) store8_guarded(p.out + static_cast<uint64_t>(g) * kTile, idx, rem, v);
          if (REENC) {
            *reinterpret_cast<uint4*>(gbase + kRYtile + 2 * idx) = v;  // team 0's rounded tile
            asm volatile("bar.sync 5, 512;" ::: "memory");
          }
        }
      } else if (has) {
        // the P copies of this block, added in rank order
        for (int r = 0; r < p.P; r++) {
          const uint32_t s = k_item % kRedStages;
          const uint32_t bi = t * kRedStages + s;
          mbar_wait_bounded(&full_bar[bi], (k_item / kRedStages) & 1u, p.status);
          const StageMeta m = meta[bi];
          if (RAW && (m.ok & kMetaRaw)) {
            // RAW shard: this block's values, 16 bytes per lane and chunk
            const uint8_t* tiles = tile_ptr(p.s[m.shard].main, p.ntiles, 0);
            const uint64_t region = static_cast<uint64_t>(kTileBytes) * p.ntiles;
            const uint64_t b0 = 2 * (static_cast<uint64_t>(g) * kTile + b * kBlock + lane * 8);
            uint4 v[4];
#pragma unroll
            for (int k = 0; k < 4; k++) v[k] = raw_load16(tiles, p.s[m.shard].esc, region, 2 * p.n, b0 + 512 * k);
#pragma unroll
            for (int k = 0; k < 4; k++) accumulate8(acc[k], v[k]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[bi]);
            k_item++;
            continue;
          }
          const uint32_t tile_s = sbase + kRStage + bi * kRedStageBytes;
          const uint32_t blk_s = tile_s + b * kBlockBytes;
          const uint32_t w0 = lds32(blk_s + 1024 + lane * 4);
          const uint32_t w1 = lds32(blk_s + 1152 + lane * 4);
          const uint32_t w2 = lds32(blk_s + 1280 + lane * 4);
          uint32_t z = ~(w0 | w1 | w2);
          if (n_tile < kTile) z &= lane_valid_mask(b, n_tile, lane);
          // the block's escape ranks: a scan inside the block, and the totals of
          // the tile's earlier blocks from the team's other three warps
          const uint32_t c = __popc(z);
          const uint32_t inc = warp_inclusive_scan(c);
          const uint32_t total = __shfl_sync(kFull, inc, 31);
          const uint32_t tot_s = sbase + kRTot + (t * 2 + (k_item & 1u)) * 16;
          if (lane == 0) asm volatile("st.shared.u32 [%0], %1;" ::"r"(tot_s + 4 * b), "r"(total) : "memory");
          // code planes -> permute selectors -> rotated exponents, while the totals meet
          uint4 exa, exb;
          {
            uint32_t sel[4];
#pragma unroll
            for (uint32_t k = 0; k < 4; k++) sel[k] = spread_sel<kSpreadCopies>(w0, w1, w2, k, spread_lb);
            const uint32_t t0 = si[m.shard].t0, t1 = si[m.shard].t1;
            exa.x = __byte_perm(t0, t1, sel[0]);
            exa.y = __byte_perm(t0, t1, sel[0] >> 16);
            exa.z = __byte_perm(t0, t1, sel[1]);
            exa.w = __byte_perm(t0, t1, sel[1] >> 16);
            exb.x = __byte_perm(t0, t1, sel[2]);
            exb.y = __byte_perm(t0, t1, sel[2] >> 16);
            exb.z = __byte_perm(t0, t1, sel[3]);
            exb.w = __byte_perm(t0, t1, sel[3] >> 16);
          }
          // the team's four warps: every block total of this copy is written
          // (the two buffers alternate; a buffer is rewritten only after all
          // four warps have passed the next copy's barrier, so after their reads)
          asm volatile("bar.sync %0, 128;" ::"r"(1 + t) : "memory");
          const uint4 tt = lds128(tot_s);
          const uint32_t first = (b > 0 ? tt.x : 0u) + (b > 1 ? tt.y : 0u) + (b > 2 ? tt.z : 0u);
          if (b == 3 && m.ok && first + total != m.cnt && lane == 0) set_status(p.status, ZC_ERR_CORRUPT_STREAM);
          if (z) {
            // patch escapes through the lane's 32 scratch bytes (bit q of z <-> byte q)
            EscSource es;
            es.smem = gbase + kRStage + bi * kRedStageBytes + kTileBytes + (m.a & 15u);
            es.glob = p.s[m.shard].esc + m.a;
            es.staged = m.staged;
            es.count = m.cnt;
            uint32_t rank = first + inc - c;
            // bytes 0..15 of the lane at scratch[16 lane], bytes 16..31 at scratch[512 + 16 lane]:
            // each 16-byte access of the warp then touches every bank once per quarter
            uint4* sp = reinterpret_cast<uint4*>(scratch + lane * 16);
            sp[0] = exa;
            sp[32] = exb;
            uint32_t mz = z;
            uint8_t* dst = scratch + lane * 16;  // byte q at dst[(q & 15) + 32 (q & 16)]
            if (first + total <= es.staged) {  // (warp-uniform) every escape of the block is staged
              const uint8_t* src = es.smem + rank;
              do {
                const uint32_t q = __ffs(mz) - 1;
                mz &= mz - 1;
                dst[(q & 15u) + 32u * (q & 16u)] = static_cast<uint8_t>(rot_exp(*src++));
              } while (mz);
            } else {
              while (mz) {
                const uint32_t q = __ffs(mz) - 1;
                mz &= mz - 1;
                dst[(q & 15u) + 32u * (q & 16u)] = static_cast<uint8_t>(rot_exp(esc_byte(es, rank)));
                rank++;
              }
            }
            exa = sp[0];
            exb = sp[32];
          }
          uint4 v[4];
#pragma unroll
          for (uint32_t k = 0; k < 4; k++) {
            const uint2 sm = lds64(blk_s + k * 256 + lane * 8);
            const uint32_t r0 = k == 0 ? exa.x : k == 1 ? exa.z : k == 2 ? exb.x : exb.z;
            const uint32_t r1 = k == 0 ? exa.y : k == 1 ? exa.w : k == 2 ? exb.y : exb.w;
            bf16_quad(sm.x, r0, v[k].x, v[k].y);
            bf16_quad(sm.y, r1, v[k].z, v[k].w);
          }
#pragma unroll
          for (int k = 0; k < 4; k++) accumulate8(acc[k], v[k]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[bi]);  // release the stage to the producer
          k_item++;
        }
      }
      RedPending cur;
      cur.has = has;
      cur.spilled = false;
      cur.done = false;
      cur.g = g;
      cur.te.total = 0;
      if (REENC && !prev.done && prev.spilled) {  // its escapes still sit in the rounded tile
        finish(j - 1, prev);
        prev.done = true;
      }
      if (has && !split) {
        uint16_t* out = p.out ? p.out + static_cast<uint64_t>(g) * kTile : nullptr;
#pragma unroll
        for (uint32_t k = 0; k < 4; k++) {
          const uint32_t idx = b * kBlock + k * 256 + lane * 8;  // tile-local element index
          uint4 v = round_pack(acc[k]);
          if (n_tile < kTile) {
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (uint32_t jj = 0; jj < 8; jj++)
              if (idx + jj >= n_tile) w[jj >> 1] &= (jj & 1) ? 0x0000FFFFu : 0xFFFF0000u;
            v = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (out) store8_guarded(out, idx, rem, v);
          if (REENC) *reinterpret_cast<uint4*>(ytile + idx) = v;
        }
      }
      if (REENC) {
        if (has) {
          __syncwarp();
          encode_blocks<1>(ytile_s + b * 2048, b, n_tile, lut_s, tile_ptr(p.out_main, p.ntiles, g) + b * kBlockBytes,
                           cur.te);
          cur.spilled = cur.te.total > kRedEbuf;
          if (!cur.spilled) stage_escapes_smem<1>(ytile_s + b * 2048, cur.te, ebuf + (j & 1u) * kRedEbuf);
        }
        const int sl = static_cast<int>(j & 1u);
        if (lane == 0) {
          rs->cnt[sl][warp] = cur.te.total;
          const uint32_t old = atomicAdd(&rs->agg[sl], (1u << 16) | cur.te.total);
          if ((old >> 16) == kRedCons - 1 && hold != G + 1) {
            const uint32_t agg = (old & 0xFFFFu) + cur.te.total;
            const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
            st_relaxed(&p.flags[G].agg, tag | agg);
          }
          mbar_arrive(&rs->cnt_bar[sl]);
        }
        __syncwarp();
        if (!prev.done) finish(j - 1, prev);
        prev = cur;
      }
    }
    if (REENC && j > 0 && !prev.done) finish(j - 1, prev);
  }
  if (REENC && skip && warp == kRedScan) exit_scan();  // (nothing was run)
}

cudaError_t launch_reduce(const Shard* shards, int P, uint64_t n, uint16_t* out, const uint8_t* out_cb,
                          uint8_t* out_main, uint8_t* out_esc, uint64_t out_cap, WsHeader* ws, Flag* flags,
                          int32_t* status, cudaStream_t stream, const DeviceInfo& dev) {
  RedParams p;
  for (int r = 0; r < P; r++) p.s[r] = shards[r];
  p.P = P;
  p.n = n;
  p.ntiles = static_cast<uint32_t>(num_tiles(n));
  p.out = out;
  p.out_cb = out_cb;
  p.out_main = out_main;
  p.out_esc = out_esc;
  p.out_cap = out_cap;
  p.ws = ws;
  p.flags = flags;
  p.status = status;
  // Inputs of at most two tiles per SM take one tile per group, and the four
  // teams of a CTA share each tile's P copies (SPLIT): with four tiles per CTA
  // a team decodes a tile's copies one after another, so on few tiles the
  // launch would be as long as P serial copies on a quarter of the SMs.
  const bool split = p.ntiles <= 2u * static_cast<uint32_t>(dev.sm_count);
  p.gt = split ? 1u : kGroupTilesR;
  const uint32_t ngroups = (p.ntiles + p.gt - 1) / p.gt;
  uint32_t ctas = ngroups;
  if (ctas > static_cast<uint32_t>(dev.sm_count)) ctas = dev.sm_count;
  if (ctas == 0) ctas = 1;
  // The all-coded launch, then the RAW-capable one; exactly one of them works.
  // A grid of at most one group per CTA, and the SPLIT shape, get the
  // RAW-capable launch alone.
  p.single = split || ngroups <= static_cast<uint32_t>(dev.sm_count) ? 1 : 0;
  // [re-encode][kind]: all-coded, RAW-capable, RAW-capable with one tile per CTA (the teams share its copies)
  static KernelPrep prep[2][3];
  const void* const fns[2][3] = {
      {reinterpret_cast<const void*>(reduce_kernel<false, false, false>),
       reinterpret_cast<const void*>(reduce_kernel<false, true, false>),
       reinterpret_cast<const void*>(reduce_kernel<false, true, true>)},
      {reinterpret_cast<const void*>(reduce_kernel<true, false, false>),
       reinterpret_cast<const void*>(reduce_kernel<true, true, false>),
       reinterpret_cast<const void*>(reduce_kernel<true, true, true>)}};
  const int re = out_cb ? 1 : 0;
  if (!re && p.ntiles == 0) return cudaSuccess;
  for (int raw = p.single; raw < 2; raw++) {
    const int kind = raw == 0 ? 0 : (p.gt == 1 ? 2 : 1);
    int per_sm = 0;
    cudaError_t err = prepare_kernel(prep[re][kind], fns[re][kind], kRedThreads, kRedSmem, dev, &per_sm);
    if (err != cudaSuccess) return err;
    void* args[] = {&p};
    err = launch_kernel(fns[re][kind], dim3(ctas), dim3(kRedThreads), kRedSmem, stream, args, re != 0);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace zc
