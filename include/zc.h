/*
 * zc.h -- C ABI of libzc: lossless BF16 exponent coding on one GB300 (sm_103a).
 *
 * The method is the one described in the technical summary of "ZipCCL:
 * Efficient Lossless Data Compression of Communication Collectives for
 * Accelerating LLM Training" (Lin, Pan, Fan, Shi, Chu, 2026), cited below as
 * [ZipCCL §x]:
 *   §2.A  LLM tensors are near-Gaussian, so BF16 exponents concentrate: the
 *         seven most frequent exponents cover about 97% of values, and they
 *         can be predicted from the layer's standard deviation sigma instead
 *         of an online histogram.
 *   §2.B  each value is split into sign-mantissa bits and exponent bits; an
 *         exponent among the top 7 becomes a 3-bit code 001..111, any other
 *         exponent becomes code 000 and its full 8 bits go to a separate
 *         escape ("zero-point") array; 16 -> 11 bits per value.
 *   §2.C  the 3-bit codes are kept as three 1-bit arrays in a column-major
 *         layout, blocks padded to 128-byte boundaries.
 *   §2.D  a zipped reduce-scatter is an all-to-all of compressed shards plus a
 *         local reduction; MoE all-to-all sends a fixed-size part first and a
 *         variable-size part after it.
 * and [CCCL §x] cites the jsqmd.com article on CCCL, an in-GPU
 * compression-coupled collective communication library: §3.2 (chunked
 * compress / transfer / decompress on separate streams), §3.3 (adaptive
 * choice of whether to compress), §5.2 (falling back to uncompressed data).
 *
 * ------------------------------------------------------------------------
 * Stream format "ZC1" (all integers little-endian)
 * ------------------------------------------------------------------------
 * A tensor of n bfloat16 values (n < 2^32) becomes two buffers:
 *
 * MAIN stream, exactly zc_main_bytes(n) = 128 + R + 5632 * ntiles bytes,
 * ntiles = ceil(n / 4096), R = roundup(4 * ntiles, 128).  Its size depends on
 * n alone, so it can be sent before the escape stream's size is known (the
 * fixed-size part of [ZipCCL §2.D]).
 *   [0, 128)     header: u32 magic 0x3142435A (bytes "ZCB1") @0, u16 version 1
 *                @4, u16 flags 0 @6, u64 n @8, u32 tile_elems 4096 @16,
 *                u32 ntiles @20, u64 n_esc @24, u8 codebook[7] @32, zeros to 128.
 *   [128, 128+R) u32 esc_off[ntiles]: exclusive prefix sum of the per-tile
 *                escape counts; zero padding up to R.
 *   tiles        tile t at 128 + R + 5632 t holds elements [4096 t, 4096 t + 4096)
 *                as four 1408-byte blocks of 1024 elements.  Block layout:
 *                  [0, 1024)     sign-mantissa byte of element i = sign<<7 | mantissa
 *                  [1024, 1152)  code plane 0 (bit 0 of every code)
 *                  [1152, 1280)  code plane 1
 *                  [1280, 1408)  code plane 2
 *                A plane is a 4 x 32 byte matrix stored column-major: plane
 *                byte q, bit j (LSB first) belongs to block element
 *                256 * (q % 4) + 8 * (q / 4) + j.
 *                Positions >= n in the last tile hold sign-mantissa 0 and code
 *                0 and are not escapes.
 * ESCAPE stream, n_esc bytes (header field): the 8-bit exponents of all values
 *   whose exponent is not in the codebook.  Tile t's escapes occupy
 *   [esc_off[t], esc_off[t] + count_t); inside a tile, blocks in order, inside
 *   a block in ascending plane-bit position (q, j).
 * CODEBOOK: 7 distinct exponent bytes in rank order; codebook[k] <-> code k+1,
 *   code 0 <-> escape.  It travels in the header, so decoding needs no codebook.
 * RAW streams (header flags bit 0 = ZC_FLAG_RAW): the raw bypass for data the
 *   coding does not shrink ([CCCL §3.3]: tiny tensors are left uncompressed;
 *   [CCCL §5.2]: a ratio near or above 1 falls back to the data as is).  The
 *   main stream keeps its size and header; its offset table is zero; the
 *   2n little-endian bytes of the values fill the tile region in order
 *   (5632 * ntiles bytes, zero beyond 2n) and the rest, the "spill"
 *   max(0, 2n - 5632 * ntiles) bytes, forms the escape stream (n_esc = spill).
 *   Only the adaptive encoders write RAW streams, exactly when the coded
 *   form's escape count exceeds the spill (RAW is then strictly smaller);
 *   every decoder reads both kinds.
 *
 * ------------------------------------------------------------------------
 * Conventions for every entry point
 * ------------------------------------------------------------------------
 * - Pointers named d_* are device pointers owned by the caller (for example
 *   tensors allocated by PyTorch); h_* are host pointers.  libzc never
 *   allocates, never frees and never synchronises the host.  All device work
 *   is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * - Launches: every kernel is launched as a programmatic dependent launch
 *   (CUDA's programmatic stream serialization), so it may be scheduled while
 *   the kernel before it on the stream finishes; it reads and writes global
 *   memory only after that kernel has completed and its writes are visible,
 *   so stream order holds for all data.  Each kernel also lets the launch
 *   after it start early: a caller's kernel that follows on the same stream
 *   with the programmatic attribute must wait for its prerequisites
 *   (cudaGridDependencySynchronize) before it reads libzc's outputs, as that
 *   attribute always requires; launches without it see plain stream order.
 * - Alignment: bfloat16 buffers, main streams and escape streams must be
 *   16-byte aligned; the workspace 16-byte aligned; d_status 4-byte aligned.
 * - Argument errors are returned synchronously and enqueue nothing.  A failed
 *   kernel launch returns ZC_ERR_CUDA.
 * - Data-dependent errors (corrupt stream, escape overflow, ...) cannot be
 *   known on the host without a synchronisation, so the device writes them to
 *   *d_status.  The caller zeroes that int32 before use; the first error wins
 *   and later errors do not overwrite it.  Read it (after the stream has
 *   finished) when convenient.
 * - Workspace: calls that need one take (d_ws, ws_bytes).  Size it with
 *   zc_workspace_size and fill it with zeros ONCE before its first use; every
 *   call that completes without a device error leaves it ready for the next
 *   call (no per-call memset is needed).  After a call that reported a device
 *   error, zero it again.  Calls that share a workspace must be ordered on one
 *   stream; concurrent calls need separate workspaces.
 */
#ifndef ZC_H
#define ZC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZC_TILE_ELEMS 4096
#define ZC_BLOCK_ELEMS 1024
#define ZC_BLOCK_BYTES 1408
#define ZC_TILE_BYTES 5632
#define ZC_HEADER_BYTES 128
#define ZC_MAGIC 0x3142435Au
#define ZC_VERSION 1
#define ZC_FLAG_RAW 1u
#define ZC_MAX_SHARDS 64
#define ZC_WORKSPACE_HEADER_BYTES 4096
#define ZC_WORKSPACE_BYTES_PER_TILE 16

typedef enum zc_status {
  ZC_OK = 0,
  /* synchronous (returned) */
  ZC_ERR_INVALID_ARG = 1,     /* null pointer, bad count, sigma not finite and positive, ... */
  ZC_ERR_ALIGNMENT = 2,       /* a pointer violates the alignment rules above */
  ZC_ERR_TOO_LARGE = 3,       /* n >= 2^32 */
  ZC_ERR_WORKSPACE = 4,       /* ws_bytes smaller than zc_workspace_size */
  ZC_ERR_CODEBOOK = 5,        /* host codebook with duplicate entries */
  ZC_ERR_CUDA = 6,            /* a CUDA runtime call or kernel launch failed */
  /* asynchronous (written to *d_status by the device) */
  ZC_ERR_ESCAPE_OVERFLOW = 7, /* more escapes than esc_capacity; the count in the header is still exact */
  ZC_ERR_BAD_HEADER = 8,      /* magic, version, tile size, ntiles, codebook or n_esc invalid */
  ZC_ERR_CORRUPT_STREAM = 9,  /* offset table inconsistent with the code planes or the escape stream */
  ZC_ERR_SIZE_MISMATCH = 10,  /* header n differs from the n passed in */
  ZC_ERR_TIMEOUT = 11,        /* an inter-block wait gave up (about one second); output invalid */
  ZC_ERR_DUP_CODEBOOK = 12,   /* a device codebook holds a repeated exponent; nothing was encoded */
  ZC_ERR_OUT_OF_ROOM = 13     /* the output buffer is smaller than the stream (QLC) */
} zc_status;

/* Human-readable name of a status value (static string, never NULL). */
const char* zc_status_string(int status);

/* Version of the library and of the stream format, as "libzc <x.y> ZC1". */
const char* zc_version(void);

/*
 * sigma -> codebook, the closed form of [ZipCCL §2.A] (host arithmetic, pure).
 * The pages derive the top-7 exponents from the layer's weight standard
 * deviation without printing the formula; libzc takes the plainest reading:
 * p_e = P(exponent field of RNE_bf16(X) == e) for X ~ N(0, sigma^2), with the
 * binade edges moved down by half an ulp for round-to-nearest-even, computed
 * in double with erf/erfc; the 7 exponents with the largest p_e (ties: the
 * smaller exponent first) in rank order.
 * sigma must be finite and > 0 (else ZC_ERR_INVALID_ARG).  cb_out: 7 bytes, host.
 */
zc_status zc_codebook_from_sigma(double sigma, uint8_t cb_out[7]);

/*
 * Sizes of the two streams for n elements (pure).  *main_bytes is exact (see
 * the format above); *max_escape_bytes = n is the worst case (every value an
 * escape).  Either output pointer may be NULL.  n >= 2^32 -> ZC_ERR_TOO_LARGE.
 */
zc_status zc_compressed_size(uint64_t n, uint64_t* main_bytes, uint64_t* max_escape_bytes);

/*
 * Workspace bytes needed by a call that encodes `count` tensors of sizes
 * h_ns[0..count-1] (compress, compress_batched, decompress_reduce with
 * re-encoding) or computes a histogram (count = 1, any n):
 * ZC_WORKSPACE_HEADER_BYTES + ZC_WORKSPACE_BYTES_PER_TILE * sum(ceil(n_i / 4096)).
 */
zc_status zc_workspace_size(const uint64_t* h_ns, int count, uint64_t* bytes);

/*
 * Exact exponent histogram -> top-7 codebook, the online alternative that
 * [ZipCCL §2.A] avoids; kept for tensors whose sigma is unknown and for
 * non-Gaussian payloads.  Counts all n exponent fields (0 and 255 included),
 * orders (count desc, exponent asc) and writes the first 7 to d_cb_out (7
 * bytes, device).  d_hist_out (256 x u32, device) receives the counts when
 * not NULL.  One launch; the codebook never leaves the device, so it can feed
 * zc_compress without a host round trip.  n = 0 yields codebook 0..6.
 * d_in: n bf16 values, 16-byte aligned.  Workspace: zc_workspace_size(&n, 1).
 */
zc_status zc_histogram_topk(const void* d_in, uint64_t n, uint8_t* d_cb_out, uint32_t* d_hist_out,
                            void* d_ws, uint64_t ws_bytes, int32_t* d_status, void* stream);

/*
 * Encode n bf16 values [ZipCCL §2.B, §2.C] into the ZC1 main stream d_main
 * (zc_main_bytes(n) bytes, fully written, padding included) and the escape
 * stream d_esc (esc_capacity bytes available).  d_cb: 7 distinct exponents,
 * DEVICE memory (from zc_histogram_topk, or zc_codebook_from_sigma copied
 * over).  The escape count is the header's n_esc; if it exceeds esc_capacity,
 * only the first esc_capacity escapes are stored and *d_status gets
 * ZC_ERR_ESCAPE_OVERFLOW.  A codebook with repeated entries sets
 * ZC_ERR_DUP_CODEBOOK and writes nothing else.  One kernel launch: the escape
 * offsets come from a single-pass scan inside it (each group of tiles adds the
 * counts published since its block's previous group), whose waits are
 * bounded (ZC_ERR_TIMEOUT).
 */
zc_status zc_compress(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                      uint64_t esc_capacity, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                      void* stream);

/*
 * Escape bytes of a RAW stream of n values, max(0, 2n - 5632 * ceil(n/4096))
 * (about 0.625 n).  An adaptive compression never needs a larger escape
 * capacity: with esc_capacity >= this bound it cannot overflow.
 * n >= 2^32 -> ZC_ERR_TOO_LARGE.
 */
zc_status zc_raw_spill(uint64_t n, uint64_t* bytes);

/*
 * zc_compress with the raw bypass ([CCCL §3.3], [CCCL §5.2]): encodes like
 * zc_compress; then, in the same launch, once every CTA has encoded its tiles
 * (a grid barrier of the cooperative launch), the escape count is read on the
 * device and the tensor is rewritten as a RAW stream (format above) when that
 * is strictly smaller, i.e. when n_esc > zc_raw_spill(n) -- no host
 * synchronisation.  The header's flags tell which form was stored and n_esc
 * the escape bytes to send.  A coded form that overflows esc_capacity is not
 * an error when the RAW form fits; ZC_ERR_ESCAPE_OVERFLOW is reported only
 * when neither fits (then the coded output stands, as in zc_compress).
 * Arguments, alignment, workspace and other errors as in zc_compress.
 */
zc_status zc_compress_adaptive(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                               uint64_t esc_capacity, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                               void* stream);

/*
 * Decode a ZC1 stream back to n bf16 values, bit for bit (the inverse of
 * zc_compress and zc_compress_adaptive; coded and RAW streams alike).
 * esc_bytes: the readable size of d_esc (at least the header's n_esc).  The
 * header and every tile's escape range are validated on the device before
 * use; a bad header writes nothing, a corrupt tile skips that tile; errors go
 * to *d_status.  No workspace.
 */
zc_status zc_decompress(const void* d_main, const void* d_esc, uint64_t esc_bytes, uint64_t n,
                        void* d_out, int32_t* d_status, void* stream);

/*
 * Local stage of a zipped reduce-scatter [ZipCCL §2.D]: decode P received
 * shards of n elements each, add them in fp32 in rank order 0..P-1
 * (acc = x_0; acc += x_r; IEEE round-to-nearest, subnormals kept), round to
 * bf16 (round-to-nearest-even; a NaN sum becomes 0x7FC0), and optionally
 * re-encode the result with the output codebook d_out_cb.
 *   h_mains, h_escs, h_esc_bytes: host arrays of P device pointers / sizes.
 *   d_out: n bf16 results, or NULL to skip writing them.
 *   d_out_cb: device codebook for re-encoding, or NULL for no re-encoding (then
 *     d_out must be non-NULL and d_out_main/d_out_esc/d_ws may be NULL).
 *   d_out_main / d_out_esc / out_esc_capacity: as in zc_compress.
 * 1 <= P <= ZC_MAX_SHARDS.  Every shard's header must carry n
 * (ZC_ERR_SIZE_MISMATCH otherwise); shards may be coded or RAW.  The
 * re-encoded output is always coded.  One fused kernel launch.
 */
zc_status zc_decompress_reduce(int P, const void* const* h_mains, const void* const* h_escs,
                               const uint64_t* h_esc_bytes, uint64_t n, void* d_out,
                               const uint8_t* d_out_cb, void* d_out_main, void* d_out_esc,
                               uint64_t out_esc_capacity, void* d_ws, uint64_t ws_bytes,
                               int32_t* d_status, void* stream);

/*
 * zc_compress without a workspace argument, for callers that cannot allocate
 * device memory: hooks of a communication or training framework that receive
 * only the tensors to send, and latency-critical paths that must never call
 * cudaMalloc (it can synchronise the device).  The method pages have no counterpart; it
 * is a deployment convenience.  Output is identical to zc_compress.
 *   - The scratch is a fixed 1 MiB + 4 KiB device array inside libzc
 *     (every GPU that loads the library holds it until the process exits), so
 *     n is limited to 2^28 values (512 MiB of bf16); larger n returns
 *     ZC_ERR_WORKSPACE and enqueues nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents; the call clears the counters that must start at zero with an
 *     8-byte cudaMemsetAsync on `stream`.  Calls that overlap on the GPU (two
 *     streams at once) race: order them on one stream.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 * Arguments, alignment and device errors as in zc_compress, except that no
 * reset is needed after a device error (a caller could not reset the internal
 * array anyway): each call clears the two counters itself, and the kernel
 * advances the launch epoch on every path, a timeout included, so flags left
 * by an earlier call never match a later one.
 */
zc_status zc_compress_noalloc(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_main, void* d_esc,
                              uint64_t esc_capacity, int32_t* d_status, void* stream);

/*
 * One tensor of a batched call.  compress: bf16 = input (n values), main/esc =
 * outputs, esc_bytes = escape capacity, cb = device codebook.  decompress:
 * main/esc = inputs, esc_bytes = readable escape bytes, bf16 = output, cb unused.
 */
typedef struct zc_tensor {
  void* bf16;
  void* main;
  void* esc;
  const uint8_t* cb;
  uint64_t n;
  uint64_t esc_bytes;
} zc_tensor;

/*
 * Encode / decode many tensors in one launch over the flattened tile space,
 * each tensor with its own codebook and its own escape scan (the per-layer
 * bucket of [ZipCCL §4]'s Llama3-8B runs, or the per-destination chunks of an
 * MoE all-to-all).  h_tensors: host array of `count` descriptors (count >= 1);
 * the library splits very large counts into several launches.
 * compress_batched needs a workspace of zc_workspace_size over all n.
 */
zc_status zc_compress_batched(int count, const zc_tensor* h_tensors, void* d_ws, uint64_t ws_bytes,
                              int32_t* d_status, void* stream);
/*
 * Zipped transfer pipeline ([CCCL §3.2]; the static/dynamic split of
 * [ZipCCL §2.D]): moves n bf16 values from d_in to d_out the way a compressed
 * collective moves them over a link -- in chunks of chunk_elems values, with
 * three stages overlapped on three streams:
 *   stream_compress    chunk k      zc_compress_adaptive into send slot k % 2
 *   stream_link        chunk k - 1  one copy kernel: the fixed-size main
 *                                   stream (the static part, its size known
 *                                   on the host) and exactly n_esc escape
 *                                   bytes, n_esc read on the device from the
 *                                   sender's header (the dynamic part)
 *   stream_decompress  chunk k - 2  zc_decompress from receive slot k % 2
 *                                   into d_out
 * On one GPU the receive slots (in the workspace) stand in for the peer's
 * buffers and the copy for the link.  Send and receive slots are double
 * buffered: compressing chunk k waits until the link has taken chunk k - 2
 * out of the send slot, and the link waits until chunk k - 2 has been decoded
 * out of the receive slot.  Each chunk is compressed adaptively (a chunk the
 * coding does not shrink travels RAW), so its escape slot (5/8 of a chunk's
 * values in bytes) never overflows.
 *   - The stages start after all work already enqueued on stream_compress;
 *     when the call's work on stream_decompress is done, d_out holds the
 *     values, and stream_compress and stream_link also wait for that point.
 *     The three streams may be the same stream (then nothing overlaps).
 *   - chunk_elems: a positive multiple of 8; d_in, d_out 16-byte aligned.
 *   - d_ws: zc_pipeline_workspace_size(chunk_elems) bytes, 256-byte aligned,
 *     zero-filled before its first use (like every workspace).  Calls that
 *     share it must be ordered.
 *   - The call creates and releases seven CUDA events (no device memory).
 *   - Device errors of any stage go to *d_status.
 */
zc_status zc_pipeline_workspace_size(uint64_t chunk_elems, uint64_t* bytes);
zc_status zc_pipelined_transfer(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_out,
                                uint64_t chunk_elems, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                void* stream_compress, void* stream_link, void* stream_decompress);

/*
 * Pipeline plan: the launch sequence of one zc_pipelined_transfer call (same
 * arguments, same checks, same errors), captured once into an instantiated
 * CUDA graph and replayed by zc_pipeline_plan_launch with a single launch.
 * Each chunk costs three kernel launches and up to seven event operations; once chunks
 * are small the host submits them more slowly than the GPU runs them, and a
 * replay removes that cost.
 *   - overlap != 0: captured from three private streams, so the graph keeps
 *     the three stages' overlap; overlap == 0: one stream, nothing overlaps.
 *   - The plan holds the pointers it was made with (not their contents): a
 *     launch reads d_in, d_cb and the workspace as they are when it runs and
 *     writes d_out and *d_status.  The buffers must outlive the plan's last
 *     launch; launches that share the workspace must be ordered (one stream).
 *   - zc_pipeline_plan_create enqueues no device work; it creates and releases
 *     streams and events and instantiates the graph (driver memory, no
 *     library allocation of the caller's buffers).  On error *plan is NULL.
 *   - zc_pipeline_plan_launch(plan, stream): the whole pipeline runs after the
 *     work already on `stream`, and later work on `stream` sees d_out.  The
 *     current device must be the one the plan was made on
 *     (else ZC_ERR_INVALID_ARG).  A plan of n == 0 launches nothing.
 *   - zc_pipeline_plan_destroy: releases the plan (NULL is accepted); a launch
 *     still in flight completes.
 */
typedef struct zc_pipeline_plan_s* zc_pipeline_plan;
zc_status zc_pipeline_plan_create(const void* d_in, uint64_t n, const uint8_t* d_cb, void* d_out,
                                  uint64_t chunk_elems, void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                  int overlap, zc_pipeline_plan* plan);
zc_status zc_pipeline_plan_launch(zc_pipeline_plan plan, void* stream);
zc_status zc_pipeline_plan_destroy(zc_pipeline_plan plan);

/*
 * Cost models for deciding, on the host, whether compressing pays
 * ([CCCL §2.2]: compression pays only while the time to compress plus the
 * time to send the compressed data stays below the time to send the raw
 * data; [ZipCCL §2.D]: the reduce-scatter switcher profiles bandwidth,
 * latency and ratio once and picks the native reduce-scatter or the zipped
 * all-to-all with a local reduction).  Plain arithmetic, no device work.
 *   link:  bandwidth (GB/s per rank and direction) and latency (us) of a message.
 *   codec: compress / decompress throughput in GB/s of uncompressed data (the
 *          decompress figure stands for decompress-reduce in the
 *          reduce-scatter model, per byte of its P inputs) and the expected
 *          ratio (uncompressed / compressed bytes, e.g. from a sample).
 * zc_transfer_pays: one message of `bytes`:
 *   t_raw = latency + bytes / bandwidth
 *   t_zipped = bytes / compress + latency + bytes / ratio / bandwidth + bytes / decompress
 * zc_reduce_scatter_choose: P ranks, `bytes` per rank before the reduction:
 *   native ring: (P - 1) steps of latency + bytes / P / bandwidth
 *   zipped: compress bytes, one all-to-all step of latency +
 *           (P - 1) / P * bytes / ratio / bandwidth, decompress-reduce of the
 *           P received shards (P * bytes / P = bytes of inputs)
 * Outputs (any may be NULL): the decision (1 = compress) and both times (us).
 * Non-positive bandwidth, throughputs or ratio, negative latency, P < 1 ->
 * ZC_ERR_INVALID_ARG.
 */
typedef struct zc_link_model {
  double bandwidth_gbps;
  double latency_us;
} zc_link_model;
typedef struct zc_codec_model {
  double compress_gbps;
  double decompress_gbps;
  double ratio;
} zc_codec_model;
zc_status zc_transfer_pays(uint64_t bytes, const zc_link_model* link, const zc_codec_model* codec, int* pays,
                           double* t_raw_us, double* t_zipped_us);
zc_status zc_reduce_scatter_choose(uint64_t bytes, int P, const zc_link_model* link, const zc_codec_model* codec,
                                   int* use_zipped, double* t_native_us, double* t_zipped_us);

/* zc_compress_batched with the raw bypass of zc_compress_adaptive, decided per tensor. */
zc_status zc_compress_batched_adaptive(int count, const zc_tensor* h_tensors, void* d_ws, uint64_t ws_bytes,
                                       int32_t* d_status, void* stream);
zc_status zc_decompress_batched(int count, const zc_tensor* h_tensors, int32_t* d_status, void* stream);

/*
 * ------------------------------------------------------------------------
 * Quad Length Codes for FP8 (e4m3) bytes -- [QLC §x] cites the ijyty.com
 * article on QLC for lossless compression of e4m3 tensors in LLM training:
 * §3.1 a 3-bit prefix splits the frequency-ranked symbol space into 8
 * regions with only four code lengths, §3.2 the static table (6/7/8/11-bit
 * codes), §3.3 dynamic tables per layer, §4.1-§4.2 one lookup per symbol.
 * ------------------------------------------------------------------------
 * TABLE: width[r] (r = 0..7) = bits after the prefix in region r; sym[k] = the
 *   byte value of frequency rank k (a permutation of 0..255).  Region r holds
 *   ranks [s_r, s_r + 2^width[r]), s_0 = 0, s_(r+1) = s_r + 2^width[r]; rank k
 *   in region r is coded as r (3 bits) then k - s_r (width[r] bits), most
 *   significant bit first.  Valid when every width <= 8 and
 *   sum 2^width[r] >= 256.  Every byte value (NaN, Inf included) has a code.
 * STREAM "ZQ1" of n bytes (one buffer, little-endian):
 *   [0, 384)   header: u32 magic 0x3142515A ("ZQB1") @0, u16 version 1 @4,
 *              u16 flags 0 @6, u64 n @8, u32 4096 @16, u32 nblocks @20,
 *              u64 payload_words @24, u8 width[8] @64, u8 sym[256] @128.
 *   [384, 384+R)  u32 word offset of each block in the payload, zero padding
 *              to R = roundup(4 * nblocks, 128).
 *   payload    payload_words u32 words; block b = 8 words of lane word counts
 *              (byte l = words of lane l) then the words of lanes 0..31.  The
 *              block's symbols [4096 b, 4096 b + 4096) form 256 runs of 16;
 *              lane l codes runs l, l + 32, ..., l + 224 in that order (the
 *              symbols below n), first code at bit 31 of its first word, the
 *              last word zero-padded.
 *   Stream bytes = 384 + R + 4 * payload_words, at most zq_max_bytes(n).
 */
#define ZQ_BLOCK_SYMBOLS 4096
#define ZQ_HEADER_BYTES 384

typedef struct zq_table {
  uint8_t width[8];
  uint8_t sym[256];
} zq_table;

/* The static widths {3,3,3,3,3,4,5,8}: regions of 8,8,8,8,8,16,32 ranks and the
 * rest (ranks 88-255), code lengths 6/7/8/11 ([QLC §3.2]).  Host. */
zc_status zq_default_widths(uint8_t widths[8]);

/* A table from a 256-bin byte histogram (host): ranks by (count desc, byte
 * asc) ([QLC §4.1]); widths NULL = the static widths.  An invalid widths set
 * returns ZC_ERR_CODEBOOK. */
zc_status zq_table_from_histogram(const uint64_t* h_hist, const uint8_t* widths, zq_table* out);

/* Largest stream of n bytes: 384 + R + 5664 * nblocks. */
zc_status zq_max_bytes(uint64_t n, uint64_t* bytes);

/* Encode n bytes (d_in, 16-byte aligned) into the ZQ1 stream d_out (16-byte
 * aligned, out_capacity bytes; zq_max_bytes(n) always suffices).  h_table:
 * host table (validated: ZC_ERR_CODEBOOK), embedded in the stream.  One
 * cooperative launch with the single-pass block-offset scan of zc_compress;
 * workspace zc_workspace_size(&n, 1) bytes, zeroed before first use.  A
 * stream larger than out_capacity sets ZC_ERR_OUT_OF_ROOM (the header's
 * payload_words is still exact); other device errors as in zc_compress. */
zc_status zq_compress(const void* d_in, uint64_t n, const zq_table* h_table, void* d_out, uint64_t out_capacity,
                      void* d_ws, uint64_t ws_bytes, int32_t* d_status, void* stream);

/* Decode a ZQ1 stream of in_bytes readable bytes back to n bytes (d_out,
 * 16-byte aligned).  The header (magic, sizes, table) is validated on the
 * device: a bad header writes nothing; a block whose words do not add up sets
 * ZC_ERR_CORRUPT_STREAM.  No workspace. */
zc_status zq_decompress(const void* d_in, uint64_t in_bytes, uint64_t n, void* d_out, int32_t* d_status,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ZC_H */
