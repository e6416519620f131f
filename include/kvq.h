/*
 * kvq.h -- C ABI of libkvq: quantized KV cache encoders and attention over an
 * MLA latent cache (the latent row is both key and value), on one GB300 GPU.
 *
 * The pages that define the operations are cited by title:
 *   [P1] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant (KV_TQ) on CPU,
 *         CUDA, and Metal" (colibri pull request 399)
 *   [P2] "CPU: KV cache quantization -- KV8 (fp8 e4m3) + KV_TQ (rotated-int4 /
 *         PolarQuant)" (colibri pull request 553)
 *   [P3] "KV cache: FP16 sliding window + attention sinks, and an optional
 *         2-bit K / 4-bit V cache scheme (--kv q2k)" (Strata pull request 2318)
 *
 * Conventions for every call:
 *   - Ownership: the caller allocates and owns all memory.  The library
 *     allocates nothing on the device and frees nothing; scratch space is the
 *     caller's `workspace`, sized by the matching *_workspace_size call.
 *   - Pointers are device pointers (any memory the GPU can address), except the
 *     layout structs, which are read on the host during the call.  The
 *     attention entry points read and write with vector instructions and
 *     return KVQ_ERR_ARG for a misaligned pointer: the code pool must be
 *     32-byte aligned (then every row is, as rows are 576 or 288 bytes),
 *     queries, outputs and new rows 16-byte aligned, scales, cu_seqlens and
 *     dst_rows 8-byte aligned.  Allocations from cudaMalloc (and PyTorch) are.
 *   - Execution is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Nothing is synchronized unless stated.
 *   - Errors: arguments are validated on the host before any launch and
 *     reported as a kvq_status; nothing is thrown across the ABI.  A launch
 *     failure returns KVQ_ERR_CUDA.  Conditions only the device can see (a
 *     ragged batch larger than the bound it was sized for, a non-monotone
 *     cu_seqlens) set an error word in the workspace (its first 4 bytes),
 *     read with kvq_read_device_error; the kernels never trap.  The word is
 *     sticky: it keeps the first error of any call until read with `clear`,
 *     and a decode/prefill workspace must start with it zero (allocate the
 *     workspace zeroed, or clear it once with kvq_read_device_error).
 *   - The library keeps no global state besides the opt-in launch timing
 *     (kvq_timing_enable, off by default); calls on different streams with
 *     different workspaces are independent.
 *   - Encoders are bit-exact by construction: IEEE f32 arithmetic in a fixed
 *     order, no fast-math, no fused multiply-add except where the definition
 *     names one.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_ARG = 1,          /* null pointer, negative size, bad enum */
    KVQ_ERR_SHAPE = 2,        /* a TQ4 block width that is not a power of two >= 2 */
    KVQ_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    KVQ_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
    KVQ_ERR_UNSUPPORTED = 5,  /* valid arguments this build has no kernel for */
    KVQ_ERR_DEVICE = 6,       /* the device error word was set (see kvq_read_device_error) */
    KVQ_ERR_MISMATCH = 7,     /* cache file of another tier, codec, bit width or layout: refused */
    KVQ_ERR_IO = 8,           /* cache file missing, unreadable, corrupt or of the wrong size */
    KVQ_ERR_NONFINITE = 9,    /* device word: an encoder met a NaN or infinite value (or an
                                 infinite TQ4 radius); that row's codes and scale are unspecified */
    KVQ_ERR_TIMEOUT = 10      /* device word: a bounded wait inside a kernel ran out; the kernel
                                 drained its tensor-core work, freed its tensor memory and wrote
                                 no result for its work item */
} kvq_status;

/* Row codecs of the MLA cache.  KV8: fp8 e4m3 codes + f32 scale per block.
 * TQ4: rotated-int4 (codec 1 of the TQ tier).  KVQ_PQ2 .. KVQ_PQ6: PolarQuant
 * (codec 0 of the TQ tier) with b = 2 .. 6 bits per angle ([P1] Summary:
 * "PolarQuant ... variable 2-6 bit"; [P2] "What's in it": KV_TQ = 2|3|5|6, or
 * 4 with KV_TQ_POLAR = 1); the format value is 10 + b. */
typedef enum kvq_format {
    KVQ_KV8 = 1,
    KVQ_TQ4 = 2,
    KVQ_PQ2 = 12,
    KVQ_PQ3 = 13,
    KVQ_PQ4 = 14,
    KVQ_PQ5 = 15,
    KVQ_PQ6 = 16
} kvq_format;
typedef enum kvq_dtype { KVQ_F32 = 0, KVQ_BF16 = 1 } kvq_dtype;

/* Which attention kernel family runs.  AUTO picks the fastest available;
 * SIMT is the fp32 CUDA-core path (outputs within 1e-5 of exact attention);
 * TENSOR is the tensor-core path (16-bit operands, within 2e-3). */
typedef enum kvq_path { KVQ_PATH_AUTO = 0, KVQ_PATH_SIMT = 1, KVQ_PATH_TENSOR = 2 } kvq_path;

/* Row layout of the MLA latent cache.  A row of D = block_dim[0] (+
 * block_dim[1]) f32 values is split into scale blocks; each block gets one f32
 * scale ([P1] Summary: "fp8 e4m3 + per-row scale"; two blocks, latent 512 and
 * rope 64, give the 584-byte KV8 row and the 296-byte TQ4 row behind the
 * "~3.9x" and "~7.8x" of [P1] Summary).  v_dim leading dims form the value
 * (must lie in block 0).  seed selects the TQ4 rotation signs. */
typedef struct kvq_mla_layout {
    int32_t n_blocks;       /* 1 or 2 */
    int32_t block_dim[2];   /* widths of the scale blocks; block_dim[1] ignored if n_blocks == 1 */
    int32_t v_dim;          /* value width, <= block_dim[0] */
    uint64_t seed;          /* TQ4 sign seed (ignored by KV8) */
} kvq_mla_layout;

/* Human-readable name of a status. */
const char* kvq_status_string(kvq_status status);

/* Library version as "major.minor.patch". */
const char* kvq_version(void);

/* Copies the f32 codebook the kernels use: which = 16 gives the TQ4 levels
 * (16) and decision thresholds (15); which = 4 gives the K2 levels (4) and
 * thresholds (3).  Host memory, host call, no GPU needed.  These are the
 * N(0,1) Lloyd-Max quantizers of [P1] "Why rotated-int4 for the 4-bit tier"
 * and of [P3] "Why per-channel K and per-token V". */
kvq_status kvq_codebook(int32_t which, float* levels, float* thresholds);

/* ------------------------------------------------------------------------ */
/* Producers                                                                */
/* ------------------------------------------------------------------------ */

/* KV8 encode ([P1] Commits, item 1; [P2] "What's in it").  For every row and
 * scale block: s = amax/448 (f32 division), code_i = e4m3(x_i / s) with one
 * round-to-nearest-even, saturating at +-448.  A block whose s is 0 stores
 * s = 0 and codes 0x00.
 *   x         [n_rows][D] f32, row-major
 *   dst_rows  NULL, or device int64 [n_rows]: input row i is stored as pool
 *             row dst_rows[i] (the decode-step append: one new row per
 *             sequence, each at the end of its own range)
 *   codes     pool [*][D] bytes (e4m3 bit patterns), rows written
 *   scales    pool [*][n_blocks] f32, rows written
 *   err_word  NULL, or a device int32 error word (for instance the first 4
 *             bytes of an attention workspace): a row holding a NaN or an
 *             infinity sets it to KVQ_ERR_NONFINITE if it is still 0 (the
 *             pages define no code for such values; that row's codes and
 *             scales are then unspecified, the other rows are unaffected)
 * Any block widths with D <= 4096.  n_rows == 0 is a no-op. */
kvq_status kv8_encode(const float* x, int64_t n_rows, const kvq_mla_layout* layout,
                      const int64_t* dst_rows, uint8_t* codes, float* scales, int32_t* err_word,
                      void* stream);

/* TQ4 (rotated-int4) encode ([P1] "Why rotated-int4 for the 4-bit tier";
 * [P2] "What's in it").  Per block of n dims (a power of two, 2..1024):
 *   y = (1/sqrt n) H_n (sigma . x)   (f32 radix-2 FWHT, stages h = 1,2,4,..)
 *   s = ||x|| / sqrt(n)              (sum of squares in a fixed order: 32
 *                                     interleaved fma partials, then halving)
 *   code_i = number of codebook thresholds strictly below y_i / s
 *   byte j of the block = code_2j | code_(2j+1) << 4
 * sigma comes from layout->seed: splitmix64 words from state = seed, each
 * block taking ceil(n/64) words in order, sign i = -1 when bit i%64 of word
 * i/64 is set.  A block with s == 0 stores s = 0 and codes 0.
 *   x         [n_rows][D] f32
 *   dst_rows  NULL, or device int64 [n_rows] destination pool rows (as kv8_encode)
 *   packed    pool [*][D/2] bytes, rows written (block 0 first)
 *   scales    pool [*][n_blocks] f32, rows written
 *   err_word  NULL, or a device int32 error word set to KVQ_ERR_NONFINITE
 *             (if still 0) by a block whose sum of squares is not finite (a
 *             NaN or infinite input, or a radius past the f32 range)
 * Returns KVQ_ERR_SHAPE for a width that is not a power of two >= 2 ([P1]
 * rebase comment and [P2] review-pass item 1: such rows would all become
 * inert, so the codec refuses). */
kvq_status tq4_encode(const float* x, int64_t n_rows, const kvq_mla_layout* layout,
                      const int64_t* dst_rows, uint8_t* packed, float* scales, int32_t* err_word,
                      void* stream);

/* The TQ4 rotation applied to whole vectors, f32 ([P1] "Ready for review"
 * comment, finding 2: rotate the query once per head, unrotate the
 * accumulated context once).  inverse = 0: out = (1/sqrt n) H_n (sigma . in)
 * per block; inverse = 1: out = sigma . ((1/sqrt n) H_n in).
 *   in   [n_vecs][D] (f32 or bf16 per in_dtype);  out [n_vecs][D] f32. */
kvq_status tq4_rotate(const void* in, kvq_dtype in_dtype, int64_t n_vecs, const kvq_mla_layout* layout,
                      int32_t inverse, float* out, void* stream);

/* PolarQuant encode (codec 0 of the TQ tier; [P1] Summary and Commits item
 * 6: "randomized-Hadamard rotation + recursive polar"; the steps of the
 * published method, Han et al. 2025).  fmt = KVQ_PQ2 .. KVQ_PQ6 gives the
 * width b.  Per block of n dims (a power of two, 2..1024):
 *   y = (1/sqrt n) H_n (sigma . x)       (the TQ4 rotation, same signs)
 *   level 1: pair j = (y_2j, y_2j+1) -> radius sqrtf(a*a + c*c) and an angle
 *            in [0, 2 pi), coded into 2^b uniform cells [2 pi k / 2^b, ...)
 *   level l = 2 .. log2 n: pair (lo, hi) of level-(l-1) radii -> radius
 *            sqrtf(lo*lo + hi*hi) and the angle atan2(hi, lo) in [0, pi/2],
 *            coded with the level's Lloyd-Max codebook for the density
 *            sin(2 psi)^(2^(l-1) - 1)
 *   radii     the one radius left (f32) -> radii[row][block]
 *   codes     the n - 1 angle codes, level 1 first, b bits each, least
 *             significant bit first: ceil(n b / 8) bytes per block, blocks in
 *             order (72 b bytes for the 512 + 64 row; 288 + 8 at b = 4, the
 *             TQ4 footprint)
 * Each decision is taken in f32 without an angle: psi > t when
 * hi * cos(t) > lo * sin(t) (f32 products of the tables' f32 cos and sin),
 * after turning a level-1 pair into its quadrant by exact sign swaps; a tie
 * goes to the lower cell, a zero pair to code 0.  An all-zero block stores
 * radius 0 and codes 0.
 *   x, dst_rows, err_word   as tq4_encode (err_word: KVQ_ERR_NONFINITE for a
 *                           block whose radius is not finite)
 *   codes     pool [*][kvq_row_bytes(fmt, layout)] bytes, rows written
 *   radii     pool [*][n_blocks] f32, rows written
 * KVQ_ERR_SHAPE for a width that is not a power of two >= 2; KVQ_ERR_ARG for
 * a format that is not PolarQuant. */
kvq_status pq_encode(kvq_format fmt, const float* x, int64_t n_rows, const kvq_mla_layout* layout,
                     const int64_t* dst_rows, uint8_t* codes, float* radii, int32_t* err_word, void* stream);

/* PolarQuant decode (the dequantizing consumer): each row rebuilt from its
 * radius down the tree with the cells' centroids, in f32; rotated != 0 leaves
 * it in the rotated domain, else it is unrotated (sigma . (1/sqrt n) H_n y).
 *   codes, radii  as written by pq_encode;  out  [n_rows][D] f32 (device). */
kvq_status pq_decode(kvq_format fmt, const uint8_t* codes, const float* radii, int64_t n_rows,
                     const kvq_mla_layout* layout, int32_t rotated, float* out, void* stream);

/* Bytes of one encoded row (the scales or radii excluded): KV8 D, TQ4 D/2,
 * PolarQuant the sum over blocks of ceil(n b / 8).  0 for an invalid format
 * or layout.  Host call. */
int64_t kvq_row_bytes(kvq_format fmt, const kvq_mla_layout* layout);

/* Copies the f32 PolarQuant tables the kernels use for width bits (2..6) and
 * level (1..10): centroids [2^bits][2] (cos, sin of each cell's centroid) and
 * thresholds [2^bits - 1][2] (cos, sin of each decision threshold; level 1:
 * the 2^(bits-2) - 1 in-quadrant thresholds j pi / 2^(bits-1), the rest left
 * untouched).  Host memory, host call, no GPU needed. */
kvq_status kvq_pq_codebook(int32_t bits, int32_t level, float* centroids, float* thresholds);

/* ------------------------------------------------------------------------ */
/* Consumers                                                                */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace kv_attn_decode needs for at most max_total_rows cached
 * rows across `batch` sequences.  Returns 0 for invalid arguments. */
size_t kv_attn_workspace_size(kvq_format fmt, const kvq_mla_layout* layout, int32_t batch,
                              int32_t n_heads, int64_t max_total_rows, kvq_path path);

/* Ragged decode attention over quantized rows, never reconstructing the cache
 * ([P2] "What's in it": KV8 dequantizes inline with the row scale factored
 * out of the score and context sums; TQ4 rotates the query once per head,
 * dots it with the codebook levels and unrotates the context once).  For
 * sequence b with rows [cu_seqlens[b], cu_seqlens[b+1]) of the packed pool and
 * head h:
 *   z_t = sm_scale * (q_bh . x_hat_t)   over all D dims
 *   out[b][h][:] = sum_t softmax(z)_t x_hat_t[0:v_dim]
 * where x_hat is the row's reconstruction (never materialized).  Long
 * sequences are split into chunks whose partial softmax states are merged
 * (split-T).  An empty sequence yields zeros.
 *   q           [batch][n_heads][D] in q_dtype
 *   codes       packed row pool: KV8 [rows][D] bytes, TQ4 [rows][D/2] bytes,
 *               PolarQuant [rows][kvq_row_bytes(fmt, layout)] bytes
 *   scales      [rows][n_blocks] f32 (PolarQuant: the block radii)
 *   cu_seqlens  [batch+1] int64, device, non-decreasing, cu[0] = 0
 *   max_total_rows  host-side bound on cu_seqlens[batch] (sizes the launch)
 *   out         [batch][n_heads][v_dim] f32, written
 * Supported attention layout: D = 576 as blocks (512, 64) or (576) for KV8,
 * (512, 64) for TQ4 and PolarQuant; v_dim = 512.  Others return
 * KVQ_ERR_UNSUPPORTED.  PolarQuant runs on the fp32 path under KVQ_PATH_AUTO
 * (it rebuilds each row's tree in the rotated domain in shared memory, tile by
 * tile, and unrotates the context once as TQ4 does).  KVQ_PATH_TENSOR with
 * KVQ_PQ4 runs the tensor-core consumer: the trees are rebuilt into f16
 * operands, each leaf rounded once (up to 2^-11 relative), so its outputs are
 * within 4e-3 rather than 2e-3; KVQ_PATH_TENSOR with another PolarQuant width
 * returns KVQ_ERR_UNSUPPORTED. */
kvq_status kv_attn_decode(kvq_format fmt, const kvq_mla_layout* layout,
                          const void* q, kvq_dtype q_dtype, int32_t batch, int32_t n_heads,
                          const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                          int64_t max_total_rows, float sm_scale, float* out,
                          void* workspace, size_t workspace_bytes, kvq_path path, void* stream);

/* One decode step together with the step's new rows: encodes x_new[b] into
 * pool row dst_rows[b] exactly as kv8_encode / tq4_encode with dst_rows would,
 * then runs kv_attn_decode over the pool with those rows included.  The
 * producer writes each new row before the consumer attends over it ([P2]
 * rebase comment, point 1, the KV producer loop; [P3] "Attention error under
 * the engine's append patterns": decode appends to the cache at every step).
 * For KV8 with a bf16 query on the tensor-core path both run in one launch:
 * the CTAs whose chunk holds row dst_rows[b] encode it themselves, use it in
 * place and (one of them) store it; other formats and paths launch the
 * encoder and then the decode.
 *   x_new     [batch][D] f32
 *   dst_rows  [batch] int64, device; dst_rows[b] must lie in [cu[b], cu[b+1])
 *             (the one-launch path sets KVQ_ERR_ARG in the device error word
 *             and skips a row outside it; elsewhere the result is undefined)
 *   codes, scales  the pool: rows dst_rows[b] written, rows of cu_seqlens read
 * Other arguments, the workspace (kv_attn_workspace_size) and the results are
 * those of kv_attn_decode; max_total_rows must be at least batch. */
kvq_status kv_attn_decode_append(kvq_format fmt, const kvq_mla_layout* layout,
                                 const float* x_new, const int64_t* dst_rows,
                                 const void* q, kvq_dtype q_dtype, int32_t batch, int32_t n_heads,
                                 uint8_t* codes, float* scales, const int64_t* cu_seqlens,
                                 int64_t max_total_rows, float sm_scale, float* out,
                                 void* workspace, size_t workspace_bytes, kvq_path path, void* stream);

/* Bytes of workspace kv_attn_decode_gather needs for at most
 * max_total_selected selected rows across `batch` sequences (the path choice,
 * and so the split, depends on q_dtype here).  Returns 0 for invalid or
 * unsupported arguments. */
size_t kv_attn_gather_workspace_size(kvq_format fmt, const kvq_mla_layout* layout, kvq_dtype q_dtype,
                                     int32_t batch, int32_t n_heads, int64_t max_total_selected, kvq_path path);

/* Decode attention over selected rows only: the top-k rows a sparse-attention
 * indexer picked for each sequence, read in place by absolute index ([P1]
 * Commits item 2 and the rebase comment's point 1: the KV8 shadow's
 * absolute-index gather for DSA selection).  For sequence b the rows are the
 * pool rows sel_rows[cu_sel[b]] .. sel_rows[cu_sel[b+1] - 1]; otherwise as
 * kv_attn_decode (same formulas, same output).
 *   pool_rows   number of rows in the pool; an index outside [0, pool_rows)
 *               sets KVQ_ERR_ARG in the device error word and is clamped
 *               (never read out of bounds)
 *   sel_rows    [cu_sel[batch]] int64, device, absolute pool rows (any order,
 *               repeats allowed)
 *   cu_sel      [batch+1] int64, device, non-decreasing, cu_sel[0] = 0
 *   max_total_selected  host-side bound on cu_sel[batch]
 * Paths: the tensor-core kernel for KV8 with bf16 queries, the fp32 kernels
 * otherwise (KVQ_PATH_TENSOR with another format or query type returns
 * KVQ_ERR_UNSUPPORTED). */
kvq_status kv_attn_decode_gather(kvq_format fmt, const kvq_mla_layout* layout,
                                 const void* q, kvq_dtype q_dtype, int32_t batch, int32_t n_heads,
                                 const uint8_t* codes, const float* scales, int64_t pool_rows,
                                 const int64_t* sel_rows, const int64_t* cu_sel, int64_t max_total_selected,
                                 float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                                 kvq_path path, void* stream);

/* kv_attn_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a convenience of this library.
 *
 * Who needs it: a caller that records the decode into a CUDA graph while the
 * stream is being captured (an allocation made then is not part of the graph,
 * and cudaMalloc synchronizes the whole device), a plugin whose host engine
 * owns every device allocation, or a real-time loop that must never block in
 * an allocator.  Such a caller cannot provide kv_attn_decode's workspace.
 *
 * Same arguments and results as kv_attn_decode, without workspace: the split-T
 * scratch lives in a fixed 32 MiB array inside the library's device memory
 * (held on every GPU that loads the library, until the process exits).  A
 * request whose kv_attn_workspace_size exceeds 32 MiB returns
 * KVQ_ERR_WORKSPACE and launches nothing (the scratch grows with the number
 * of sequences, not their length: 32 MiB covers 128 heads for batches of up
 * to 76 sequences (KV8) or 114 (TQ4) of any length on the tensor-core path).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, which may load the library's device code), and so
 * does the first call after the device's context was re-created (a device
 * reset loads the library's device code anew); make that first call before
 * any stream capture.  Argument checks and their statuses are those of
 * kv_attn_decode, made before the size check.  All calls share the one array, which keeps the last call's
 * contents: calls that can overlap on the GPU (other streams, other host
 * threads) race and must be serialized by the caller.  The device error word
 * of kv_attn_decode is not readable here; a ragged batch larger than
 * max_total_rows yields zero outputs for the sequences past the bound. */
kvq_status kv_attn_decode_noalloc(kvq_format fmt, const kvq_mla_layout* layout,
                                  const void* q, kvq_dtype q_dtype, int32_t batch, int32_t n_heads,
                                  const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                                  int64_t max_total_rows, float sm_scale, float* out,
                                  kvq_path path, void* stream);

/* Bytes of workspace kv_attn_prefill needs. */
size_t kv_attn_prefill_workspace_size(kvq_format fmt, const kvq_mla_layout* layout, int32_t n_heads,
                                      int64_t n_past, int64_t n_new, kvq_path path);

/* Chunked causal prefill of one sequence: first encodes the n_new new rows
 * into pool rows [n_past, n_past + n_new) (kv8_encode / tq4_encode), then
 * attends each new token j over pool rows [0, n_past + j] in quantized form,
 * its own row included (the producer runs before the consumer, [P2] review
 * thread on the producer loop).
 *   x_new   [n_new][D] f32
 *   q       [n_new][n_heads][D] in q_dtype
 *   codes, scales  the pool, capacity >= n_past + n_new rows; rows
 *           [0, n_past) are read, rows [n_past, n_past + n_new) written
 *   out     [n_new][n_heads][v_dim] f32, written */
kvq_status kv_attn_prefill(kvq_format fmt, const kvq_mla_layout* layout,
                           const float* x_new, const void* q, kvq_dtype q_dtype,
                           int64_t n_past, int64_t n_new, int32_t n_heads,
                           uint8_t* codes, float* scales, float sm_scale, float* out,
                           void* workspace, size_t workspace_bytes, kvq_path path, void* stream);

/* Opt-in launch timing, for kernel-level rooflines (instrumentation, not part
 * of the pages' method).  With capacity > 0, every kv_attn_decode,
 * kv_attn_decode_append, kv_attn_decode_gather, kv_attn_prefill and
 * kv_attn_decode_k2v4 call records three CUDA events on its stream -- before
 * its partial kernel, before its merge, after its merge -- into the next of
 * `capacity` slots (a ring: older calls are overwritten); capacity 0 turns it
 * off and frees the events.  The record between the two kernels ends the
 * merge's programmatic overlap with the partial kernel, so timed calls run a
 * little slower than untimed ones.  Process-wide state, not thread-safe.
 * Returns KVQ_ERR_ARG for a negative capacity, KVQ_ERR_CUDA if the events
 * cannot be created (then timing is off). */
kvq_status kvq_timing_enable(int32_t capacity);

/* Waits for the recorded calls and returns the summed milliseconds of their
 * partial kernels (from the first record to the second: launch to end of the
 * partial kernel, and for the fused append the row encoding inside it) and of
 * their merges, and how many calls were complete; then empties the ring.
 * KVQ_ERR_ARG for a null pointer, KVQ_ERR_CUDA if an event query fails. */
kvq_status kvq_timing_read(double* partial_ms, double* merge_ms, int32_t* n_calls);

/* Reads the device error word of a decode/prefill workspace (synchronizes
 * `stream`).  Returns 0 when clear, else the kvq_status value of the first
 * error recorded since it was last cleared; clears it when `clear` is
 * non-zero. */
int32_t kvq_read_device_error(void* workspace, int32_t clear, void* stream);

/* Diagnostic of the tensor-core attention kernels: how many tiles after the
 * first of a work item took the exact path of the lagged running maxima (a
 * score passing the running reference by more than the lag: column maxima,
 * then the context accumulator rescaled in tensor memory) since the counter
 * was last cleared.  The counter is bytes 16..19 of a decode/prefill
 * workspace (zero in a zeroed workspace; wraps at 2^32).  Synchronizes
 * `stream`; clears the counter when `clear` is non-zero.  Returns -1 for a
 * null workspace or a failed copy. */
int64_t kvq_read_exact_rescales(void* workspace, int32_t clear, void* stream);

/* Testing hook for the timeout path of the tensor-core attention kernels (the
 * KV8, KV8 f32-query and TQ4 decode/prefill kernels).  Process-wide, not
 * thread-safe, off by default.  With polls > 0, every later launch of those
 * kernels first waits, for at most `polls` polls, on a barrier that nothing
 * arrives on, and its other tile-loop waits give up after `polls` polls too:
 * the wait runs out, the kernel leaves its tile loop, waits (with the normal
 * bound) for the tensor-core operations it issued, frees its tensor memory
 * and sets KVQ_ERR_TIMEOUT in the workspace's error word; no partial result
 * of that launch is meaningful.  polls = 0 restores normal operation.
 * Returns KVQ_ERR_ARG for a negative count. */
kvq_status kvq_test_stall_waits(int64_t polls);

/* ------------------------------------------------------------------------ */
/* K2/V4 GQA cache with an exact FP16 window ([P3])                          */
/* ------------------------------------------------------------------------ */

/* [P3] Summary: K at 2 bits with per-channel scales (one fp16 scale per dim
 * per 32-cell group, a 4-level Lloyd-Max codebook, stored scale = k_gain x
 * the rule's scale with the codes chosen against the un-gained scale), V at 4
 * bits per token (q4_0: 32-dim blocks of fp16 d + 16 bytes, value = (code-8)
 * d, element j < 16 the low nibble of byte j, j >= 16 the high nibble of byte
 * j-16), and an FP16 overlay holding exact copies of the first n_sink cells
 * and the last n_window cells (n_slack spare slots, 16 on the page). */
typedef struct kvq_k2v4_layout {
    int32_t n_kv_heads;
    int32_t head_dim;       /* multiple of 32, <= 512 */
    int32_t group;          /* must be 32 */
    float k_gain;           /* 1.10 on the page */
    int32_t n_sink, n_window, n_slack;
} kvq_k2v4_layout;

/* Encodes whole sequences of n_cells cells (a multiple of 32) and writes the
 * overlay for the sink and window cells.
 *   k, v      [batch][n_kv_heads][n_cells][head_dim] f32 (already rotated; the
 *             Hadamard rotation of the page's cache happens before this call)
 *   k_codes   [batch][n_kv_heads][capacity][head_dim/4] bytes: dim d is bits
 *             2(d%4) of byte d/4, code c reads level c of the K2 codebook
 *   k_scales  [batch][n_kv_heads][capacity/32][head_dim] fp16 bits
 *   v_blocks  [batch][n_kv_heads][capacity][head_dim/32][18] bytes (q4_0)
 *   k_win, v_win [batch][n_kv_heads][n_sink+n_window+n_slack][head_dim] fp16
 *   err_word  NULL, or a device int32 error word set to KVQ_ERR_NONFINITE (if
 *             still 0) by a NaN or infinite K or V value (or K squares past
 *             the f32 range); the codes of the group or block holding it are
 *             then unspecified, the others are encoded as usual
 * Overlay slot of cell c: c < n_sink -> c; c >= n_cells - n_window ->
 * n_sink + c mod (n_window + n_slack). */
kvq_status k2v4_encode(const kvq_k2v4_layout* layout, const float* k, const float* v,
                       int32_t batch, int64_t n_cells, int64_t capacity,
                       uint8_t* k_codes, uint16_t* k_scales, uint8_t* v_blocks,
                       uint16_t* k_win, uint16_t* v_win, int32_t* err_word, void* stream);

/* Appends n_new cells to every sequence at cells n_past .. n_past + n_new - 1
 * (the engine's append patterns of [P3] "Attention error under the engine's
 * append patterns": decode steps, speculative-verify windows, prefill chunks
 * that start or end inside a 32-cell group).
 *   k_new, v_new  [batch][n_kv_heads][n_new][head_dim] f32
 *   pools         as for k2v4_encode; cells < n_past are left as they are
 * K scale of a group ([P3] "Review fixes", "Fresh partial-group scale"):
 *   - first written by this call with all 32 cells: the encoder's rule;
 *   - first written by this call with n < 32 cells:
 *       s = sqrt((ss + (32 - n) prev^2) / 32), ss the sum of squares of the n
 *       cells, prev = fp16(stored scale of the previous group) / k_gain, the
 *       same bits whether that group was stored by an earlier call or in this
 *       one (two calls split at a group boundary store what one call stores);
 *     group 0 with n < 32 cells: s = sqrt(ss / n);
 *   - already holding cells from an earlier call: the stored scale is kept
 *     and the new cells are coded against fp16(stored) / k_gain.
 * Stored scale fp16(k_gain * s), codes against s, as in the encoder.  V and
 * the overlay of the new cells as in the encoder, the window taken at
 * n_past + n_new.  Requires n_past + n_new <= capacity (a multiple of 32);
 * returns KVQ_ERR_ARG otherwise.  err_word as for k2v4_encode. */
kvq_status k2v4_append(const kvq_k2v4_layout* layout, const float* k_new, const float* v_new,
                       int32_t batch, int64_t n_past, int64_t n_new, int64_t capacity,
                       uint8_t* k_codes, uint16_t* k_scales, uint8_t* v_blocks,
                       uint16_t* k_win, uint16_t* v_win, int32_t* err_word, void* stream);

size_t kv_attn_decode_k2v4_workspace_size(const kvq_k2v4_layout* layout, int32_t batch,
                                          int32_t n_q_heads, int64_t n_cells, kvq_path path);

/* GQA decode over the K2/V4 cache: q head h reads kv head h / (n_q_heads /
 * n_kv_heads); cells in the overlay read fp16 exactly, the rest the bulk.
 * n_cells may end inside a 32-cell group (after appends); capacity is a
 * multiple of 32.  k_codes, k_scales and v_blocks are 16-byte aligned
 * (KVQ_ERR_ARG otherwise): tiles are staged by bulk copies of whole groups.
 *   q    [batch][n_q_heads][head_dim] f32;  out [batch][n_q_heads][head_dim] f32 */
kvq_status kv_attn_decode_k2v4(const kvq_k2v4_layout* layout, const float* q, int32_t batch,
                               int32_t n_q_heads, int64_t n_cells, int64_t capacity,
                               const uint8_t* k_codes, const uint16_t* k_scales, const uint8_t* v_blocks,
                               const uint16_t* k_win, const uint16_t* v_win, float sm_scale, float* out,
                               void* workspace, size_t workspace_bytes, kvq_path path, void* stream);


/* ------------------------------------------------------------------------ */
/* Persistence of quantized row pools ([P1] "KV persistence across mode      */
/* changes"; [P2] "What's in it", the .coli_kv bullet)                       */
/* ------------------------------------------------------------------------ */

/* Files are versioned by their magic, which names the tier: "COLIKV" (v1,
 * f32 rows), "COLIKV2" (v2, KV8 codes), "COLIKV3" (v3, TQ codes); eight int64
 * header words follow: rows, row dimension, scale blocks, the two block dims,
 * v_dim, the TQ sign seed and, in h[7], codec << 8 | bits (TQ4: codec 1, 4
 * bits; PolarQuant: codec 0, 2..6 bits, [P1] Commits item 6: "COLIKV3,
 * h[7]=codec<<8|bits").  Then one record per row: its codes, then its f32
 * scales or radii (v1: its f32 values).  All pointers here are HOST pointers; copy device pools to the host
 * first.  Files are written to "<path>.tmp" and renamed over `path`.
 * `msg` (optional, msg_len bytes) receives the reason of a refusal. */

/* Writes a KV8, TQ4 or PolarQuant pool of n_rows rows (codes
 * [n][kvq_row_bytes(fmt, layout)], scales [n][n_blocks]). */
kvq_status kvq_cache_save(const char* path, kvq_format fmt, const kvq_mla_layout* layout, int64_t n_rows,
                          const uint8_t* codes, const float* scales);

/* Writes f32 rows [n][D] as a v1 file (the unquantized tier). */
kvq_status kvq_cache_save_f32(const char* path, const kvq_mla_layout* layout, int64_t n_rows, const float* rows);

/* Reads a file's tier (1, 2, 3), row count and the 8 header words. */
kvq_status kvq_cache_info(const char* path, int32_t* version, int64_t* n_rows, int64_t* header_words, char* msg,
                          size_t msg_len);

/* Reads a KV8 / TQ4 pool into codes / scales (room for `capacity` rows).  A
 * file of another tier, TQ codec, bit width, rotation seed or layout returns
 * KVQ_ERR_MISMATCH (e.g. "file is fp8 (KV8), current mode is KV_TQ: refused")
 * and reads nothing; a size that disagrees with the header returns KVQ_ERR_IO;
 * more rows than `capacity` returns KVQ_ERR_WORKSPACE. */
kvq_status kvq_cache_load(const char* path, kvq_format fmt, const kvq_mla_layout* layout, int64_t capacity,
                          uint8_t* codes, float* scales, int64_t* n_rows, char* msg, size_t msg_len);

/* Reads a v1 (f32) file: a quantized mode loads it by encoding these rows
 * (kv8_encode / tq4_encode) and keeps the file unchanged until it saves. */
kvq_status kvq_cache_load_f32(const char* path, const kvq_mla_layout* layout, int64_t capacity, float* rows,
                              int64_t* n_rows, char* msg, size_t msg_len);

/* Appends n_new rows to a KV8 / TQ4 file in place: the records are written,
 * flushed, and only then counted in the header.  Bytes past the header's
 * count -- an append interrupted before its header update -- are dropped
 * first (and `msg` says so).  Mode checks as kvq_cache_load. */
kvq_status kvq_cache_append(const char* path, kvq_format fmt, const kvq_mla_layout* layout, int64_t n_new,
                            const uint8_t* codes, const float* scales, int64_t* n_rows, char* msg, size_t msg_len);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
