/*
 * mosaickv.h -- C ABI of libmosaickv.so, the GB300 (sm_103a) decode-time hot
 * path of MosaicKV's dynamic two-D KV-cache compression.
 *
 * Sources cited below:
 *  [N] "MosaicKV：面向超长上下文LLM服务的动态二维KV缓存压缩——阅读笔记"
 *      (reading notes, zhongzhuzhou.org).
 *  [S] "MosaicKV: Serving Long-Context LLM with Dynamic Two-D KV Cache
 *      Compression" (paperlayer.ai summary of arXiv 2607.00760v1).
 *
 * Conventions for every call
 *  - Device pointers are plain CUDA device addresses owned by the caller.
 *    The library never allocates device memory: the caller provides one
 *    persistent "arena" (the compressed cache) and one "workspace" (scratch
 *    reused by every call) sized by mk_arena_bytes / mk_workspace_bytes.
 *  - bf16 tensors are passed as void* to raw 16-bit bf16 words.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    validate on the host and enqueue kernels; they do not synchronise.
 *  - Errors found on the host return at once and change no state.  Errors
 *    found by a kernel (capacity overrun, bad block id) set a sticky device
 *    error word, make later kernels of the context return early, and are read
 *    with mk_poll_error.  No call aborts, throws or traps.
 *  - One context must be used by one host thread at a time, and its calls
 *    must be ordered on the device (one stream, or events between streams).
 *  - The decode kernels use programmatic dependent launch: each may start its
 *    prologue while the previous kernel in the stream finishes.  Before its
 *    wait point a kernel reads only the rotations and, for mk_block_select,
 *    the query; so the query must be complete when the stream's previous
 *    kernel finishes (true whenever it is written before the preceding
 *    mk_append_compress, or by any kernel that does not itself trigger early).
 *  - Positions: a sequence holds tokens 0..T-1.  Sink tokens [0, S) and the
 *    recent window [T-W, T) are stored uncompressed (rotated bf16); the
 *    middle [S, T-W) is cut into blocks of B tokens from position S.
 */
#ifndef MOSAICKV_H
#define MOSAICKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_HEAD_DIM 128      /* head dimension d; the only one supported */
#define MK_MAX_SEGMENTS 4    /* strategy segments per sequence */
#define MK_MAX_GROUP 8       /* query heads per kv head (GQA group) */
#define MK_MAX_CALL_SEQS 256 /* sequences per call */
#define MK_MAX_SPLITS 64     /* split-T work items per (sequence, kv head) */
#define MK_MAX_META_CHANNELS 48 /* channels a compressed per-block key may keep */

typedef enum mk_status {
  MK_OK = 0,
  MK_EINVAL = 1,   /* bad argument or configuration */
  MK_ENOMEM = 2,   /* arena/workspace too small, or capacity exceeded */
  MK_ESTATE = 3,   /* call out of order (e.g. attention before a rotation) */
  MK_ECUDA = 4,    /* a CUDA runtime call failed */
  MK_EDEVICE = 5,  /* a kernel set the device error word */
  MK_ETIMEOUT = 6, /* a bounded device-side wait gave up */
  MK_ENOTSUP = 7   /* valid but not supported by the library */
} mk_status;

typedef struct mk_ctx mk_ctx;
typedef void* mk_stream;

/* One middle strategy segment ([S] sec. 4.3: each segment has its own channel
 * retention and sequence retention).  It starts at the first block boundary
 * at or after begin_permille/1000 of the sequence's prefill length (the first
 * segment must start at 0); the last segment is open-ended and receives the
 * tokens appended during decode. */
typedef struct mk_segment {
  int32_t begin_permille; /* 0..1000 */
  int32_t r;              /* channels kept per vector, 1..128 */
  int32_t always;         /* 1: attended in full, never scored; 0: top-k */
  int32_t keep_channels;  /* 0 (= 128) or r..128: the per-vector top-r of the
                             compressed middle picks among the first
                             keep_channels rotated channels only, the bottom
                             ones being truncated ([S] sec. 5.2 truncates the
                             bottom 25%: 96).  Sinks and window stay whole. */
  int32_t elem_group;     /* MK_PAGES_BITMAP only (else 0): this segment's
                             element-group size, 1, 2, 4 or 8 ([S] sec. 4.3:
                             each segment's strategy has its own); 0 takes
                             mk_config.elem_group.  r and keep_channels must be
                             multiples of it.  A segment keeps it when it is
                             re-compressed (mk_swap_segment). */
  int32_t retain_permille; /* 0, or 1..1000 for a scored segment: its own
                             sequence retention ([S] sec. 4.3).  When any scored
                             segment gives one, each scored segment keeps its
                             own ceil(rate * n / 1000) best blocks (n: its blocks
                             present; clamped to [1, n]; rate: its own, else
                             mk_config.retain_permille), ties to the lower id,
                             and the ids of all segments come in ascending order
                             in one row; mk_config.topk_fixed must then be 0.
                             Must be 0 for an always-attended segment. */
} mk_segment;

typedef struct mk_config {
  int32_t head_dim;        /* must be 128 */
  int32_t n_q_heads;       /* query heads per layer */
  int32_t n_kv_heads;      /* kv heads per layer; n_q_heads/n_kv_heads <= 8 */
  int32_t n_layers;
  int32_t max_seqs;        /* sequence slots, <= MK_MAX_CALL_SEQS */
  int32_t max_tokens;      /* capacity per sequence (every layer) */
  int32_t n_sink;          /* S >= 0 */
  int32_t window;          /* W >= 1 */
  int32_t block;           /* B: 16, 32 or 64 tokens */
  int32_t topk_fixed;      /* > 0: keep min(topk_fixed, n) scored blocks */
  int32_t retain_permille; /* else keep ceil(retain*n/1000), clamped to [1, n] */
  int32_t n_segments;      /* 1..MK_MAX_SEGMENTS */
  mk_segment seg[MK_MAX_SEGMENTS];
  int32_t meta_channels;   /* 0: full per-block keys (min and max over all 128
                              channels).  1..MK_MAX_META_CHANNELS: the keys are
                              channel-compressed too ([S] sec. 5.2): each block
                              keeps the meta_channels channels with the largest
                              bound magnitude max(|min|, |max|), ties to the
                              lower channel, and the scores use those only (the
                              others count as zero). */
  int32_t page_format;     /* MK_PAGES_PACKED (0): the method's per-vector top-r
                              pages.  MK_PAGES_DENSE (1): the Quest comparator
                              ([S] sec. 6.1 baselines, sec. 6.3): middle blocks
                              keep every channel (page = [K bf16 B x 128][V bf16
                              B x 128]) and only the token-block selection
                              applies; every segment must then have r = 128,
                              keep_channels 0, and meta_channels must be 0.
                              Block min/max, scores, top-k and attention are the
                              same calls; with an identity rotation this is
                              Quest's page selection on the raw keys.
                              MK_PAGES_BITMAP (2): the packed format of [S]
                              sec. 5.1 with a position bitmap per vector in
                              place of the uint8 indices (see elem_group). */
  int32_t elem_group;      /* MK_PAGES_BITMAP only (else 0): the element-group
                              size g of the segments that give none, 1, 2, 4 or
                              8 (0 means 1).  Each vector
                              stores a bitmap of 128/g bits, bit j set when
                              channels g*j .. g*j+g-1 are kept (bit j in byte
                              j/8 at bit j%8), followed by nothing else: the
                              values stay r bf16 in ascending channel order.
                              g = 1 keeps the per-vector top-r of [N] Eq. (9);
                              g > 1 keeps the r/g groups with the largest
                              energy (sum of squares over the group's channels,
                              in fp32, summed in channel order), ties to the
                              lower group ([S] sec. 5.1 variable-granularity
                              bitmap, [S] sec. 4.3 element-group size).  Every
                              segment's r and nonzero keep_channels must be
                              multiples of its g. */
} mk_config;

#define MK_PAGES_PACKED 0
#define MK_PAGES_DENSE 1
#define MK_PAGES_BITMAP 2

/* Byte offsets of one (layer, sequence, kv head) inside the arena, for tests
 * and tools.  Pages: block b lives at pages + b*page_stride and holds
 * [K values B*r bf16][K positions][V values B*r bf16][V positions], r being
 * the block's segment r and the positions B*r u8 channel indices
 * (MK_PAGES_PACKED) or B bitmaps of 16/g bytes (MK_PAGES_BITMAP); token slot
 * t of the block uses row t. */
typedef struct mk_layout_info {
  int64_t rkt, rvt, rv;      /* fp32 [128][128]: R_k^T, R_v^T, R_v */
  int64_t sink_k, sink_v;    /* bf16 [S][128], rotated */
  int64_t win_k, win_v;      /* bf16 [W][128], ring: position p at slot (p-S) mod W */
  int64_t meta;              /* bf16 [nblk_cap][2][128]: per-block min, max */
  int64_t pages;             /* packed pages */
  int64_t page_stride;       /* bytes between consecutive blocks' pages */
  int32_t nblk_cap;
  int32_t T;                 /* current length (host view) */
  int32_t seg_first_block[MK_MAX_SEGMENTS];
  int32_t n_segments;
  int32_t reserved;
  int64_t cmeta;             /* compressed per-block keys (meta_channels > 0):
                                [nblk_cap] rows of cmeta_row bytes, each
                                [min bf16 x m][max bf16 x m][channel u8 x m],
                                m = meta_channels, channels ascending */
  int32_t cmeta_row;
  int32_t meta_channels;
} mk_layout_info;

/* Sizes of the caller-owned buffers for a configuration. */
mk_status mk_arena_bytes(const mk_config* cfg, size_t* bytes);
mk_status mk_workspace_bytes(const mk_config* cfg, size_t* bytes);
/* Row length of the ids buffer of mk_block_select: the largest k any call
 * can return under this configuration. */
mk_status mk_max_select(const mk_config* cfg, int32_t* k_max);

/* Creates a context over a caller-owned arena and workspace (device memory
 * of at least the sizes above, 256-byte aligned).  Zeroes the sequence
 * state; synchronises the device once.  The buffers must outlive the
 * context. */
mk_status mk_create(const mk_config* cfg, void* arena, size_t arena_bytes,
                    void* workspace, size_t workspace_bytes, mk_ctx** out);
mk_status mk_destroy(mk_ctx* ctx);

/* Installs the rotations of one (layer, seq, kv head): R_k and R_v are d x d
 * row-major fp32 host arrays whose rows are the eigenvectors of K^T K (resp.
 * V^T V) by descending eigenvalue, so that k' = k R_k^T ([N] Eq. (4), (6)-(8))
 * and output = o' R_v ([N] Eq. (14)).  Computing them (host eigensolver, once
 * per head at prefill) is the caller's job, as on the pages.  Copies the data
 * before returning.  Must precede the first append of that head. */
mk_status mk_set_rotation(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head,
                          const float* Rk_host, const float* Rv_host, mk_stream stream);

/* Appends n_new[i] tokens to sequence seq_ids[i] of `layer`, for every kv
 * head: rotates each new k, v into its head's basis (fp32 accumulation,
 * rounded to bf16), stores sink and window tokens dense, and compresses each
 * token leaving the window: per-vector top-r channels by magnitude, ties to
 * the lower channel, stored in ascending channel order ([N] Eq. (9),
 * Algorithm 1; [S] sec. 4.2, 5.1), plus the block's min/max keys.
 * k, v: device bf16 [sum(n_new)][n_kv_heads][128], sequences in call order,
 * 16-byte aligned when any n_new[i] exceeds 16 (the bulk path, whose rotation
 * of 128-token tiles runs as a tensor-core GEMM, reads 16-byte vectors).
 * The first append of a sequence is its prefill: it fixes the strategy
 * segments.  seq_ids/n_new are host arrays; n_new[i] >= 0.
 * Errors: MK_ENOMEM if a sequence would pass max_tokens; MK_ESTATE if a
 * rotation is missing; MK_EINVAL for bad ids, duplicates or misaligned k, v. */
mk_status mk_append_compress(mk_ctx* ctx, int32_t layer, int32_t n_seqs,
                             const int32_t* seq_ids, const int32_t* n_new,
                             const void* k, const void* v, mk_stream stream);

/* The decode step's append and block selection in one launch: appends one
 * new token to each listed sequence (as mk_append_compress with n_new = 1)
 * and then selects its blocks for the query q (as mk_block_select), with the
 * same results as those two calls in a row.  k, v: device bf16
 * [n_seqs][n_kv_heads][128] (one row per sequence, in call order); q, ids,
 * n_sel, scores as for mk_block_select.  Every sequence must hold its prefill
 * already.  One kernel does both: the append of each (sequence, kv head) runs
 * in the CTA that scores the blocks its evicted token can change.  This is
 * not a step of the pages' method, only a fusion of two of its steps.
 * Errors: those of the two calls it replaces. */
mk_status mk_append_select(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                           const void* k, const void* v, const void* q, int32_t* ids,
                           int32_t* n_sel, float* scores, mk_stream stream);

/* Scores every middle block of each (sequence, kv head) from its min/max
 * keys and the rotated query q' = q R_k^T:
 *   s_b = max_h (1/sqrt(d)) sum_j max(q'_hj mn_bj, q'_hj mx_bj)
 * (Quest-style bound on [N] Eq. (12)), over the group's query heads h, and
 * keeps the top-k blocks of the scored segments ([S] sec. 4.2 stage 2),
 * ties to the lower id, ids ascending.
 * q: device bf16 [n_seqs][n_q_heads][128].  ids: device int32
 * [n_seqs][n_kv_heads][k_max] (mk_max_select); n_sel: device int32
 * [n_seqs][n_kv_heads].  scores: optional device fp32
 * [n_seqs][n_kv_heads][nblk_cap] (NULL to skip).  Also stores q' in the
 * workspace for the following mk_decode_attn of the same layer. */
mk_status mk_block_select(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                          const void* q, int32_t* ids, int32_t* n_sel, float* scores,
                          mk_stream stream);

/* PackedAttention ([N] Eq. (13), (14); [S] sec. 5.3): for each query head,
 * softmax attention of q' over the sink tokens, the window, the tokens of the
 * selected blocks and of the always-attended segments, read straight from the
 * packed pages; then output = o' R_v.  Uses the q' of the last
 * mk_block_select (or mk_append_select) of the same layer, kept in the
 * workspace per layer, whose sequence list must equal this call's: MK_ESTATE
 * otherwise.  ids/n_sel: as written by that call.  out: device bf16
 * [n_seqs][n_q_heads][128]. */
mk_status mk_decode_attn(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                         const int32_t* ids, const int32_t* n_sel, void* out, mk_stream stream);

/* Uncompressed decode attention of our own, the roofline and speedup
 * reference ([N] Eq. (1)): out = softmax(q K^T / sqrt(d)) V over
 * K, V: device bf16 [n_seqs][n_kv_heads][t_stride][128], the first T[i]
 * tokens of sequence i (T: host int32, 1 <= T[i] <= t_stride).  Uses the
 * context's workspace and its head counts.  q, K, V and out must be 16-byte
 * aligned (K and V rows move by bulk copies): MK_EINVAL otherwise. */
mk_status mk_dense_decode_attn(mk_ctx* ctx, int32_t n_seqs, const int32_t* T,
                               const void* q, const void* K, const void* V, int64_t t_stride,
                               void* out, mk_stream stream);

/* Allocation-free variant of mk_dense_decode_attn.  The paper has no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory at the point where they run attention (a plugin inside a host
 * framework whose enqueue step forbids allocation, a serving runtime with a
 * fixed memory plan, a process whose allocator belongs to someone else) and
 * therefore cannot provide a context's workspace.  It takes only inputs and
 * outputs and needs no context: q [n_seqs][n_q_heads][128], K, V
 * [n_seqs][n_kv_heads][t_stride][128] (bf16, device), T host int32
 * [n_seqs] with 1 <= T[i] <= t_stride, out [n_seqs][n_q_heads][128] bf16;
 * q, K, V and out 16-byte aligned (MK_EINVAL otherwise, before any launch).
 * Its scratch (split-T partials, counters, error word) is one static device
 * array of MK_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds
 * until the process exits (about 4.3 MB).  Calls with
 * n_seqs * n_q_heads > MK_NOALLOC_MAX_QUERY_HEADS return MK_ENOMEM before
 * anything is launched.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.  Every call shares the
 * array and clears what must start at zero; calls that overlap on the GPU
 * (different streams without ordering) race on it and give wrong results.
 * The return value covers host-side checks and the launch only.  A failure
 * found on the device (a bounded wait for a copy that ran out) is recorded in
 * the array's error word, which calls do not clear: from then on every call
 * on that device leaves its output untouched until mk_noalloc_poll_error
 * reports and clears the failure. */
#define MK_NOALLOC_SCRATCH_BYTES 4456448
#define MK_NOALLOC_MAX_QUERY_HEADS 128
mk_status mk_dense_decode_attn_noalloc(int32_t n_q_heads, int32_t n_kv_heads, int32_t n_seqs,
                                       const int32_t* T, const void* q, const void* K, const void* V,
                                       int64_t t_stride, void* out, mk_stream stream);
/* Device-side status of mk_dense_decode_attn_noalloc on the current device:
 * waits for the whole device, then returns MK_OK, or MK_ETIMEOUT / MK_EDEVICE
 * with the kernel's detail code in *detail (optional), and clears the error
 * word so later calls run again.  Allocates nothing; no context needed. */
mk_status mk_noalloc_poll_error(int32_t* detail);

/* Set-up helper, not on the decode path: gram = X^T X (fp32 accumulation)
 * for X: device bf16 rows of 128 values, row i at x + i*row_stride elements
 * (x 16-byte aligned, row_stride a multiple of 8).
 * gram: device fp32 [128][128], overwritten. */
mk_status mk_gram(const void* x, int64_t n_rows, int64_t row_stride, float* gram, mk_stream stream);

/* ---- Host-side strategy generation (host memory only; no device, no context) ----
 * The CPU part of the method: the covariance a head accumulates, the
 * rotation from its eigenvectors ([N] Eq. (4), (6)), the channel count that
 * keeps the discarded energy under a loss threshold ([N] Eq. (5); [S] sec.
 * 5.5, channel parameters chosen under a loss threshold), and the per-segment
 * channel count of [N] Algorithm 2 (Eq. (10)-(11)).  All arithmetic is fp64.
 * These calls touch no GPU and may run on any thread, concurrently with the
 * decode calls. */

/* G += sum over the n rows x of x^T x.  G: d x d row-major doubles (the
 * caller's accumulator, updated in place); x: n rows of d bf16 words, row i
 * at x + i * row_stride words.  MK_EINVAL: null pointer, d < 1 or n < 0. */
mk_status mk_cov_update(double* G, const void* x, int64_t n, int64_t row_stride, int32_t d);

/* Eigen-decomposition of the symmetric d x d matrix G (row-major doubles) by
 * cyclic Jacobi rotations: lambda[i] in descending order, R (d x d floats,
 * row-major) with row i the unit eigenvector of lambda[i], so R is the
 * rotation mk_set_rotation takes (k' = k R^T).  Eigenvectors are unique up to
 * sign (and, for repeated eigenvalues, up to a rotation of their subspace).
 * MK_EINVAL: null pointer, d < 1, or G not symmetric (relative 1e-12);
 * MK_ETIMEOUT: no convergence within 100 sweeps (R and lambda still hold the
 * last iterate). */
mk_status mk_rotation_from_cov(const double* G, int32_t d, float* R, double* lambda);

/* Smallest r in [1, d] whose discarded energy sum_{i>=r} lambda_i /
 * sum_i lambda_i (lambda descending, [N] Eq. (5): 1 - Energy(r)) is at most
 * loss_max.  A zero spectrum gives r = 1; eigenvalues down to -1e-9 lambda_0
 * (roundoff) count as zero.  MK_EINVAL: null pointer, d < 1, loss_max < 0, a
 * lambda below -1e-9 lambda_0, or lambda not descending (same tolerance). */
mk_status mk_choose_r(const double* lambda, int32_t d, double loss_max, int32_t* r);

/* [N] Algorithm 2 for one rotated segment of s vectors of d channels. */
typedef struct mk_alg2_params {
  double outlier_abs;       /* |x| above this counts as an outlier element */
  double outlier_ratio_max; /* above this outlier ratio the segment is compressed harder */
  double alpha;             /* strength of the adjustment */
  int32_t r_min, r_max;     /* clamp of the result */
  int32_t hist_bins;        /* bins of the magnitude histogram (entropy) */
} mk_alg2_params;
typedef struct mk_seg_stats {
  double variance;      /* mean over channels of the channel's population variance */
  double outlier_ratio; /* #{|x| > outlier_abs} / (s d) */
  double entropy;       /* -sum p ln p over the magnitude histogram (natural log) */
} mk_seg_stats;
/* seg: s rows of d bf16 words (row stride row_stride words), already
 * rotated; budget: the segment's element budget R_budget.  With
 * u = outlier_ratio, r = budget/s * (1 - alpha u) if u > outlier_ratio_max,
 * else budget/s * (1 + alpha (1 - u)); clamped to [r_min, r_max] and rounded
 * down.  The histogram has hist_bins equal bins over [0, max |x|] (a value
 * equal to the maximum goes to the last bin; all-zero data fill bin 0).
 * stats may be NULL.  MK_EINVAL: null seg or r, s < 1, d < 1, hist_bins < 1,
 * r_min < 1, r_max < r_min, budget < 0. */
mk_status mk_alg2_segment_r(const void* seg, int64_t s, int64_t row_stride, int32_t d, double budget,
                            const mk_alg2_params* params, mk_seg_stats* stats, int32_t* r);

/* Block-size choice of [S] sec. 5.5 (block sizes chosen under a variance
 * threshold) for one segment of s vectors of d channels (seg: s rows of d
 * bf16 words, row stride row_stride words; rotated or not: the statistic
 * does not change under a rotation of the channels).  For each candidate B
 * the segment is cut into its complete blocks of B consecutive vectors; the
 * candidate's within-block variance is the mean over those blocks of the mean
 * over channels of each channel's population variance inside the block
 * (Algorithm 2's variance, per block).  *block receives the largest candidate
 * whose within-block variance is at most threshold, else the smallest
 * candidate.  within_var (optional, n_cands doubles, in the order given)
 * receives each candidate's statistic, NaN for a candidate with no complete
 * block (which never qualifies).  fp64 throughout.  MK_EINVAL: null seg or
 * block or cands, s < 1, d < 1, row_stride < d, n_cands outside [1, 16], a
 * candidate < 1 or repeated, threshold negative or NaN. */
mk_status mk_choose_block_size(const void* seg, int64_t s, int64_t row_stride, int32_t d, const int32_t* cands,
                               int32_t n_cands, double threshold, double* within_var, int32_t* block);

/* ---- Double-buffered re-compression of a closed segment ([S] sec. 5.4) ----
 * While decoding goes on with the GPU's compression of a segment, the CPU
 * re-compresses the segment's tokens exactly (fp64 rotation, rounded once to
 * bf16), possibly under a new strategy (channel count r, truncation), and the
 * result replaces the GPU's version in the arena, stream-ordered and without
 * blocking the host.  The segment may keep the head's rotation or take its
 * own (the per-segment SVD of [N] Fig. 4). */

/* Packs n_blocks complete blocks of `block` tokens on the host, in the
 * arena's formats.  k, v: the blocks' raw (unrotated) bf16 rows, row i at
 * k + i * row_stride words; R_k, R_v: the head's rotations (as given to
 * mk_set_rotation).  Each token is rotated in fp64 (k' = k R^T) and rounded
 * to nearest-even bf16; its top-r over the first keep_channels channels
 * (0 = all) is kept as in mk_append_compress, in groups of elem_group
 * channels for the bitmap format.  Outputs, all host memory: pages (n_blocks
 * x page_stride bytes: [K values B*r bf16][K positions][V values][V
 * positions], the positions being B*r u8 indices for MK_PAGES_PACKED or B
 * bitmaps of 16/g bytes for MK_PAGES_BITMAP, the rest zero), meta (n_blocks
 * x 2 x 128 bf16: per-channel min and max of the zero-filled compressed
 * keys), and, with meta_channels > 0, cmeta (n_blocks rows of ((5
 * meta_channels + 15) / 16) * 16 bytes, the compressed block keys).
 * MK_EINVAL: a null pointer, block not 16, 32 or 64, page_format not
 * MK_PAGES_PACKED or MK_PAGES_BITMAP, elem_group not as mk_config states, r
 * outside [1, 128], keep_channels outside {0} u [r, 128], r or keep_channels
 * not a multiple of g, page_stride below the page's size, meta_channels
 * outside [0, 48]. */
mk_status mk_host_pack_blocks(const float* R_k, const float* R_v, const void* k, const void* v, int64_t row_stride,
                              int32_t n_blocks, int32_t block, int32_t r, int32_t keep_channels, int64_t page_stride,
                              int32_t meta_channels, int32_t page_format, int32_t elem_group, void* pages, void* meta,
                              void* cmeta);

/* Replaces strategy segment `segment` of one (layer, sequence, kv head) with
 * pages, meta (and cmeta) packed by mk_host_pack_blocks for all of its blocks
 * (mk_layout gives the segment's first blocks), under channel count r and
 * truncation keep_channels from then on.  R_k, R_v: NULL when the pages were
 * packed with the head's rotations; else the segment's own rotations (host
 * fp32 [128][128], rows = eigenvectors of the segment's own K^T K and V^T V by
 * descending eigenvalue, the per-segment SVD of [N] Fig. 4), which the pages
 * were packed with: from then on the segment's blocks are scored with the
 * query rotated by its R_k and their weighted values un-rotated by its R_v.
 * The rotations are copied before the call returns (from pageable memory,
 * after the stream's earlier work); the pages, meta and cmeta copies and the
 * descriptor update are enqueued on `stream`, and those host buffers must stay
 * valid until they run (pinned memory makes the copies asynchronous).  The
 * segment must be closed: not the last one, which still receives appends.  r
 * may not exceed the largest r of the configuration (the page capacity).
 * The pages' positions are checked on the host before any copy: every uint8
 * index below 128, every bitmap row with exactly r/g bits set.
 * MK_EINVAL: bad ids, a null buffer, only one of R_k and R_v, r or
 * keep_channels out of range or not multiples of the element group, a
 * position outside those rules; MK_ESTATE:
 * the sequence has no prefill yet, or
 * the segment is the last or empty; MK_ENOTSUP: uncompressed pages. */
mk_status mk_swap_segment(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, int32_t segment, int32_t r,
                          int32_t keep_channels, const float* R_k, const float* R_v, const void* pages,
                          const void* meta, const void* cmeta, mk_stream stream);

/* Waits for the device and reads the sticky error word: MK_OK, MK_EDEVICE or
 * MK_ETIMEOUT; *detail (optional) receives the kernel's detail code. */
mk_status mk_poll_error(mk_ctx* ctx, int32_t* detail);
/* Clears the device error word and the workspace's arrival counters and key
 * histograms, which a kernel that gave up may have left part-way
 * (synchronising). */
mk_status mk_clear_error(mk_ctx* ctx);
/* Re-reads every sequence length from the device into the host view (needed
 * after replaying a captured CUDA graph of appends).  Synchronises. */
mk_status mk_sync_state(mk_ctx* ctx);
mk_status mk_seq_length(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t* T);
mk_status mk_layout(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, mk_layout_info* out);
const char* mk_status_str(mk_status s);

/* Measurement helper, not a step of the method: records `event` (a
 * cudaEvent_t created by the caller with timing enabled) on `stream`.  While
 * the stream is being captured into a CUDA graph the record becomes an
 * event-record node of the graph, so kernel durations can be timed inside
 * graph replays. */
mk_status mk_record_event(void* event, mk_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* MOSAICKV_H */
