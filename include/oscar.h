/*
 * oscar.h -- C ABI of liboscar: OSCAR INT2 KV-cache decode attention for
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes (cited by page title and section):
 *
 *  [News]     "Together AI 开源 OSCAR：一种面向长上下文 LLM 服务的注意力感知
 *              2 位 KV 缓存量化系统"
 *  [Blog]     "超越TurboQuant：Together AI把2-bit KV Cache推向真实服务"
 *  [Telegram] "OSCAR: открытая система двухбитного сжатия KV-кэша"
 *
 *  - Each request's KV cache has three regions: the first 64 tokens (sink) in
 *    BF16, the newest 256 tokens (recent window) in BF16, and every token in
 *    between (history) in INT2 after rotation and clipping [News, section
 *    "服务系统：混合精度缓存布局"; Telegram, paragraph on the first 64 / last
 *    256 tokens].
 *  - The rotation is R_K = U_Q·H·P_br for keys and R_V = U_S·H·P_br for values,
 *    per layer and per KV head (U: eigenvectors of the query covariance /
 *    score-weighted value covariance, H: normalised Sylvester Hadamard, P_br:
 *    bit-reversal permutation) [News, section "OSCAR 的不同之处"; Blog, section
 *    "OSCAR把旋转对准attention"].
 *  - A new token is written to the recent window; the oldest recent token is
 *    rotated, clipped, quantised (asymmetric INT2 with an fp16 scale and zero
 *    point per group) and packed 4 codes per byte into history.  Decoding runs
 *    the INT2 segment and the BF16 segments separately and merges them by
 *    online softmax [Blog, pipeline figure "从离线校准到在线推理的pipeline" and
 *    the paragraph under it].
 *
 * Conventions
 *  - Every call returns an oscar_status; no exception crosses the ABI.
 *  - Device pointers are raw CUDA device addresses; host pointers are marked
 *    "host".  BF16 and FP16 data are passed as their 16-bit patterns (void*).
 *    All arrays are dense, row-major, and must be 16-byte aligned.
 *  - The per-step operands of the append and decode calls (k_new, v_new, q,
 *    out, lse) may also be pinned host memory (cudaHostAlloc, or
 *    cudaHostRegister'ed), passed by its host address: with unified addressing
 *    the kernels read and write it in place over the host link (NVLink-C2C on
 *    Grace), with no copy call.  Results written there are complete once the
 *    stream has been synchronised.  Pools, page tables, windows, lengths and
 *    scratch must be device memory.
 *  - Calls that take a stream are asynchronous on that stream (NULL = legacy
 *    default stream).  Argument errors are detected on the host and reported
 *    before anything is launched.  Errors found by a kernel (a page-table
 *    entry that is -1 or out of range, a window overflow, a scale out of the
 *    kernel's range, a wait that timed out) are written to a per-context
 *    device error word; kernels never trap.  oscar_get_error reads it.
 *  - Tracing: each call that launches device work runs inside an NVTX range
 *    named after the call (NVTX 3, header-only: free unless a tool attaches).
 *  - Ownership: the caller allocates and owns every device buffer it passes
 *    (page pools, page tables, windows, lengths, q, out, scratch).  The
 *    context owns only its rotation tables and its error word, which
 *    oscar_destroy frees.
 *  - Fixed shape: head_dim = 128, page_size = 64, sink = 64, recent = 256.
 *    group_size is 32, 64 or 128; num_q_heads / num_kv_heads is 1, 2, 4 or 8.
 *
 * Page layouts (one pool per layer; a page holds the same 64 history token
 * slots for every KV head):
 *  INT2 page  = num_kv_heads blocks, one per KV head, each
 *     [K codes 64 x 32 B][V codes 128 x 16 B][K s/z 64 x (128/g) x 4 B]
 *     [V s/z 64 x (128/g) x 4 B]
 *   = 4608 B per head at g = 128, 5120 B at g = 64, 6144 B at g = 32.
 *   A code at bit position b of a little-endian 32-bit word sits in byte b/8
 *   at bits b%8 and b%8+1.
 *   K codes are token-major: 8 words per token.  Rotated channel
 *     c = 64A + 16B + 8C + 2D + E is stored in word 2D + A at bit 16E + 2(2B + C).
 *   V codes are channel-major: 4 words per rotated channel per page.  Token
 *     slot t = 16S + 8A + 2T + E is stored in word T at bit 16E + 2(2S + A).
 *   s/z: one (scale, zero) fp16 pair per token and group, scale first.
 *   Groups are g consecutive rotated channels.  Dequantisation: x' = code*s + z.
 *  BF16 page (baseline history) = num_kv_heads blocks of
 *     [K 64 x 128 bf16][V 64 x 128 bf16] = 32768 B per head.
 *  Windows: sink_k/sink_v bf16 [max_batch][num_kv_heads][64][128];
 *           ring_k/ring_v bf16 [max_batch][num_kv_heads][256][128];
 *  absolute position p of request b lives in sink[p] (p < 64), in history
 *  slot p - 64 (64 <= p < 64 + hist_lens[b]) or in ring slot (p - 64) % 256.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSCAR_HEAD_DIM 128
#define OSCAR_PAGE_SIZE 64
#define OSCAR_SINK_TOKENS 64
#define OSCAR_RECENT_TOKENS 256

/* Same type as cudaStream_t. */
typedef struct CUstream_st* oscar_stream_t;

typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer     */
  OSCAR_ERR_UNSUPPORTED = 2, /* head_dim != 128, group size or GQA ratio      */
  OSCAR_ERR_NO_PAGE = 3,     /* device: page-table entry is -1                */
  OSCAR_ERR_RANGE = 4,       /* device: page id, length or scale out of range */
  OSCAR_ERR_TIMEOUT = 5,     /* device: a bounded wait ran out                */
  OSCAR_ERR_CUDA = 6,        /* a CUDA runtime call failed                    */
  OSCAR_ERR_STATE = 7,       /* device: cache state does not allow the call   */
  OSCAR_ERR_TOO_LARGE = 8    /* request needs more than the built-in scratch  */
} oscar_status;

typedef enum {
  OSCAR_ROT_OSCAR = 0,    /* R = U·H·P_br                          */
  OSCAR_ROT_HADAMARD = 1, /* R = H (Hadamard-only baseline)        */
  OSCAR_ROT_NONE = 2      /* R = I (naive INT2)                    */
} oscar_rot_mode;

/* INT2 history decode kernels (the BF16-history baseline has one kernel). */
typedef enum {
  OSCAR_DECODE_TENSOR = 0,        /* tensor cores; with at most 4 query heads per kv head a warp
                                     takes two pages per tile as two softmax streams (default) */
  OSCAR_DECODE_CUDA_CORE = 1,     /* fp32 CUDA cores, one page per warp at a time */
  OSCAR_DECODE_TENSOR_SINGLE = 2, /* tensor cores, one page per tile at any group size */
  OSCAR_DECODE_TCGEN05 = 3        /* tcgen05.mma with the codes unpacked into tensor memory:
                                     warp-specialised, one CTA per SM, 128-token tiles, an even
                                     static split of the work over the SMs */
} oscar_decode_impl;
/* (A layer with a Lloyd-Max codebook, oscar_set_codebook, always decodes with
 * the codebook kernel: tensor cores, one page per tile.) */

/* Prefill attention kernels (oscar_prefill). */
typedef enum {
  OSCAR_PREFILL_TCGEN05 = 0, /* tcgen05.mma, S/P/O in tensor memory, warp-specialised (default) */
  OSCAR_PREFILL_MMA_SYNC = 1 /* mma.sync, eight warps share each dequantised page */
} oscar_prefill_impl;

typedef enum {
  OSCAR_OPT_DECODE_IMPL = 0, /* an oscar_decode_impl value (default OSCAR_DECODE_TENSOR) */
  OSCAR_OPT_CTAS_PER_SM = 1, /* persistent decode CTAs per SM, 1..4 (default 4), capped by occupancy */
  OSCAR_OPT_ITEMS_PER_CTA = 2, /* work items per decode CTA the scheduler aims for, 1..8, or 0
                                  (default): automatic -- one item per CTA while items stay small,
                                  else up to 4 per CTA of at least 28 pages, balanced at run time */
  OSCAR_OPT_PREFILL_IMPL = 3, /* an oscar_prefill_impl value (default OSCAR_PREFILL_TCGEN05) */
  OSCAR_OPT_WAIT_POLLS = 4,    /* iteration budget of the first wait for each history page of the
                                  mma.sync and CUDA-core decode kernels (default 4194304 polls).
                                  A wait that runs out records OSCAR_ERR_TIMEOUT; the kernel then
                                  waits, with the full budget, for the copies it has in flight and
                                  leaves.  0 makes every such wait give up at once: a way to
                                  exercise that path.  Values < 0 are OSCAR_ERR_INVALID_ARG. */
  OSCAR_OPT_DECODE_PARTITION = 5 /* how the mma.sync and CUDA-core decode kernels split the work:
                                    0 (default) automatic -- balanced when the call has at least
                                    16 (request, kv head) pairs, or when a CTA would get more than
                                    96 history pages of the item list (40 for the BF16-history
                                    decode), else the item list; 1 the
                                    item list (OSCAR_OPT_ITEMS_PER_CTA); 2 balanced: CTA i takes an
                                    equal share of all history pages and window chunks, in order.
                                    The outputs do not depend on the partition beyond rounding. */
} oscar_option;

typedef struct {
  int num_layers;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;          /* must be 128 */
  int group_size;        /* 32, 64 or 128 */
  int page_size;         /* must be 64 */
  int sink_tokens;       /* must be 64 */
  int recent_tokens;     /* must be 256 */
  int max_batch;         /* largest batch any call will pass */
  int max_pages_per_req; /* row length of every page table */
  int num_pages;         /* pages in each layer's pool */
} oscar_config;

typedef struct {
  size_t int2_head_bytes;   /* one KV head's block in an INT2 page          */
  size_t int2_page_bytes;   /* whole INT2 page (num_kv_heads blocks)        */
  size_t off_k_codes;       /* offsets inside a head block                  */
  size_t off_v_codes;
  size_t off_k_sz;
  size_t off_v_sz;
  size_t bf16_head_bytes;   /* one KV head's block in a BF16 page (32768)   */
  size_t bf16_page_bytes;
  size_t sink_bytes;        /* bytes of sink_k (or sink_v) at max_batch     */
  size_t ring_bytes;        /* bytes of ring_k (or ring_v) at max_batch     */
  size_t decode_scratch_bytes; /* scratch oscar_decode* needs at max_batch  */
  size_t prefill_scratch_bytes; /* scratch oscar_prefill needs, any batch up to
                                   max_batch and any chunk up to 64 tokens  */
} oscar_layout_info;

/* One layer's cache.  Every pointer is a device pointer owned by the caller.
 * seq_lens[b] = tokens cached for request b; hist_lens[b] = how many of them
 * are in INT2 history.  Both are read and updated by the kernels, so each
 * layer needs its own pair of arrays. */
typedef struct {
  void* pool;              /* INT2 pool (or BF16 pool for the baseline calls) */
  const int32_t* page_table; /* [max_batch][max_pages_per_req]; -1 = no page */
  void* sink_k;
  void* sink_v;
  void* ring_k;
  void* ring_v;
  int32_t* seq_lens;       /* [max_batch] */
  int32_t* hist_lens;      /* [max_batch] */
} oscar_cache;

typedef struct oscar_ctx oscar_ctx;

/* Library version (major*10000 + minor*100 + patch). */
int oscar_version(void);

/* Static text for a status code. */
const char* oscar_status_string(int status);

/* Sizes and offsets of every buffer for a configuration.  Host only; needs
 * no GPU.  Returns OSCAR_ERR_UNSUPPORTED / OSCAR_ERR_INVALID_ARG for
 * configurations the kernels do not support. */
oscar_status oscar_layout(const oscar_config* cfg, oscar_layout_info* out);

/* Create a context on the current CUDA device: validates cfg, allocates the
 * rotation tables (identity rotation, clip 1.0 for every layer and head) and
 * the error word.  *out receives the context. */
oscar_status oscar_create(const oscar_config* cfg, oscar_ctx** out);

/* Free a context and everything it owns.  Synchronises the device first. */
oscar_status oscar_destroy(oscar_ctx* ctx);

/* Set a tuning option (oscar_option).  Host only. */
oscar_status oscar_set_option(oscar_ctx* ctx, int option, int value);

/* Load one layer's rotation and clip ratios [News, "OSCAR 的不同之处";
 * Blog, "OSCAR把旋转对准attention": fixed per layer and head after offline
 * calibration].
 *   U_K, U_V : host float [num_kv_heads][128][128], row-major; column i is
 *              the i-th eigenvector (descending eigenvalue).  The rotation
 *              applied is x' = x·U·H·P_br (OSCAR mode).  Ignored (may be NULL)
 *              in HADAMARD and NONE modes.
 *   clip_k, clip_v : host float [num_kv_heads], ratios in (0, 1].
 *   rot_mode : oscar_rot_mode.
 * R = U·H·P_br (or H, or I) is composed on the host in double precision and
 * stored in fp32; every kernel applies it as one 128x128 product, so the
 * demotion, the bulk import and oscar_debug_rotate share one arithmetic.
 * Copies host memory on `stream` and synchronises it before returning. */
oscar_status oscar_set_rotation(oscar_ctx* ctx, int layer, const float* U_K,
                                const float* U_V, const float* clip_k,
                                const float* clip_v, int rot_mode,
                                oscar_stream_t stream);

/* Append one token per request [Blog, pipeline figure paragraph]: for each
 * b < batch and KV head, if the recent window already holds 256 tokens, its
 * oldest token is first rotated, clipped, quantised and packed into history
 * slot hist_lens[b] (page page_table[b][slot/64], row slot%64; hist_lens[b]
 * += 1); then the new token is written to sink[L] (L < 64) or ring slot
 * (L - 64) % 256, and seq_lens[b] += 1.
 *   k_new, v_new : device bf16 [batch][num_kv_heads][128].
 * Device errors: OSCAR_ERR_NO_PAGE if the history page is -1,
 * OSCAR_ERR_RANGE if the page id is >= num_pages or the slot is beyond
 * max_pages_per_req; the request is then left unchanged. */
oscar_status oscar_append(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                          const void* k_new, const void* v_new, int batch,
                          oscar_stream_t stream);

/* Demote the oldest recent token of every request into history without
 * appending (the window shrinks by one).  Requests with an empty window are
 * left unchanged. */
oscar_status oscar_demote(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                          int batch, oscar_stream_t stream);

/* Bulk import of n tokens into empty requests (seq_lens[b] must be 0):
 * the same cache state as n appends.  K, V: device bf16 [batch][num_kv_heads]
 * [n][128].  Device error OSCAR_ERR_STATE if a request is not empty. */
oscar_status oscar_import_tokens(oscar_ctx* ctx, int layer,
                                 const oscar_cache* cache, const void* K,
                                 const void* V, int batch, int n,
                                 oscar_stream_t stream);

/* Decode attention for one new query token per request over the three
 * regions [Blog, pipeline figure paragraph: INT2 kernel unpack + scale/zero
 * dequantisation + float accumulation, BF16 kernel for sink/recent, online
 * softmax merge].  q' = q·R_K is formed on the device; the history partial
 * is un-rotated by R_V^T before the merge.
 *   q   : device bf16 [batch][num_q_heads][128]
 *   out : device bf16 [batch][num_q_heads][128]
 *   lse : device float [batch][num_q_heads] natural-log log-sum-exp of the
 *         scaled logits, or NULL
 *   scratch : device buffer of at least decode_scratch_bytes
 *             (oscar_layout) bytes, 256-byte aligned; no initial contents
 *             needed; not to be shared by calls that may overlap.
 * Requests with seq_lens[b] == 0 produce zeros and lse = -inf. */
oscar_status oscar_decode(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                          const void* q, void* out, float* lse, void* scratch,
                          size_t scratch_bytes, int batch,
                          oscar_stream_t stream);

/* One decode step of one layer: exactly oscar_append(k_new, v_new) followed by
 * oscar_decode(q) on `stream` (the new token takes part in the attention),
 * as the pages' serving loop runs them each step [Blog, pipeline figure
 * paragraph: the new token is written to the recent window, the oldest one
 * demoted, then attention over sink, INT2 history and recent window].  The
 * query rotation does not depend on the append, so the library runs the two
 * side by side in one kernel instead of one after the other.  Arguments,
 * layouts, ownership and errors are those of the two calls; k_new, v_new and q
 * must all be complete when the call's work starts on `stream`. */
oscar_status oscar_decode_step(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                               const void* k_new, const void* v_new, const void* q, void* out,
                               float* lse, void* scratch, size_t scratch_bytes, int batch,
                               oscar_stream_t stream);

/* Chunked prefill over the cache (prefix-hit extension) [News,
 * "服务系统：混合精度缓存布局": the mixed-precision layout serves prefix-cache
 * reuse; Blog, pipeline figure paragraph: attention over sink, INT2 history
 * and recent window].  For each b < batch, the T new tokens of request b
 * attend to the request's cache as it stands (BF16 sink and recent window;
 * the INT2 history with q' = q·R_K, its output un-rotated by R_V^T) and
 * causally to the chunk itself: chunk token t sees chunk tokens 0..t.  One
 * softmax over all of them per (token, query head).  The chunk is NOT stored:
 * append it afterwards (oscar_append per token, or oscar_import_tokens into an
 * empty request) if it is to stay in the cache.
 *   q   : device bf16 [batch][T][num_q_heads][128]
 *   k, v: device bf16 [batch][T][num_kv_heads][128], the chunk's keys and values
 *   T   : 1..64 tokens per request (the same for every request of the call)
 *   out : device bf16 [batch][T][num_q_heads][128]
 *   lse : device float [batch][T][num_q_heads] natural-log log-sum-exp of the
 *         scaled logits, or NULL
 *   scratch : device buffer of at least prefill_scratch_bytes (oscar_layout)
 *             bytes, 256-byte aligned, no initial contents needed; not to be
 *             shared by calls that may overlap.
 * q, k, v, out 16-byte aligned.  Returns OSCAR_ERR_INVALID_ARG for T outside
 * 1..64.  On a layer with a non-uniform Lloyd-Max codebook
 * (oscar_set_codebook) the mma.sync kernel runs whatever OSCAR_OPT_PREFILL_IMPL
 * says, dequantising s·level(code) + z.  Device errors as oscar_decode (OSCAR_ERR_NO_PAGE / OSCAR_ERR_RANGE
 * for a bad history page, whose tokens are then left out). */
oscar_status oscar_prefill(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* q,
                           const void* k, const void* v, int T, void* out, float* lse,
                           void* scratch, size_t scratch_bytes, int batch,
                           oscar_stream_t stream);

/* Offline calibration on the GPU for one (layer, kv head) [News, "OSCAR 的不同之处":
 * keys are rotated into the eigenbasis of the query covariance
 * C_Q = (1/N) Σ qᵀq, values into that of C_S = (1/N) VᵀSᵀSV with S the
 * attention scores; Blog, "OSCAR把旋转对准attention": fixed offline per layer
 * and head].  From N calibration tokens:
 *   C_Q = (1/(G N)) Σ_h Σ_n q_{h,n}ᵀ q_{h,n}   (the G query heads of the kv head pooled)
 *   C_S = (1/(G N)) Σ_h (S_h V)ᵀ (S_h V),  S_h = causal softmax(Q_h Kᵀ / √d)
 * and their eigenvectors (cuSOLVER dsyevd in fp64; the library opens cuSOLVER
 * at the first call and returns OSCAR_ERR_UNSUPPORTED if it cannot).
 *   Q : device bf16 [G][N][128], G = num_q_heads / num_kv_heads
 *   K, V : device bf16 [N][128]
 *   U_K, U_V : host float [128][128] out, row-major, column i = eigenvector of
 *              the i-th largest eigenvalue of C_Q (C_S), signed so that its
 *              largest-magnitude entry (lowest index on ties) is positive: the
 *              U_K / U_V that oscar_set_rotation takes
 *   C_Q, C_S : host double [128][128] out, or NULL
 *   scratch : device, at least oscar_calibration_scratch_bytes(G, N, 0) bytes,
 *             256-byte aligned.
 * Synchronises `stream`.  Allocates cuSOLVER's workspace (this call is
 * offline; the decode path allocates nothing). */
size_t oscar_calibration_scratch_bytes(int G, int N, int M);
oscar_status oscar_calibrate(oscar_ctx* ctx, const void* Q, const void* K, const void* V, int N,
                             float* U_K, float* U_V, double* C_Q, double* C_S, void* scratch,
                             size_t scratch_bytes, oscar_stream_t stream);

/* Clip search for one (layer, kv head) with the rotation loaded by
 * oscar_set_rotation [Blog, "OSCAR把旋转对准attention": clipping thresholds are
 * fixed offline].  For each candidate ratio c_m the calibration keys and values
 * are rotated (x' = x·R, fp32) and quantised and dequantised by the
 * demotion's quantiser at ratio c_m, and the error left in what attention
 * computes is measured (the library's reading; the pages name no objective):
 *   err_k[m] = ||Q' K'ᵀ - Q' K̂'ᵀ||²_F, Q' = Q·R_K over the G heads' queries
 *              (computed as Σ_n e_n (Q'ᵀQ') e_nᵀ, e_n = k'_n - k̂'_n)
 *   err_v[m] = Σ_h ||S_h (V' - V̂')||²_F, S_h the causal scores of head h
 * best_k, best_v = the index of the smallest error (first on ties).
 *   Q, K, V as in oscar_calibrate; ratios : host float [M] in (0, 1], M >= 1;
 *   err_k, err_v : host double [M] out; best_k, best_v : host int out (or NULL);
 *   scratch : at least oscar_calibration_scratch_bytes(G, N, M) bytes.
 * Synchronises `stream`. */
oscar_status oscar_clip_errors(oscar_ctx* ctx, int layer, int kv_head, const void* Q, const void* K,
                               const void* V, int N, const float* ratios, int M, double* err_k,
                               double* err_v, int* best_k, int* best_v, void* scratch,
                               size_t scratch_bytes, oscar_stream_t stream);

/* Lloyd-Max codebook [Blog, closing paragraph on TurboQuant: the released
 * code pairs the attention-aware rotation with a Lloyd-Max codebook; the
 * pages give no formula, so the following is the library's reading].
 * A group keeps the uniform quantiser's fp16 scale s and zero point z and its
 * normalised value t = (x - z)/s (fp32); only the four values t is rounded to
 * change.  They are symmetric about 1.5,
 *   level(code) = {1.5 - b, 1.5 - a, 1.5 + a, 1.5 + b},  0 <= a < b <= 3,
 * and x_hat = level(code)·s + z.  A code is the nearest level, ties to the
 * even code: code = [t > 1.5 - m] + [t >= 1.5] + [t > 1.5 + m], m = (a + b)/2
 * in fp32.  (a, b) = (0.5, 1.5) is the uniform quantiser exactly. */
#define OSCAR_CODEBOOK_MAX_ROWS (1 << 20)

/* Sets the codebooks of one layer, per kv head, for keys and for values:
 *   k_ab, v_ab : host float [num_kv_heads][2] = (a, b) pairs, or NULL for the
 *                uniform levels (0.5, 1.5) on that side.
 * From then on the demotion, the bulk import, oscar_clip_errors and the decode
 * of this layer use them.  While any head of the layer has a non-uniform
 * codebook the decode runs the codebook kernel (two tensor-core products per
 * operand, whatever OSCAR_OPT_DECODE_IMPL says) and oscar_prefill runs its
 * mma.sync kernel.  Codes already in the cache are not
 * re-quantised: set the codebook before the layer's tokens are written.
 * OSCAR_ERR_INVALID_ARG if a pair is outside 0 <= a < b <= 3 or not finite
 * (nothing is changed then).  Synchronises `stream`. */
oscar_status oscar_set_codebook(oscar_ctx* ctx, int layer, const float* k_ab, const float* v_ab,
                                oscar_stream_t stream);

/* Fits the codebook of one (layer, kv head) for keys (which = 0) or values
 * (which = 1) by Lloyd-Max: the N calibration rows are rotated by the layer's
 * R_K or R_V (x' = x·R, fp32) and every group is normalised to t at the
 * head's clip ratio (groups with a zero scale are left out); with the folded
 * value f = |t - 1.5| the two levels alternate between a = mean of f <= m and
 * b = mean of f > m, m = (a + b)/2 (fp64), from (0.5, 1.5) until the inner
 * cell's count repeats or max_iters updates ran.  The layer's codebook is not
 * changed (pass the result to oscar_set_codebook; b above 3 is refused there).
 *   X : device bf16 [N][128], 1 <= N <= OSCAR_CODEBOOK_MAX_ROWS
 *   scratch : device, 256-byte aligned, at least oscar_codebook_scratch_bytes(N)
 *   ab : host float [2] out = (a, b);  updates : host int out (or NULL), the
 *        number of centroid updates.
 * Synchronises `stream`. */
size_t oscar_codebook_scratch_bytes(int N);
oscar_status oscar_fit_codebook(oscar_ctx* ctx, int layer, int kv_head, int which, const void* X, int N,
                                int max_iters, void* scratch, size_t scratch_bytes, float* ab, int* updates,
                                oscar_stream_t stream);

/* Test hook: the demotion's quantiser with codebook (a, b) on given rotated
 * fp32 vectors; arguments and layouts as oscar_quantize_rotated_f32. */
oscar_status oscar_quantize_codebook_f32(const float* x, int n, int group_size, float clip, float a, float b,
                                         int which, uint8_t* codes, void* sz, oscar_stream_t stream);

/* Decode without any device allocation (the pages have no counterpart: this
 * is a deployment convenience of this library).  Same computation, arguments
 * and results as oscar_decode, but the working memory comes from a buffer of
 * OSCAR_NOALLOC_SCRATCH_BYTES that the library itself holds in device memory,
 * so the caller passes no scratch.  It is meant for callers that cannot or
 * must not call cudaMalloc on the decode path: engines that reserve (nearly)
 * all device memory for their KV pools at start-up and forbid later
 * allocations so that serving can never fail for lack of memory, code paths
 * where an allocation would block on or synchronise with other work on the
 * device, and plain C callers with no device allocator of their own.
 *  - Every GPU that loads the library holds this buffer until the process
 *    exits, whether or not the call is used.
 *  - The context's device must be the current device
 *    (OSCAR_ERR_INVALID_ARG otherwise).  The first call on each device looks
 *    up the buffer's device address once and keeps it; make that first call
 *    before any stream capture begins.  The kept address belongs to the
 *    device's primary context: after a device reset it is stale, so do not
 *    call this entry point again in that process.
 *  - All calls share the one buffer and it keeps the last call's contents.
 *    The kernels reset everything that must start at zero themselves.  Calls
 *    that may run at the same time on the GPU (different streams, different
 *    host threads) race on it: serialise them.
 *  - Returns OSCAR_ERR_TOO_LARGE, launching nothing, if the request's working
 *    memory (decode_scratch_bytes for `batch` at the context's current
 *    options) exceeds OSCAR_NOALLOC_SCRATCH_BYTES.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define OSCAR_NOALLOC_SCRATCH_BYTES (8u << 20)
oscar_status oscar_decode_noalloc(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                                  const void* q, void* out, float* lse, int batch,
                                  oscar_stream_t stream);

/* Baseline with the same split-K design, over a BF16 history pool (no
 * rotation, no quantisation): the comparison point for the speedup the
 * pages report against BF16 KV [News, "结果"; Blog, paragraph after
 * "精度只是第一关"].  Same arguments as oscar_decode; cache->pool is a
 * BF16 pool. */
oscar_status oscar_decode_bf16_history(oscar_ctx* ctx, const oscar_cache* cache,
                                       const void* q, void* out, float* lse,
                                       void* scratch, size_t scratch_bytes,
                                       int batch, oscar_stream_t stream);

/* Bulk import of n tokens into empty requests of a BF16-history cache
 * (history stored unrotated in bf16).  Arguments as oscar_import_tokens. */
oscar_status oscar_import_bf16_history(oscar_ctx* ctx, const oscar_cache* cache,
                                       const void* K, const void* V, int batch,
                                       int n, oscar_stream_t stream);

/* One token per request appended to a BF16-history cache (cache->pool a BF16
 * pool; the baseline's counterpart of oscar_append, no rotation and no
 * quantisation): if the recent window holds 256 tokens, its oldest token
 * (ring slot hist_lens[b] % 256) is first copied into history slot
 * hist_lens[b] (hist_lens[b] += 1); then the new token is written to sink[L]
 * (L < 64) or ring slot (L - 64) % 256, and seq_lens[b] += 1.
 *   k_new, v_new : device bf16 [batch][num_kv_heads][128].
 * Device errors: OSCAR_ERR_NO_PAGE / OSCAR_ERR_RANGE for a missing or bad
 * history page; the request is then left unchanged. */
oscar_status oscar_append_bf16_history(oscar_ctx* ctx, const oscar_cache* cache, const void* k_new,
                                       const void* v_new, int batch, oscar_stream_t stream);

/* Test hook: the demotion's quantiser and packer on given rotated fp32
 * vectors, so that codes and bytes can be compared bit for bit.
 *   x : device float [n][128] rotated channels
 *   which = 0: codes -> device uint8 [n][32] K rows (K layout);
 *   which = 1: codes -> device uint8 [n/64][2048] V blocks (token i in slot
 *              i%64 of block i/64); n must be a multiple of 64.
 *   sz : device fp16 pairs [n][128/group_size][2] (scale, zero). */
oscar_status oscar_quantize_rotated_f32(const float* x, int n, int group_size,
                                        float clip, int which, uint8_t* codes,
                                        void* sz, oscar_stream_t stream);

/* Test hook: rotate n bf16 vectors of one KV head with the layer's R_K
 * (which = 0) or R_V (which = 1): x_rot = x·R.  x: device bf16 [n][128];
 * x_rot: device float [n][128]. */
oscar_status oscar_debug_rotate(oscar_ctx* ctx, int layer, int which,
                                int kv_head, const void* x, float* x_rot,
                                int n, oscar_stream_t stream);

/* Debug aid: checks host copies of a cache's lengths and page table against
 * the configuration, without touching the device.  For every request b < batch:
 *   max(L - 320, 0) <= H <= max(L - 64, 0), L = seq_lens[b], H = hist_lens[b]
 *   (the recent window holds 0..256 tokens), ceil(H / 64) <= max_pages_per_req,
 *   and each of its first ceil(H / 64) page-table entries is in [0, num_pages)
 *   and used by no other history slot of the batch.
 *   seq_lens, hist_lens : host int32 [batch]
 *   page_table : host int32 [batch][max_pages_per_req]
 *   bad_request : host int out (or NULL), the first failing request, -1 if none.
 * Returns OSCAR_OK, OSCAR_ERR_STATE (lengths), OSCAR_ERR_NO_PAGE (a -1 entry)
 * or OSCAR_ERR_RANGE (an id out of range, shared, or too many pages). */
oscar_status oscar_check_cache_host(const oscar_config* cfg, const int32_t* seq_lens, const int32_t* hist_lens,
                                    const int32_t* page_table, int batch, int* bad_request);

/* Synchronise `stream`, return the first device-side error recorded since
 * the last call in *code (OSCAR_OK if none) and clear it. */
oscar_status oscar_get_error(oscar_ctx* ctx, oscar_stream_t stream, int* code);

/* The CUDA runtime error code (a cudaError_t value) behind the most recent
 * OSCAR_ERR_CUDA returned to the calling host thread, 0 if there was none.
 * The pages describe no error reporting; this is the library's own. */
int oscar_last_cuda_error(void);

/* Kernel timing (tracing).  The pages describe no profiler; this is the
 * library's own instrumentation.  While enabled, every kernel the context
 * launches is bracketed by a pair of CUDA events recorded on the launching
 * stream (at most 65536 launches are kept).  oscar_profile_read waits for the
 * recorded events, returns for kernel `kernel_id` (oscar_kernel) the number
 * of launches and their summed device time in milliseconds, and with
 * reset != 0 forgets everything recorded so far. */
typedef enum {
  OSCAR_KERNEL_APPEND = 0,      /* append / demote                      */
  OSCAR_KERNEL_IMPORT = 1,      /* all bulk-import kernels              */
  OSCAR_KERNEL_DECODE_PREP = 2, /* q rotation, work-counter reset       */
  OSCAR_KERNEL_DECODE_MAIN = 3, /* split-K decode over history + window */
  OSCAR_KERNEL_DECODE_MERGE = 4,/* partial merge + un-rotation          */
  OSCAR_KERNEL_STEP = 5,        /* oscar_decode_step's append + q rotation */
  OSCAR_KERNEL_PREFILL_PREP = 6,  /* prefill: q rotation and scaling       */
  OSCAR_KERNEL_PREFILL_ATTN = 7,  /* prefill: split attention over regions */
  OSCAR_KERNEL_PREFILL_MERGE = 8, /* prefill: split merge + un-rotation    */
  OSCAR_KERNEL_COUNT = 9
} oscar_kernel;

oscar_status oscar_profile_enable(oscar_ctx* ctx, int enable);
oscar_status oscar_profile_read(oscar_ctx* ctx, int kernel_id, int* launches,
                                double* total_ms, int reset);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
