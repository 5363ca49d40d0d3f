/*
 * cacheblend.h — C ABI of the GB300 (sm_103a) selective-KV-recompute library.
 *
 * The library fuses key/value caches that were precomputed for each document chunk in
 * isolation into one long-context prefill, recomputing only the tokens whose KV deviates
 * most (CacheBlend).  Sources cited below by short tag:
 *   [CB-A] "論文解説: CacheBlend — RAGシステム向けKV Cache融合による高速LLMサービング"
 *          (0h-n0.github.io/posts/paper-2312-03052)
 *   [CB-B] CacheBlend explainer, abeam.tech (2026-09-20-cacheblend-rag-cached-knowledge-fusion)
 *   [PC]   "論文解説: Prompt Cache — モジュラーAttention再利用による低レイテンシ推論"
 *          (0h-n0.github.io/posts/paper-2402-01008)
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Memory: the caller allocates every device buffer; the library allocates nothing on
 *    the call path.  Scratch comes from a caller-provided device workspace whose size
 *    cb_workspace_bytes() returns.  Pointers named *_host are host memory; all others
 *    are device memory.  The library never frees caller memory.
 *  - Alignment: device buffers start on a 16-byte boundary (cudaMalloc and the PyTorch
 *    allocator return 256-byte aligned blocks); the kernels move rows in 16- and 32-byte
 *    vectors.  A misaligned buffer is refused with CB_ERR_INVALID_ARG before any launch.
 *    Exceptions: cb_gather_rows and cb_scatter_kv need 4 bytes, 8-bit codes 8 bytes, and
 *    arrays of row indices, positions or scores 4 bytes.
 *  - Streams: every call takes a cudaStream_t (passed as void*, NULL = legacy default
 *    stream), enqueues its kernels on it and returns without synchronising, unless the
 *    description says otherwise.
 *  - Errors: an int status.  All argument checks run on the host before any launch, so a
 *    call that returns an error has enqueued nothing.  Kernels that detect bad data at run
 *    time (a non-finite deviation score, an index out of range) set a sticky device error
 *    word that cb_sync() returns; they never trap.
 *  - Row indices: every call that takes a device array of row indices also takes the row
 *    count of the buffer they index (n_*_rows).  An index outside [0, that count) is not
 *    followed: the kernel skips that row (its output row is left unwritten), records the
 *    error and cb_sync() returns CB_ERR_DEVICE.
 *  - Layout: row-major, token-major.  A K or V cache is [n_rows, n_kv_heads * head_dim]
 *    (heads contiguous inside a row).  Hidden rows are [n, d_model].  Weights are stored
 *    output-major, [out_features, in_features], so a projection is y = x W^T.
 *  - Positions: in a blended sequence the row index is the token's position.  RoPE pairs
 *    are interleaved (x[2i], x[2i+1]) and rotate by pos * theta_i, theta_i =
 *    base^(-2i/head_dim) ([CB-A] §RoPE).  A cos/sin table built by cb_rope_table() is
 *    passed to every call that rotates.
 *  - Element type: dims->dtype (CB_F32 or CB_BF16) applies to every floating tensor of a
 *    call except where a parameter says float (fp32); arithmetic is fp32 in both.
 */
#ifndef CACHEBLEND_H
#define CACHEBLEND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------- */
#define CB_OK               0
#define CB_ERR_INVALID_ARG  1   /* null pointer, negative size, bad enum               */
#define CB_ERR_SHAPE        2   /* sizes inconsistent with each other or the dims      */
#define CB_ERR_DTYPE        3   /* unsupported element type                            */
#define CB_ERR_WORKSPACE    4   /* workspace smaller than cb_workspace_bytes() asks    */
#define CB_ERR_NONFINITE    5   /* NaN/Inf deviation score (reported by cb_sync)       */
#define CB_ERR_CUDA         6   /* a CUDA runtime/driver call failed                   */
#define CB_ERR_TIMEOUT      7   /* cb_sync waited longer than its limit                */
#define CB_ERR_UNSUPPORTED  8   /* a shape the kernels do not handle (see message)     */
#define CB_ERR_DEVICE       9   /* a kernel recorded an out-of-range index             */
#define CB_ERR_IO          10   /* a storage read failed (cb_io_error_message says why) */

#define CB_F32   0
#define CB_BF16  1

#define CB_DEV_KV  0   /* deviation over K and V                                     */
#define CB_DEV_K   1   /* deviation over K only (the page's select_hkvd_tokens code)  */

#define CB_LAYER_PRECHECK 0   /* layer before the check layer: every row            */
#define CB_LAYER_CHECK    1   /* HKVD selection over all cached rows                 */
#define CB_LAYER_STEADY   2   /* reuse the incoming row set (fixed mode)             */
#define CB_LAYER_GRADUAL  3   /* re-select inside the incoming row set               */

typedef struct {
    int32_t d_model;      /* d                                                       */
    int32_t n_heads;      /* H  query heads                                          */
    int32_t n_kv_heads;   /* Hkv  (GQA: H % Hkv == 0; query head h reads h / (H/Hkv)) */
    int32_t head_dim;     /* hd (even)                                               */
    int32_t d_ff;         /* F  SwiGLU width                                         */
    int32_t vocab;        /* lm_head rows                                            */
    double  rope_base;    /* RoPE base (1e4 Llama, 5e6 Yi)                           */
    float   rms_eps;      /* RMSNorm epsilon                                         */
    int32_t dtype;        /* CB_F32 or CB_BF16                                       */
} cb_dims;

/* One decoder layer's weights (device, dims->dtype).  Pre-norm Llama layer, no biases.
 * attn_norm / ffn_norm may be NULL: unit gains (a caller with other gains may fold them
 * into the columns of wqkv / w_gate_up and pass NULL).  With a NULL ffn_norm the bf16 path
 * folds the FFN norm into the GEMMs: the O-projection's epilogue leaves each row's partial
 * sums of squares and the gate/up GEMM scales its rows by 1/rms in its epilogue. */
typedef struct {
    const void* attn_norm;   /* [d]                                                 */
    const void* wqkv;        /* [(H + 2 Hkv) hd, d]: rows of Wq, then Wk, then Wv    */
    const void* wo;          /* [d, H hd]                                           */
    const void* ffn_norm;    /* [d]                                                 */
    const void* w_gate_up;   /* [2F, d]: rows 0..F-1 gate, rows F..2F-1 up           */
    const void* w_down;      /* [d, F]                                              */
} cb_layer_w;

/* ---- housekeeping ----------------------------------------------------------------- */

/* Human-readable text for a status code (static storage). */
const char* cb_status_string(int status);

/* Detail of the last error raised on the calling thread (static, thread-local). */
const char* cb_last_error_message(void);

/* The last failing CUDA runtime call on the calling thread (the one behind the latest
 * CB_ERR_CUDA): error name, text and the call; "" if there has been none.  Static,
 * thread-local. */
const char* cb_last_cuda_error(void);

/* Waits for `stream` (polling, up to timeout_s seconds; <= 0 means no limit), then reads
 * and clears the sticky device error word.  Returns CB_OK, CB_ERR_TIMEOUT (nothing was
 * cancelled; the work is still queued), CB_ERR_NONFINITE, CB_ERR_DEVICE or CB_ERR_CUDA.
 * The pages' synchronize() ([CB-A] §vLLM integration). */
int cb_sync(void* stream, double timeout_s);

/* Failure-path self test of the device-side bounded waits (every mbarrier wait of the
 * tensor-core kernels is bounded): one tiny kernel waits on an mbarrier that is completed
 * (arrive != 0) or that nothing completes.  In the second case the wait gives up after
 * max_polls (1..2^20) tries, records the timeout in the device error word and returns;
 * the next cb_sync reports CB_ERR_DEVICE ("bounded wait expired") and the context stays
 * usable.  No trap, no hang. */
int cb_selftest_wait(int32_t max_polls, int32_t arrive, void* stream);

/* Releases the library's host-side per-device state: the cached SM counts, occupancy and
 * CTA-pair figures, the kernels' shared-memory attribute flags, the allocation-free entry
 * point's cached scratch address, and the calling thread's profiler events.  Every later
 * call rebuilds what it needs, so the library stays usable.  Call it with no library work
 * in flight (after cb_sync on every stream that ran library calls), e.g. before the
 * process resets its device context.  Frees no caller memory. */
void cb_shutdown(void);

/* Device workspace (bytes) large enough for every call below on rows up to n_tok and a
 * selected set of up to m_max rows, for these dims.  Host-only. */
int cb_workspace_bytes(const cb_dims* dims, int64_t n_tok, int64_t m_max, size_t* out_host);

/* HKVD budget: k = floor(n_cached * ratio) in double, at least 1 when ratio > 0, 0 when
 * ratio == 0, at most n_cand ([CB-A] §HKVD selection code: max(int(N*r), 1)).
 * Host-only.  Returns k, or -1 for a ratio outside [0, 1] or a negative size. */
int64_t cb_hkvd_budget(int64_t n_cached, double ratio, int64_t n_cand);

/* Gradual-filtering ratio of `layer`: r_l = r + (r1 - r) 2^-(layer - check_layer),
 * r1 = min(1, r1_factor * r) ([CB-A] §Gradual filtering: r1 slightly above r, r_i
 * approaching r).  Host-only.  Returns -1 for layer < check_layer. */
double cb_gradual_ratio(double r, int32_t layer, int32_t check_layer, double r1_factor);

/* Load-controller ratio r* = max(r_min, T_load / T_prefill) ([CB-A] §Pipelining and load
 * controller).  Host-only. */
double cb_load_controller_ratio(double r_min, double t_load_s, double t_prefill_s);

/* ---- RoPE --------------------------------------------------------------------------- */

/* Fills cos_sin [max_pos][head_dim/2][2] (fp32: cos, sin) with cos/sin(p theta_i) for
 * p in [0, max_pos), the angle formed in fp64 on the device and rounded once
 * ([CB-A] §RoPE rotation matrix R(m)).  Negative rotations use the same table with the
 * sine negated. */
int cb_rope_table(float* cos_sin, int32_t max_pos, int32_t head_dim, double base,
                  void* stream);

/* Re-positions cached keys: k_dst[i] = R(delta[i]) k_src[src_row[i]], and copies values
 * v_dst[i] = v_src[src_row[i]] ([PC] §RoPE position adjustment, k(p) = R(p-p') k(p');
 * [CB-B] position correction when loading chunk KV).
 *   k_src, v_src : [n_src_rows, Hkv hd] source rows (e.g. a pool of precomputed chunk caches)
 *   src_row      : [n_rows] int32 source row per destination row, each in [0, n_src_rows),
 *                  or NULL (row i; then n_src_rows >= n_rows)
 *   delta        : [n_rows] int32 position offset p - p', |delta| < max_pos
 *   k_dst, v_dst : [n_rows, Hkv hd]; v_src/v_dst may both be NULL (keys only).
 * In-place (k_dst == k_src) is allowed only with src_row == NULL.  The sources may be
 * pinned host memory mapped at the same device address (read over the host link, no
 * landing copy); any other host pointer is rejected before launch. */
int cb_rope_shift(void* k_dst, void* v_dst, const void* k_src, const void* v_src,
                  const int32_t* src_row, int64_t n_src_rows, const int32_t* delta,
                  int64_t n_rows, const cb_dims* dims, const float* cos_sin, int32_t max_pos,
                  void* stream);

/* ---- 8-bit chunk KV ([CG] §Step 1 per-channel quantization; entropy coding is not done) */

/* Quantizes one chunk's K (or V) of one layer per channel c (column): z_c = min over the
 * rows, s_c = max((max - z_c) / 255, 1e-8), code = round-half-even((x - z_c) / s_c)
 * clipped to [0, 255]; every step is one IEEE fp32 operation, so the codes are
 * reproducible bit for bit.  A non-finite input sets the device error word.
 *   x : [n_rows, W] of `dtype`;  codes : [n_rows, W] uint8;  scale, zero : [W] fp32. */
int cb_kv_quantize(const void* x, int64_t n_rows, int32_t W, int32_t dtype, uint8_t* codes,
                   float* scale, float* zero, void* stream);

/* cb_rope_shift from an 8-bit chunk store, decoding as it re-positions:
 *   x = code * s + z (fp32 product rounded before the sum), s and z from row qrow[i] of
 *   the per-chunk tables; k_dst[i] = R(delta[i]) x_k[src_row[i]], v_dst[i] = x_v[src_row[i]].
 *   k_codes, v_codes : [n_src_rows, Hkv hd] uint8 (8-byte aligned)
 *   k_scale, k_zero, v_scale, v_zero : [n_qrows, Hkv hd] fp32 (16-byte aligned)
 *   src_row : [n_rows] or NULL (row i);  qrow : [n_rows] in [0, n_qrows)
 *   delta, cos_sin, max_pos as in cb_rope_shift;  v_* all NULL = keys only.
 * Half the bytes of the bf16 store cross the host link and are read by this pass; the
 * codes may be pinned host memory mapped at the same device address (as cb_rope_shift). */
int cb_rope_shift_q8(void* k_dst, void* v_dst, const uint8_t* k_codes, const uint8_t* v_codes,
                     const float* k_scale, const float* k_zero, const float* v_scale,
                     const float* v_zero, const int32_t* src_row, int64_t n_src_rows,
                     const int32_t* qrow, int32_t n_qrows, const int32_t* delta, int64_t n_rows,
                     const cb_dims* dims, const float* cos_sin, int32_t max_pos, void* stream);

/* ---- HKVD selection ----------------------------------------------------------------- */

/* Per-candidate deviation and top-k ([CB-A] §KV deviation; §HKVD selection code):
 *   scores[c] = sum_e (k_new[new_row[c]][e] - k_ref[ref_row[c]][e])^2
 *             (+ the same over V when dev_mode == CB_DEV_KV), fp32 accumulation;
 *   sel       = the k candidates with the largest scores, ties to the lower candidate
 *               index, written ascending as ref_row values (length k).
 *   k_new/v_new : [n_new_rows, Hkv hd] freshly computed rows
 *   k_ref/v_ref : [n_ref_rows, Hkv hd] the cache
 *   new_row/ref_row : [n_cand] int32 ascending row maps into those, or NULL (identity: then
 *                     the buffer holds at least n_cand rows)
 *   scores : [n_cand] fp32 (output, may be NULL)
 * 0 <= k <= n_cand.  A non-finite score sets CB_ERR_NONFINITE (cb_sync). */
int cb_kv_deviation_topk(const void* k_new, const void* v_new, int64_t n_new_rows,
                         const void* k_ref, const void* v_ref, int64_t n_ref_rows,
                         const int32_t* new_row, const int32_t* ref_row, int32_t n_cand,
                         int32_t k, int32_t dev_mode, const cb_dims* dims, float* scores,
                         int32_t* sel, void* ws, size_t ws_bytes, void* stream);

/* Allocation-free variant of cb_kv_deviation_topk, for callers that cannot hand the
 * library device memory: for example a plugin running inside a host program that owns and
 * pre-partitions all device memory, or a latency-critical caller that must not call
 * cudaMalloc (which can synchronise the device).  The pages have no counterpart: this is
 * a deployment convenience, not a step of the method.
 * Same arguments and results as cb_kv_deviation_topk, without the workspace.  Its scratch
 * (a score and an ordinal per candidate) is a fixed 512 KiB array in the library's device
 * memory, held by every GPU that loads the library until the process exits.
 *   - n_cand is limited to 65536; larger returns CB_ERR_UNSUPPORTED before any launch.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current, in the context current then: the device's primary context
 *     for callers of the runtime API) and keeps it until cb_shutdown(); make that first
 *     call before any stream capture, and call cb_shutdown() after resetting the device.
 *   - Every call shares the one array and it keeps the last call's contents: calls that
 *     may overlap on the GPU (different streams, or different host threads, on the same
 *     device) race with each other.  Serialise them. */
int cb_kv_deviation_topk_noalloc(const void* k_new, const void* v_new, int64_t n_new_rows,
                                 const void* k_ref, const void* v_ref, int64_t n_ref_rows,
                                 const int32_t* new_row, const int32_t* ref_row,
                                 int32_t n_cand, int32_t k, int32_t dev_mode,
                                 const cb_dims* dims, float* scores, int32_t* sel,
                                 void* stream);

/* Top-k of given fp32 scores (>= 0, finite), ties to the lower index, output ascending
 * as cand[c] (cand NULL = c).  The selection step alone, for bit-exact checks. */
int cb_topk_from_scores(const float* scores, const int32_t* cand, int32_t n_cand,
                        int32_t k, int32_t* sel, void* ws, size_t ws_bytes, void* stream);

/* ---- row movement ------------------------------------------------------------------- */

/* RMSNorm of rows: out[i] = x[rows[i]] / sqrt(mean(x[rows[i]]^2) + eps) * gain (rows NULL:
 * row i), the pre-norm of every layer ([CB-A] model: RMSNorm before attention and FFN).
 *   x : [n_x_rows, d] of dtype_in;  rows : [n] in [0, n_x_rows), or NULL (n <= n_x_rows)
 *   gain : [d] of dtype_in;  out : [n, d] of dtype_out
 *   (bf16 -> bf16, bf16 -> fp32 or fp32 -> fp32);  d a multiple of 8.  Sums in fp32. */
int cb_rmsnorm(void* out, const void* x, int64_t n_x_rows, const int32_t* rows, int64_t n,
               int32_t d, const void* gain, float eps, int32_t dtype_in, int32_t dtype_out,
               void* stream);

/* dst[i] = src[idx[i]] for i < n; rows of row_bytes bytes (a multiple of 4); src holds
 * n_src_rows rows and every idx[i] must lie in [0, n_src_rows) (e.g. token ids into an
 * embedding table of vocab rows); idx NULL means i ([CB-A] §Selective recomputation,
 * Step 1: restrict the input to S).  dst and src must not overlap (rows are copied in
 * parallel, in no fixed order). */
int cb_gather_rows(void* dst, const void* src, int64_t n_src_rows, const int32_t* idx,
                   int64_t n, int64_t row_bytes, void* stream);

/* KV expansion ([CB-A] §Selective recomputation, Step 3: K_new = Concat(K_pre[not S],
 * K_recomp[S])):  k_cache[dst_idx[i]] = k_rows[src_idx[i]] and the same for V, i < n.
 * Rows are [Hkv hd]; the caches hold n_cache_rows rows, the row buffers n_src_rows rows;
 * dst_idx[i] < n_cache_rows, src_idx[i] < n_src_rows (src_idx NULL means i).  The caches
 * must not overlap the row buffers (rows are copied in parallel, in no fixed order). */
int cb_scatter_kv(void* k_cache, void* v_cache, int64_t n_cache_rows, const void* k_rows,
                  const void* v_rows, int64_t n_src_rows, const int32_t* dst_idx,
                  const int32_t* src_idx, int64_t n, const cb_dims* dims, void* stream);

/* ---- selective layer pieces --------------------------------------------------------- */

/* Q/K/V of selected rows ([CB-A] §Selective recomputation, Step 2; [CB-B] §技術の仕組み):
 *   a = RMSNorm(x[rows[i]]) * attn_norm;  q = a Wq^T, k = a Wk^T, v = a Wv^T;
 *   RoPE on q and k at position pos[i].
 *   x : [n_x_rows, d];  rows : [M] int32 in [0, n_x_rows), or NULL (i; M <= n_x_rows)
 *   pos : [M] int32 (< max_pos);  q : [M, H hd] or NULL;  k, v : [M, Hkv hd] or both NULL. */
int cb_selective_qkv(const void* x, int64_t n_x_rows, const int32_t* rows, const int32_t* pos,
                     int32_t M, const cb_dims* dims, const cb_layer_w* w, const float* cos_sin,
                     int32_t max_pos, void* q, void* k, void* v, void* ws, size_t ws_bytes,
                     void* stream);

/* Selected queries over the whole causal KV ([CB-A] §Selective recomputation, Step 4;
 * [CB-B]: the selected tokens attend over the entire input):
 *   out[j, h] = softmax_t<=q_pos[j]( q[j,h] . k_cache[t, g(h)] / sqrt(hd) ) v_cache[t, g(h)]
 *   q : [M, H hd];  q_pos : [M] int32 causal bound (row index = position), each < n_kv
 *   k_cache, v_cache : [n_kv, Hkv hd];  out : [M, H hd]. */
int cb_partial_attention(const void* q, const int32_t* q_pos, int32_t M,
                         const void* k_cache, const void* v_cache, int64_t n_kv,
                         const cb_dims* dims, void* out, void* ws, size_t ws_bytes,
                         void* stream);

/* O-projection with residual and SwiGLU FFN with residual, on M rows
 * ([CB-A] §Selective recomputation, Step 4, the next layer's input):
 *   h = x_res + attn Wo^T;  y = h + (SiLU(b Wg^T) * (b Wu^T)) Wd^T,  b = RMSNorm(h) g.
 *   attn : [M, H hd];  x_res : [M, d];  x_out : [M, d] (may alias x_res). */
int cb_o_proj_ffn(const void* attn, const void* x_res, int32_t M, const cb_dims* dims,
                  const cb_layer_w* w, void* x_out, void* ws, size_t ws_bytes, void* stream);

/* One layer of the blend ([CB-A] §Selective recomputation Steps 1-4, §HKVD selection,
 * §Gradual filtering).  Rows of the sequence are 0..n_tok-1; rows < n_cached come from
 * chunk caches already re-positioned into k_cache/v_cache ([n_tok, Hkv hd], updated in
 * place); rows >= n_cached are the uncached suffix.  Forced rows F = [n_cached, n_tok)
 * plus row n_tok-1 are always recomputed.
 *   x_in [m_in, d] : hidden rows of the incoming set s_in (ascending, each in [0, n_tok);
 *                    NULL = 0..m_in-1; a row outside is not followed, see Row indices)
 *   mode PRECHECK  : all rows (m_in == n_tok); Q for every row, K/V only for rows
 *                    >= n_cached; output all rows.
 *   mode CHECK     : all rows in; K/V for every row; deviation over the cached,
 *                    unforced rows; S = top-k_budget U F.
 *   mode STEADY    : S = s_in.
 *   mode GRADUAL   : K/V for s_in; deviation over its cached, unforced rows;
 *                    S = top-k_budget U F (a subset of s_in).
 *   For CHECK/STEADY/GRADUAL: K/V of S are written into the cache (Step 3), then Q of S,
 *   attention of S over the cache, O-proj and FFN give x_out [m_out, d] for the rows
 *   s_out [m_out] (ascending).
 *   sel_override : [k_budget] ascending cache rows that replace the top-k choice (the
 *                  forced rows are still added), or NULL.
 *   scores_out   : [n_cand] fp32 deviation scores, or NULL (CHECK/GRADUAL only).  For
 *                  bf16 the squared differences are taken in the K/V GEMM's epilogue as
 *                  the new rows are produced (one fp32 partial per 128 columns, summed in
 *                  column order); fp32 runs the standalone deviation kernel.
 *   m_out_host   : receives m_out (known on the host before any launch: no sync).
 *   opts         : optional extras (NULL = none), see cb_layer_opts.
 * x_out must not alias x_in. */
typedef struct {
  /* Uncached rows anywhere in the request (a system prompt, separators, several query
   * spans): [n_tok] device bytes, nonzero = forced row (recomputed at every layer).  It
   * must mark row n_tok-1; n_forced is its count.  NULL = the default layout (forced
   * rows = [n_cached, n_tok) plus row n_tok-1).  With a mask, n_cached is not used (the
   * caller's k_budget already counts the cached rows), candidates are the unmarked rows
   * of the incoming set, and m_out = k_budget + n_forced. */
  const uint8_t* forced_mask;
  int32_t n_forced;
  /* A cudaEvent_t marking when the cached rows of k_cache/v_cache have been written (e.g.
   * re-positioned on a loading stream), or NULL.  The layer waits for it just before its
   * first access to the cached rows: in PRECHECK after the Q and uncached-row K/V GEMMs,
   * which touch only forced rows, so those overlap the load ([CB-A] §Pipelining). */
  void* kv_ready;
  /* PRECHECK only: nonzero = compute K/V for every row (one Q/K/V GEMM over all rows)
   * instead of reusing the re-positioned cache for the cached rows.  At the pre-check
   * layer the two agree up to rounding (its input is the context-free embedding, R5), so a
   * caller that loads chunk KV over a slow link can skip that layer's load entirely. */
  int32_t recompute_kv;
  /* PRECHECK only, without forced_mask and recompute_kv: 0 = off; r in [1, n_cached] =
   * compute K/V for rows [r, n_tok) (the cached rows from r on and the uncached suffix) and
   * read the cache only for rows [0, r), so that a caller loading chunk KV over a slow link
   * loads only the first r rows of this layer while the GEMMs run (the split that balances
   * the two is the load controller's choice at this layer, [CB-A] §Pipelining and load
   * controller).  kv_ready then marks rows [0, r) only. */
  int32_t recompute_from;
  /* PRECHECK only: input row i is row x_rows[i] (in [0, n_x_rows)) of x_in instead of row i,
   * e.g. x_in = the embedding table [vocab, d] and x_rows = the token ids, so the layer reads
   * the embedding rows in place (no gather of the input rows).  NULL = rows 0..n_tok-1. */
  const int32_t* x_rows;
  int64_t n_x_rows;
  /* CHECK/GRADUAL: a second stream (cudaStream_t) and two events (cudaEvent_t) owned by the
   * caller, all three set or all NULL.  With them the KV expansion of the selected rows (Step
   * 3) runs on aux_stream while the main stream computes the selected rows' queries; the
   * main stream waits for it (aux_join) before attention.  The call forks at aux_fork.  A
   * gradual layer that computes Q for every incoming row in its K/V GEMM has no Q GEMM to
   * overlap and expands on the main stream.  The caller must not use the three concurrently
   * elsewhere. */
  void* aux_stream;
  void* aux_fork;
  void* aux_join;
  /* Row statistics passed from layer to layer, so that the bf16 path with unit attention-norm
   * gains (attn_norm NULL) needs no separate norm pass.
   *   x_out_ssq : caller memory of n_tok * 2 * ceil(d / 192) floats, or NULL.  The call writes
   *     there each x_out row's partial sums of squares (a layout private to the library) and
   *     their count to *x_out_ssq_parts_host (0 when it wrote none: fp32).
   *   x_in_ssq / x_in_ssq_parts : the same from the call that produced x_in (x_in_ssq_parts 0
   *     or NULL x_in_ssq: none).  CHECK, GRADUAL and STEADY then read x_in un-normalised and
   *     scale each row by 1/rms in their Q/K/V GEMMs' epilogues. */
  float* x_out_ssq;
  int32_t* x_out_ssq_parts_host;
  const float* x_in_ssq;
  int32_t x_in_ssq_parts;
} cb_layer_opts;

int cb_blend_layer(const cb_dims* dims, const cb_layer_w* w, int32_t mode,
                   const void* x_in, const int32_t* s_in, int32_t m_in,
                   int64_t n_tok, int64_t n_cached, void* k_cache, void* v_cache,
                   const float* cos_sin, int32_t max_pos, int32_t k_budget, int32_t dev_mode,
                   const int32_t* sel_override, void* x_out, int32_t* s_out,
                   int32_t* m_out_host, float* scores_out, const cb_layer_opts* opts, void* ws,
                   size_t ws_bytes, void* stream);

/* A steady layer (fixed mode, S_l = S_c) of n_req requests at once ([CB-A] §Selective
 * recomputation Steps 2-4 for each request; the batch of independent requests shares the
 * weights).  The selected rows of all requests are one set of GEMM rows, so the Q/K/V,
 * O-projection and FFN GEMMs run once over all of them and read each weight once; attention
 * runs per request over that request's own cache.  Per row the arithmetic is that of
 * cb_blend_layer(STEADY).
 *   row0_host : [n_req + 1] host prefix offsets: request r owns rows [row0[r], row0[r+1])
 *               (row0[0] = 0, non-decreasing, at most n_tok rows per request, n_req <= 64)
 *   x_in  : [row0[n_req], d] hidden rows of every request's selection, request by request
 *   s_in  : [row0[n_req]] each row's position in its request (ascending within a request,
 *           each in [0, n_tok); a row outside is not followed, see Row indices)
 *   k_cache, v_cache : [n_req * n_tok, Hkv hd] the requests' caches of this layer back to back
 *           (request r's row j at r * n_tok + j), updated in place at the selected rows
 *   x_out : [row0[n_req], d] (must not alias x_in).  n_req * n_tok must fit in int32. */
int cb_blend_steady_batch(const cb_dims* dims, const cb_layer_w* w, int32_t n_req,
                          const int32_t* row0_host, const void* x_in, const int32_t* s_in,
                          int64_t n_tok, void* k_cache, void* v_cache, const float* cos_sin,
                          int32_t max_pos, void* x_out, void* ws, size_t ws_bytes, void* stream);

/* Standard causal prefill of n tokens at positions pos0..pos0+n-1 through n_layers
 * layers: the quality reference (KV^full, [CB-A] §KV cache definitions; [CB-B] "full KV
 * recompute") and the per-chunk precompute (KV^pre, pos0 = 0).
 *   layers_host : host array of n_layers cb_layer_w;  embed : [vocab, d]
 *   tokens : [n] int32 device;  k_out_host/v_out_host : host arrays of n_layers device
 *   pointers, each [n, Hkv hd];  h_last : [d] hidden row n-1 after the last layer;
 *   x_all : [n, d] final hidden rows, or NULL. */
int cb_full_prefill(const cb_dims* dims, int32_t n_layers, const cb_layer_w* layers_host,
                    const void* embed, const int32_t* tokens, int32_t n, int32_t pos0,
                    void* const* k_out_host, void* const* v_out_host, void* h_last,
                    void* x_all, const float* cos_sin, int32_t max_pos, void* ws,
                    size_t ws_bytes, void* stream);

/* First answer token: token[0] = argmax_v (RMSNorm(h) final_norm) . w_lm[v], lowest v on
 * ties.  h : [d];  w_lm : [vocab, d];  logits : [vocab] fp32 or NULL;  token : [1] int32
 * device. */
int cb_lmhead_argmax(const void* h, const void* final_norm, const void* w_lm,
                     const cb_dims* dims, float* logits, int32_t* token, void* ws,
                     size_t ws_bytes, void* stream);

/* ---- layer-ahead loading ------------------------------------------------------------ */

/* Starts the copy of one layer's cached chunk KV from pinned host memory to the device on
 * `side_stream` and records `done_event` (a cudaEvent_t) behind it, so the next layer's KV
 * loads while the current layer recomputes ([CB-A] §Pipelining and load controller: layer
 * i+1's KV is fetched during layer i's selective recompute; [CB-B] §ロードと再計算を重ねる).
 * dev_dst and pinned_src must not overlap; bytes may be 0. */
int cb_prefetch_layer(void* dev_dst, const void* pinned_src, size_t bytes, void* side_stream,
                      void* done_event);

/* Stream-ordered copy between any two CUDA-visible buffers (direction from the pointers,
 * e.g. token ids from pinned host memory, the first-token id back to it); capturable in a
 * CUDA graph like every call of this library. */
int cb_copy_async(void* dst, const void* src, size_t bytes, void* stream);

/* Makes `stream` wait (on the device, without blocking the host) for `event`, typically the
 * done_event of cb_prefetch_layer, before its next launch. */
int cb_stream_wait(void* stream, void* event);

/* ---- launch accounting and per-launch timing ---------------------------------------- */

/* Kernel families reported by the profiler. */
#define CB_PROF_ROPE_SHIFT 0
#define CB_PROF_COPY_ROWS  1
#define CB_PROF_RMSNORM    2
#define CB_PROF_GEMM       3
#define CB_PROF_ATTENTION  4
#define CB_PROF_DEVIATION  5
#define CB_PROF_TOPK       6
#define CB_PROF_INDEX      7
#define CB_PROF_LMHEAD     8
#define CB_PROF_ARGMAX     9
#define CB_PROF_ROPE_TABLE 10
#define CB_PROF_QUANT      11

typedef struct {
    int32_t kind;      /* CB_PROF_*                                                     */
    int32_t aux;       /* GEMM: epilogue kind; otherwise 0                              */
    int64_t m, n, k;   /* launch sizes (GEMM: M, N, K; attention: queries, keys, heads) */
    double  flops;     /* algorithmic floating-point operations (0 if not known on host) */
    double  bytes;     /* algorithmic HBM bytes (compulsory reads + writes)             */
    float   ms;        /* device time between events recorded around the launch (-1 in
                        * span mode)                                                    */
    float   span_ms;   /* span mode: from the first CTA past its wait on the preceding
                        * launch to the last CTA's end, from the GPU's global timer; -1
                        * for kernels that do not record spans, and in event mode         */
} cb_prof_record;

/* Number of kernels this library has launched in the process (host-side count). */
int64_t cb_kernel_launch_count(void);

/* Starts recording a CUDA-event pair around every kernel launch made by the calling
 * thread, up to max_records launches.  Not for use while a stream is being captured. */
int cb_profile_begin(int32_t max_records);

/* Starts span profiling for the calling thread, up to max_records launches (at most 8192):
 * no events are recorded between launches, so programmatic dependent launch overlaps them as
 * in an unprofiled run.  Instead each tensor-core GEMM and attention kernel, and the
 * re-positioning (bf16/fp32), multi-row copy and lm_head GEMV kernels, record in their
 * launch's slot of a library-owned device buffer the global-timer time at which its first CTA
 * passed the wait on the preceding launch and the time at which its last CTA finished.  The
 * result is that launch's execution window inside the launch chain.  Synchronises the device.
 * The buffer is the current device's and serves one host thread at a time: while another
 * thread is in span mode the call fails with CB_ERR_INVALID_ARG.  Not for use while a stream
 * is being captured. */
int cb_profile_begin_spans(int32_t max_records);

/* Stops recording (either mode), waits for the recorded events (event mode) or for the
 * device (span mode), writes up to max_records records (host memory) and their count. */
int cb_profile_end(cb_prof_record* out_host, int32_t max_records, int32_t* n_out_host);

/* Plain projection y = x W^T on the same GEMM kernels the layer calls use (tcgen05/TMEM
 * for bf16, exact-fp32 SIMT for fp32); the "Q/K/V transform" primitive of [CB-A]
 * §Selective recomputation Step 2 without an epilogue.  x : [M, K], w : [N, K], y : [M, N],
 * all of element type `dtype`.  bf16 needs N % 16 == 0 and K % 8 == 0; fp32 N % 4 == 0. */
int cb_linear(const void* x, const void* w, void* y, int32_t M, int32_t N, int32_t K, int32_t dtype,
              void* stream);

/* ---- storage tier ---------------------------------------------------------------------- */

/* Reads bytes [offset, offset + bytes) of the file at path into dst_host (typically pinned
 * memory, so a following cb_prefetch_layer streams it to the device), with up to n_threads
 * parallel positional reads of at least 4 MB each: the storage-to-host leg of layer-wise
 * KV loading ([CB-A] §Pipelining and load controller).  Synchronous, host only.  Returns
 * CB_OK or CB_ERR_IO (short file, open/read failure; cb_io_error_message gives the reason,
 * for the calling thread). */
int cb_file_read(const char* path, uint64_t offset, void* dst_host, size_t bytes, int32_t n_threads);
const char* cb_io_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* CACHEBLEND_H */
