/*
 * path_attn.h - C ABI of the GB300 PaTH attention library (libpath_attn.so).
 *
 * PaTH attention ("PaTH Attention: Position Encoding via Accumulating Householder
 * Transformations", summarised on the review page "거리에서 경로로, PaTH Attention"
 * §3-§4 and §9, and on the technical summary "技術要約: PaTH Attention" §2-§3):
 * per token s and head, a transition H_s = I - beta_s w_s w_s^T (w_s unit-norm,
 * beta_s in (0, 2)); query i attends causally to key j with logit
 *     scale * k_j^T (H_{j+1} ... H_i) q_i                      (PaTH)
 *     scale * k_j^T (H_{j+1} ... H_i) q_i + sum_{s=j+1..i} log f_s   (PaTH-FoX)
 * followed by softmax over j <= i and the weighted sum of v_j.
 *
 * Conventions shared by every entry point
 *  - Device pointers, contiguous row-major: q, k, v, w, out are (B, H, L, d);
 *    beta, log_f, lse are (B, H, L) fp32. Element type of q, k, v, w, out and of
 *    the decode caches is given by `dtype` (PATH_F32 or PATH_BF16).
 *  - d must be 64 (the head size the pages benchmark); the forward (path_attn_fwd,
 *    path_fox_fwd, path_fwd_prepare, path_fwd_scan) and the decode steps also take
 *    d = 128 (the larger head the pages mention; the forward then runs on fp32 CUDA-core
 *    kernels for either dtype; the PaTH-FoX scan decides its early exit as it goes).
 *    Anything else returns PATH_ERR_SHAPE.
 *  - Every tensor pointer and the workspace must be 16-byte aligned
 *    (PATH_ERR_ALIGN); the workspace must be 256-byte aligned.
 *  - The caller owns every buffer, the workspace included. The library
 *    allocates no device memory and keeps no state between calls.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Every call is
 *    asynchronous on it; argument checks are synchronous and run before any
 *    launch: on an error nothing is launched and nothing is written.
 *  - Errors detected after launch: PATH_ERR_CUDA (a launch failed; returned by
 *    the call) and PATH_ERR_TIMEOUT (a kernel gave up a bounded wait; read it
 *    with path_check_workspace after the stream has reached the call).
 *  - Empty problems (B, H or L equal to 0; decode with B or H equal to 0) are
 *    valid and launch nothing.
 *  - No C++ exception crosses this interface.
 */
#ifndef PATH_ATTN_H
#define PATH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PATH_OK = 0,
    PATH_ERR_NULL = 1,      /* a required pointer is NULL */
    PATH_ERR_SHAPE = 2,     /* negative size, d != 64, or a size above the limits */
    PATH_ERR_DTYPE = 3,     /* dtype is not PATH_F32 or PATH_BF16 */
    PATH_ERR_ALIGN = 4,     /* a pointer is not 16-byte (workspace: 256-byte) aligned */
    PATH_ERR_WORKSPACE = 5, /* ws_bytes below path_workspace_bytes() */
    PATH_ERR_CAPACITY = 6,  /* decode: cache_len + 1 > cache_cap */
    PATH_ERR_TIMEOUT = 7,   /* a kernel gave up a bounded wait (see path_check_workspace) */
    PATH_ERR_CUDA = 8,      /* a CUDA call failed */
    PATH_ERR_ARG = 9        /* a scalar argument is out of range (e.g. non-finite scale) */
} path_status;

typedef enum { PATH_F32 = 0, PATH_BF16 = 1 } path_dtype;

typedef enum {
    PATH_OP_FWD = 0,
    PATH_OP_FOX_FWD = 1,
    PATH_OP_DECODE = 2,
    PATH_OP_FOX_DECODE = 3,
    PATH_OP_BWD = 4,
    PATH_OP_FOX_BWD = 5
} path_op;

/* Largest sizes accepted: B*H <= PATH_MAX_HEADS, L <= PATH_MAX_LEN. */
#define PATH_MAX_HEADS 65535
#define PATH_MAX_LEN (1 << 22)

/*
 * Workspace bytes that `op` needs for the given sizes (L = cache capacity and d = 64 or
 * 128 for PATH_OP_DECODE and PATH_OP_FOX_DECODE). Returns 0 for invalid arguments. The workspace holds the
 * per-block factors of the forward (boundary-adjusted queries and keys, the
 * dense block transitions, the diagonal-block logits, the FoX prefix sums),
 * the split partial results of decode, or the fp32 factors, per-block gradients
 * and carried query blocks of the backward, plus a 256-byte status header.
 */
size_t path_workspace_bytes(int op, int B, int H, int L, int d, int dtype);

/*
 * PaTH forward: out = softmax_j(scale * k_j^T (H_{j+1}...H_i) q_i) v, causal.
 * Defined in review "거리에서 경로로, PaTH Attention" §3 (the data-dependent transition
 * H_s = I - beta_s w_s w_s^T and the logit through the product of the transitions between
 * key and query) and §4 (softmax attention over those logits); technical summary
 * "技術要約: PaTH Attention" §2 "コアメカニズム". Computed blockwise as in technical
 * summary §3 (UT-form block factors, boundary-adjusted queries and keys, a right-to-left
 * scan with online softmax).
 *   q, k, v, w : (B, H, L, d) dtype      beta : (B, H, L) fp32
 *   out        : (B, H, L, d) dtype      lse  : (B, H, L) fp32, natural-log
 *                                               log-sum-exp of the logits; may be NULL
 *   scale      : softmax scale, any finite value (1/sqrt(d) is the usual one)
 *   ws         : workspace of ws_bytes >= path_workspace_bytes(PATH_OP_FWD, ...)
 * Equivalent to path_fwd_prepare followed by path_fwd_scan on the same stream.
 */
path_status path_attn_fwd(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, void *out, float *lse, int B, int H, int L,
                          int d, int dtype, float scale, void *ws, size_t ws_bytes,
                          void *stream);

/*
 * PaTH-FoX forward: as path_attn_fwd with the additive forget-gate bias
 * sum_{s=j+1..i} log f_s (added after scaling) on every logit.
 *   log_f : (B, H, L) fp32 per-token log forget gate (<= 0 in practice; any finite value)
 * ws must hold path_workspace_bytes(PATH_OP_FOX_FWD, ...).
 * Early exit (exact within rounding): since every H_s is a contraction, a PaTH logit
 * is at most |scale| |q~_i| |k~_j|; the scan of a 128-row tile stops above the key
 * blocks whose every key, bias included, weighs below e^-40 relative to the largest
 * logit of the row's own block (with the bound doubled for rounding). See
 * path_fox_first_blocks. At d = 128 the same bound is tested inside the scan against each
 * row's running maximum before every key block (the scan of a 64-row query block stops once
 * all its rows pass it), and the bias of a key in an earlier block is formed from in-block
 * prefix sums, block totals summed in fp64 and the key's in-block tail sum.
 */
path_status path_fox_fwd(const void *q, const void *k, const void *v, const void *w,
                         const float *beta, const float *log_f, void *out, float *lse,
                         int B, int H, int L, int d, int dtype, float scale, void *ws,
                         size_t ws_bytes, void *stream);

/*
 * First stage of the forward (the per-block UT preprocessing): for every block
 * of 64 tokens it forms the block's compact Householder-product factors and
 * writes into ws the boundary-adjusted queries and keys, the dense block
 * transition and the diagonal-block logits; with log_f (PaTH-FoX; NULL for
 * PaTH) also the prefix sums of log f. Reads q, k, w, beta[, log_f].
 */
path_status path_fwd_prepare(const void *q, const void *k, const void *w, const float *beta,
                             const float *log_f, int B, int H, int L, int d, int dtype,
                             float scale, void *ws, size_t ws_bytes, void *stream);

/*
 * PaTH backward (plain PaTH): gradients of a loss L with respect to q, k, v, w and beta,
 * given dL/d out. The pages give no backward pass (review "거리에서 경로로, PaTH
 * Attention" §9 and technical summary "技術要約: PaTH Attention" §3 only say the blockwise
 * algorithm makes training efficient); this is the chain rule applied to the forward of
 * path_attn_fwd, with the softmax gradient dS_ij = p_ij (d_out_i . v_j - d_out_i . out_i).
 *   q, k, v, w : (B, H, L, d) dtype     beta : (B, H, L) fp32    (the forward's inputs)
 *   out        : (B, H, L, d) dtype     lse  : (B, H, L) fp32    (the forward's outputs)
 *   d_out      : (B, H, L, d) dtype, the gradient of the loss with respect to out
 *   dq, dk, dv, dw : (B, H, L, d) fp32 outputs;  dbeta : (B, H, L) fp32 output
 *   d          : 64 or 128 (other head sizes return PATH_ERR_SHAPE)
 *   scale      : the forward's softmax scale (finite)
 *   ws         : ws_bytes >= path_workspace_bytes(PATH_OP_BWD, B, H, L, d, dtype), which
 *                grows as B H (L / 64)^2 (the query pass keeps every carried query block
 *                and its logit gradient: per block pair 32 KB for fp32 inputs at d = 64,
 *                e.g. 1.0 GB at B H = 64, L = 2048, and 48 KB at d = 128; half of that for
 *                bf16 inputs, which keep them in bf16)
 * Gradients are fp32 whatever dtype is (bf16 inputs are widened on load). bf16 inputs take
 * bf16 tensor-core products with fp32 accumulation in the query pass (tcgen05 at d = 64,
 * warp-level MMAs at d = 128) and tf32 tensor-core products in the block pass; fp32 inputs
 * take fp32 products throughout. w is used as given (no renormalisation). Gradients of several query blocks meet in dv and in
 * internal per-block sums through fp32 atomic adds, so their rounding order (not their
 * value beyond fp32 rounding) varies between runs. Outputs are written from zero: no
 * accumulation into the caller's buffers.
 */
path_status path_attn_bwd(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, const void *out, const float *lse, const void *d_out,
                          int B, int H, int L, int d, int dtype, float scale, float *dq, float *dk,
                          float *dv, float *dw, float *dbeta, void *ws, size_t ws_bytes,
                          void *stream);

/*
 * PaTH-FoX backward: as path_attn_bwd for the forward of path_fox_fwd, plus the gradient of
 * the per-token log forget gate:
 *   log_f  : (B, H, L) fp32, the forward's gate        dlog_f : (B, H, L) fp32 output,
 *            d log f_s = sum over pairs j < s <= i of dS_ij (the bias sum_{s=j+1..i} log f_s
 *            enters logit (i, j) once for every s in that range)
 *   out, lse : the outputs of path_fox_fwd on the same inputs
 *   ws     : ws_bytes >= path_workspace_bytes(PATH_OP_FOX_BWD, B, H, L, d, dtype)
 * Every key block is visited (no early exit): blocks whose weights vanish contribute dS = 0.
 */
path_status path_fox_bwd(const void *q, const void *k, const void *v, const void *w,
                         const float *beta, const float *log_f, const void *out, const float *lse,
                         const void *d_out, int B, int H, int L, int d, int dtype, float scale,
                         float *dq, float *dk, float *dv, float *dw, float *dbeta, float *dlog_f,
                         void *ws, size_t ws_bytes, void *stream);

/*
 * Second stage of the forward: the right-to-left scan over key blocks with
 * online softmax. Reads v and the factors path_fwd_prepare left in ws (which
 * must come from a prepare call with the same sizes, dtype, scale and log_f
 * presence); writes out and lse (may be NULL).
 */
path_status path_fwd_scan(const void *v, void *out, float *lse, int fox, int B, int H, int L,
                          int d, int dtype, float scale, void *ws, size_t ws_bytes,
                          void *stream);

/*
 * PaTH-FoX early-exit extents, for inspection. After path_fwd_prepare with log_f on ws
 * (and until ws is reused), copies asynchronously on `stream`, into the device buffer
 * first_block (B * H * ceil(L / 64) int32, row-major (B, H, L / 64)), for every query
 * block of 64 rows the lowest 64-token key block any of its rows needs; the scan visits
 * key blocks from the tile's own down to the lower of its two query blocks' values.
 * Values lie in [0, query block]. Returns PATH_ERR_WORKSPACE if ws_bytes is below
 * path_workspace_bytes(PATH_OP_FOX_FWD, ...). The pages give no such call: it exposes
 * the rule of review "거리에서 경로로, PaTH Attention" §4 / technical summary
 * "技術要約: PaTH Attention" §2 (the gate makes distant keys vanish) for testing.
 * d = 64 only (the d = 128 scan decides its exit as it runs): other head sizes return
 * PATH_ERR_SHAPE.
 */
path_status path_fox_first_blocks(const void *ws, size_t ws_bytes, int B, int H, int L,
                                  int d, int dtype, int *first_block, void *stream);

/*
 * One PaTH decode step (the inference scheme of review "거리에서 경로로, PaTH Attention"
 * §9 and technical summary "技術要約: PaTH Attention" §3 "推論": the new token's
 * transition updates the cached keys in place, no w/beta cache is kept):
 *   1. k_j <- H_t k_j = k_j - beta_t (w_t . k_j) w_t for every cached j < cache_len,
 *      written back into k_cache (rounded to dtype);
 *   2. k_t, v_t are appended untransformed at index cache_len;
 *   3. out = softmax_j(scale * q_t . k_j) v_j over j <= cache_len.
 *   q, k, v, w : (B, H, d) dtype         beta : (B, H) fp32      d = 64 or 128
 *   k_cache, v_cache : (B, H, cache_cap, d) dtype, updated in place
 *   out : (B, H, d) dtype
 * On return the caches hold cache_len + 1 valid entries; the caller advances its
 * length. Requires cache_len >= 0 and cache_len + 1 <= cache_cap
 * (PATH_ERR_CAPACITY otherwise). Calls on the same caches must be ordered on
 * one stream: each step rewrites every cached key.
 */
path_status path_decode_step(const void *q, const void *k, const void *v, const void *w,
                             const float *beta, void *k_cache, void *v_cache, int B, int H,
                             int cache_len, int cache_cap, int d, int dtype, float scale,
                             void *out, void *ws, size_t ws_bytes, void *stream);

/*
 * One PaTH-FoX decode step: path_decode_step with the forget-gate bias of PaTH-FoX
 * (review "거리에서 경로로, PaTH Attention" §4; technical summary "技術要約: PaTH
 * Attention" §2 "拡張: PaTH-FoX"): the logit of cached key j gains
 * sum_{s=j+1..t} log f_s. The cache keeps that sum per key, updated in place like the
 * keys (review §9; technical summary §3 "推論"):
 *   g_cache : (B, H, cache_cap) fp32. On entry g_cache[j] (j < cache_len) holds
 *             sum_{s=j+1..cache_len-1} log f_s, the gate sum from key j to the last
 *             cached token (0 for the last one).
 *   log_f   : (B, H) fp32, the new token's log forget gate (any finite value).
 *   1. k_j <- H_t k_j and g_j <- g_j + log f_t for every cached j < cache_len;
 *   2. k_t, v_t are appended untransformed at index cache_len with g = 0;
 *   3. out = softmax_j(scale * q_t . k_j + g_j) v_j over j <= cache_len.
 * Other arguments, the results and the error behaviour as path_decode_step; ws must
 * hold path_workspace_bytes(PATH_OP_FOX_DECODE, B, H, cache_cap, d, dtype) bytes and
 * g_cache must be 16-byte aligned.
 */
path_status path_fox_decode_step(const void *q, const void *k, const void *v, const void *w,
                                 const float *beta, const float *log_f, void *k_cache,
                                 void *v_cache, float *g_cache, int B, int H, int cache_len,
                                 int cache_cap, int d, int dtype, float scale, void *out,
                                 void *ws, size_t ws_bytes, void *stream);

/*
 * path_decode_step without a workspace, for callers that cannot allocate device memory
 * for this library: for instance a plugin inside an inference engine that owns all
 * device memory through an allocator the plugin cannot reach, or a latency-bound loop
 * that must not call cudaMalloc because it can synchronise the device. The paper has no
 * counterpart; this is an interface convenience only.
 * Same arguments and results as path_decode_step, minus ws/ws_bytes. The split partial
 * results go to a fixed PATH_NOALLOC_SCRATCH_BYTES array compiled into the library, held
 * by every GPU that loads the library until the process exits. Limit:
 * B * H * ceil(cache_len / 1024) * (d + 2) * 4 bytes <= PATH_NOALLOC_SCRATCH_BYTES (for example
 * B*H = 1024 heads with up to 63488 cached keys); larger problems return
 * PATH_ERR_WORKSPACE before any launch. The call allocates nothing. The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call outside any stream capture. The address is kept per
 * device together with the id of the context it was looked up in: after a device reset
 * (cudaDeviceReset, or the primary context released and made again) the next call looks
 * it up again, and that call, too, should come before any stream capture. All calls on a device share
 * the array: calls that may overlap on the GPU (different streams or host threads) race
 * and must be serialised by the caller. No part of the array needs to start at zero.
 */
#define PATH_NOALLOC_SCRATCH_BYTES (16u << 20)
path_status path_decode_step_noalloc(const void *q, const void *k, const void *v, const void *w,
                                     const float *beta, void *k_cache, void *v_cache, int B,
                                     int H, int cache_len, int cache_cap, int d, int dtype,
                                     float scale, void *out, void *stream);

/*
 * Producer of the per-token Householder directions w and strengths beta (review
 * "거리에서 경로로, PaTH Attention" §3: a low-dimensional linear projection and a short
 * convolution of size 3 give w, which is L2-normalised, and beta is twice a sigmoid;
 * technical summary "技術要約: PaTH Attention" §2: beta_s = 2 sigmoid(u^T x_s + b), §6: beta
 * is clipped for bf16). For every token t of sequence b and head h:
 *   y_t   = w_up (w_down x_t)                             (H*d channels)
 *   y'_t  = conv[:,2] y_t + conv[:,1] y_{t-1} + conv[:,0] y_{t-2}  (depthwise, causal,
 *           zero before the first token of each sequence)
 *   w_out[b,h,t,:] = y'_t,h / max(|y'_t,h|, 1e-12)        (per head of d channels)
 *   beta_out[b,h,t] = min(2 sigmoid(u_h . x_t + bias_h), beta_max)
 *   x      : (B, L, D) bf16 activations
 *   w_down : (R, D) bf16, w_up : (H*d, R) bf16, u : (H, D) bf16 (rows = output features)
 *   conv   : (H*d, 3) fp32 taps; bias : (H) fp32; beta_max: clip (2 or more: none)
 *   w_out  : (B, H, L, d) bf16, beta_out : (B, H, L) fp32 -- the layouts path_attn_fwd takes
 *   ws     : path_wbeta_workspace_bytes(B, L, D, R, H, d, dtype) bytes (intermediate
 *            z = w_down x and the tap-scaled w_up, bf16)
 * Supported: dtype PATH_BF16 (else PATH_ERR_DTYPE); d = 64; D a positive multiple of 64;
 * R a multiple of 64 with R + (H rounded up to 16) <= 256; H >= 1 (else PATH_ERR_SHAPE).
 * beta_max must be positive and finite (PATH_ERR_ARG). Contractions use bf16 operands with
 * fp32 accumulation; z and the tap-scaled w_up are rounded to bf16.
 */
size_t path_wbeta_workspace_bytes(int B, int L, int D, int R, int H, int d, int dtype);
path_status path_wbeta_produce(const void *x, const void *w_down, const void *w_up,
                               const float *conv, const void *u, const float *bias,
                               float beta_max, void *w_out, float *beta_out, int B, int L,
                               int D, int R, int H, int d, int dtype, void *ws, size_t ws_bytes,
                               void *stream);

/*
 * Waits for `stream`, then reads and clears the status word that kernels of
 * earlier calls on this workspace wrote. Returns PATH_OK, PATH_ERR_TIMEOUT or
 * PATH_ERR_CUDA (if the synchronisation or the read failed).
 */
path_status path_check_workspace(void *ws, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *path_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PATH_ATTN_H */
