// Host side of the C ABI declared in include/path_attn.h: argument checks (synchronous,
// before any launch), workspace sizing and kernel dispatch on the caller's stream.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "path_attn.h"

namespace path {
size_t ut_prepare_smem_bytes();
template <typename T>
cudaError_t launch_ut_prepare(const void *q, const void *k, const void *w, const float *beta,
                              const float *log_f, int BH, int L, float scale, void *ws,
                              cudaStream_t stream);
cudaError_t launch_fox_prepare(const float *log_f, int BH, int L, int elt_bytes, float scale,
                               void *ws, cudaStream_t stream);
cudaError_t launch_ut_prepare_tc(const void *q, const void *k, const void *w, const float *beta,
                                 const float *log_f, int BH, int L, float scale, void *ws,
                                 uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_pair_combine(int BH, int L, void *ws, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_scan_tc_fox(const void *v, void *out, float *lse, int BH, int L, float scale,
                               void *ws, uint64_t limit_ns, int force_timeout,
                               cudaStream_t stream);
cudaError_t launch_scan_tc(const void *v, void *out, float *lse, int BH, int L,
                           float scale, void *ws, uint64_t limit_ns, int force_timeout,
                           cudaStream_t stream);
cudaError_t launch_scan_f32(const void *v, void *out, float *lse, bool fox, int BH, int L,
                            float scale, void *ws, cudaStream_t stream);
template <typename T>
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, void *k_cache, void *v_cache, int BH, int cache_len,
                          int cap, int d, float scale, void *out, void *ws, cudaStream_t stream);
template <typename T>
cudaError_t launch_fox_decode(const void *q, const void *k, const void *v, const void *w,
                              const float *beta, const float *log_f, void *k_cache,
                              void *v_cache, float *gc, int BH, int cache_len, int cap, int d,
                              float scale, void *out, void *ws, cudaStream_t stream);
size_t producer_ws_bytes(int B, int L, int R, int H);
cudaError_t launch_producer(const void *x, const void *w_down, const void *w_up, const float *conv,
                            const void *u, const float *bias, float beta_max, void *w_out,
                            float *beta_out, int B, int L, int D, int R, int H, void *ws,
                            uint64_t limit_ns, cudaStream_t stream);
template <typename T>
cudaError_t launch_path_bwd(const void *q, const void *k, const void *v, const void *w,
                            const float *beta, const float *log_f, const void *o,
                            const float *lse, const void *dout, int B, int H, int L, float scale,
                            float *dq, float *dk, float *dv, float *dw, float *dbeta, float *dlogf,
                            void *ws, cudaStream_t stream);
template <typename T>
cudaError_t launch_prep_d128(const void *q, const void *k, const void *w, const float *beta,
                             const float *log_f, int B, int H, int L, float scale, void *ws,
                             cudaStream_t stream);
template <typename T>
cudaError_t launch_scan_d128(const void *v, void *out, float *lse, bool fox, int B, int H, int L,
                             float scale, void *ws, cudaStream_t stream);
cudaError_t launch_fox_exit_d128(const float *log_f, int BH, int L, float scale, void *ws,
                                 cudaStream_t stream);
cudaError_t launch_ut_prepare_tc128(const void *q, const void *k, const void *w,
                                    const float *beta, const float *log_f, int BH, int L,
                                    float scale, void *ws, uint64_t limit_ns,
                                    cudaStream_t stream);
cudaError_t launch_scan_tc128(const void *v, void *out, float *lse, bool fox, int BH, int L,
                              float scale, void *ws, uint64_t limit_ns, cudaStream_t stream);
size_t bwd_tc_ws_bytes(int B, int H, int L, bool fox);
size_t bwd128_ws_bytes(int B, int H, int L, bool fox);
size_t bwd_tc128_ws_bytes(int B, int H, int L, bool fox);
cudaError_t launch_path_bwd128_tc(const void *q, const void *k, const void *v, const void *w,
                                  const float *beta, const float *log_f, const void *o,
                                  const float *lse, const void *dout, int B, int H, int L,
                                  float scale, float *dq, float *dk, float *dv, float *dw,
                                  float *dbeta, float *dlogf, void *ws, uint64_t limit_ns,
                                  cudaStream_t stream);
template <typename T>
cudaError_t launch_path_bwd128(const void *q, const void *k, const void *v, const void *w,
                               const float *beta, const float *log_f, const void *o,
                               const float *lse, const void *dout, int B, int H, int L,
                               float scale, float *dq, float *dk, float *dv, float *dw,
                               float *dbeta, float *dlogf, void *ws, cudaStream_t stream);
cudaError_t launch_path_bwd_tc(const void *q, const void *k, const void *v, const void *w,
                               const float *beta, const float *log_f, const void *o,
                               const float *lse, const void *dout, int B, int H, int L,
                               float scale, float *dq, float *dk, float *dv, float *dw,
                               float *dbeta, float *dlogf, void *ws, uint64_t limit_ns,
                               cudaStream_t stream);
size_t decode_static_scratch_bytes();
size_t decode_static_scratch_needed(int BH, int cache_len, int d);
template <typename T>
cudaError_t launch_decode_static(const void *q, const void *k, const void *v, const void *w,
                                 const float *beta, void *k_cache, void *v_cache, int BH,
                                 int cache_len, int cap, int d, float scale, void *out,
                                 cudaStream_t stream);
}  // namespace path

namespace {

using namespace path;

// Bounded waits inside the tensor-core scan give up after this long.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// Test hook: PATH_ATTN_DEBUG_FORCE_TIMEOUT=1 makes the scan's MMA lane wait on a barrier
// that nothing arrives at, with a 2 ms limit, to exercise the timeout path without a fault.
constexpr uint64_t kDebugWaitLimitNs = 2000000ull;

bool debug_force_timeout() {
    const char *e = std::getenv("PATH_ATTN_DEBUG_FORCE_TIMEOUT");
    return e != nullptr && e[0] == '1';
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elt_bytes(int dtype) { return dtype == PATH_BF16 ? 2 : 4; }

path_status check_sizes(int B, int H, int L, int d, int dtype) {
    if (B < 0 || H < 0 || L < 0) return PATH_ERR_SHAPE;
    if (d != kD) return PATH_ERR_SHAPE;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_DTYPE;
    if ((long long)B * H > PATH_MAX_HEADS || L > PATH_MAX_LEN) return PATH_ERR_SHAPE;
    return PATH_OK;
}

// The forward and the backward (PaTH and PaTH-FoX) also take d = 128.
path_status check_fwd_sizes(int B, int H, int L, int d, int dtype) {
    return check_sizes(B, H, L, d == 128 ? kD : d, dtype);
}

// Decode works on head sizes 64 and 128.
path_status check_decode_sizes(int B, int H, int cap, int d, int dtype) {
    return check_sizes(B, H, cap, d == 128 ? kD : (d == kD ? kD : -1), dtype);
}

path_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PATH_OK : PATH_ERR_CUDA; }

path_status check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr) return PATH_ERR_NULL;
    if (!aligned(ws, 256)) return PATH_ERR_ALIGN;
    if (ws_bytes < need) return PATH_ERR_WORKSPACE;
    return PATH_OK;
}

// Forward workspace size for a (d, dtype) pair.
size_t fwd_ws_bytes(int B, int H, int L, int d, int dtype, bool fox) {
    if (d == 128)
        return dtype == PATH_BF16 ? d128_tc_layout(B, H, L, fox).total
                                  : d128_layout(B, H, L, fox).total;
    return fwd_layout(B, H, L, elt_bytes(dtype), fox).total;
}

path_status prepare_impl(const void *q, const void *k, const void *w, const float *beta,
                         const float *log_f, bool fox, int B, int H, int L, int d, int dtype,
                         float scale, void *ws, size_t ws_bytes, cudaStream_t stream) {
    path_status st = check_fwd_sizes(B, H, L, d, dtype);
    if (st != PATH_OK) return st;
    if (!std::isfinite(scale)) return PATH_ERR_ARG;
    if ((long long)B * H * L == 0) return PATH_OK;
    if (!q || !k || !w || !beta || (fox && !log_f)) return PATH_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(w, 16) || !aligned(beta, 16) ||
        (fox && !aligned(log_f, 16)))
        return PATH_ERR_ALIGN;
    if (d == 128) {
        if ((st = check_ws(ws, ws_bytes, fwd_ws_bytes(B, H, L, d, dtype, fox))) != PATH_OK) return st;
        const float *lf = fox ? log_f : nullptr;
        // bf16: tensor-core preparation (PaTH-FoX: then the early-exit extents); fp32: the
        // fp32 CUDA-core kernel (the fp32 bar), whose scan decides its exit as it runs
        if (dtype != PATH_BF16)
            return from_cuda(launch_prep_d128<float>(q, k, w, beta, lf, B, H, L, scale, ws, stream));
        cudaError_t e = launch_ut_prepare_tc128(q, k, w, beta, lf, B * H, L, scale, ws,
                                                kWaitLimitNs, stream);
        if (e == cudaSuccess && fox) e = launch_fox_exit_d128(lf, B * H, L, scale, ws, stream);
        return from_cuda(e);
    }
    const FwdLayout lay = fwd_layout(B, H, L, elt_bytes(dtype), fox);
    if ((st = check_ws(ws, ws_bytes, lay.total)) != PATH_OK) return st;
    const float *lf = fox ? log_f : nullptr;
    cudaError_t e = (dtype == PATH_BF16)
                        ? launch_ut_prepare_tc(q, k, w, beta, lf, B * H, L, scale, ws,
                                               kWaitLimitNs, stream)
                        : launch_ut_prepare<float>(q, k, w, beta, lf, B * H, L, scale, ws, stream);
    // bf16 PaTH: the block-pair products the two-block scan steps use
    if (e == cudaSuccess && dtype == PATH_BF16 && !fox)
        e = launch_pair_combine(B * H, L, ws, kWaitLimitNs, stream);
    // FoX: gate prefix sums and the scan's early-exit extents (reads K1's q~, k~ and table)
    if (e == cudaSuccess && fox)
        e = launch_fox_prepare(lf, B * H, L, elt_bytes(dtype), scale, ws, stream);
    return from_cuda(e);
}

path_status scan_impl(const void *v, void *out, float *lse, bool fox, int B, int H, int L, int d,
                      int dtype, float scale, void *ws, size_t ws_bytes, cudaStream_t stream) {
    path_status st = check_fwd_sizes(B, H, L, d, dtype);
    if (st != PATH_OK) return st;
    if (!std::isfinite(scale)) return PATH_ERR_ARG;
    if ((long long)B * H * L == 0) return PATH_OK;
    if (!v || !out) return PATH_ERR_NULL;
    if (!aligned(v, 16) || !aligned(out, 16) || (lse && !aligned(lse, 16))) return PATH_ERR_ALIGN;
    if (d == 128) {
        if ((st = check_ws(ws, ws_bytes, fwd_ws_bytes(B, H, L, d, dtype, fox))) != PATH_OK) return st;
        return from_cuda(dtype == PATH_BF16
                             ? launch_scan_tc128(v, out, lse, fox, B * H, L, scale, ws,
                                                 kWaitLimitNs, stream)
                             : launch_scan_d128<float>(v, out, lse, fox, B, H, L, scale, ws, stream));
    }
    const FwdLayout lay = fwd_layout(B, H, L, elt_bytes(dtype), fox);
    if ((st = check_ws(ws, ws_bytes, lay.total)) != PATH_OK) return st;
    if (dtype == PATH_BF16) {
        const bool force = debug_force_timeout();
        const uint64_t lim = force ? kDebugWaitLimitNs : kWaitLimitNs;
        cudaError_t e = fox ? launch_scan_tc_fox(v, out, lse, B * H, L, scale, ws, lim,
                                                 force ? 1 : 0, stream)
                            : launch_scan_tc(v, out, lse, B * H, L, scale, ws, lim,
                                             force ? 1 : 0, stream);
        return from_cuda(e);
    }
    return from_cuda(launch_scan_f32(v, out, lse, fox, B * H, L, scale, ws, stream));
}

}  // namespace

namespace {
size_t bwd_ws_bytes(int B, int H, int L, int d, int dtype, bool fox) {
    if (d == 128)
        return dtype == PATH_BF16 ? bwd_tc128_ws_bytes(B, H, L, fox) : bwd128_ws_bytes(B, H, L, fox);
    return dtype == PATH_BF16 ? bwd_tc_ws_bytes(B, H, L, fox) : bwd_layout(B, H, L, fox).total;
}

path_status bwd_impl(const void *q, const void *k, const void *v, const void *w, const float *beta,
                     const float *log_f, const void *out, const float *lse, const void *d_out,
                     int B, int H, int L, int d, int dtype, float scale, float *dq, float *dk,
                     float *dv, float *dw, float *dbeta, float *dlog_f, bool fox, void *ws,
                     size_t ws_bytes, void *stream) {
    path_status st = check_fwd_sizes(B, H, L, d, dtype);
    if (st != PATH_OK) return st;
    if (!std::isfinite(scale)) return PATH_ERR_ARG;
    if ((long long)B * H * L == 0) return PATH_OK;
    const void *in[] = {q, k, v, w, beta, out, lse, d_out, dq, dk, dv, dw, dbeta,
                        fox ? (const void *)log_f : q, fox ? (const void *)dlog_f : q};
    for (const void *p : in)
        if (!p) return PATH_ERR_NULL;
    for (const void *p : in)
        if (!aligned(p, 16)) return PATH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, bwd_ws_bytes(B, H, L, d, dtype, fox))) != PATH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float *lf = fox ? log_f : nullptr;
    float *dlf = fox ? dlog_f : nullptr;
    // d = 128: bf16 inputs take the warp-level tensor-core query pass, fp32 inputs the fp32
    // CUDA-core kernels
    if (d == 128)
        return from_cuda(dtype == PATH_BF16
                             ? launch_path_bwd128_tc(q, k, v, w, beta, lf, out, lse, d_out, B, H, L,
                                                     scale, dq, dk, dv, dw, dbeta, dlf, ws,
                                                     kWaitLimitNs, s)
                             : launch_path_bwd128<float>(q, k, v, w, beta, lf, out, lse, d_out, B,
                                                         H, L, scale, dq, dk, dv, dw, dbeta, dlf,
                                                         ws, s));
    // bf16 inputs: tensor-core query pass; fp32 inputs: the fp32 CUDA-core kernels, whose
    // accuracy the fp32 bar needs
    cudaError_t e = dtype == PATH_BF16
                        ? launch_path_bwd_tc(q, k, v, w, beta, lf, out, lse, d_out, B, H, L,
                                             scale, dq, dk, dv, dw, dbeta, dlf, ws, kWaitLimitNs,
                                             s)
                        : launch_path_bwd<float>(q, k, v, w, beta, lf, out, lse, d_out, B, H, L,
                                                 scale, dq, dk, dv, dw, dbeta, dlf, ws, s);
    return from_cuda(e);
}
}  // namespace

extern "C" {

size_t path_workspace_bytes(int op, int B, int H, int L, int d, int dtype) {
    switch (op) {
        case PATH_OP_FWD:
        case PATH_OP_FOX_FWD:
            if (check_fwd_sizes(B, H, L, d, dtype) != PATH_OK) return 0;
            return fwd_ws_bytes(B, H, L, d, dtype, op == PATH_OP_FOX_FWD);
        default: break;
    }
    if (op == PATH_OP_BWD || op == PATH_OP_FOX_BWD) {
        if (check_fwd_sizes(B, H, L, d, dtype) != PATH_OK) return 0;
        return bwd_ws_bytes(B, H, L, d, dtype, op == PATH_OP_FOX_BWD);
    }
    if (check_decode_sizes(B, H, L, d, dtype) != PATH_OK) return 0;
    switch (op) {
        case PATH_OP_DECODE: return decode_ws_bytes(B, H, L, d);
        case PATH_OP_FOX_DECODE: return decode_ws_bytes(B, H, L, d);
        default: return 0;
    }
}

path_status path_fwd_prepare(const void *q, const void *k, const void *w, const float *beta,
                             const float *log_f, int B, int H, int L, int d, int dtype,
                             float scale, void *ws, size_t ws_bytes, void *stream) {
    return prepare_impl(q, k, w, beta, log_f, log_f != nullptr, B, H, L, d, dtype, scale, ws,
                        ws_bytes, static_cast<cudaStream_t>(stream));
}

path_status path_fox_first_blocks(const void *ws, size_t ws_bytes, int B, int H, int L,
                                  int d, int dtype, int *first_block, void *stream) {
    path_status st = check_sizes(B, H, L, d, dtype);
    if (st != PATH_OK) return st;
    if ((long long)B * H * L == 0) return PATH_OK;
    if (!first_block) return PATH_ERR_NULL;
    if (!aligned(first_block, 4)) return PATH_ERR_ALIGN;
    const FwdLayout lay = fwd_layout(B, H, L, elt_bytes(dtype), true);
    if ((st = check_ws(const_cast<void *>(ws), ws_bytes, lay.total)) != PATH_OK) return st;
    const int nq = (L + kC - 1) / kC;
    return from_cuda(cudaMemcpy2DAsync(first_block, (size_t)nq * sizeof(int),
                                       static_cast<const char *>(ws) + lay.off_fb,
                                       (size_t)lay.nblk * sizeof(int), (size_t)nq * sizeof(int),
                                       (size_t)B * H, cudaMemcpyDeviceToDevice,
                                       static_cast<cudaStream_t>(stream)));
}

path_status path_attn_bwd(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, const void *out, const float *lse, const void *d_out,
                          int B, int H, int L, int d, int dtype, float scale, float *dq, float *dk,
                          float *dv, float *dw, float *dbeta, void *ws, size_t ws_bytes,
                          void *stream) {
    return bwd_impl(q, k, v, w, beta, nullptr, out, lse, d_out, B, H, L, d, dtype, scale, dq, dk,
                    dv, dw, dbeta, nullptr, false, ws, ws_bytes, stream);
}

path_status path_fox_bwd(const void *q, const void *k, const void *v, const void *w,
                         const float *beta, const float *log_f, const void *out, const float *lse,
                         const void *d_out, int B, int H, int L, int d, int dtype, float scale,
                         float *dq, float *dk, float *dv, float *dw, float *dbeta, float *dlog_f,
                         void *ws, size_t ws_bytes, void *stream) {
    return bwd_impl(q, k, v, w, beta, log_f, out, lse, d_out, B, H, L, d, dtype, scale, dq, dk,
                    dv, dw, dbeta, dlog_f, true, ws, ws_bytes, stream);
}

path_status path_fwd_scan(const void *v, void *out, float *lse, int fox, int B, int H, int L,
                          int d, int dtype, float scale, void *ws, size_t ws_bytes,
                          void *stream) {
    return scan_impl(v, out, lse, fox != 0, B, H, L, d, dtype, scale, ws, ws_bytes,
                     static_cast<cudaStream_t>(stream));
}

path_status path_attn_fwd(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, void *out, float *lse, int B, int H, int L, int d,
                          int dtype, float scale, void *ws, size_t ws_bytes, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every argument of both stages is checked before the first launch
    path_status st = check_fwd_sizes(B, H, L, d, dtype);
    if (st != PATH_OK) return st;
    if ((long long)B * H * L > 0) {
        if (!v || !out) return PATH_ERR_NULL;
        if (!aligned(v, 16) || !aligned(out, 16) || (lse && !aligned(lse, 16)))
            return PATH_ERR_ALIGN;
    }
    st = prepare_impl(q, k, w, beta, nullptr, false, B, H, L, d, dtype, scale, ws, ws_bytes, s);
    if (st != PATH_OK) return st;
    return scan_impl(v, out, lse, false, B, H, L, d, dtype, scale, ws, ws_bytes, s);
}

path_status path_fox_fwd(const void *q, const void *k, const void *v, const void *w,
                         const float *beta, const float *log_f, void *out, float *lse, int B,
                         int H, int L, int d, int dtype, float scale, void *ws, size_t ws_bytes,
                         void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    path_status st = check_fwd_sizes(B, H, L, d, dtype);
    if (st != PATH_OK) return st;
    if ((long long)B * H * L > 0) {
        if (!v || !out || !log_f) return PATH_ERR_NULL;
        if (!aligned(v, 16) || !aligned(out, 16) || (lse && !aligned(lse, 16)))
            return PATH_ERR_ALIGN;
    }
    st = prepare_impl(q, k, w, beta, log_f, true, B, H, L, d, dtype, scale, ws, ws_bytes, s);
    if (st != PATH_OK) return st;
    return scan_impl(v, out, lse, true, B, H, L, d, dtype, scale, ws, ws_bytes, s);
}

path_status path_decode_step(const void *q, const void *k, const void *v, const void *w,
                             const float *beta, void *k_cache, void *v_cache, int B, int H,
                             int cache_len, int cache_cap, int d, int dtype, float scale,
                             void *out, void *ws, size_t ws_bytes, void *stream) {
    path_status st = check_decode_sizes(B, H, cache_cap, d, dtype);
    if (st != PATH_OK) return st;
    if (cache_len < 0) return PATH_ERR_SHAPE;
    if (!std::isfinite(scale)) return PATH_ERR_ARG;
    if ((long long)B * H == 0) return PATH_OK;
    if (cache_len + 1 > cache_cap) return PATH_ERR_CAPACITY;
    if (!q || !k || !v || !w || !beta || !k_cache || !v_cache || !out) return PATH_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(w, 16) ||
        !aligned(beta, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return PATH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, decode_ws_bytes(B, H, cache_cap, d))) != PATH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == PATH_BF16)
        return from_cuda(launch_decode<__nv_bfloat16>(q, k, v, w, beta, k_cache, v_cache, B * H,
                                                      cache_len, cache_cap, d, scale, out, ws, s));
    return from_cuda(launch_decode<float>(q, k, v, w, beta, k_cache, v_cache, B * H, cache_len,
                                          cache_cap, d, scale, out, ws, s));
}

path_status path_fox_decode_step(const void *q, const void *k, const void *v, const void *w,
                                 const float *beta, const float *log_f, void *k_cache,
                                 void *v_cache, float *g_cache, int B, int H, int cache_len,
                                 int cache_cap, int d, int dtype, float scale, void *out,
                                 void *ws, size_t ws_bytes, void *stream) {
    path_status st = check_decode_sizes(B, H, cache_cap, d, dtype);
    if (st != PATH_OK) return st;
    if (cache_len < 0) return PATH_ERR_SHAPE;
    if (!std::isfinite(scale)) return PATH_ERR_ARG;
    if ((long long)B * H == 0) return PATH_OK;
    if (cache_len + 1 > cache_cap) return PATH_ERR_CAPACITY;
    if (!q || !k || !v || !w || !beta || !log_f || !k_cache || !v_cache || !g_cache || !out)
        return PATH_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(w, 16) ||
        !aligned(beta, 4) || !aligned(log_f, 4) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(g_cache, 16) || !aligned(out, 16))
        return PATH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, decode_ws_bytes(B, H, cache_cap, d))) != PATH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == PATH_BF16)
        return from_cuda(launch_fox_decode<__nv_bfloat16>(q, k, v, w, beta, log_f, k_cache,
                                                          v_cache, g_cache, B * H, cache_len,
                                                          cache_cap, d, scale, out, ws, s));
    return from_cuda(launch_fox_decode<float>(q, k, v, w, beta, log_f, k_cache, v_cache, g_cache,
                                              B * H, cache_len, cache_cap, d, scale, out, ws, s));
}

path_status path_decode_step_noalloc(const void *q, const void *k, const void *v, const void *w,
                                     const float *beta, void *k_cache, void *v_cache, int B,
                                     int H, int cache_len, int cache_cap, int d, int dtype,
                                     float scale, void *out, void *stream) {
    path_status st = check_decode_sizes(B, H, cache_cap, d, dtype);
    if (st != PATH_OK) return st;
    if (cache_len < 0) return PATH_ERR_SHAPE;
    if (!std::isfinite(scale)) return PATH_ERR_ARG;
    if ((long long)B * H == 0) return PATH_OK;
    if (cache_len + 1 > cache_cap) return PATH_ERR_CAPACITY;
    if (!q || !k || !v || !w || !beta || !k_cache || !v_cache || !out) return PATH_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(w, 16) ||
        !aligned(beta, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return PATH_ERR_ALIGN;
    if (decode_static_scratch_needed(B * H, cache_len, d) > decode_static_scratch_bytes())
        return PATH_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == PATH_BF16)
        return from_cuda(launch_decode_static<__nv_bfloat16>(q, k, v, w, beta, k_cache, v_cache,
                                                             B * H, cache_len, cache_cap, d,
                                                             scale, out, s));
    return from_cuda(launch_decode_static<float>(q, k, v, w, beta, k_cache, v_cache, B * H,
                                                 cache_len, cache_cap, d, scale, out, s));
}

namespace {
path_status check_producer_sizes(int B, int L, int D, int R, int H, int d, int dtype) {
    if (B < 0 || L < 0 || D <= 0 || R <= 0 || H <= 0) return PATH_ERR_SHAPE;
    if (dtype != PATH_BF16) return PATH_ERR_DTYPE;
    if (d != kD || D % 64 != 0 || R % 64 != 0 || R + ((H + 15) & ~15) > 256) return PATH_ERR_SHAPE;
    if ((long long)B * H > PATH_MAX_HEADS || L > PATH_MAX_LEN || D > (1 << 16) ||
        (long long)B * L > (1LL << 30))
        return PATH_ERR_SHAPE;
    return PATH_OK;
}
}  // namespace

size_t path_wbeta_workspace_bytes(int B, int L, int D, int R, int H, int d, int dtype) {
    if (check_producer_sizes(B, L, D, R, H, d, dtype) != PATH_OK) return 0;
    return producer_ws_bytes(B, L, R, H);
}

path_status path_wbeta_produce(const void *x, const void *w_down, const void *w_up,
                               const float *conv, const void *u, const float *bias,
                               float beta_max, void *w_out, float *beta_out, int B, int L,
                               int D, int R, int H, int d, int dtype, void *ws, size_t ws_bytes,
                               void *stream) {
    path_status st = check_producer_sizes(B, L, D, R, H, d, dtype);
    if (st != PATH_OK) return st;
    if (!std::isfinite(beta_max) || !(beta_max > 0.f)) return PATH_ERR_ARG;
    if ((long long)B * L == 0) return PATH_OK;
    if (!x || !w_down || !w_up || !conv || !u || !bias || !w_out || !beta_out) return PATH_ERR_NULL;
    if (!aligned(x, 16) || !aligned(w_down, 16) || !aligned(w_up, 16) || !aligned(u, 16) ||
        !aligned(conv, 4) || !aligned(bias, 4) || !aligned(w_out, 16) || !aligned(beta_out, 4))
        return PATH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, producer_ws_bytes(B, L, R, H))) != PATH_OK) return st;
    return from_cuda(launch_producer(x, w_down, w_up, conv, u, bias, beta_max, w_out, beta_out, B,
                                     L, D, R, H, ws, kWaitLimitNs,
                                     static_cast<cudaStream_t>(stream)));
}

path_status path_check_workspace(void *ws, void *stream) {
    if (ws == nullptr) return PATH_ERR_NULL;
    if (!aligned(ws, 256)) return PATH_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return PATH_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PATH_ERR_CUDA;
    if (word != 0 && cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return PATH_ERR_CUDA;
    return word == 0 ? PATH_OK : (word == kStatusTimeout ? PATH_ERR_TIMEOUT : PATH_ERR_CUDA);
}

const char *path_status_string(int status) {
    switch (status) {
        case PATH_OK: return "PATH_OK";
        case PATH_ERR_NULL: return "PATH_ERR_NULL: a required pointer is NULL";
        case PATH_ERR_SHAPE: return "PATH_ERR_SHAPE: unsupported or negative size";
        case PATH_ERR_DTYPE: return "PATH_ERR_DTYPE: unsupported dtype";
        case PATH_ERR_ALIGN: return "PATH_ERR_ALIGN: misaligned pointer";
        case PATH_ERR_WORKSPACE: return "PATH_ERR_WORKSPACE: workspace too small";
        case PATH_ERR_CAPACITY: return "PATH_ERR_CAPACITY: decode cache is full";
        case PATH_ERR_TIMEOUT: return "PATH_ERR_TIMEOUT: a kernel gave up a bounded wait";
        case PATH_ERR_CUDA: return "PATH_ERR_CUDA: a CUDA call failed";
        case PATH_ERR_ARG: return "PATH_ERR_ARG: scalar argument out of range";
        default: return "PATH_ERR_UNKNOWN";
    }
}

}  // extern "C"
