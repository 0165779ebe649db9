// K3: PaTH decode step with the in-place key-cache update.
//
// Technical summary "技術要約: PaTH Attention" §3 "推論" and review "거리에서 경로로, PaTH
// Attention" §9: at inference the transition of the new token t updates every cached key
// in place, k_j <- H_t k_j = k_j - beta_t (w_t . k_j) w_t, so no w/beta history is kept
// and ordinary softmax decoding follows (FlashDecoding-style). The new token's own key
// and value are appended untransformed (the diagonal logit uses the empty product).
//
// Split-K layout: grid (splits, heads); each CTA streams kDecodeChunk cached keys of one
// head. A key is one 128-byte row (bf16) handled by 8 lanes with one 16-byte load each
// (16 lanes x 16 bytes for fp32), so every warp load covers whole cache lines. Per key:
// load k, v; reduce w.k over the key's lanes; write back the updated key; reduce q.k;
// online softmax and o += p v in registers. The CTA merges its warps' partial softmax
// states and writes (m, l, o) of the split. A second kernel (one CTA per head) appends
// the new key/value, scores it and merges the splits.
//
// PaTH-FoX decode (review §4 and technical summary §2 "拡張: PaTH-FoX": the forget gate
// adds sum_{s=j+1..t} log f_s to the logit of key j): the cache keeps, per cached key, its
// running gate sum g_j = sum_{s=j+1..N-1} log f_s up to the last cached token, updated in
// place like the keys: g_j <- g_j + log f_t for j < N, and the new key enters with g = 0.
// Recent keys, the ones whose weight matters, hold small sums, so fp32 keeps them exact to
// within a few ulps however long the cache grows. The gate makes old keys vanish: a key
// whose logit lies more than 64 (log2 units) below the new token's own logit, itself a
// lower bound of the row's largest logit, weighs below 2^-64 of the largest weight, so its
// value row is not read (the key is still updated in place). Even 2^22 such keys move the
// softmax sum by less than 2^-42 of itself: exact within fp32 rounding.
#include <mutex>

#include "common.cuh"

namespace path {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int E = 8;
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&x)[8]) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = unpack_bf16x2(w[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ uint4 load_raw(const __nv_bfloat16 *p) {
        return *reinterpret_cast<const uint4 *>(p);
    }
    static __device__ __forceinline__ void unpack(const uint4 &u, float (&x)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = unpack_bf16x2(w[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&x)[8]) {
        uint4 u;
        u.x = pack_bf16x2(x[0], x[1]);
        u.y = pack_bf16x2(x[2], x[3]);
        u.z = pack_bf16x2(x[4], x[5]);
        u.w = pack_bf16x2(x[6], x[7]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};
template <> struct Vec<float> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void load(const float *p, float (&x)[4]) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    }
    static __device__ __forceinline__ uint4 load_raw(const float *p) {
        return *reinterpret_cast<const uint4 *>(p);
    }
    static __device__ __forceinline__ void unpack(const uint4 &u, float (&x)[4]) {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ void store(float *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

// Both variants hold rows of several passes in registers; three CTAs per SM keep enough
// bytes in flight (the bound caps them at 80 registers).
template <typename T, bool FOX, int D>
__global__ void __launch_bounds__(kThreads, 3)
decode_split_kernel(const T *__restrict__ q, const T *__restrict__ w,
                    const float *__restrict__ beta, T *__restrict__ kc, const T *__restrict__ vc,
                    int cache_len, int cap, int nsplit, float scale_log2, float *__restrict__ part,
                    const T *__restrict__ k_new, const float *__restrict__ log_f,
                    float *__restrict__ gc) {
    constexpr int E = Vec<T>::E;
    constexpr int TPK = D / E;    // lanes per key (16 B each)
    constexpr int KPW = 32 / TPK; // keys per warp pass
    __shared__ float sm_m[kWarps * KPW], sm_l[kWarps * KPW];
    __shared__ float sm_o[kWarps * KPW][D];

    const int sp = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / TPK, e0 = (lane % TPK) * E;
    const size_t head = (size_t)bh;

    float qv[E], wv[E];
    Vec<T>::load(q + head * D + e0, qv);
    Vec<T>::load(w + head * D + e0, wv);
    const float bt = beta[head];
    const float lf = FOX ? log_f[head] : 0.f;
    float *const grow = FOX ? gc + head * cap : nullptr;
    float thr = -INFINITY;  // FoX: keys scoring below it skip their value row
    if (FOX) {
        float kn[E], dn = 0.f;
        Vec<T>::load(k_new + head * D + e0, kn);
#pragma unroll
        for (int e = 0; e < E; ++e) dn = fmaf(qv[e], kn[e], dn);
#pragma unroll
        for (int off = 1; off < TPK; off <<= 1) dn += __shfl_xor_sync(0xffffffffu, dn, off);
        thr = dn * scale_log2 - 64.f;
    }

    const int j0 = sp * kDecodeChunk;
    const int j1 = min(j0 + kDecodeChunk, cache_len);
    float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;

    T *krow = kc + head * cap * D + e0;
    const T *vrow = vc + head * cap * D + e0;
    // The arithmetic of one cached key whose row kv is in registers: update it in place,
    // score it (bias gj, log2 units) and fold it into the lane's online softmax. Every lane
    // calls it (the shuffles are warp-wide); lanes whose key is past the end store nothing.
    // vv holds the value row, or for FoX is loaded here once the key is known to matter.
    auto key_math = [&](int j, bool valid, float gj, float (&kv)[E], float (&vv)[E]) {
        float dw = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dw = fmaf(wv[e], kv[e], dw);
#pragma unroll
        for (int off = 1; off < TPK; off <<= 1) dw += __shfl_xor_sync(0xffffffffu, dw, off);
        const float a = bt * dw;
        float dq = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            kv[e] = fmaf(-a, wv[e], kv[e]);
            dq = fmaf(qv[e], kv[e], dq);
        }
        if (valid) Vec<T>::store(krow + (size_t)j * D, kv);
#pragma unroll
        for (int off = 1; off < TPK; off <<= 1) dq += __shfl_xor_sync(0xffffffffu, dq, off);
        if (!valid) return;
        const float xl = FOX ? fmaf(gj, kLog2e, dq * scale_log2) : dq * scale_log2;
        if (FOX) {
            if (xl < thr) return;  // uniform over the key's lanes (they share dq and gj)
            Vec<T>::load(vrow + (size_t)j * D, vv);
        }
        const float m_new = fmaxf(m, xl);
        const float sc = exp2f(m - m_new);  // 0 while m is -inf
        const float p = exp2f(xl - m_new);
        l = l * sc + p;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf(p, vv[e], o[e] * sc);
        m = m_new;
    };
    if (!FOX) {
        // warp-uniform trip count: every lane joins the shuffles, lanes past the end idle.
        // Two passes' key and value rows are loaded together (raw, 16 bytes per lane each)
        // so that each warp keeps twice the bytes in flight.
        constexpr int kStride = kWarps * KPW;
        for (int jb = j0 + warp * KPW; jb < j1; jb += 2 * kStride) {
            uint4 kr[2], vr[2];
#pragma unroll
            for (int pb = 0; pb < 2; ++pb) {
                const int j = jb + pb * kStride + g;
                const bool valid = j < j1;
                kr[pb] = valid ? Vec<T>::load_raw(krow + (size_t)j * D) : make_uint4(0u, 0u, 0u, 0u);
                vr[pb] = valid ? Vec<T>::load_raw(vrow + (size_t)j * D) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int pb = 0; pb < 2; ++pb) {
                const int j = jb + pb * kStride + g;
                float kv[E], vv[E];
                Vec<T>::unpack(kr[pb], kv);
                Vec<T>::unpack(vr[pb], vv);
                key_math(j, j < j1, 0.f, kv, vv);
            }
        }
    } else {
        // Each warp owns runs of 32 consecutive keys: lane i reads, advances and writes
        // back the gate sum of key run + i (one coalesced 128-byte load and store per
        // run), and the key's lanes fetch it by shuffle. Most value rows are skipped, so
        // the key rows of a batch of passes are loaded up front (raw, 16 bytes per lane
        // and pass) to keep enough bytes in flight.
        constexpr int kPasses = 32 / KPW;
        constexpr int kBatch = kPasses < 4 ? kPasses : 4;
        for (int rb = j0 + warp * 32; rb < j1; rb += kWarps * 32) {
            const int jl = rb + lane;
            // the gate sums' load and the first key rows' loads are in flight together; the
            // advanced sums are stored once they arrive, after those loads are issued
            const float g_old = (jl < j1) ? grow[jl] : 0.f;
            float gl = 0.f;
#pragma unroll
            for (int b0 = 0; b0 < kPasses; b0 += kBatch) {
                uint4 kraw[kBatch];
#pragma unroll
                for (int pb = 0; pb < kBatch; ++pb) {
                    const int j = rb + (b0 + pb) * KPW + g;
                    kraw[pb] = (j < j1) ? Vec<T>::load_raw(krow + (size_t)j * D)
                                        : make_uint4(0u, 0u, 0u, 0u);
                }
                if (b0 == 0) {
                    gl = g_old + lf;
                    if (jl < j1) grow[jl] = gl;
                }
#pragma unroll
                for (int pb = 0; pb < kBatch; ++pb) {
                    const int src = (b0 + pb) * KPW + g;
                    const float gj = __shfl_sync(0xffffffffu, gl, src);
                    const int j = rb + src;
                    float kv[E], vv[E];
                    Vec<T>::unpack(kraw[pb], kv);
                    key_math(j, j < j1, gj, kv, vv);
                }
            }
        }
    }
    // ---- merge the kWarps * KPW partial states of this split
    const int slot = warp * KPW + g;
    if ((lane % TPK) == 0) {
        sm_m[slot] = m;
        sm_l[slot] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sm_o[slot][e0 + e] = o[e];
    __syncthreads();
    if (threadIdx.x < D) {
        const int c = threadIdx.x;
        float M = -INFINITY;
        for (int s = 0; s < kWarps * KPW; ++s) M = fmaxf(M, sm_m[s]);
        float Ls = 0.f, Oc = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < kWarps * KPW; ++s) {
                const float f = exp2f(sm_m[s] - M);
                Ls += sm_l[s] * f;
                Oc += sm_o[s][c] * f;
            }
        }
        float *dst = part + (head * nsplit + sp) * (D + 2);
        dst[2 + c] = Oc;
        if (c == 0) {
            dst[0] = M;
            dst[1] = Ls;
        }
    }
}

// One CTA of D threads per head: append (k_t, v_t) (and, for PaTH-FoX, the new key's
// gate sum 0: its logit has no bias), score the new key and merge splits.
template <typename T, bool FOX, int D>
__global__ void __launch_bounds__(D)
decode_merge_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    T *__restrict__ kc, T *__restrict__ vc, int cache_len, int cap, int nsplit,
                    float scale_log2, const float *__restrict__ part, T *__restrict__ out,
                    float *__restrict__ gc) {
    __shared__ float red[D / 32];
    const int bh = blockIdx.x, c = threadIdx.x;
    const size_t head = (size_t)bh;
    const T kt = k[head * D + c], vt = v[head * D + c];
    kc[(head * cap + cache_len) * D + c] = kt;
    vc[(head * cap + cache_len) * D + c] = vt;
    if (FOX && c == 0) gc[head * cap + cache_len] = 0.f;
    float d = Elt<T>::to_f(q[head * D + c]) * Elt<T>::to_f(kt);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if ((c & 31) == 0) red[c >> 5] = d;
    __syncthreads();
    float dsum = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < D / 32; ++w2) dsum += red[w2];
    const float x_new = dsum * scale_log2;
    const float *pp = part + head * nsplit * (D + 2);
    float M = x_new;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pp[s * (D + 2)]);
    const float f_new = exp2f(x_new - M);
    float Ls = f_new, Oc = f_new * Elt<T>::to_f(vt);
    for (int s = 0; s < nsplit; ++s) {
        const float ms = pp[s * (D + 2)];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        Ls += pp[s * (D + 2) + 1] * f;
        Oc += pp[s * (D + 2) + 2 + c] * f;
    }
    out[head * D + c] = Elt<T>::from_f(Oc / Ls);
}

// Both kernels of one step with the split partials at `part`; log_f and gc are used only
// when FOX is set.
template <typename T, bool FOX, int D>
cudaError_t launch_decode_kernels(const void *q, const void *k, const void *v, const void *w,
                                  const float *beta, const float *log_f, void *k_cache,
                                  void *v_cache, float *gc, int BH, int cache_len, int cap,
                                  float scale, void *out, float *part, cudaStream_t stream) {
    const float sl2 = scale * kLog2e;
    const int used = (cache_len + kDecodeChunk - 1) / kDecodeChunk;
    if (used > 0) {
        dim3 grid(used, BH);
        decode_split_kernel<T, FOX, D><<<grid, kThreads, 0, stream>>>(
            static_cast<const T *>(q), static_cast<const T *>(w), beta, static_cast<T *>(k_cache),
            static_cast<const T *>(v_cache), cache_len, cap, used, sl2, part,
            static_cast<const T *>(k), log_f, gc);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    decode_merge_kernel<T, FOX, D><<<BH, D, 0, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<T *>(k_cache), static_cast<T *>(v_cache), cache_len, cap, used, sl2, part,
        static_cast<T *>(out), gc);
    return cudaGetLastError();
}

template <typename T, bool FOX>
cudaError_t launch_decode_d(int d, const void *q, const void *k, const void *v, const void *w,
                            const float *beta, const float *log_f, void *k_cache, void *v_cache,
                            float *gc, int BH, int cache_len, int cap, float scale, void *out,
                            float *part, cudaStream_t stream) {
    if (d == 128)
        return launch_decode_kernels<T, FOX, 128>(q, k, v, w, beta, log_f, k_cache, v_cache, gc,
                                                  BH, cache_len, cap, scale, out, part, stream);
    return launch_decode_kernels<T, FOX, 64>(q, k, v, w, beta, log_f, k_cache, v_cache, gc, BH,
                                             cache_len, cap, scale, out, part, stream);
}

}  // namespace

template <typename T>
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, void *k_cache, void *v_cache, int BH, int cache_len,
                          int cap, int d, float scale, void *out, void *ws, cudaStream_t stream) {
    float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + 256);
    return launch_decode_d<T, false>(d, q, k, v, w, beta, nullptr, k_cache, v_cache, nullptr, BH,
                                     cache_len, cap, scale, out, part, stream);
}

// PaTH-FoX decode: as launch_decode, plus the in-place gate sums gc (BH, cap) fp32 and the
// new token's log forget gate log_f (BH).
template <typename T>
cudaError_t launch_fox_decode(const void *q, const void *k, const void *v, const void *w,
                              const float *beta, const float *log_f, void *k_cache,
                              void *v_cache, float *gc, int BH, int cache_len, int cap, int d,
                              float scale, void *out, void *ws, cudaStream_t stream) {
    float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + 256);
    return launch_decode_d<T, true>(d, q, k, v, w, beta, log_f, k_cache, v_cache, gc, BH,
                                    cache_len, cap, scale, out, part, stream);
}

// ---------------------------------------------------------------- no-allocation variant
// Callers that cannot give this library any device memory of their own (a plugin inside
// an engine whose allocator is not exposed to it, or a real-time loop that may not call
// cudaMalloc because the call can synchronise the device) use this variant: its split
// partials live in a fixed array compiled into the library. Every GPU that loads the
// library holds these 16 MiB until the process exits. All calls on a device share the
// array, so calls that overlap on that GPU (other streams, other host threads) race and
// must be serialised by the caller. Nothing in the array has to start at zero: each call
// writes every partial entry it later reads.
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context id the pointer belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Id of the calling thread's current context (unique for the life of the process, so a
// context created after a device reset never matches one from before it).
cudaError_t current_context_id(unsigned long long *id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &r1) != cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) !=
                cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess)
            return cudaErrorNotSupported;
        get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        get_id = reinterpret_cast<CtxGetIdFn>(q);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
    if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}
}  // namespace

// Device address of the static scratch on the current device. The first call on a
// device (with that device current) looks it up: host code only holds a stand-in for
// the symbol, never its device address. The pointer is cached together with the id of
// the context it was looked up in; after a device reset the runtime makes a new context
// (and reloads the module), the ids differ and the address is looked up again.
static cudaError_t static_scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // no context may be current yet on this thread (the runtime makes the primary context
    // current on first use, which the symbol lookup below is)
    std::lock_guard<std::mutex> lock(g_scratch_mu);  // also guards the entry-point lookup
    unsigned long long ctx_id = 0;
    const bool have_id = current_context_id(&ctx_id) == cudaSuccess;
    if (!have_id || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx_id) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        if (!have_id) {
            e = current_context_id(&ctx_id);
            if (e != cudaSuccess) return e;
        }
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx_id;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

size_t decode_static_scratch_bytes() { return kStaticScratchBytes; }

size_t decode_static_scratch_needed(int BH, int cache_len, int d) {
    const size_t used = (size_t)((cache_len + kDecodeChunk - 1) / kDecodeChunk);
    return (size_t)BH * used * (d + 2) * sizeof(float);
}

// Same kernels as launch_decode, with the partials in the static scratch. The caller
// has checked decode_static_scratch_needed() <= decode_static_scratch_bytes().
template <typename T>
cudaError_t launch_decode_static(const void *q, const void *k, const void *v, const void *w,
                                 const float *beta, void *k_cache, void *v_cache, int BH,
                                 int cache_len, int cap, int d, float scale, void *out,
                                 cudaStream_t stream) {
    void *scratch = nullptr;
    cudaError_t err = static_scratch_address(&scratch);
    if (err != cudaSuccess) return err;
    float *part = static_cast<float *>(scratch);
    return launch_decode_d<T, false>(d, q, k, v, w, beta, nullptr, k_cache, v_cache, nullptr, BH,
                                     cache_len, cap, scale, out, part, stream);
}

template cudaError_t launch_decode_static<float>(const void *, const void *, const void *,
                                                 const void *, const float *, void *, void *,
                                                 int, int, int, int, float, void *, cudaStream_t);
template cudaError_t launch_decode_static<__nv_bfloat16>(const void *, const void *,
                                                         const void *, const void *,
                                                         const float *, void *, void *, int, int,
                                                         int, int, float, void *, cudaStream_t);

template cudaError_t launch_decode<float>(const void *, const void *, const void *, const void *,
                                          const float *, void *, void *, int, int, int, int,
                                          float, void *, void *, cudaStream_t);
template cudaError_t launch_decode<__nv_bfloat16>(const void *, const void *, const void *,
                                                  const void *, const float *, void *, void *,
                                                  int, int, int, int, float, void *, void *,
                                                  cudaStream_t);
template cudaError_t launch_fox_decode<float>(const void *, const void *, const void *,
                                              const void *, const float *, const float *, void *,
                                              void *, float *, int, int, int, int, float, void *,
                                              void *, cudaStream_t);
template cudaError_t launch_fox_decode<__nv_bfloat16>(const void *, const void *, const void *,
                                                      const void *, const float *, const float *,
                                                      void *, void *, float *, int, int, int, int,
                                                      float, void *, void *, cudaStream_t);

}  // namespace path
