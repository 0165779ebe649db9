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
    static __device__ __forceinline__ void store(float *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(const T *__restrict__ q, const T *__restrict__ w,
                    const float *__restrict__ beta, T *__restrict__ kc, const T *__restrict__ vc,
                    int cache_len, int cap, int nsplit, float scale_log2, float *__restrict__ part) {
    constexpr int E = Vec<T>::E;
    constexpr int TPK = kD / E;   // lanes per key
    constexpr int KPW = 32 / TPK; // keys per warp pass
    __shared__ float sm_m[kWarps * KPW], sm_l[kWarps * KPW];
    __shared__ float sm_o[kWarps * KPW][kD];

    const int sp = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / TPK, e0 = (lane % TPK) * E;
    const size_t head = (size_t)bh;

    float qv[E], wv[E];
    Vec<T>::load(q + head * kD + e0, qv);
    Vec<T>::load(w + head * kD + e0, wv);
    const float bt = beta[head];

    const int j0 = sp * kDecodeChunk;
    const int j1 = min(j0 + kDecodeChunk, cache_len);
    float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;

    T *krow = kc + head * cap * kD + e0;
    const T *vrow = vc + head * cap * kD + e0;
    // warp-uniform trip count: every lane joins the shuffles, lanes past the end idle
    for (int jb = j0 + warp * KPW; jb < j1; jb += kWarps * KPW) {
        const int j = jb + g;
        const bool valid = j < j1;
        float kv[E], vv[E];
        if (valid) {
            Vec<T>::load(krow + (size_t)j * kD, kv);
            Vec<T>::load(vrow + (size_t)j * kD, vv);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) kv[e] = vv[e] = 0.f;
        }
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
        if (valid) Vec<T>::store(krow + (size_t)j * kD, kv);
#pragma unroll
        for (int off = 1; off < TPK; off <<= 1) dq += __shfl_xor_sync(0xffffffffu, dq, off);
        if (!valid) continue;
        const float xl = dq * scale_log2;
        const float m_new = fmaxf(m, xl);
        const float sc = exp2f(m - m_new);  // 0 while m is -inf
        const float p = exp2f(xl - m_new);
        l = l * sc + p;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf(p, vv[e], o[e] * sc);
        m = m_new;
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
    if (threadIdx.x < kD) {
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
        float *dst = part + (head * nsplit + sp) * (kD + 2);
        dst[2 + c] = Oc;
        if (c == 0) {
            dst[0] = M;
            dst[1] = Ls;
        }
    }
}

// One CTA of 64 threads per head: append (k_t, v_t), score the new key and merge splits.
template <typename T>
__global__ void __launch_bounds__(kD)
decode_merge_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    T *__restrict__ kc, T *__restrict__ vc, int cache_len, int cap, int nsplit,
                    float scale_log2, const float *__restrict__ part, T *__restrict__ out) {
    __shared__ float red[2];
    const int bh = blockIdx.x, c = threadIdx.x;
    const size_t head = (size_t)bh;
    const T kt = k[head * kD + c], vt = v[head * kD + c];
    kc[(head * cap + cache_len) * kD + c] = kt;
    vc[(head * cap + cache_len) * kD + c] = vt;
    float d = Elt<T>::to_f(q[head * kD + c]) * Elt<T>::to_f(kt);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if ((c & 31) == 0) red[c >> 5] = d;
    __syncthreads();
    const float x_new = (red[0] + red[1]) * scale_log2;
    const float *pp = part + head * nsplit * (kD + 2);
    float M = x_new;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pp[s * (kD + 2)]);
    const float f_new = exp2f(x_new - M);
    float Ls = f_new, Oc = f_new * Elt<T>::to_f(vt);
    for (int s = 0; s < nsplit; ++s) {
        const float ms = pp[s * (kD + 2)];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        Ls += pp[s * (kD + 2) + 1] * f;
        Oc += pp[s * (kD + 2) + 2 + c] * f;
    }
    out[head * kD + c] = Elt<T>::from_f(Oc / Ls);
}

}  // namespace

template <typename T>
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *w,
                          const float *beta, void *k_cache, void *v_cache, int BH, int cache_len,
                          int cap, float scale, void *out, void *ws, cudaStream_t stream) {
    const int nsplit = decode_splits(cap);
    float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + 256);
    const float sl2 = scale * kLog2e;
    const int used = (cache_len + kDecodeChunk - 1) / kDecodeChunk;
    if (used > 0) {
        dim3 grid(used, BH);
        decode_split_kernel<T><<<grid, kThreads, 0, stream>>>(
            static_cast<const T *>(q), static_cast<const T *>(w), beta, static_cast<T *>(k_cache),
            static_cast<const T *>(v_cache), cache_len, cap, used, sl2, part);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    decode_merge_kernel<T><<<BH, kD, 0, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<T *>(k_cache), static_cast<T *>(v_cache), cache_len, cap, used, sl2, part,
        static_cast<T *>(out));
    return cudaGetLastError();
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
}  // namespace

// Device address of the static scratch on the current device. The first call on a
// device looks it up (host code only holds a stand-in for the symbol, never its device
// address) and caches it; later calls reuse the cached pointer.
static cudaError_t static_scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

size_t decode_static_scratch_bytes() { return kStaticScratchBytes; }

size_t decode_static_scratch_needed(int BH, int cache_len) {
    const size_t used = (size_t)((cache_len + kDecodeChunk - 1) / kDecodeChunk);
    return (size_t)BH * used * (kD + 2) * sizeof(float);
}

// Same kernels as launch_decode, with the partials in the static scratch. The caller
// has checked decode_static_scratch_needed() <= decode_static_scratch_bytes().
template <typename T>
cudaError_t launch_decode_static(const void *q, const void *k, const void *v, const void *w,
                                 const float *beta, void *k_cache, void *v_cache, int BH,
                                 int cache_len, int cap, float scale, void *out,
                                 cudaStream_t stream) {
    void *scratch = nullptr;
    cudaError_t err = static_scratch_address(&scratch);
    if (err != cudaSuccess) return err;
    float *part = static_cast<float *>(scratch);
    const float sl2 = scale * kLog2e;
    const int used = (cache_len + kDecodeChunk - 1) / kDecodeChunk;
    if (used > 0) {
        dim3 grid(used, BH);
        decode_split_kernel<T><<<grid, kThreads, 0, stream>>>(
            static_cast<const T *>(q), static_cast<const T *>(w), beta, static_cast<T *>(k_cache),
            static_cast<const T *>(v_cache), cache_len, cap, used, sl2, part);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    decode_merge_kernel<T><<<BH, kD, 0, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<T *>(k_cache), static_cast<T *>(v_cache), cache_len, cap, used, sl2, part,
        static_cast<T *>(out));
    return cudaGetLastError();
}

template cudaError_t launch_decode_static<float>(const void *, const void *, const void *,
                                                 const void *, const float *, void *, void *,
                                                 int, int, int, float, void *, cudaStream_t);
template cudaError_t launch_decode_static<__nv_bfloat16>(const void *, const void *,
                                                         const void *, const void *,
                                                         const float *, void *, void *, int, int,
                                                         int, float, void *, cudaStream_t);

template cudaError_t launch_decode<float>(const void *, const void *, const void *, const void *,
                                          const float *, void *, void *, int, int, int, float,
                                          void *, void *, cudaStream_t);
template cudaError_t launch_decode<__nv_bfloat16>(const void *, const void *, const void *,
                                                  const void *, const float *, void *, void *,
                                                  int, int, int, float, void *, void *,
                                                  cudaStream_t);

}  // namespace path
