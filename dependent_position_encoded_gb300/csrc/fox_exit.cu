// PaTH-FoX: the forget-gate prefix sums and the scan's exact-within-rounding early exit.
//
// Review "거리에서 경로로, PaTH Attention" §4 and technical summary "技術要約: PaTH
// Attention" §2 ("拡張: PaTH-FoX"): the FoX logit of row i against key j adds the data-
// dependent forget-gate bias sum_{s=j+1..i} log f_s = c_i - c_j with c the inclusive
// prefix sum of log f. Everything here is in log2 units (c2 = log2(e) * c), like the
// scan's logits.
//
// Early exit. Every H_s = I - beta_s w_s w_s^T with beta_s in [0, 2] and unit w_s is a
// contraction, so the state a row carries down the scan, x = P_{b+1} ... q~_i, has
// |x| <= |q~_i|, and every PaTH logit against a key of block b is bounded by
// |scale| |q~_i| max_{j in b} |k~_j|. The bias against block b is at most c_i - min_{j in b}
// c_j. Hence if, for every key block b' <= b,
//     c2_i - Mpre(b) + 2 |scale| log2(e) |q~_i| Kpre(b) < m_i - 40 log2(e),
// with Mpre(b) the minimum of c2 over blocks 0..b, Kpre(b) the maximum of |k~_j| over
// blocks 0..b and m_i any lower bound of the row's running maximum, every key in blocks
// 0..b weighs less than e^-40 relative to the row's largest weight and the scan may stop
// above block b. The factor 2 covers the rounding of the bf16 state and keys (their
// transitions are contractions only up to rounding). m_i here is the row's largest
// diagonal-block logit, which the running maximum can only exceed, so every scan role
// knows its extent before it starts. The left side grows with b, so the first block a
// query block needs is found by bisection.
#include "common.cuh"

namespace path {

namespace {

constexpr float kExitLog2 = 40.f * kLog2e;  // e^-40 relative weight, in log2 units

// Squared Euclidean norm of one 64-element row (16-byte loads).
__device__ __forceinline__ float row_norm2(const __nv_bfloat16 *row) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = __ldg(p + c);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            s = fmaf(f.x, f.x, s);
            s = fmaf(f.y, f.y, s);
        }
    }
    return s;
}
__device__ __forceinline__ float row_norm2(const float *row) {
    const float4 *p = reinterpret_cast<const float4 *>(row);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float4 f = __ldg(p + c);
        s = fmaf(f.x, f.x, s);
        s = fmaf(f.y, f.y, s);
        s = fmaf(f.z, f.z, s);
        s = fmaf(f.w, f.w, s);
    }
    return s;
}

// Largest entry of one 64-element row of the diagonal-block table (entries above the
// diagonal and beyond L hold -inf).
__device__ __forceinline__ float row_max(const __half *row) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row);
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = __ldg(p + c);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
            m = fmaxf(m, fmaxf(f.x, f.y));
        }
    }
    return m;
}
__device__ __forceinline__ float row_max(const float *row) {
    const float4 *p = reinterpret_cast<const float4 *>(row);
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float4 f = __ldg(p + c);
        m = fmaxf(m, fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w)));
    }
    return m;
}

// Per head (one CTA of 1024 threads, 16 blocks of 64 tokens per pass):
//   c2[t]   = log2(e) * sum_{s<=t} log f_s   (padded positions repeat the last value)
//   mpre[b] = min of c2 over blocks 0..b,  kpre[b] = max of |k~_j| over real tokens of
//   blocks 0..b (k~ from the preprocessing workspace, which must already be written).
template <typename T>
__global__ void __launch_bounds__(1024)
fox_bounds_kernel(const float *__restrict__ log_f, const T *__restrict__ kp, int L, int Lp,
                  int nblk, float *__restrict__ c2, float *__restrict__ mpre,
                  float *__restrict__ kpre) {
    __shared__ float warp_tot[32], warp_min[32], warp_max[32];
    __shared__ float carry_s, cmin_s, kmax_s;
    const int bh = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float *src = log_f + (size_t)bh * L;
    float *dst = c2 + (size_t)bh * Lp;
    if (tid == 0) {
        carry_s = 0.f;
        cmin_s = INFINITY;
        kmax_s = 0.f;
    }
    __syncthreads();
    for (int base = 0; base < Lp; base += 1024) {
        const int t = base + tid;
        float x = (t < L) ? src[t] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            float y = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) y += n;
            }
            warp_tot[lane] = y;
        }
        __syncthreads();
        const float v = carry_s + x + (wid > 0 ? warp_tot[wid - 1] : 0.f);
        const float cv = kLog2e * v;
        if (t < Lp) dst[t] = cv;
        float kn = 0.f;
        if (t < L) {
            const T *row = kp + (((size_t)bh * nblk + (t >> 6)) * (2 * kC) + (t & 63)) * kD;
            kn = sqrtf(row_norm2(row));
        }
        float cm = (t < Lp) ? cv : INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            cm = fminf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            kn = fmaxf(kn, __shfl_xor_sync(0xffffffffu, kn, o));
        }
        if (lane == 0) {
            warp_min[wid] = cm;
            warp_max[wid] = kn;
        }
        __syncthreads();
        if (tid == 1023) carry_s = v;
        if (tid == 0) {
            // blocks of 64 tokens = warp pairs; running minimum / maximum across blocks
            float cmin = cmin_s, kmax = kmax_s;
            for (int k = 0; k < 16; ++k) {
                const int b = (base >> 6) + k;
                if (b >= nblk) break;
                cmin = fminf(cmin, fminf(warp_min[2 * k], warp_min[2 * k + 1]));
                kmax = fmaxf(kmax, fmaxf(warp_max[2 * k], warp_max[2 * k + 1]));
                mpre[(size_t)bh * nblk + b] = cmin;
                kpre[(size_t)bh * nblk + b] = kmax;
            }
            cmin_s = cmin;
            kmax_s = kmax;
        }
        __syncthreads();
    }
}

// first[bh][qb]: the lowest key block any row of query block qb needs (qb itself when no
// earlier block is needed). One CTA of 64 threads (one row each) per query block.
template <typename T, typename D>
__global__ void __launch_bounds__(64)
fox_exit_kernel(const T *__restrict__ qt, const D *__restrict__ dg,
                const float *__restrict__ c2, const float *__restrict__ mpre,
                const float *__restrict__ kpre, int L, int Lp, int nblk, float abs_scale_log2,
                int *__restrict__ first) {
    __shared__ int warp_first[2];
    const int qb = blockIdx.x, bh = blockIdx.y, r = threadIdx.x;
    const int i = qb * kC + r;
    int lo = qb;
    if (i < L && qb > 0) {
        const float qn = sqrtf(row_norm2(qt + ((size_t)bh * Lp + i) * kD));
        const float dmax = row_max(dg + (((size_t)bh * nblk + qb) * kC + r) * kC);
        const float rhs = dmax - kExitLog2;
        const float ci = c2[(size_t)bh * Lp + i];
        const float qk = 2.f * abs_scale_log2 * qn;
        const float *mp = mpre + (size_t)bh * nblk;
        const float *kq = kpre + (size_t)bh * nblk;
        // smallest b in [0, qb) whose prefix bound is not below rhs (qb if there is none);
        // a NaN anywhere makes nothing skippable
        int hi = qb;
        lo = 0;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const bool skippable = (ci - mp[mid] + qk * kq[mid]) < rhs;
            if (skippable) lo = mid + 1;
            else hi = mid;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    if ((r & 31) == 0) warp_first[r >> 5] = lo;
    __syncthreads();
    if (r == 0) first[(size_t)bh * nblk + qb] = min(warp_first[0], warp_first[1]);
}

}  // namespace

cudaError_t launch_fox_prepare(const float *log_f, int BH, int L, int elt_bytes, float scale,
                               void *ws, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, elt_bytes, true);
    char *basep = static_cast<char *>(ws);
    float *c2 = reinterpret_cast<float *>(basep + lay.off_c2);
    float *mpre = reinterpret_cast<float *>(basep + lay.off_mpre);
    float *kpre = reinterpret_cast<float *>(basep + lay.off_kpre);
    int *first = reinterpret_cast<int *>(basep + lay.off_fb);
    const float s = fabsf(scale) * kLog2e;
    const dim3 grid(lay.nblk, BH);
    if (elt_bytes == 2) {
        fox_bounds_kernel<__nv_bfloat16><<<BH, 1024, 0, stream>>>(
            log_f, reinterpret_cast<const __nv_bfloat16 *>(basep + lay.off_kp), L, lay.Lp,
            lay.nblk, c2, mpre, kpre);
        fox_exit_kernel<__nv_bfloat16, __half><<<grid, 64, 0, stream>>>(
            reinterpret_cast<const __nv_bfloat16 *>(basep + lay.off_qt),
            reinterpret_cast<const __half *>(basep + lay.off_dg), c2, mpre, kpre, L, lay.Lp,
            lay.nblk, s, first);
    } else {
        fox_bounds_kernel<float><<<BH, 1024, 0, stream>>>(
            log_f, reinterpret_cast<const float *>(basep + lay.off_kp), L, lay.Lp, lay.nblk, c2,
            mpre, kpre);
        fox_exit_kernel<float, float><<<grid, 64, 0, stream>>>(
            reinterpret_cast<const float *>(basep + lay.off_qt),
            reinterpret_cast<const float *>(basep + lay.off_dg), c2, mpre, kpre, L, lay.Lp,
            lay.nblk, s, first);
    }
    return cudaGetLastError();
}

}  // namespace path
