// PaTH-FoX: the forget-gate prefix sums and the scan's exact-within-rounding early exit.
//
// Review "거리에서 경로로, PaTH Attention" §4 and technical summary "技術要約: PaTH
// Attention" §2 ("拡張: PaTH-FoX"): the FoX logit of row i against key j adds the data-
// dependent forget-gate bias sum_{s=j+1..i} log f_s = c_i - c_j with c the inclusive
// prefix sum of log f. Everything here is in log2 units (c2 = log2(e) * c), like the
// scan's logits. The sums are accumulated in fp64 (per block, then over block totals): c_i
// itself can reach thousands over a long sequence, and one fp32 difference c_i - c_j would
// carry an error of about ulp(|c_i|) even for neighbouring tokens. So each token stores
// c2 relative to the base of its pair of 64-token blocks (small, fp32), and each pair its
// base as an fp32 pair hi + lo; the scan forms c2_i - c2_j as
//     [(hi_P(i) - hi_u) + (lo_P(i) - lo_u) + rel_i] - rel_j      (j in pair u),
// the bracket once per row and step, accurate to the size of the bias.
// Three passes: per key block (fp64 total, in-block minimum, key-norm maximum; for bf16
// inputs the tensor-core preparation forms these as it goes, so this pass runs for fp32
// inputs only), per head over the block totals (offsets and prefix bounds), per query
// block (its c2 values and its early-exit extent).
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

// Inclusive prefix sum of log f within one 64-token block, in fp64 (64 threads, one token
// each; tokens at or beyond L contribute 0).
__device__ __forceinline__ double block_prefix(const float *__restrict__ log_f, int L, int bh,
                                               int blk, double *warp_tot) {
    const int r = threadIdx.x, lane = r & 31, wid = r >> 5;
    const int t = blk * kC + r;
    double x = (t < L) ? (double)log_f[(size_t)bh * L + t] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += n;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 1) x += warp_tot[0];
    return x;
}

// Per key block (64 threads): its total of log f, the minimum of its in-block prefix sums
// (both fp64) and, with ROWS, the largest |k~_j| over its real tokens (k~ from the
// preprocessing workspace, which must already be written; without ROWS the bf16
// preprocessing has written that maximum itself).
template <typename T, bool ROWS>
__global__ void __launch_bounds__(64)
fox_block_kernel(const float *__restrict__ log_f, const T *__restrict__ kp, int L, int nblk,
                 double *__restrict__ btot, double *__restrict__ bmin, float *__restrict__ bkmax) {
    __shared__ double warp_tot[2], warp_min[2];
    __shared__ float warp_kmax[2];
    const int b = blockIdx.x, bh = blockIdx.y, r = threadIdx.x, lane = r & 31, wid = r >> 5;
    const double loc = block_prefix(log_f, L, bh, b, warp_tot);
    const int t = b * kC + r;
    float kn = 0.f;
    if (ROWS && t < L) kn = sqrtf(row_norm2(kp + (((size_t)bh * nblk + b) * (2 * kC) + r) * kD));
    double m = loc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = fmin(m, __shfl_xor_sync(0xffffffffu, m, o));
        kn = fmaxf(kn, __shfl_xor_sync(0xffffffffu, kn, o));
    }
    __syncthreads();  // warp_tot was read by block_prefix
    if (lane == 0) {
        warp_min[wid] = m;
        warp_kmax[wid] = kn;
    }
    __syncthreads();
    if (r == kC - 1) btot[(size_t)bh * nblk + b] = loc;
    if (r == 0) {
        bmin[(size_t)bh * nblk + b] = fmin(warp_min[0], warp_min[1]);
        if (ROWS) bkmax[(size_t)bh * nblk + b] = fmaxf(warp_kmax[0], warp_kmax[1]);
    }
}

// Per head (256 threads over its key blocks): the fp64 offset of every block (the sum of
// log f over all earlier blocks), and in log2 units the prefix bounds
//   mpre[b] = min of c2 over blocks 0..b,   kpre[b] = max of |k~_j| over blocks 0..b.
__global__ void __launch_bounds__(256)
fox_prefix_kernel(const double *__restrict__ btot, const double *__restrict__ bmin,
                  const float *__restrict__ bkmax, int nblk, double *__restrict__ boff,
                  float *__restrict__ mpre, float *__restrict__ kpre) {
    __shared__ double w_sum[8], w_min[8];
    __shared__ float w_max[8];
    __shared__ double c_off, c_min;
    __shared__ float c_max;
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        c_off = 0.0;
        c_min = INFINITY;
        c_max = 0.f;
    }
    __syncthreads();
    for (int base = 0; base < nblk; base += 256) {
        const int b = base + tid;
        const size_t g = (size_t)bh * nblk + b;
        const double tot = (b < nblk) ? btot[g] : 0.0;
        // exclusive prefix of the block totals
        double x = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        if (lane == 31) w_sum[wid] = x;
        __syncthreads();
        double before = c_off;
        for (int w = 0; w < wid; ++w) before += w_sum[w];
        const double off = before + x - tot;
        // prefix minimum of the block minima of c, prefix maximum of |k~|
        double m = (b < nblk) ? off + bmin[g] : INFINITY;
        float k = (b < nblk) ? bkmax[g] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double nm = __shfl_up_sync(0xffffffffu, m, o);
            const float nk = __shfl_up_sync(0xffffffffu, k, o);
            if (lane >= o) {
                m = fmin(m, nm);
                k = fmaxf(k, nk);
            }
        }
        if (lane == 31) {
            w_min[wid] = m;
            w_max[wid] = k;
        }
        __syncthreads();
        double pm = c_min;
        float pk = c_max;
        for (int w = 0; w < wid; ++w) {
            pm = fmin(pm, w_min[w]);
            pk = fmaxf(pk, w_max[w]);
        }
        pm = fmin(pm, m);
        pk = fmaxf(pk, k);
        if (b < nblk) {
            boff[g] = off;
            mpre[g] = (float)(pm * (double)kLog2e);
            kpre[g] = pk;
        }
        __syncthreads();
        if (tid == 255) {
            c_off = off + tot;
            c_min = pm;
            c_max = pk;
        }
        __syncthreads();
    }
}

// Per query block (64 threads, one row each): with C2 first writes c2 of its 64 positions,
// c2_i = log2(e) (offset of the block + in-block prefix), as an fp32 pair hi + lo (so that
// differences c2_i - c2_j stay accurate to their own size however large the sums grow; the
// head-size-128 scan forms its bias from its own sums and needs none); then
// first[bh][qb], the lowest key block any of its rows needs (qb itself when no earlier
// block is needed). With ROWS the row norms |q~_i| and diagonal-table maxima are read from
// the rows; without, from the per-row values the bf16 preprocessing wrote.
template <typename T, typename D, bool ROWS, bool C2 = true>
__global__ void __launch_bounds__(64)
fox_exit_kernel(const float *__restrict__ log_f, const double *__restrict__ boff,
                const T *__restrict__ qt, const D *__restrict__ dg,
                const float *__restrict__ qn_row, const float *__restrict__ dmax_row,
                float *__restrict__ c2,
                float *__restrict__ pbase, const float *__restrict__ mpre,
                const float *__restrict__ kpre, int L, int Lp, int nblk, float abs_scale_log2,
                int *__restrict__ first) {
    __shared__ int warp_first[2];
    __shared__ double warp_tot[2];
    const int qb = blockIdx.x, bh = blockIdx.y, r = threadIdx.x;
    const int i = qb * kC + r;
    const double loc = block_prefix(log_f, L, bh, qb, warp_tot);
    const double own = boff[(size_t)bh * nblk + qb], base = boff[(size_t)bh * nblk + (qb & ~1)];
    const double cd = (own + loc) * (double)kLog2e;
    const float c_hi = (float)cd;
    if (C2) c2[(size_t)bh * Lp + i] = (float)((own - base + loc) * (double)kLog2e);
    if (C2 && r == 0 && (qb & 1) == 0) {
        const double bd = base * (double)kLog2e;
        const float bh_hi = (float)bd;
        float *pb = pbase + ((size_t)bh * (nblk >> 1) + (qb >> 1)) * 2;
        pb[0] = bh_hi;
        pb[1] = (float)(bd - (double)bh_hi);
    }
    int lo = qb;
    if (i < L && qb > 0) {
        const float qn = ROWS ? sqrtf(row_norm2(qt + ((size_t)bh * Lp + i) * kD))
                              : qn_row[(size_t)bh * Lp + i];
        const float dmax = ROWS ? row_max(dg + (((size_t)bh * nblk + qb) * kC + r) * kC)
                                : dmax_row[(size_t)bh * Lp + i];
        const float rhs = dmax - kExitLog2;
        const float ci = c_hi;
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

// Head size 128 (bf16, tensor-core preparation): the same prefix and extent passes over the
// d128_tc_layout workspace, from the per-row and per-block values the preparation wrote.
cudaError_t launch_fox_exit_d128(const float *log_f, int BH, int L, float scale, void *ws,
                                 cudaStream_t stream) {
    const D128TcLayout y = d128_tc_layout(1, BH, L, true);
    char *basep = static_cast<char *>(ws);
    double *btot = reinterpret_cast<double *>(basep + y.off_btot);
    double *bmin = reinterpret_cast<double *>(basep + y.off_bmin);
    double *boff = reinterpret_cast<double *>(basep + y.off_boff);
    float *bkmax = reinterpret_cast<float *>(basep + y.off_bkmax);
    float *mpre = reinterpret_cast<float *>(basep + y.off_mpre);
    float *kpre = reinterpret_cast<float *>(basep + y.off_kpre);
    fox_prefix_kernel<<<BH, 256, 0, stream>>>(btot, bmin, bkmax, y.nblk, boff, mpre, kpre);
    fox_exit_kernel<__nv_bfloat16, __half, false, false><<<dim3(y.nblk, BH), 64, 0, stream>>>(
        log_f, boff, nullptr, nullptr, reinterpret_cast<const float *>(basep + y.off_qn),
        reinterpret_cast<const float *>(basep + y.off_dmax), nullptr, nullptr, mpre, kpre, L,
        y.Lp, y.nblk, fabsf(scale) * kLog2e, reinterpret_cast<int *>(basep + y.off_first));
    return cudaGetLastError();
}

cudaError_t launch_fox_prepare(const float *log_f, int BH, int L, int elt_bytes, float scale,
                               void *ws, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, elt_bytes, true);
    char *basep = static_cast<char *>(ws);
    float *c2 = reinterpret_cast<float *>(basep + lay.off_c2);
    float *pbase = reinterpret_cast<float *>(basep + lay.off_pbase);
    float *mpre = reinterpret_cast<float *>(basep + lay.off_mpre);
    float *kpre = reinterpret_cast<float *>(basep + lay.off_kpre);
    int *first = reinterpret_cast<int *>(basep + lay.off_fb);
    double *btot = reinterpret_cast<double *>(basep + lay.off_btot);
    double *bmin = reinterpret_cast<double *>(basep + lay.off_bmin);
    double *boff = reinterpret_cast<double *>(basep + lay.off_boff);
    float *bkmax = reinterpret_cast<float *>(basep + lay.off_bkmax);
    const float *qn = reinterpret_cast<const float *>(basep + lay.off_qn);
    const float *dmax = reinterpret_cast<const float *>(basep + lay.off_dmax);
    const float s = fabsf(scale) * kLog2e;
    const dim3 grid(lay.nblk, BH);
    // bf16: the tensor-core preprocessing has written |q~|, the table maxima, the key-norm
    // maxima and the blocks' fp64 gate totals and minima; fp32: a per-block pass forms them
    if (elt_bytes != 2)
        fox_block_kernel<float, true><<<grid, 64, 0, stream>>>(
            log_f, reinterpret_cast<const float *>(basep + lay.off_kp), L, lay.nblk, btot, bmin,
            bkmax);
    fox_prefix_kernel<<<BH, 256, 0, stream>>>(btot, bmin, bkmax, lay.nblk, boff, mpre, kpre);
    if (elt_bytes == 2)
        fox_exit_kernel<__nv_bfloat16, __half, false><<<grid, 64, 0, stream>>>(
            log_f, boff, reinterpret_cast<const __nv_bfloat16 *>(basep + lay.off_qt),
            reinterpret_cast<const __half *>(basep + lay.off_dg), qn, dmax, c2, pbase, mpre, kpre,
            L, lay.Lp,
            lay.nblk, s, first);
    else
        fox_exit_kernel<float, float, true><<<grid, 64, 0, stream>>>(
            log_f, boff, reinterpret_cast<const float *>(basep + lay.off_qt),
            reinterpret_cast<const float *>(basep + lay.off_dg), qn, dmax, c2, pbase, mpre, kpre, L,
            lay.Lp,
            lay.nblk, s, first);
    return cudaGetLastError();
}

}  // namespace path
