// The UT factor's triangular inverse on the CUDA cores' tensor path (mma.sync, tf32),
// shared by the bf16 preparation and the bf16 backward's block pass.
//
// Technical summary "技術要約: PaTH Attention" §3 ("UT変換による表現"): a block's
// transitions combine as I - W^T A W with A = (I + D strictly-upper(W W^T))^{-1} D, so
// both need (I + E)^{-1} for a strictly upper triangular E. It is formed blockwise: the
// four 16 x 16 diagonal blocks by back-substitution, then X12 = -X11 E12 X22 for the
// 16-blocks and for the 32-blocks, each 16 x 8 output tile one warp's mma.sync with tf32
// operands. Every factor is bounded (X_su = A_su / beta_u), so no intermediate grows.
#pragma once
#include "common.cuh"

namespace path {
namespace ut_inverse {

constexpr int XLD = 68;  // row stride (floats) of the 64 x 64 fp32 matrix being inverted
constexpr int YLD = 40;  // B-fragment loads of the 32 x 32 scratch Y (rows t, columns g) hit 32 banks

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One warp: the 16 x 8 tile acc = A (16 x K, row-major, stride lda) x B (K x 8, row-major,
// stride ldb) on the tensor cores with tf32 operands (one product per k-step: the products
// feed A, which later MMAs take as fp16, so a 10-bit operand significand is enough).
// Fragment layout of m16n8k8: g = lane / 4, t = lane % 4; A rows g, g + 8 and columns
// t, t + 4; B rows t, t + 4 and column g; acc rows g (0, 1), g + 8 (2, 3), columns 2t, 2t + 1.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

template <int K>
__device__ __forceinline__ void warp_tile_16x8(const float *A, int lda, const float *B, int ldb,
                                               int lane, float (&acc)[4]) {
    const int g = lane >> 2, t = lane & 3;
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint32_t a[4] = {to_tf32(A[g * lda + k0 + t]), to_tf32(A[(g + 8) * lda + k0 + t]),
                               to_tf32(A[g * lda + k0 + t + 4]),
                               to_tf32(A[(g + 8) * lda + k0 + t + 4])};
        const uint32_t b[2] = {to_tf32(B[(k0 + t) * ldb + g]), to_tf32(B[(k0 + t + 4) * ldb + g])};
        mma_tf32(acc, a, b);
    }
}

// (I + E)^{-1} in place over E (upper triangle; E is zero on and below the diagonal),
// all 256 threads. On return X[s][u] (s <= u) holds the inverse.
__device__ __forceinline__ void blocked_unit_upper_inverse(float *X, float *Y, int r) {
    // level 0: the four 16 x 16 diagonal blocks, one column per thread (threads 0-63).
    // Column u of the inverse solves x_l = -sum_{m>l} E_lm x_m (x_lu = 1, x_l = 0 below);
    // right-looking: once x_m is final it is folded into the partial sums of every row
    // above, so the dependent chain is one FMA per row instead of a whole dot product.
    float x[16];
    const int u = r & 63, b0 = (u >> 4) << 4, lu = u & 15;
    if (r < 64) {
#pragma unroll
        for (int l = 0; l < 16; ++l) x[l] = 0.f;
#pragma unroll
        for (int m = 15; m >= 0; --m) {
            x[m] = (m == lu) ? 1.f : ((m < lu) ? -x[m] : 0.f);
#pragma unroll
            for (int l = 0; l < m; ++l) x[l] = fmaf(X[(b0 + l) * XLD + b0 + m], x[m], x[l]);
        }
    }
    __syncthreads();
    if (r < 64) {
#pragma unroll
        for (int l = 0; l < 16; ++l) X[(b0 + l) * XLD + u] = x[l];
    }
    __syncthreads();
    const int warp = r >> 5, lane = r & 31, g = lane >> 2, t = lane & 3;
    float acc[4];
    // level 1: X[o:o+16, o+16:o+32] = -X11 E12 X22 for the two 32-blocks (o = 0, 32);
    // warps 0-3, warp = (block p, 8-column tile n)
    if (warp < 4) {
        const int o = 32 * (warp >> 1), n0 = 8 * (warp & 1);
        warp_tile_16x8<16>(X + o * XLD + o + 16, XLD, X + (o + 16) * XLD + o + 16 + n0, XLD,
                           lane, acc);
        float *y = Y + (o >> 1) * YLD + n0;  // rows 16 p .. 16 p + 15 of Y
        *reinterpret_cast<float2 *>(y + g * YLD + 2 * t) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2 *>(y + (g + 8) * YLD + 2 * t) = make_float2(acc[2], acc[3]);
    }
    __syncthreads();
    if (warp < 4) {
        const int o = 32 * (warp >> 1), n0 = 8 * (warp & 1);
        warp_tile_16x8<16>(X + o * XLD + o, XLD, Y + (o >> 1) * YLD + n0, YLD, lane, acc);
        float *x12 = X + o * XLD + o + 16 + n0;
        *reinterpret_cast<float2 *>(x12 + g * XLD + 2 * t) = make_float2(-acc[0], -acc[1]);
        *reinterpret_cast<float2 *>(x12 + (g + 8) * XLD + 2 * t) = make_float2(-acc[2], -acc[3]);
    }
    __syncthreads();
    // level 2: X[0:32, 32:64] = -X[0:32, 0:32] E[0:32, 32:64] X[32:64, 32:64];
    // warp = (16-row tile m, 8-column tile n)
    {
        const int m0 = 16 * (warp >> 2), n0 = 8 * (warp & 3);
        warp_tile_16x8<32>(X + m0 * XLD + 32, XLD, X + 32 * XLD + 32 + n0, XLD, lane, acc);
        float *y = Y + m0 * YLD + n0;
        *reinterpret_cast<float2 *>(y + g * YLD + 2 * t) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2 *>(y + (g + 8) * YLD + 2 * t) = make_float2(acc[2], acc[3]);
        __syncthreads();
        warp_tile_16x8<32>(X + m0 * XLD, XLD, Y + n0, YLD, lane, acc);
        float *x12 = X + m0 * XLD + 32 + n0;
        *reinterpret_cast<float2 *>(x12 + g * XLD + 2 * t) = make_float2(-acc[0], -acc[1]);
        *reinterpret_cast<float2 *>(x12 + (g + 8) * XLD + 2 * t) = make_float2(-acc[2], -acc[3]);
    }
    __syncthreads();
}


}  // namespace ut_inverse
}  // namespace path
