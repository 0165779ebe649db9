// fp32 64 x 64 tile products on the CUDA cores, shared by the backward's fp32 query passes
// (head sizes 64 and 128: a 64 x 128 operand is two 64-column halves, a 128 x 128 one four
// quadrants, so every product is a sum of these tile products).
#pragma once

#include "common.cuh"

namespace path {
namespace bwd_f32 {

constexpr int LD = 68;          // padded row stride (floats) of a 64 x 64 shared buffer
constexpr int BUF = kC * LD;
constexpr int kThreads = 256;
constexpr int kBlkTile = kC * kD;  // floats in one 64 x 64 tile

// 64 x 64 fp32 tile from global (row-major, ld floats per row) into shared memory, as is
// (dst[r][c]) or transposed (dst[c][r]). Each thread issues all four of its 16-byte loads
// before the first store, so the tile costs one memory latency.
__device__ __forceinline__ void load_tile(float *dst, const float *__restrict__ src, bool transpose,
                                          int ld = kD) {
    constexpr int kIt = kBlkTile / 4 / kThreads;
    float4 x[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = 4 * (threadIdx.x + it * kThreads);
        x[it] = *reinterpret_cast<const float4 *>(src + (e / kD) * ld + e % kD);
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = 4 * (threadIdx.x + it * kThreads), r = e / kD, c = e % kD;
        if (transpose) {
            dst[c * LD + r] = x[it].x;
            dst[(c + 1) * LD + r] = x[it].y;
            dst[(c + 2) * LD + r] = x[it].z;
            dst[(c + 3) * LD + r] = x[it].w;
        } else {
            *reinterpret_cast<float4 *>(dst + r * LD + c) = x[it];
        }
    }
}

// Rows t0 .. t0 + 63, 64 columns, of a row-major tensor of type T with ld elements per row,
// zero past L, as is and transposed (either may be null); four elements per thread and step,
// all loads issued first.
template <typename T>
__device__ __forceinline__ void load_rows(float *dst, float *dst_t, const T *__restrict__ src,
                                          int t0, int L, int ld = kD) {
    constexpr int kIt = kBlkTile / 4 / kThreads;
    float x[kIt][4];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = 4 * (threadIdx.x + it * kThreads), r = e / kD, c = e % kD;
        const bool in = t0 + r < L;
        const T *p = src + (size_t)(t0 + r) * ld + c;
#pragma unroll
        for (int q = 0; q < 4; ++q) x[it][q] = in ? Elt<T>::to_f(p[q]) : 0.f;
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = 4 * (threadIdx.x + it * kThreads), r = e / kD, c = e % kD;
        if (dst) *reinterpret_cast<float4 *>(dst + r * LD + c) = make_float4(x[it][0], x[it][1], x[it][2], x[it][3]);
        if (dst_t)
#pragma unroll
            for (int q = 0; q < 4; ++q) dst_t[(c + q) * LD + r] = x[it][q];
    }
}

// Four groups of 64 threads; a group computes half (32 rows) of a 64 x 64 x 64 product as
// a 4 x 8 register tile per thread. Every operand stays in its stored row-major layout
// (no transposed copies); the three forms of product are
//   mm48:   A row-major (rows r0 + 8i), B k-major (columns col48(c0, j))     e.g. G P_b
//   mmrb48: A and B row-major, the contraction index contiguous in both (rows r0 + 8i,
//           columns n0 + 8j)                                                  e.g. X K~_b^T
//   mmkk48: A and B k-major (rows m0 + i, columns col48(c0, j))               e.g. dT^T X
// With ty, tx = the thread's row and column in its group (8 x 8), r0 = rb + ty,
// m0 = rb + 4 ty, c0 = 4 tx and n0 = tx (rb = 0 or 32, the group's half). The lanes of a
// quarter warp share the A rows (broadcast loads) and read eight distinct 16-byte pieces of
// B (contiguous, or eight consecutive rows at a stride of 68 floats).
__device__ __forceinline__ int col48(int c0, int j) { return c0 + (j < 4 ? j : 28 + j); }

// acc[i][j] += sum_k A[r0 + 8i][k] * B[k][col48(c0, j)]
__device__ __forceinline__ void mm48(const float *__restrict__ A, const float *__restrict__ B,
                                     int r0, int c0, float (&acc)[4][8]) {
#pragma unroll 2
    for (int k = 0; k < kC; k += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 8 * i) * LD + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 b0 = *reinterpret_cast<const float4 *>(B + (k + kk) * LD + c0);
            const float4 b1 = *reinterpret_cast<const float4 *>(B + (k + kk) * LD + c0 + 32);
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
            }
        }
    }
}

// acc[i][j] += sum_k A[r0 + 8i][k] * B[n0 + 8j][k]
__device__ __forceinline__ void mmrb48(const float *__restrict__ A, const float *__restrict__ B,
                                       int r0, int n0, float (&acc)[4][8]) {
#pragma unroll 1
    for (int k = 0; k < kC; k += 4) {
        float4 a[4], b[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 8 * i) * LD + k);
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = *reinterpret_cast<const float4 *>(B + (n0 + 8 * j) * LD + k);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float t = acc[i][j];
                t = fmaf(a[i].x, b[j].x, t);
                t = fmaf(a[i].y, b[j].y, t);
                t = fmaf(a[i].z, b[j].z, t);
                acc[i][j] = fmaf(a[i].w, b[j].w, t);
            }
    }
}

// acc[i][j] += sum_k A[k][m0 + i] * B[k][col48(c0, j)]
__device__ __forceinline__ void mmkk48(const float *__restrict__ A, const float *__restrict__ B,
                                       int m0, int c0, float (&acc)[4][8]) {
#pragma unroll 4
    for (int k = 0; k < kC; ++k) {
        const float4 a = *reinterpret_cast<const float4 *>(A + k * LD + m0);
        const float4 b0 = *reinterpret_cast<const float4 *>(B + k * LD + c0);
        const float4 b1 = *reinterpret_cast<const float4 *>(B + k * LD + c0 + 32);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

__device__ __forceinline__ void zero48(float (&a)[4][8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) a[i][j] = 0.f;
}

// an mm48 tile (rows r0 + 8i, columns col48) into shared memory
__device__ __forceinline__ void put48(float *dst, const float (&v)[4][8], int r0, int c0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + 8 * i;
        *reinterpret_cast<float4 *>(dst + r * LD + c0) = make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
        *reinterpret_cast<float4 *>(dst + r * LD + c0 + 32) = make_float4(v[i][4], v[i][5], v[i][6], v[i][7]);
    }
}

// an mm48 tile stored into a row-major global tile (ld floats per row)
__device__ __forceinline__ void st48(float *dst, const float (&v)[4][8], int r0, int c0, int ld = kC) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + 8 * i;
        *reinterpret_cast<float4 *>(dst + r * ld + c0) = make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
        *reinterpret_cast<float4 *>(dst + r * ld + c0 + 32) = make_float4(v[i][4], v[i][5], v[i][6], v[i][7]);
    }
}

// an mmrb48 tile (rows r0 + 8i, columns n0 + 8j) into a row-major buffer of stride ld
__device__ __forceinline__ void put_rb(float *dst, int ld, const float (&v)[4][8], int r0, int n0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[(r0 + 8 * i) * ld + n0 + 8 * j] = v[i][j];
}

// an mmkk48 tile (rows m0 + i, columns col48) added into a row-major global tile (ld
// floats per row)
__device__ __forceinline__ void red_kk(float *dst, const float (&v)[4][8], int m0, int c0, int ld = kC) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) atomicAdd(dst + (m0 + i) * ld + col48(c0, j), v[i][j]);
}

// PaTH-FoX: the dS row sums rp of a lead group's thread (its four rows, each then summed over
// the eight lanes that share the row) join rs_acc; the column sums cp go to csum_blk (the
// key block's 64 entries) with one atomic per column and warp.
__device__ __forceinline__ void fox_tile_sums(float (&rp)[4], float (&cp)[8], float (&rs_acc)[4],
                                              float *csum_blk, int n0) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) rp[i] += __shfl_xor_sync(0xffffffffu, rp[i], o);
        rs_acc[i] += rp[i];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        cp[j] += __shfl_xor_sync(0xffffffffu, cp[j], 8);
        cp[j] += __shfl_xor_sync(0xffffffffu, cp[j], 16);
        if (lane < 8) atomicAdd(csum_blk + n0 + 8 * j, cp[j]);
    }
}

}  // namespace bwd_f32
}  // namespace path
