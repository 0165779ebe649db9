// K2 (fp32 dtype): the right-to-left block scan of PaTH attention in fp32 FFMA.
//
// Same algorithm as the tensor-core scan (technical summary "技術要約: PaTH Attention" §3;
// review "거리에서 경로로, PaTH Attention" §9), for fp32 inputs whose tolerance rules out
// bf16 operands: one CTA per 64-row query block of one head holds the state
// X = (q~_i)_i in shared memory and, for key block b = ib, ib-1, ..., 0, forms the
// logits (diagonal block: precomputed; earlier blocks: X K~_b^T), updates the online
// softmax, accumulates O += P V_b and advances X <- X P_b^T.
#include "common.cuh"

namespace path {

namespace {

constexpr int LD = 68;
constexpr int BUF = kC * LD;
constexpr int kThreads = 256;

// acc1[i][j] += sum_k A[r0 + 16i][k] B1[n0 + 16j][k] and acc2 likewise with B2: all three
// row-major with the contraction (the head dimension) contiguous, each A piece loaded once
// for both products. The eight lanes of a quarter warp read eight consecutive B rows: at a
// stride of LD = 68 floats their 16-byte pieces fall in distinct bank groups.
__device__ __forceinline__ void mm_rows2(const float *__restrict__ A, const float *__restrict__ B1,
                                         const float *__restrict__ B2, int r0, int n0,
                                         float (&acc1)[4][4], float (&acc2)[4][4]) {
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 16 * i) * LD + k);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 b = *reinterpret_cast<const float4 *>((j < 4 ? B1 : B2) + (n0 + 16 * (j & 3)) * LD + k);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float t = j < 4 ? acc1[i][j & 3] : acc2[i][j & 3];
                t = fmaf(a[i].x, b.x, t);
                t = fmaf(a[i].y, b.y, t);
                t = fmaf(a[i].z, b.z, t);
                t = fmaf(a[i].w, b.w, t);
                if (j < 4) acc1[i][j & 3] = t;
                else acc2[i][j & 3] = t;
            }
        }
    }
}

// acc[i][j] += sum_k A[r0 + 16i][k] B[k][c0 + j]: A row-major, B with the contraction as
// its row index (k-major).
__device__ __forceinline__ void mm_rowk(const float *__restrict__ A, const float *__restrict__ B,
                                        int r0, int c0, float (&acc)[4][4]) {
#pragma unroll 2
    for (int k = 0; k < kC; k += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 16 * i) * LD + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 b = *reinterpret_cast<const float4 *>(B + (k + kk) * LD + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                acc[i][0] = fmaf(av, b.x, acc[i][0]);
                acc[i][1] = fmaf(av, b.y, acc[i][1]);
                acc[i][2] = fmaf(av, b.z, acc[i][2]);
                acc[i][3] = fmaf(av, b.w, acc[i][3]);
            }
        }
    }
}

// 64 rows of 64 floats (row-major in global memory) into shared rows of stride LD; rows at
// or past `valid` are zero. Four 16-byte loads per thread, all in flight before the stores.
__device__ __forceinline__ void load_rows64(float *dst, const float *__restrict__ src, int valid) {
    float4 x[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int e = (int)threadIdx.x + it * kThreads, r = e >> 4;
        x[it] = r < valid ? reinterpret_cast<const float4 *>(src)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int e = (int)threadIdx.x + it * kThreads, r = e >> 4, c = 4 * (e & 15);
        *reinterpret_cast<float4 *>(dst + r * LD + c) = x[it];
    }
}

// Thread (ty, tx) owns rows ty + 16i of every 64 x 64 product: columns tx + 16j of the
// logits and the new state, columns 4tx .. 4tx + 3 of the output.
template <bool FOX>
__global__ void __launch_bounds__(kThreads)
path_scan_f32_kernel(const float *__restrict__ v, const float *__restrict__ qt,
                     const float *__restrict__ kp, const float *__restrict__ dg,
                     const float *__restrict__ c2, const float *__restrict__ pbase,
                     const int *__restrict__ first_blk,
                     float *__restrict__ out, float *__restrict__ lse, int L, int Lp, int nblk,
                     float scale_log2, int heads_fast) {
    extern __shared__ __align__(16) float sm[];
    float *Xr = sm;          // state X[i][c]
    float *KB = Xr + BUF;    // k~_b [j][c]
    float *PB = KB + BUF;    // P_b [n][c]
    float *Vs = PB + BUF;    // V_b [j][c]
    float *Ss = Vs + BUF;    // logits S[i][j] (log2 units)
    float *Pm = Ss + BUF;    // probabilities [i][j]
    float *alpha_s = Pm + BUF;
    float *c2k = alpha_s + kC;

    const int tid = threadIdx.x;
    // longest walks (the last query blocks) first, heads fastest or head by head
    // (heads_fastest)
    const int nq = (int)(heads_fast ? gridDim.y : gridDim.x);
    const int ib = nq - 1 - (int)(heads_fast ? blockIdx.y : blockIdx.x);
    const int bh = heads_fast ? blockIdx.x : blockIdx.y;
    if (ib * kC >= L) return;
    const size_t head = (size_t)bh;
    const int ty = tid / 16, tx = tid % 16, c0 = 4 * tx;
    const int row = tid >> 2, part = tid & 3;  // softmax: 4 threads per row
    float m_run = -INFINITY, l_run = 0.f;
    // gate sums relative to the base of their pair of blocks; per key block the row's
    // offset against pair b / 2 is (base_own - base) in fp32-pair arithmetic + rel_row
    const float rel_row = FOX ? c2[head * Lp + ib * kC + row] : 0.f;
    const int npair = nblk >> 1;
    const float2 base_own = FOX ? *reinterpret_cast<const float2 *>(pbase + (head * npair + (ib >> 1)) * 2)
                                : make_float2(0.f, 0.f);

    load_rows64(Xr, qt + (head * Lp + (size_t)ib * kC) * kD, kC);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    // PaTH-FoX stops above the blocks whose keys all weigh below e^-40 (see fox_exit.cu)
    const int b_last = FOX ? first_blk[head * nblk + ib] : 0;
    for (int b = ib; b >= b_last; --b) {
        __syncthreads();
        load_rows64(Vs, v + (head * L + (size_t)b * kC) * kD, L - b * kC);
        if (b < ib) {
            const float *blk = kp + ((head * nblk + b) * 2 * kC) * kD;
            load_rows64(KB, blk, kC);
            load_rows64(PB, blk + kC * kD, kC);
        } else {
            load_rows64(Ss, dg + (head * nblk + b) * kC * kC, kC);
        }
        if (FOX && b < ib && tid < kC) c2k[tid] = c2[head * Lp + b * kC + tid];
        float c2_row = 0.f;
        if (FOX && b < ib) {
            const float2 bb = *reinterpret_cast<const float2 *>(pbase + (head * npair + (b >> 1)) * 2);
            c2_row = ((base_own.x - bb.x) + (base_own.y - bb.y)) + rel_row;
        }
        __syncthreads();
        if (b < ib) {
            float s[4][4], xn[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = xn[i][j] = 0.f;
            mm_rows2(Xr, KB, PB, ty, tx, s, xn);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) Ss[(ty + 16 * i) * LD + tx + 16 * j] = s[i][j] * scale_log2;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) Xr[(ty + 16 * i) * LD + tx + 16 * j] = xn[i][j];
        }
        __syncthreads();
        // ---- online softmax, 4 threads per row, 16 columns each
        {
            float x[16];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                x[j] = Ss[row * LD + part * 16 + j];
                if (FOX && b < ib) x[j] += c2_row - c2k[part * 16 + j];
                mx = fmaxf(mx, x[j]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                float pj[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    pj[q] = exp2f(x[j + q] - m_use);
                    sum += pj[q];
                }
                *reinterpret_cast<float4 *>(Pm + row * LD + part * 16 + j) = make_float4(pj[0], pj[1], pj[2], pj[3]);
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            l_run = l_run * alpha + sum;
            m_run = m_new;
            if (part == 0) alpha_s[row] = alpha;
        }
        __syncthreads();
        {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float al = alpha_s[ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] *= al;
            }
            mm_rowk(Pm, Vs, ty, c0, acc);
        }
    }
    __syncthreads();
    if (part == 0) alpha_s[row] = (l_run > 0.f) ? 1.f / l_run : 0.f;
    if (lse != nullptr && part == 0 && ib * kC + row < L)
        lse[head * L + ib * kC + row] = (m_run + log2f(l_run)) * 0.69314718055994531f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty + 16 * i, t = ib * kC + r;
        if (t < L) {
            const float inv = alpha_s[r];
            *reinterpret_cast<float4 *>(out + (head * L + t) * kD + c0) =
                make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
        }
    }
}

}  // namespace

cudaError_t launch_scan_f32(const void *v, void *out, float *lse, bool fox, int BH, int L,
                            float scale, void *ws, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 4, fox);
    char *basep = static_cast<char *>(ws);
    const size_t smem = (size_t)(6 * BUF + 2 * kC) * sizeof(float);
    auto kern = fox ? path_scan_f32_kernel<true> : path_scan_f32_kernel<false>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    // shared per token: k~, P_b rows and v (256 B each)
    const bool hf = heads_fastest((size_t)BH, (size_t)L, 768);
    const int nq = (L + kC - 1) / kC;
    const dim3 grid = hf ? dim3(BH, nq) : dim3(nq, BH);
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const float *>(v), reinterpret_cast<const float *>(basep + lay.off_qt),
        reinterpret_cast<const float *>(basep + lay.off_kp),
        reinterpret_cast<const float *>(basep + lay.off_dg),
        fox ? reinterpret_cast<const float *>(basep + lay.off_c2) : nullptr,
        fox ? reinterpret_cast<const float *>(basep + lay.off_pbase) : nullptr,
        fox ? reinterpret_cast<const int *>(basep + lay.off_fb) : nullptr,
        static_cast<float *>(out), lse, L, lay.Lp, lay.nblk, scale * kLog2e, hf ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace path
