// Backward block pass of PaTH attention for bf16 inputs, in matrix form on the tensor
// cores (mma.sync, tf32 operands, fp32 accumulation).
//
// The pages give no backward (review "거리에서 경로로, PaTH Attention" §9 and technical
// summary "技術要約: PaTH Attention" §3 only say the block-wise algorithm makes training
// efficient). The query pass hands each 64-token block the gradients of its
// boundary-adjusted queries dq~, keys dk~, dense transition dP and diagonal-block logits dT
// (j <= i). The block's forward, in the UT form of summary §3 (D = diag(beta)):
//     G = W W^T,  A = (I + D strictly-upper(G))^{-1} D,
//     Lq = lower-incl(Q W^T),  Rk = strictly-upper(K W^T),  U = A^T W,  V = A W,
//     q~ = Q - Lq U,  k~ = K - Rk V,  P = I - W^T V,  T = Q K^T - Lq A^T Rk^T,
// so reverse mode gives dense 64 x 64 products only (Y = Lq A^T, dY = -dT Rk, X = the
// inverse, dX = dA D, dTT the gradient of I + D strictly-upper(G)):
//     dLq = tril(-dq~ U^T + dY A)             dRk = striu(-dk~ V^T - dT^T Y)
//     dU = -Lq^T dq~                          dV = -Rk^T dk~ - W dP
//     dA = dY^T Lq + W dU^T + dV W^T          dbeta_u += sum_s dA_su X_su
//     dTT = -X^T dX X^T                       dbeta_s += sum_{v>s} dTT_sv G_sv
//     dG = D strictly-upper(dTT)
//     dq = dq~ + dT K + dLq W                 dk = dk~ + dT^T Q + dRk W
//     dw = -V dP^T + dLq^T Q + dRk^T K + A dU + A^T dV + (dG + dG^T) W
// The same gradient as the token-level sweeps of backward.cu, which stay for fp32 inputs
// (the fp32 bar): those walk 192 sweeps of up to 64 dependent steps per block, whereas here
// each block is 31 products on the tensor cores. The products are small and on one
// dependent chain, so each is a warp-level mma.sync over fp32 tiles in shared memory (any
// operand read transposed by its fragment addressing); tf32 keeps the fp32 range with a
// 10-bit significand, well inside the bf16 inputs' error.
// One CTA of 256 threads per (block, head), twelve 64 x 64 fp32 tiles (204 KB), one CTA per
// SM. Warp w computes rows 16 (w >> 1) .. + 15 and columns 32 (w & 1) .. + 31 of every
// product (four m16n8k8 tiles). Padded tokens (past L) have zero q, k, w and beta, so their
// transitions are the identity; the inputs the sweeps ignore are zero here too: dP of the
// first and last block, dk~ of the last block, dT above the diagonal.
#include "common.cuh"
#include "ut_inverse.cuh"

namespace path {

namespace {

using ut_inverse::blocked_unit_upper_inverse;
using ut_inverse::mma_tf32;
using ut_inverse::XLD;
using ut_inverse::YLD;

constexpr int kThreads = 256;
constexpr int LD = XLD;                               // row stride of every tile (floats)
constexpr uint32_t kTile = 64 * LD * 4;               // one fp32 tile
constexpr int kTiles = 12;
constexpr uint32_t kYOff = kTiles * kTile;            // the inverse's 32 x YLD scratch
constexpr uint32_t kBetaOff = kYOff + 32 * YLD * 4;   // beta (64), d beta (64)
constexpr uint32_t kSmem = kBetaOff + 2 * 64 * 4;
static_assert(kSmem <= 227u * 1024u, "block-pass shared memory");

using Acc = float[4][4];  // four m16n8 tiles: [n-tile][c0, c1, c2, c3]

__device__ __forceinline__ void zero(Acc &a) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) a[j][e] = 0.f;
}

// Row and column of accumulator element (j, e) for the calling thread.
struct Frag {
    int m0, n0, g, t;
    __device__ Frag() {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        m0 = 16 * (w >> 1);
        n0 = 32 * (w & 1);
        g = lane >> 2;
        t = lane & 3;
    }
    __device__ __forceinline__ int row(int e) const { return m0 + g + 8 * (e >> 1); }
    __device__ __forceinline__ int col(int j, int e) const { return n0 + 8 * j + 2 * t + (e & 1); }
};

// Fragments of the tf32 m16n8k8 MMA from fp32 tiles. A non-transposed operand (A stored
// [i][k], B stored [j][k]: the contraction index contiguous) is read with ldmatrix: an 8 x 8
// matrix of 16-bit elements is 8 rows x 4 fp32, and the element a thread receives (row
// lane / 4, 16-bit columns 2 (lane % 4) and + 1) is exactly fp32 column lane % 4, the tf32
// fragment's; one ldmatrix.x4 replaces four scalar loads. Transposed operands keep scalar
// loads (ldmatrix transposes 16-bit elements, not 32-bit ones).
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Operand fetchers for one k-step (k0) of a warp's 16 x 32 block.
template <bool TA, bool NEG>
struct OpA {
    const float *A;
    uint32_t lsm;  // ldmatrix row address of this lane (non-transposed)
    __device__ OpA(const float *A_, const Frag &f) : A(A_) {
        const int lane = threadIdx.x & 31;
        lsm = TA ? 0u : smem_u32(A + (f.m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LD + 4 * (lane >> 4));
    }
    __device__ __forceinline__ void get(int k0, const Frag &f, uint32_t (&a)[4]) const {
        if constexpr (!TA) {
            ldsm4(lsm + 4u * (uint32_t)k0, a);
        } else {
            const float av[4] = {A[(k0 + f.t) * LD + f.m0 + f.g], A[(k0 + f.t) * LD + f.m0 + f.g + 8],
                                 A[(k0 + f.t + 4) * LD + f.m0 + f.g],
                                 A[(k0 + f.t + 4) * LD + f.m0 + f.g + 8]};
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] = __float_as_uint(av[e]);
        }
        if constexpr (NEG) {
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] ^= 0x80000000u;
        }
    }
};
template <bool TB>
struct OpB {
    const float *B;
    uint32_t lsm;  // ldmatrix row address of this lane for n-tiles 0 and 1 (non-transposed)
    __device__ OpB(const float *B_, const Frag &f) : B(B_) {
        const int lane = threadIdx.x & 31;
        lsm = TB ? smem_u32(B + (f.n0 + (lane & 7) + 8 * (lane >> 4)) * LD + 4 * ((lane >> 3) & 1)) : 0u;
    }
    // b[j] for the four n-tiles j of the block
    __device__ __forceinline__ void get(int k0, const Frag &f, uint32_t (&b)[4][2]) const {
        if constexpr (TB) {
            uint32_t r[4];
            ldsm4(lsm + 4u * (uint32_t)k0, r);
            b[0][0] = r[0]; b[0][1] = r[1]; b[1][0] = r[2]; b[1][1] = r[3];
            ldsm4(lsm + 4u * (uint32_t)(16 * LD + k0), r);
            b[2][0] = r[0]; b[2][1] = r[1]; b[3][0] = r[2]; b[3][1] = r[3];
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = f.n0 + 8 * j + f.g;
                b[j][0] = __float_as_uint(B[(k0 + f.t) * LD + n]);
                b[j][1] = __float_as_uint(B[(k0 + f.t + 4) * LD + n]);
            }
        }
    }
};

// acc += (NEG ? -1 : 1) * opA x opB over K = 64, with opA(i, k) = TA ? A[k][i] : A[i][k] and
// opB(k, j) = TB ? B[j][k] : B[k][j] (tiles row-major at stride LD). The operands go to the
// tf32 MMA as their fp32 bits, which it reads truncated to a 10-bit significand.
template <bool TA, bool TB, bool NEG = false>
__device__ __forceinline__ void mm(const float *A, const float *B, const Frag &f, Acc &acc) {
    const OpA<TA, NEG> oa(A, f);
    const OpB<TB> ob(B, f);
#pragma unroll 2
    for (int k0 = 0; k0 < 64; k0 += 8) {
        uint32_t a[4], b[4][2];
        oa.get(k0, f, a);
        ob.get(k0, f, b);
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_tf32(acc[j], a, b[j]);
    }
}

// Two independent products in one loop (twice the independent MMA chains per warp):
// acc1 += op1, acc2 += op2, each as in mm.
template <bool TA1, bool TB1, bool NEG1, bool TA2, bool TB2, bool NEG2>
__device__ __forceinline__ void mm2(const float *A1, const float *B1, Acc &acc1,
                                    const float *A2, const float *B2, Acc &acc2, const Frag &f) {
    const OpA<TA1, NEG1> oa1(A1, f);
    const OpB<TB1> ob1(B1, f);
    const OpA<TA2, NEG2> oa2(A2, f);
    const OpB<TB2> ob2(B2, f);
#pragma unroll 2
    for (int k0 = 0; k0 < 64; k0 += 8) {
        uint32_t a1[4], a2[4], b1[4][2], b2[4][2];
        oa1.get(k0, f, a1);
        oa2.get(k0, f, a2);
        ob1.get(k0, f, b1);
        ob2.get(k0, f, b2);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            mma_tf32(acc1[j], a1, b1[j]);
            mma_tf32(acc2[j], a2, b2[j]);
        }
    }
}

// tile[r][c] = acc (where keep(r, c)), else 0
template <typename Keep>
__device__ __forceinline__ void put(float *tile, const Acc &acc, const Frag &f, Keep keep) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = f.row(e), c = f.col(j, e);
            tile[r * LD + c] = keep(r, c) ? acc[j][e] : 0.f;
        }
}
__device__ __forceinline__ void get(const float *tile, const Frag &f, Acc &acc) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = tile[f.row(e) * LD + f.col(j, e)];
}
// rows r < nvalid of a (64-row) global fp32 block, row-major at ld floats per row
__device__ __forceinline__ void store_rows(float *dst, const Acc &acc, const Frag &f, int nvalid,
                                           int ld = kD) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const int r = f.row(e);
            if (r < nvalid)
                *reinterpret_cast<float2 *>(dst + (size_t)r * ld + f.col(j, e)) =
                    make_float2(acc[j][e], acc[j][e + 1]);
        }
}
// acc = the same positions read back (zero at rows r >= nvalid)
__device__ __forceinline__ void load_rows(const float *src, Acc &acc, const Frag &f, int nvalid,
                                          int ld) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const int r = f.row(e);
            const float2 v = r < nvalid
                                 ? *reinterpret_cast<const float2 *>(src + (size_t)r * ld + f.col(j, e))
                                 : make_float2(0.f, 0.f);
            acc[j][e] = v.x;
            acc[j][e + 1] = v.y;
        }
}

// 64 x 64 fp32 tile from 64 rows of global memory at stride ld floats, zero past nvalid or
// everywhere if !use: asynchronous 16-byte copies (zero-filled where not used), waited for
// by cp_async_wait
__device__ __forceinline__ void load_tile_async(float *tile, const float *src, int nvalid, bool use,
                                                int ld = kD) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int e = threadIdx.x + it * kThreads, r = e >> 4, c = (e & 15) * 4;
        const bool in = use && r < nvalid;
        const uint32_t dst = smem_u32(tile + r * LD + c);
        const float *g = in ? src + (size_t)r * ld + c : src;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(g),
                     "r"(in ? 16 : 0)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// N bf16 64 x 64 tiles (rows of bf16 tensors at ld elements per row, zero past nvalid) as
// fp32: every load is issued before the first conversion
template <int N>
__device__ __forceinline__ void load_bf16_tiles(float *const (&dst)[N],
                                                const __nv_bfloat16 *const (&src)[N], int nvalid,
                                                int ld = kD) {
    uint2 u[N][4];
#pragma unroll
    for (int m = 0; m < N; ++m)
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = threadIdx.x + it * kThreads, r = e >> 4, c = (e & 15) * 4;
            u[m][it] = r < nvalid ? *reinterpret_cast<const uint2 *>(src[m] + (size_t)r * ld + c)
                                  : make_uint2(0u, 0u);
        }
#pragma unroll
    for (int m = 0; m < N; ++m)
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = threadIdx.x + it * kThreads, r = e >> 4, c = (e & 15) * 4;
            const float2 a = unpack_bf16x2(u[m][it].x), b = unpack_bf16x2(u[m][it].y);
            *reinterpret_cast<float4 *>(dst[m] + r * LD + c) = make_float4(a.x, a.y, b.x, b.y);
        }
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_block_mm_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                    const __nv_bfloat16 *__restrict__ w, const float *__restrict__ beta,
                    const float *__restrict__ dqt, const float *__restrict__ dkt,
                    const float *__restrict__ dP, const float *__restrict__ dTd,
                    float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dw,
                    float *__restrict__ dbeta, int L, int Lp, int nblk) {
    extern __shared__ __align__(16) float sm[];
    float *S[kTiles];
#pragma unroll
    for (int i = 0; i < kTiles; ++i) S[i] = sm + i * (kTile / 4);
    float *const Ys = sm + kYOff / 4;
    float *const bs = sm + kBetaOff / 4;
    float *const dbs = bs + 64;

    const int tid = threadIdx.x;
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t hL = (size_t)bh * L;
    const int nvalid = min(kC, L - t0);
    const bool last = blk == nblk - 1;
    const Frag f;

    // tiles: 0 W, 1 Q, 2 K, 3 dq~, 4 dk~, 5 dP, 6 dT, then 7-11 as noted per step
    float *const W = S[0], *const Q = S[1], *const K = S[2];
    load_tile_async(S[3], dqt + ((size_t)bh * Lp + t0) * kD, nvalid, true);
    load_tile_async(S[4], dkt + ((size_t)bh * Lp + t0) * kD, nvalid, !last);
    load_tile_async(S[5], dP + ((size_t)bh * nblk + blk) * kC * kC, kC, blk > 0 && !last);
    load_tile_async(S[6], dTd + ((size_t)bh * nblk + blk) * kC * kC, nvalid, true);
    {
        float *const dst[3] = {W, Q, K};
        const __nv_bfloat16 *const src[3] = {w + (hL + t0) * kD, q + (hL + t0) * kD,
                                             k + (hL + t0) * kD};
        load_bf16_tiles(dst, src, nvalid);
    }
    cp_async_wait();
    if (tid < kC) {
        bs[tid] = tid < nvalid ? beta[hL + t0 + tid] : 0.f;
        dbs[tid] = 0.f;
    }
    __syncthreads();
    // dT only where j <= i
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, c = e & 63;
        if (c > r) S[6][r * LD + c] = 0.f;
    }

    Acc a0, a1, a2;
    // ---- G = W W^T -> E = D strictly-upper(G) (tile 10); Lq (8), Rk (9)
    zero(a0);
    mm<false, true>(W, W, f, a0);
    put(S[10], a0, f, [](int, int) { return true; });
    zero(a1);
    zero(a2);
    mm2<false, true, false, false, true, false>(Q, W, a1, K, W, a2, f);
    put(S[8], a1, f, [](int r, int c) { return c <= r; });
    put(S[9], a2, f, [](int r, int c) { return c > r; });
    __syncthreads();
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, c = e & 63;
        S[10][r * LD + c] = c > r ? bs[r] * S[10][r * LD + c] : 0.f;
    }
    __syncthreads();
    // ---- X = (I + E)^{-1} in place (tile 10), A = X D (tile 11)
    blocked_unit_upper_inverse(S[10], Ys, tid);
    float *const X = S[10], *const A = S[11], *const Lq = S[8], *const Rk = S[9];
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, c = e & 63;
        A[r * LD + c] = X[r * LD + c] * bs[c];
    }
    __syncthreads();

    // ---- U = A^T W (tile 7); dLq = -dq~ U^T; dU = -Lq^T dq~ (tile 7); dq = dq~ + ...
    Acc dLq, dQ, dRk, dK, dW, dA;
    zero(a0);
    mm<true, false>(A, W, f, a0);
    put(S[7], a0, f, [](int, int) { return true; });
    get(S[3], f, dQ);
    __syncthreads();
    zero(dLq);
    zero(a0);
    mm2<false, true, true, true, false, true>(S[3], S[7], dLq, Lq, S[3], a0, f);  // dLq, dU
    __syncthreads();
    put(S[7], a0, f, [](int, int) { return true; });
    float *const dU = S[7];
    // ---- V = A W (tile 3); dRk = -dk~ V^T; dV = -Rk^T dk~ - W dP (tile 4 after); dw = -V dP^T
    zero(a0);
    mm<false, false>(A, W, f, a0);
    put(S[3], a0, f, [](int, int) { return true; });
    get(S[4], f, dK);
    __syncthreads();
    zero(dRk);
    zero(a1);
    mm2<false, true, true, true, false, true>(S[4], S[3], dRk, Rk, S[4], a1, f);
    zero(dW);
    mm2<false, false, true, false, true, true>(W, S[5], a1, S[3], S[5], dW, f);
    __syncthreads();
    put(S[4], a1, f, [](int, int) { return true; });
    float *const dV = S[4];
    // ---- with dT (tile 6): dq += dT K; dk += dT^T Q; dY = -dT Rk (tile 3); Y = Lq A^T (5)
    mm2<false, false, false, true, false, false>(S[6], K, dQ, S[6], Q, dK, f);
    zero(a0);
    zero(a1);
    mm2<false, false, true, false, true, false>(S[6], Rk, a0, Lq, A, a1, f);  // dY, Y
    put(S[3], a0, f, [](int, int) { return true; });
    put(S[5], a1, f, [](int, int) { return true; });
    __syncthreads();
    float *const dY = S[3];
    mm2<true, false, true, false, false, false>(S[6], S[5], dRk, dY, A, dLq, f);  // -dT^T Y, dY A
    zero(dA);
    mm<true, false>(dY, Lq, f, dA);             // dY^T Lq
    __syncthreads();
    // ---- dLq = tril (tile 5), dRk = striu (tile 6); dq, dk complete
    put(S[5], dLq, f, [](int r, int c) { return c <= r; });
    put(S[6], dRk, f, [](int r, int c) { return c > r; });
    __syncthreads();
    mm2<false, false, false, false, false, false>(S[5], W, dQ, S[6], W, dK, f);
    mm<true, false>(S[5], Q, f, dW);
    mm<true, false>(S[6], K, f, dW);
    store_rows(dq + (hL + t0) * kD, dQ, f, nvalid);
    store_rows(dk + (hL + t0) * kD, dK, f, nvalid);
    // ---- dA += W dU^T + dV W^T; dw += A dU + A^T dV
    mm2<false, true, false, false, false, false>(W, dU, dA, A, dU, dW, f);
    mm2<false, true, false, true, false, false>(dV, W, dA, A, dV, dW, f);
    // ---- A = X D: dbeta_u += sum_s dA_su X_su, dX = dA D (tile 1)
    {
        float cs[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) cs[j][0] = cs[j][1] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = f.row(e), c = f.col(j, e);
                cs[j][e & 1] = fmaf(dA[j][e], X[r * LD + c], cs[j][e & 1]);
                dA[j][e] *= bs[c];
            }
        // column sums over the warp's 16 rows: lanes with the same t hold the same columns
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = cs[j][h];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (f.g == 0) atomicAdd(&dbs[f.n0 + 8 * j + 2 * f.t + h], v);
            }
    }
    __syncthreads();  // Q no longer read: tile 1 takes dX
    put(S[1], dA, f, [](int, int) { return true; });
    __syncthreads();
    // ---- dTT = -X^T dX X^T (P1 = X^T dX in tile 2)
    zero(a0);
    mm<true, false>(X, S[1], f, a0);
    __syncthreads();  // K no longer read
    put(S[2], a0, f, [](int, int) { return true; });
    __syncthreads();
    zero(a1);
    zero(a2);
    mm2<false, true, true, false, true, false>(S[2], X, a1, W, W, a2, f);  // dTT, G again
    // ---- T = I + D strictly-upper(G): dbeta_s += sum_{v>s} dTT_sv G_sv, dG = D su(dTT)
    {
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = f.row(e), c = f.col(j, e);
                const bool up = c > r;
                rs[e >> 1] = fmaf(up ? a1[j][e] : 0.f, a2[j][e], rs[e >> 1]);
                a1[j][e] = up ? bs[r] * a1[j][e] : 0.f;
            }
        // row sums over the warp's 32 columns: the four lanes with the same g
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v = rs[h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (f.t == 0) atomicAdd(&dbs[f.m0 + f.g + 8 * h], v);
        }
    }
    put(S[3], a1, f, [](int, int) { return true; });  // dG
    __syncthreads();
    zero(a0);
    mm2<false, false, false, true, false, false>(S[3], W, dW, S[3], W, a0, f);  // dG W, dG^T W
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) dW[j][e] += a0[j][e];
    store_rows(dw + (hL + t0) * kD, dW, f, nvalid);
    if (tid < nvalid) dbeta[hL + t0 + tid] = dbs[tid];
}

// Head size 128: the same gradient with every d-side matrix (W, Q, K, dq~, dk~, U, V, dU,
// dV and the outputs) as two 64-column halves h and dP_b as four 64 x 64 quadrants dP[h'][h]
// (rows h', columns h). G, Lq, Rk, dLq, dRk and dA sum their contractions over both halves;
//     dV_h = -Rk^T dk~_h - sum_h' W_h' dP[h'][h],     dw_h' -= V_h dP[h'][h]^T for each h,
// and every other d-side product is one per half. Twelve fp32 tiles as in head size 64: W's
// halves, dT, X, A, Lq and Rk stay resident while q, k, dq~, dk~ and the dP quadrants stream
// through the others; dw's halves accumulate in registers, dq and dk are formed last.
__global__ void __launch_bounds__(kThreads, 1)
bwd_block_mm128_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                       const __nv_bfloat16 *__restrict__ w, const float *__restrict__ beta,
                       const float *__restrict__ dqt, const float *__restrict__ dkt,
                       const float *__restrict__ dP, const float *__restrict__ dTd,
                       float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dw,
                       float *__restrict__ dbeta, int L, int Lp, int nblk) {
    constexpr int D = 128;
    extern __shared__ __align__(16) float sm[];
    float *S[kTiles];
#pragma unroll
    for (int i = 0; i < kTiles; ++i) S[i] = sm + i * (kTile / 4);
    float *const Ys = sm + kYOff / 4;
    float *const bs = sm + kBetaOff / 4;
    float *const dbs = bs + 64;

    const int tid = threadIdx.x;
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t hL = (size_t)bh * L;
    const int nvalid = min(kC, L - t0);
    const bool last = blk == nblk - 1;
    const Frag f;
    const __nv_bfloat16 *const qr = q + (hL + t0) * D, *const kr = k + (hL + t0) * D,
                               *const wr = w + (hL + t0) * D;
    const float *const dqr = dqt + ((size_t)bh * Lp + t0) * D;
    const float *const dkr = dkt + ((size_t)bh * Lp + t0) * D;

    // tiles: 0, 1 W's halves, 2 dT, 5 E then X, 6 Lq, 7 Rk, 8 A; 3, 4, 9, 10, 11 stream
    float *const W0 = S[0], *const W1 = S[1], *const dT = S[2];
    load_tile_async(dT, dTd + ((size_t)bh * nblk + blk) * kC * kC, nvalid, true);
    {
        float *const d1[3] = {W0, W1, S[3]};
        const __nv_bfloat16 *const s1[3] = {wr, wr + 64, qr};
        load_bf16_tiles(d1, s1, nvalid, D);
        float *const d2[3] = {S[9], S[4], S[10]};
        const __nv_bfloat16 *const s2[3] = {qr + 64, kr, kr + 64};
        load_bf16_tiles(d2, s2, nvalid, D);
    }
    cp_async_wait();
    if (tid < kC) {
        bs[tid] = tid < nvalid ? beta[hL + t0 + tid] : 0.f;
        dbs[tid] = 0.f;
    }
    __syncthreads();
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, c = e & 63;
        if (c > r) dT[r * LD + c] = 0.f;
    }

    Acc a0, a1, a2;
    // ---- G = W W^T, Lq = tril(Q W^T), Rk = striu(K W^T), each over both halves
    zero(a0);
    zero(a1);
    zero(a2);
    mm2<false, true, false, false, true, false>(W0, W0, a0, S[3], W0, a1, f);
    mm2<false, true, false, false, true, false>(W1, W1, a0, S[9], W1, a1, f);
    mm<false, true>(S[4], W0, f, a2);
    mm<false, true>(S[10], W1, f, a2);
    put(S[5], a0, f, [](int, int) { return true; });
    put(S[6], a1, f, [](int r, int c) { return c <= r; });
    put(S[7], a2, f, [](int r, int c) { return c > r; });
    __syncthreads();
    // dq~ and dk~ halves stream in under the inverse (the q and k tiles are dead)
    load_tile_async(S[3], dqr, nvalid, true, D);
    load_tile_async(S[9], dqr + 64, nvalid, true, D);
    load_tile_async(S[4], dkr, nvalid, !last, D);
    load_tile_async(S[10], dkr + 64, nvalid, !last, D);
    cp_async_commit();
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, c = e & 63;
        S[5][r * LD + c] = c > r ? bs[r] * S[5][r * LD + c] : 0.f;
    }
    __syncthreads();
    // ---- X = (I + E)^{-1} in place (tile 5), A = X D (tile 8)
    blocked_unit_upper_inverse(S[5], Ys, tid);
    float *const X = S[5], *const A = S[8], *const Lq = S[6], *const Rk = S[7];
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int r = e >> 6, c = e & 63;
        A[r * LD + c] = X[r * LD + c] * bs[c];
    }
    cp_async_wait();
    __syncthreads();

    Acc dLq, dRk, dA, dW0, dW1;
    zero(dLq);
    zero(dRk);
    zero(dA);
    zero(dW0);
    zero(dW1);
    float *const Ut = S[11];  // U_h, dU_h, V_h, dV_h in turn
    // ---- per half: U_h = A^T W_h; dLq -= dq~_h U_h^T; dU_h = -Lq^T dq~_h;
    //      dA += W_h dU_h^T; dw_h += A dU_h
    auto qside = [&](const float *Wh, const float *dqh, Acc &dWh) {
        zero(a0);
        mm<true, false>(A, Wh, f, a0);
        put(Ut, a0, f, [](int, int) { return true; });
        __syncthreads();
        zero(a0);
        mm2<false, true, true, true, false, true>(dqh, Ut, dLq, Lq, dqh, a0, f);
        __syncthreads();
        put(Ut, a0, f, [](int, int) { return true; });
        __syncthreads();
        mm2<false, true, false, false, false, false>(Wh, Ut, dA, A, Ut, dWh, f);
        __syncthreads();
    };
    qside(W0, S[3], dW0);
    qside(W1, S[9], dW1);
    // ---- per half: V_h = A W_h; dRk -= dk~_h V_h^T; dV_h = -Rk^T dk~_h - sum_h' W_h' dP[h'][h];
    //      dw_h' -= V_h dP[h'][h]^T; dA += dV_h W_h^T; dw_h += A^T dV_h
    const float *const dPb = dP + ((size_t)bh * nblk + blk) * D * D;
    const bool useP = blk > 0 && !last;  // P_0 and the last P_b reach no logit
    auto kside = [&](int h, const float *Wh, const float *dkh, Acc &dWh) {
        load_tile_async(S[3], dPb + 64 * h, kC, useP, D);           // dP[0][h]
        load_tile_async(S[9], dPb + 64 * D + 64 * h, kC, useP, D);  // dP[1][h]
        cp_async_commit();
        zero(a0);
        mm<false, false>(A, Wh, f, a0);
        put(Ut, a0, f, [](int, int) { return true; });
        cp_async_wait();
        __syncthreads();
        zero(a1);
        mm2<false, true, true, true, false, true>(dkh, Ut, dRk, Rk, dkh, a1, f);
        mm<false, false, true>(W0, S[3], f, a1);
        mm<false, false, true>(W1, S[9], f, a1);
        mm2<false, true, true, false, true, true>(Ut, S[3], dW0, Ut, S[9], dW1, f);
        __syncthreads();
        put(Ut, a1, f, [](int, int) { return true; });
        __syncthreads();
        mm2<false, true, false, true, false, false>(Ut, Wh, dA, A, Ut, dWh, f);
        __syncthreads();
    };
    kside(0, W0, S[4], dW0);
    kside(1, W1, S[10], dW1);
    // ---- with dT: dY = -dT Rk (tile 3), Y = Lq A^T (tile 9); dRk -= dT^T Y; dLq += dY A;
    //      dA += dY^T Lq
    zero(a0);
    zero(a1);
    mm2<false, false, true, false, true, false>(dT, Rk, a0, Lq, A, a1, f);
    put(S[3], a0, f, [](int, int) { return true; });
    put(S[9], a1, f, [](int, int) { return true; });
    __syncthreads();
    mm2<true, false, true, false, false, false>(dT, S[9], dRk, S[3], A, dLq, f);
    mm<true, false>(S[3], Lq, f, dA);
    __syncthreads();
    // ---- dLq = tril (tile 3), dRk = striu (tile 9); q and k again (tiles 6, 7, 4, 10: Lq,
    //      Rk and dk~ are dead); per half dq_h = dq~_h + dT K_h + dLq W_h,
    //      dk_h = dk~_h + dT^T Q_h + dRk W_h, dw_h += dLq^T Q_h + dRk^T K_h
    put(S[3], dLq, f, [](int r, int c) { return c <= r; });
    put(S[9], dRk, f, [](int r, int c) { return c > r; });
    {
        float *const d1[2] = {S[6], S[7]};
        const __nv_bfloat16 *const s1[2] = {qr, kr};
        load_bf16_tiles(d1, s1, nvalid, D);
        float *const d2[2] = {S[4], S[10]};
        const __nv_bfloat16 *const s2[2] = {qr + 64, kr + 64};
        load_bf16_tiles(d2, s2, nvalid, D);
    }
    __syncthreads();
    auto outs = [&](int h, const float *Wh, const float *Qh, const float *Kh, Acc &dWh) {
        load_rows(dqr + 64 * h, a0, f, nvalid, D);
        load_rows(dkr + 64 * h, a1, f, last ? 0 : nvalid, D);
        mm2<false, false, false, true, false, false>(dT, Kh, a0, dT, Qh, a1, f);
        mm2<false, false, false, false, false, false>(S[3], Wh, a0, S[9], Wh, a1, f);
        mm<true, false>(S[3], Qh, f, dWh);
        mm<true, false>(S[9], Kh, f, dWh);
        store_rows(dq + (hL + t0) * D + 64 * h, a0, f, nvalid, D);
        store_rows(dk + (hL + t0) * D + 64 * h, a1, f, nvalid, D);
    };
    outs(0, W0, S[6], S[7], dW0);
    outs(1, W1, S[4], S[10], dW1);
    // ---- A = X D: dbeta_u += sum_s dA_su X_su, dX = dA D (tile 11)
    {
        float cs[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) cs[j][0] = cs[j][1] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = f.row(e), c = f.col(j, e);
                cs[j][e & 1] = fmaf(dA[j][e], X[r * LD + c], cs[j][e & 1]);
                dA[j][e] *= bs[c];
            }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = cs[j][h];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (f.g == 0) atomicAdd(&dbs[f.n0 + 8 * j + 2 * f.t + h], v);
            }
    }
    put(Ut, dA, f, [](int, int) { return true; });
    __syncthreads();  // also: tiles 3 and 9 (dLq, dRk) are no longer read
    // ---- dTT = -X^T dX X^T (P1 = X^T dX in tile 3); G again
    zero(a0);
    mm<true, false>(X, Ut, f, a0);
    put(S[3], a0, f, [](int, int) { return true; });
    __syncthreads();
    zero(a1);
    zero(a2);
    mm2<false, true, true, false, true, false>(S[3], X, a1, W0, W0, a2, f);
    mm<false, true>(W1, W1, f, a2);
    // ---- T = I + D strictly-upper(G): dbeta_s += sum_{v>s} dTT_sv G_sv, dG = D su(dTT)
    {
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = f.row(e), c = f.col(j, e);
                const bool up = c > r;
                rs[e >> 1] = fmaf(up ? a1[j][e] : 0.f, a2[j][e], rs[e >> 1]);
                a1[j][e] = up ? bs[r] * a1[j][e] : 0.f;
            }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v = rs[h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (f.t == 0) atomicAdd(&dbs[f.m0 + f.g + 8 * h], v);
        }
    }
    put(S[9], a1, f, [](int, int) { return true; });  // dG
    __syncthreads();
    // dw_h += (dG + dG^T) W_h
    mm<false, false>(S[9], W0, f, dW0);
    mm<true, false>(S[9], W0, f, dW0);
    mm<false, false>(S[9], W1, f, dW1);
    mm<true, false>(S[9], W1, f, dW1);
    store_rows(dw + (hL + t0) * D, dW0, f, nvalid, D);
    store_rows(dw + (hL + t0) * D + 64, dW1, f, nvalid, D);
    if (tid < nvalid) dbeta[hL + t0 + tid] = dbs[tid];
}

}  // namespace

// The block pass for bf16 inputs: dq, dk, dw (B, H, L, 64) and dbeta (B, H, L), fp32, from
// the query pass's dq~, dk~ (BH, Lp, 64), dP and the diagonal dT (BH, nblk, 64, 64).
cudaError_t launch_bwd_block_mm(const void *q, const void *k, const void *w, const float *beta,
                                const float *dqt, const float *dkt, const float *dP,
                                const float *dTd, float *dq, float *dk, float *dw,
                                float *dbeta, int BH, int L, int Lp, int nblk,
                                cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd_block_mm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    bwd_block_mm_kernel<<<dim3(nblk, BH), kThreads, kSmem, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(w), beta, dqt, dkt, dP, dTd, dq, dk, dw, dbeta, L, Lp,
        nblk);
    return cudaGetLastError();
}

// The block pass for bf16 inputs at head size 128: dq, dk, dw (B, H, L, 128) and dbeta
// (B, H, L), fp32, from dq~, dk~ (BH, Lp, 128), dP (BH, nblk, 128, 128) and the diagonal dT
// (BH, nblk, 64, 64).
cudaError_t launch_bwd_block_mm128(const void *q, const void *k, const void *w, const float *beta,
                                   const float *dqt, const float *dkt, const float *dP,
                                   const float *dTd, float *dq, float *dk, float *dw,
                                   float *dbeta, int BH, int L, int Lp, int nblk,
                                   cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd_block_mm128_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    bwd_block_mm128_kernel<<<dim3(nblk, BH), kThreads, kSmem, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(w), beta, dqt, dkt, dP, dTd, dq, dk, dw, dbeta, L, Lp,
        nblk);
    return cudaGetLastError();
}

}  // namespace path
