// PaTH forward at head size d = 128 for fp32 inputs, fp32 on the CUDA cores (the fp32 bar
// needs fp32 products; bf16 inputs take the tensor-core kernels of ut_prepare_tc.cu and
// scan_tc128.cu). The same algorithm as the d = 64 kernels (technical summary
// "技術要約: PaTH Attention" §3 "UT変換による表現" and the block-wise algorithm; review
// "거리에서 경로로, PaTH Attention" §9, which flags larger heads as costlier): per block of
// C = 64 tokens the UT factor A = (I + D N)^{-1} D with N = strictly-upper(W W^T), the
// boundary-adjusted q~ and k~, the dense block transition P_b = I - W^T A W (here 128 x 128)
// and the diagonal-block logits; then per 64-row query block a right-to-left scan over key
// blocks with online softmax, carrying X <- X P_b^T. Contractions over the head dimension
// run to 128; the triangular solve is unchanged (64 x 64).
//
// PaTH-FoX (technical summary §2 "拡張: PaTH-FoX"; review §4): every logit also takes the
// forget-gate bias sum_{s=j+1..i} log f_s = c_i - c_j, in log2 units like the logits. The
// preparation forms, per block and in fp64, the inclusive in-block sums lc_i of
// log2(e) log f_s and the block total T_b; the diagonal table takes lc_i - lc_j. For a key
// j of an earlier block b the scan splits the bias as
//     c_i - c_j = [lc_i + sum_{b < b' < ib} T_b'] + [T_b - lc_j],
// a per-row term with an fp64 running sum (exact where the weights are not negligible:
// its rounding grows with the bias itself) and the key's tail sum within its block, so no
// difference of two large prefix sums is ever taken.
// Early exit, exact within rounding (review §4: the gate makes distant keys vanish): every
// H_s with beta_s in [0, 2] and unit w_s is a contraction, so the state a row carries is no
// longer than q~_i, and against any key of blocks 0..b its logit is at most
//     bound_i(b) = 2 |scale| log2(e) |q~_i| Kpre(b) + c2_i - Mpre(b),
// with Kpre(b) the largest |k~_j| and Mpre(b) the smallest c2_j over blocks 0..b (the factor
// 2 covers rounding). Before visiting block b the scan stops if bound_i(b) is below the
// row's running maximum minus 40 log2(e) for every row of the query block: what remains
// weighs less than e^-40 relative to the row's largest weight. The preparation records per
// block the largest |k~_j| and the smallest in-block sum; a per-head pass forms the block
// start offsets C_b (fp64), Mpre and Kpre.
#include "common.cuh"

namespace path {

namespace {

constexpr int kD2 = 128;           // head size of this file
constexpr int LDA = kC + 4;        // stride of buffers with 64 columns
constexpr int LDB = kD2 + 4;       // stride of buffers with 128 columns
constexpr int kThreads = 256;
constexpr float kExitLog2 = 40.f * kLog2e;  // e^-40 relative weight, in log2 units

// acc[i][j] += sum_{k < K} X[k][m0 + i] * Y[k][n0 + j]  (k-major operands)
template <int K>
__device__ __forceinline__ void mmk(const float *__restrict__ X, int ldx, const float *__restrict__ Y,
                                    int ldy, int m0, int n0, float (&acc)[4][4]) {
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        const float4 a = *reinterpret_cast<const float4 *>(X + k * ldx + m0);
        const float4 b = *reinterpret_cast<const float4 *>(Y + k * ldy + n0);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

__device__ __forceinline__ void zero(float (&a)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[i][j] = 0.f;
}

// rows x 128 fp32 tile (row-major, 128 floats per row) into shared memory rows of stride
// ld; eight 16-byte loads in flight per thread before the first store
__device__ __forceinline__ void load128(float *dst, int ld, const float *__restrict__ src, int rows) {
    const int n4 = rows * (kD2 / 4);
    for (int base = 0; base < n4; base += 8 * kThreads) {
        float4 x[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int e = base + (int)threadIdx.x + it * kThreads;
            x[it] = e < n4 ? reinterpret_cast<const float4 *>(src)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int e = base + (int)threadIdx.x + it * kThreads;
            if (e < n4) {
                const int r = e / (kD2 / 4), c = 4 * (e % (kD2 / 4));
                *reinterpret_cast<float4 *>(dst + r * ld + c) = x[it];
            }
        }
    }
}

// four consecutive elements (the kernels are instantiated for fp32 inputs)
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

template <typename T> __device__ __forceinline__ void put4(T *dst, const float *v);
template <> __device__ __forceinline__ void put4<float>(float *dst, const float *v) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// ---------------------------------------------------------------- register-tiled products
// acc[i][j] += sum_{k < K} A[r0 + 16i][k] * B[k][col(j)] with A row-major and B k-major;
// col(j) = c0 + j for j < 4 and c0 + 64 + j - 4 for j >= 4 (NJ = 8). The 16 lanes of a
// half warp share the A rows (broadcast loads) and the eight lanes of a quarter warp read
// one contiguous 128-byte piece of B.
template <int K, int NJ>
__device__ __forceinline__ void mmr(const float *__restrict__ A, int lda, const float *__restrict__ B,
                                    int ldb, int r0, int c0, float (&acc)[4][NJ]) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 16 * i) * lda + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float bv[NJ];
            const float4 b0 = *reinterpret_cast<const float4 *>(B + (k + kk) * ldb + c0);
            bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
            if (NJ == 8) {
                const float4 b1 = *reinterpret_cast<const float4 *>(B + (k + kk) * ldb + c0 + 64);
                bv[NJ == 8 ? 4 : 0] = b1.x; bv[NJ == 8 ? 5 : 1] = b1.y;
                bv[NJ == 8 ? 6 : 2] = b1.z; bv[NJ == 8 ? 7 : 3] = b1.w;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
            }
        }
    }
}

// acc[i][j] += sum_{k < K} A[r0 + 16i][k] * B[n0 + 16j][k]: both operands row-major (the
// contraction index contiguous in memory), so B^T products need no transposed copy. The
// eight lanes of a quarter warp read eight consecutive B rows (n0 = tx): at a row stride of
// LDB = 132 floats their 16-byte pieces fall in eight distinct bank groups.
template <int K, int NJ>
__device__ __forceinline__ void mmrb(const float *__restrict__ A, int lda, const float *__restrict__ B,
                                     int ldb, int r0, int n0, float (&acc)[4][NJ]) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 a[4], b[NJ];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 16 * i) * lda + k);
#pragma unroll
        for (int j = 0; j < NJ; ++j) b[j] = *reinterpret_cast<const float4 *>(B + (n0 + 16 * j) * ldb + k);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                float t = acc[i][j];
                t = fmaf(a[i].x, b[j].x, t);
                t = fmaf(a[i].y, b[j].y, t);
                t = fmaf(a[i].z, b[j].z, t);
                acc[i][j] = fmaf(a[i].w, b[j].w, t);
            }
    }
}

// mmrb for two products that share the A rows: acc1 = A B1^T (NJ1 columns) and acc2 =
// A B2^T (NJ2 columns), each A piece loaded once for both.
template <int K, int NJ1, int NJ2>
__device__ __forceinline__ void mmrb2(const float *__restrict__ A, int lda,
                                      const float *__restrict__ B1, const float *__restrict__ B2,
                                      int ldb, int r0, int n0, float (&acc1)[4][NJ1],
                                      float (&acc2)[4][NJ2]) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (r0 + 16 * i) * lda + k);
#pragma unroll
        for (int j = 0; j < NJ1 + NJ2; ++j) {
            const float4 b = j < NJ1 ? *reinterpret_cast<const float4 *>(B1 + (n0 + 16 * j) * ldb + k)
                                     : *reinterpret_cast<const float4 *>(B2 + (n0 + 16 * (j - NJ1)) * ldb + k);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float t = j < NJ1 ? acc1[i][j < NJ1 ? j : 0] : acc2[i][j < NJ1 ? 0 : j - NJ1];
                t = fmaf(a[i].x, b.x, t);
                t = fmaf(a[i].y, b.y, t);
                t = fmaf(a[i].z, b.z, t);
                t = fmaf(a[i].w, b.w, t);
                if (j < NJ1) acc1[i][j < NJ1 ? j : 0] = t;
                else acc2[i][j < NJ1 ? 0 : j - NJ1] = t;
            }
        }
    }
}

// ---------------------------------------------------------------- preparation
// One CTA of 256 threads per (block, head), two CTAs per SM. Every operand stays in its
// stored row-major layout (products over the head dimension read both operands as rows):
// phase 1 holds W, Q and K and forms G = W W^T, Lq = Q W^T, Rk = K W^T and Q K^T in
// registers; then four 64 x 64 slots replace Q and K (G, A, Lq, Rk; later Qhat, Khat and
// A W), and the epilogues of q~ and k~ read q and k again from global memory.
template <typename T, bool FOX>
__global__ void __launch_bounds__(kThreads, 2)
prep_d128_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ w,
                 const float *__restrict__ beta, const float *__restrict__ log_f, int L, int Lp,
                 int nblk, float scale_log2, float *__restrict__ qt, float *__restrict__ kp,
                 float *__restrict__ dg, float *__restrict__ lc, float *__restrict__ tail,
                 double *__restrict__ tot, double *__restrict__ mlc, float *__restrict__ kmax) {
    extern __shared__ __align__(16) float sm[];
    float *Wr = sm;                  // W [s][c], 64 x LDB
    float *R = Wr + kC * LDB;        // phase 1: Q [i][c] and K [j][c] (64 x LDB each)
    float *Qr = R, *Kr = R + kC * LDB;
    float *S0 = R, *Ar = R + kC * LDA, *S2 = R + 2 * kC * LDA, *S3 = R + 3 * kC * LDA;
    float *bs = R + 4 * kC * LDA;    // beta [64]
    double *lcs = reinterpret_cast<double *>(bs + kC);  // FoX: in-block sums lc [64], fp64
    float *kn2 = reinterpret_cast<float *>(lcs + kC);    // FoX: |k~_j|^2 [64]

    const int tid = threadIdx.x, blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t head = (size_t)bh * L;
    // four elements per thread and step, all of a thread's loads issued first
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float4 wv[4], qv[4], kv[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = tid + (4 * half + it) * kThreads, s = e / (kD2 / 4), c = 4 * (e % (kD2 / 4));
            const bool in = t0 + s < L;
            const size_t g = (head + t0 + s) * kD2 + c;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            wv[it] = in ? ld4(w + g) : z;
            qv[it] = in ? ld4(q + g) : z;
            kv[it] = in ? ld4(k + g) : z;
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = tid + (4 * half + it) * kThreads, s = e / (kD2 / 4), c = 4 * (e % (kD2 / 4));
            *reinterpret_cast<float4 *>(Wr + s * LDB + c) = wv[it];
            *reinterpret_cast<float4 *>(Qr + s * LDB + c) = qv[it];
            *reinterpret_cast<float4 *>(Kr + s * LDB + c) = kv[it];
        }
    }
    if (tid < kC) bs[tid] = (t0 + tid < L) ? beta[head + t0 + tid] : 0.f;
    if (FOX && tid < kC) kn2[tid] = 0.f;
    if (FOX && tid < 32) {
        // inclusive prefix of log2(e) log f over the block (tokens past L add 0): lane l
        // holds tokens 2l and 2l + 1 and scans the pair sums over the warp
        const double f0 = (t0 + 2 * tid < L) ? (double)log_f[head + t0 + 2 * tid] * kLog2eD : 0.0;
        const double f1 = (t0 + 2 * tid + 1 < L) ? (double)log_f[head + t0 + 2 * tid + 1] * kLog2eD : 0.0;
        double x = f0 + f1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, o);
            if (tid >= o) x += y;
        }
        lcs[2 * tid] = x - f1;
        lcs[2 * tid + 1] = x;
    }
    __syncthreads();
    if (FOX && tid < kC) {
        const size_t tok = (size_t)bh * Lp + t0 + tid;
        lc[tok] = (float)lcs[tid];
        tail[tok] = (float)(lcs[kC - 1] - lcs[tid]);
        if (tid == 0) tot[(size_t)bh * nblk + blk] = lcs[kC - 1];
    }

    // thread (ty, tx): rows ty + 16a, columns tx + 16b of the 64 x 64 products (mmrb), or
    // columns 4tx .. 4tx + 3 (+ 64) of the row-times-k-major products (mmr)
    const int ty = tid / 16, tx = tid % 16;
    float g[4][4], lq[4][4], rk[4][4], qk[4][4];
    zero(g);
    zero(lq);
    zero(rk);
    zero(qk);
    mmrb<kD2, 4>(Wr, LDB, Wr, LDB, ty, tx, g);   // G[s][v] = w_s . w_v
    mmrb<kD2, 4>(Kr, LDB, Wr, LDB, ty, tx, rk);  // Rk[j][s] = k_j . w_s (s > j)
    // Lq[i][u] = q_i . w_u (u <= i) and q_i . k_j, one pass over the Q rows
    mmrb2<kD2, 4, 4>(Qr, LDB, Wr, Kr, LDB, ty, tx, lq, qk);
    __syncthreads();  // Q and K are no longer read from shared memory
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int r = ty + 16 * a, c = tx + 16 * b;
            S0[r * LDA + c] = g[a][b];
            S2[r * LDA + c] = (c <= r) ? lq[a][b] : 0.f;
            S3[r * LDA + c] = (c > r) ? rk[a][b] : 0.f;
            Ar[r * LDA + c] = 0.f;
        }
    __syncthreads();
    // A = (I + D N)^{-1} D, one column per four threads: A[u][u] = beta_u and, for s < u,
    // A[s][u] = -beta_s sum_{v = s+1..u} G[s][v] A[v][u]
    {
        const int u = tid >> 2, part = tid & 3;
        for (int s = kC - 1; s >= 0; --s) {
            float sum = 0.f;
            for (int v = s + 1 + part; v < kC; v += 4) sum = fmaf(S0[s * LDA + v], Ar[v * LDA + u], sum);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (part == 0) Ar[s * LDA + u] = (s == u) ? bs[u] : (s < u ? -bs[s] * sum : 0.f);
            __syncwarp();
        }
    }
    __syncthreads();
    // Qhat[i][s] = sum_u Lq[i][u] A[s][u] -> slot 0 (G is no longer read)
    {
        float qh[4][4];
        zero(qh);
        mmrb<kC, 4>(S2, LDA, Ar, LDA, ty, tx, qh);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) S0[(ty + 16 * a) * LDA + tx + 16 * b] = qh[a][b];
    }
    __syncthreads();
    const size_t blk_base = (size_t)bh * nblk + blk;
    // diagonal-block logits, log2 units: scale (q_i . k_j - sum_s Qhat[i][s] Rk[j][s]), j <= i
    {
        float corr[4][4];
        zero(corr);
        mmrb<kC, 4>(S0, LDA, S3, LDA, ty, tx, corr);
        float *out = dg + blk_base * kC * kC;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int ii = ty + 16 * a, jj = tx + 16 * b;
                const float bias = FOX ? (float)(lcs[ii] - lcs[jj]) : 0.f;
                out[ii * kC + jj] = (jj <= ii && t0 + jj < L)
                                        ? scale_log2 * (qk[a][b] - corr[a][b]) + bias
                                        : -INFINITY;
            }
    }
    // Khat[j][u] = sum_s Rk[j][s] A[s][u] -> slot 2 (Lq is no longer read)
    {
        float kh[4][4];
        zero(kh);
        mmr<kC, 4>(S3, LDA, Ar, LDA, ty, 4 * tx, kh);
#pragma unroll
        for (int a = 0; a < 4; ++a)
            *reinterpret_cast<float4 *>(S2 + (ty + 16 * a) * LDA + 4 * tx) =
                make_float4(kh[a][0], kh[a][1], kh[a][2], kh[a][3]);
    }
    __syncthreads();
    // q~[i][c] = q[i][c] - sum_s Qhat[i][s] W[s][c] and k~[j][c] = k[j][c] - sum_u Khat[j][u]
    // W[u][c], q and k read again from global memory
    float kq[4] = {0.f, 0.f, 0.f, 0.f};  // FoX: partial |k~_j|^2 of this thread's rows
    float *kp_blk = kp + blk_base * (kC + kD2) * kD2;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const T *src = pass == 0 ? q : k;
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
        mmr<kC, 8>(pass == 0 ? S0 : S2, LDA, Wr, LDB, ty, 4 * tx, acc);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int r = ty + 16 * a;
            const bool in = t0 + r < L;
            const size_t g0 = (head + t0 + r) * kD2 + 4 * tx;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 x0 = in ? ld4(src + g0) : z, x1 = in ? ld4(src + g0 + 64) : z;
            const float v0[4] = {x0.x - acc[a][0], x0.y - acc[a][1], x0.z - acc[a][2], x0.w - acc[a][3]};
            const float v1[4] = {x1.x - acc[a][4], x1.y - acc[a][5], x1.z - acc[a][6], x1.w - acc[a][7]};
            float *dst = pass == 0 ? qt + ((size_t)bh * Lp + t0 + r) * kD2 : kp_blk + r * kD2;
            put4<float>(dst + 4 * tx, v0);
            put4<float>(dst + 4 * tx + 64, v1);
            if (FOX && pass == 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) kq[a] = fmaf(v0[e], v0[e], fmaf(v1[e], v1[e], kq[a]));
            }
        }
    }
    if (FOX) {
#pragma unroll
        for (int a = 0; a < 4; ++a) atomicAdd(&kn2[ty + 16 * a], kq[a]);
    }
    __syncthreads();  // slots 2 and 3 (Khat, Rk) are free
    if (FOX && tid < 32) {
        // the block's largest |k~_j| and smallest in-block sum, over its tokens below L
        float km = 0.f;
        double ml = INFINITY;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = tid + 32 * h;
            if (t0 + j < L) {
                km = fmaxf(km, sqrtf(kn2[j]));
                ml = fmin(ml, lcs[j]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
            ml = fmin(ml, __shfl_xor_sync(0xffffffffu, ml, o));
        }
        if (tid == 0) {
            kmax[blk_base] = km;
            mlc[blk_base] = ml;
        }
    }
    // (A W)[s][c] = sum_u A[s][u] W[u][c] -> slots 2-3 as 64 x LDB
    float *AW = S2;
    {
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
        mmr<kC, 8>(Ar, LDA, Wr, LDB, ty, 4 * tx, acc);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float *row = AW + (ty + 16 * a) * LDB + 4 * tx;
            *reinterpret_cast<float4 *>(row) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
            *reinterpret_cast<float4 *>(row + 64) = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
        }
    }
    __syncthreads();
    // P_b[n][c] = delta(n, c) - sum_s W[s][n] (A W)[s][c], four 64 x 64 quadrants
    const int m0 = ty * 4, n0 = tx * 4;
    for (int pq = 0; pq < 4; ++pq) {
        const int nb = 64 * (pq >> 1), cb = 64 * (pq & 1);
        float acc[4][4];
        zero(acc);
        mmk<kC>(Wr, LDB, AW, LDB, nb + m0, cb + n0, acc);
        float *out = kp_blk + kC * kD2;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = ((nb + m0 + i) == (cb + n0 + j) ? 1.f : 0.f) - acc[i][j];
            put4<float>(out + (nb + m0 + i) * kD2 + cb + n0, v);
        }
    }
}

// ---------------------------------------------------------------- PaTH-FoX exit bounds
// One warp per head, 32 blocks per iteration: C_b = sum of the totals of blocks 0..b-1 (fp64),
// Mpre(b) = min over blocks b' <= b of C_b' + (smallest in-block sum of b'), and Kpre(b) =
// max over blocks b' <= b of the block's largest |k~_j|; all in log2 units.
__global__ void __launch_bounds__(128)
fox_bounds_d128_kernel(const double *__restrict__ tot, const double *__restrict__ mlc,
                       const float *__restrict__ kmax, double *__restrict__ cst,
                       double *__restrict__ mpre, float *__restrict__ kpre, int BH, int nblk) {
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (bh >= BH) return;
    const size_t h0 = (size_t)bh * nblk;
    double carry_c = 0.0, carry_m = INFINITY;
    float carry_k = 0.f;
    for (int b0 = 0; b0 < nblk; b0 += 32) {
        const int b = b0 + lane;
        const bool in = b < nblk;
        const double t = in ? tot[h0 + b] : 0.0;
        double inc = t;  // inclusive prefix of the totals within these 32 blocks
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const double c = carry_c + (inc - t);
        double m = in ? c + mlc[h0 + b] : INFINITY;
        float k = in ? kmax[h0 + b] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double ym = __shfl_up_sync(0xffffffffu, m, o);
            const float yk = __shfl_up_sync(0xffffffffu, k, o);
            if (lane >= o) {
                m = fmin(m, ym);
                k = fmaxf(k, yk);
            }
        }
        m = fmin(m, carry_m);
        k = fmaxf(k, carry_k);
        if (in) {
            cst[h0 + b] = c;
            mpre[h0 + b] = m;
            kpre[h0 + b] = k;
        }
        carry_c = __shfl_sync(0xffffffffu, carry_c + inc, 31);
        carry_m = __shfl_sync(0xffffffffu, m, 31);
        carry_k = __shfl_sync(0xffffffffu, k, 31);
    }
}

// ---------------------------------------------------------------- scan
// One CTA per (64-row query block, head): the state X = (q~_i) as rows in shared memory;
// for key block b = ib, ib-1, ..., 0 the logits (diagonal block: the table; earlier blocks:
// X K~_b^T), the online softmax, O += P V_b and X <- X P_b^T. Thread (ty, tx) owns rows
// ty + 16i (i < 4) and, of the 128-wide results, columns 4tx .. 4tx + 3 and 64 + 4tx ..
// FOX: the forget-gate bias of every earlier block's logits, [row term] + [key tail].
template <typename T, bool FOX>
__global__ void __launch_bounds__(kThreads, 1)
scan_d128_kernel(const T *__restrict__ v, const float *__restrict__ qt, const float *__restrict__ kp,
                 const float *__restrict__ dg, const float *__restrict__ lc,
                 const float *__restrict__ tail, const double *__restrict__ tot,
                 const double *__restrict__ cst, const double *__restrict__ mpre,
                 const float *__restrict__ kpre, T *__restrict__ out, float *__restrict__ lse,
                 int L, int Lp, int nblk, float scale_log2, int heads_fast) {
    extern __shared__ __align__(16) float sm[];
    float *Xr = sm;                 // X [i][c], 64 x LDB
    float *KB = Xr + kC * LDB;      // K~_b [j][c], 64 x LDB (slot of 128 x LDA)
    float *PB = KB + kD2 * LDA;     // P_b [n][c], 128 x LDB
    float *Vs = PB + kD2 * LDB;     // V_b [j][c], 64 x LDB
    float *Ss = Vs + kC * LDB;      // logits [i][j] (log2 units)
    float *Pm = Ss + kC * LDA;      // probabilities [i][j]
    float *alpha_s = Pm + kC * LDA;
    float *rbias = alpha_s + kC;    // FoX: row terms lc_i + sum of the blocks in between
    float *kbias = rbias + kC;      // FoX: tail sums T_b - lc_j of the keys of block b

    // longest walks (the last query blocks) first, heads fastest or head by head
    // (heads_fastest)
    const int tid = threadIdx.x;
    const int ib = nblk - 1 - (int)(heads_fast ? blockIdx.y : blockIdx.x);
    const int bh = heads_fast ? blockIdx.x : blockIdx.y;
    if (ib * kC >= L) return;
    const int ty = tid / 16, tx = tid % 16, r0 = ty, c0 = 4 * tx;
    const int row = tid >> 2, part = tid & 3;
    const size_t hL = (size_t)bh * L;
    load128(Xr, LDB, qt + ((size_t)bh * Lp + (size_t)ib * kC) * kD2, kC);
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    // FoX: row lc_i (threads 0-63) and the fp64 sum of the totals of blocks b + 1 .. ib - 1
    const float lci = (FOX && tid < kC) ? lc[(size_t)bh * Lp + (size_t)ib * kC + tid] : 0.f;
    double between = 0.0;
    // FoX early exit: per softmax row, 2 |scale| log2(e) |q~_i|, c2_i - C_ib and whether the
    // row lies past L (such rows never hold the scan back)
    float qk2 = 0.f, lcr = 0.f;
    double cst_ib = 0.0;
    bool pad = true;
    if (FOX) {
        __syncthreads();
        float n2 = 0.f;
#pragma unroll 8
        for (int c = 0; c < 32; ++c) {
            const float x = Xr[row * LDB + part * 32 + c];
            n2 = fmaf(x, x, n2);
        }
        n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
        n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
        qk2 = 2.f * fabsf(scale_log2) * sqrtf(n2);
        lcr = lc[(size_t)bh * Lp + (size_t)ib * kC + row];
        cst_ib = cst[(size_t)bh * nblk + ib];
        pad = ib * kC + row >= L;
    }
    for (int b = ib; b >= 0; --b) {
        if (FOX && b < ib) {
            const size_t kb = (size_t)bh * nblk + b;
            const float bound = (float)((cst_ib - mpre[kb]) + (double)lcr) + qk2 * kpre[kb];
            if (__syncthreads_and(pad || bound < m_run - kExitLog2)) break;
        }
        __syncthreads();
        {
            float4 vv[8];
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int e = tid + it * kThreads, j = e / (kD2 / 4), c = 4 * (e % (kD2 / 4));
                vv[it] = (b * kC + j < L) ? ld4(v + (hL + b * kC + j) * kD2 + c)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int e = tid + it * kThreads, j = e / (kD2 / 4), c = 4 * (e % (kD2 / 4));
                *reinterpret_cast<float4 *>(Vs + j * LDB + c) = vv[it];
            }
        }
        if (b < ib) {
            const float *blk = kp + ((size_t)bh * nblk + b) * (kC + kD2) * kD2;
            if (FOX) {
                if (tid < kC) {
                    rbias[tid] = (float)((double)lci + between);
                    between += tot[(size_t)bh * nblk + b];
                } else if (tid < 2 * kC) {
                    kbias[tid - kC] = tail[(size_t)bh * Lp + (size_t)b * kC + tid - kC];
                }
            }
            load128(KB, LDB, blk, kC);
            load128(PB, LDB, blk + kC * kD2, kD2);
        } else {
            const float *tab = dg + ((size_t)bh * nblk + b) * kC * kC;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int e = tid + it * kThreads, r = e / (kC / 4), c = 4 * (e % (kC / 4));
                *reinterpret_cast<float4 *>(Ss + r * LDA + c) = reinterpret_cast<const float4 *>(tab)[e];
            }
        }
        __syncthreads();
        if (b < ib) {
            float sv[4][4], xn[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int j = 0; j < 4; ++j) sv[i][j] = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) xn[i][j] = 0.f;
            }
            // logits and the new state, columns tx + 16j of rows r0 + 16i
            mmrb2<kD2, 4, 8>(Xr, LDB, KB, PB, LDB, r0, tx, sv, xn);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float bias = FOX ? rbias[r0 + 16 * i] + kbias[tx + 16 * j] : 0.f;
                    Ss[(r0 + 16 * i) * LDA + tx + 16 * j] = fmaf(sv[i][j], scale_log2, bias);
                }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) Xr[(r0 + 16 * i) * LDB + tx + 16 * j] = xn[i][j];
        }
        __syncthreads();
        // ---- online softmax, 4 threads per row, 16 columns each
        {
            float x[16];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                x[j] = Ss[row * LDA + part * 16 + j];
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
                *reinterpret_cast<float4 *>(Pm + row * LDA + part * 16 + j) = make_float4(pj[0], pj[1], pj[2], pj[3]);
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
                const float al = alpha_s[r0 + 16 * i];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] *= al;
            }
            mmr<kC, 8>(Pm, LDA, Vs, LDB, r0, c0, acc);
        }
    }
    __syncthreads();
    if (part == 0) alpha_s[row] = (l_run > 0.f) ? 1.f / l_run : 0.f;
    if (lse != nullptr && part == 0 && ib * kC + row < L)
        lse[hL + ib * kC + row] = (m_run + log2f(l_run)) * 0.69314718055994531f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + 16 * i, t = ib * kC + r;
        if (t < L) {
            const float inv = alpha_s[r];
            const float o0[4] = {acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv};
            const float o1[4] = {acc[i][4] * inv, acc[i][5] * inv, acc[i][6] * inv, acc[i][7] * inv};
            put4<T>(out + (hL + t) * kD2 + c0, o0);
            put4<T>(out + (hL + t) * kD2 + c0 + 64, o1);
        }
    }
}

size_t prep_d128_smem() {
    return (size_t)(kC * LDB + 4 * kC * LDA + 2 * kC) * sizeof(float) + kC * sizeof(double);
}
size_t scan_d128_smem() {
    return (size_t)(2 * kC * LDB + kD2 * LDA + kD2 * LDB + 2 * kC * LDA + 3 * kC) * sizeof(float);
}

}  // namespace

// Workspace of the d = 128 forward: 256-byte status header, fp32 q~ (BH, Lp, 128), per block
// [k~ (64 rows); P_b (128 rows)] (BH, nblk, 192, 128), diagonal logits (BH, nblk, 64, 64);
// PaTH-FoX adds the in-block sums lc and the tail sums (BH, Lp) fp32, the block totals
// (BH, nblk) fp64, all in log2 units, and the early-exit bounds per block: smallest in-block
// sum (fp64), largest |k~_j| (fp32), block start offset C_b and prefix minimum Mpre (fp64),
// prefix maximum Kpre (fp32).
D128Layout d128_layout(int B, int H, int L, bool fox) {
    D128Layout y;
    y.BH = B * H;
    y.nblk = (L + kC - 1) / kC;
    y.Lp = y.nblk * kC;
    const size_t bh = (size_t)y.BH;
    size_t off = 256;
    y.off_qt = off;
    off = align256(off + bh * y.Lp * kD2 * 4);
    y.off_kp = off;
    off = align256(off + bh * y.nblk * (kC + kD2) * kD2 * 4);
    y.off_dg = off;
    off = align256(off + bh * y.nblk * kC * kC * 4);
    y.off_lc = y.off_tail = y.off_tot = off;
    y.off_mlc = y.off_kmax = y.off_cst = y.off_mpre = y.off_kpre = off;
    if (fox) {
        const size_t nb = bh * y.nblk;
        off = align256(off + bh * y.Lp * 4);
        y.off_tail = off;
        off = align256(off + bh * y.Lp * 4);
        y.off_tot = off;
        off = align256(off + nb * 8);
        y.off_mlc = off;
        off = align256(off + nb * 8);
        y.off_kmax = off;
        off = align256(off + nb * 4);
        y.off_cst = off;
        off = align256(off + nb * 8);
        y.off_mpre = off;
        off = align256(off + nb * 8);
        y.off_kpre = off;
        off = align256(off + nb * 4);
    }
    y.total = off;
    return y;
}

// log_f non-null: PaTH-FoX (the workspace laid out with the FoX sums).
template <typename T>
cudaError_t launch_prep_d128(const void *q, const void *k, const void *w, const float *beta,
                             const float *log_f, int B, int H, int L, float scale, void *ws,
                             cudaStream_t stream) {
    const bool fox = log_f != nullptr;
    const D128Layout y = d128_layout(B, H, L, fox);
    char *base = static_cast<char *>(ws);
    cudaError_t e;
    if ((e = cudaMemsetAsync(base, 0, 4, stream)) != cudaSuccess) return e;
    const size_t sm = prep_d128_smem();
    auto kern = fox ? prep_d128_kernel<T, true> : prep_d128_kernel<T, false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) !=
        cudaSuccess)
        return e;
    kern<<<dim3(y.nblk, y.BH), kThreads, sm, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(w), beta,
        log_f, L, y.Lp, y.nblk, scale * kLog2e, reinterpret_cast<float *>(base + y.off_qt),
        reinterpret_cast<float *>(base + y.off_kp), reinterpret_cast<float *>(base + y.off_dg),
        reinterpret_cast<float *>(base + y.off_lc), reinterpret_cast<float *>(base + y.off_tail),
        reinterpret_cast<double *>(base + y.off_tot), reinterpret_cast<double *>(base + y.off_mlc),
        reinterpret_cast<float *>(base + y.off_kmax));
    if ((e = cudaGetLastError()) != cudaSuccess || !fox) return e;
    fox_bounds_d128_kernel<<<(y.BH + 3) / 4, 128, 0, stream>>>(
        reinterpret_cast<const double *>(base + y.off_tot), reinterpret_cast<const double *>(base + y.off_mlc),
        reinterpret_cast<const float *>(base + y.off_kmax), reinterpret_cast<double *>(base + y.off_cst),
        reinterpret_cast<double *>(base + y.off_mpre), reinterpret_cast<float *>(base + y.off_kpre),
        y.BH, y.nblk);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_scan_d128(const void *v, void *out, float *lse, bool fox, int B, int H, int L,
                             float scale, void *ws, cudaStream_t stream) {
    const D128Layout y = d128_layout(B, H, L, fox);
    const char *base = static_cast<const char *>(ws);
    cudaError_t e;
    const size_t sm = scan_d128_smem();
    auto kern = fox ? scan_d128_kernel<T, true> : scan_d128_kernel<T, false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) !=
        cudaSuccess)
        return e;
    // shared per token: k~ (512 B), P_b rows (1 KB), v (512 B)
    const bool hf = heads_fastest((size_t)y.BH, (size_t)L, 2048);
    kern<<<hf ? dim3(y.BH, y.nblk) : dim3(y.nblk, y.BH), kThreads, sm, stream>>>(
        static_cast<const T *>(v), reinterpret_cast<const float *>(base + y.off_qt),
        reinterpret_cast<const float *>(base + y.off_kp), reinterpret_cast<const float *>(base + y.off_dg),
        reinterpret_cast<const float *>(base + y.off_lc), reinterpret_cast<const float *>(base + y.off_tail),
        reinterpret_cast<const double *>(base + y.off_tot), reinterpret_cast<const double *>(base + y.off_cst),
        reinterpret_cast<const double *>(base + y.off_mpre), reinterpret_cast<const float *>(base + y.off_kpre),
        static_cast<T *>(out), lse, L, y.Lp, y.nblk, scale * kLog2e, hf ? 1 : 0);
    return cudaGetLastError();
}

#define PATH_D128_INST(T)                                                                        \
    template cudaError_t launch_prep_d128<T>(const void *, const void *, const void *,           \
                                             const float *, const float *, int, int, int, float, \
                                             void *, cudaStream_t);                              \
    template cudaError_t launch_scan_d128<T>(const void *, void *, float *, bool, int, int, int,  \
                                             float, void *, cudaStream_t);
PATH_D128_INST(float)
#undef PATH_D128_INST

}  // namespace path
