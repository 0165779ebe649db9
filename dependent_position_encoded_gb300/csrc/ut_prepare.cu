// K1 (fp32 dtype): per-block UT preprocessing of PaTH attention in fp32 FFMA. bf16 inputs
// use the tensor-core version (ut_prepare_tc.cu); the fp32 workload's 1e-4 tolerance
// rules out 16-bit operands, so this kernel keeps every product in fp32.
//
// For every block of C = 64 tokens of one head (technical summary "技術要約: PaTH
// Attention" §3 "UT変換による表現" and the block-wise algorithm below it; review
// "거리에서 경로로, PaTH Attention" §9) this kernel forms, in fp32:
//   G  = W W^T, N = strictly-upper(G), D = diag(beta)
//   A  = (I + D N)^{-1} D            so that H_0 ... H_63 = I - W^T A W  (UT form)
//   q~_i = (H_0 ... H_i) q_i         = q_i - sum_s (Lq A^T)[i, s] w_s,  Lq[i,u] = (q_i.w_u)[u<=i]
//   k~_j = (H_{j+1} ... H_63)^T k_j  = k_j - sum_u (Rk A)[j, u] w_u,    Rk[j,s] = (k_j.w_s)[s>j]
//   P_b  = H_0 ... H_63              = I - W^T (A W)   (dense 64 x 64 block transition)
//   diagonal-block logits, j <= i:  scale * (q_i.k_j - sum_s (Lq A^T)[i,s] Rk[j,s])
//                                    [+ sum_{s=j+1..i} log f_s]   stored in log2 units.
// Leading and trailing partial products use the matching sub-blocks of A, since
// the inverse of a triangular matrix restricted to a contiguous diagonal range
// is the inverse of that range's sub-block.
//
// One CTA of 256 threads per (block, head), two per SM (six 64 x 64 buffers). Every product
// is a 64 x 64 x 64 contraction over shared memory with W, Q, K and A kept row-major only:
// contractions over the head dimension read both operands as rows, the others read A as
// rows or both operands k-major; each thread owns a 4 x 4 output tile.
#include "common.cuh"

namespace path {

namespace {

constexpr int LD = 68;                 // padded row stride (floats), rows 16-byte aligned
constexpr int BUF = kC * LD;           // floats per 64 x 64 buffer
constexpr int kPrepThreads = 256;

// acc[i][j] += sum_{k in [k0, k1)} X[k][m0 + i] * Y[k][n0 + j]
__device__ __forceinline__ void mm_acc(const float *__restrict__ X, const float *__restrict__ Y,
                                       int m0, int n0, float (&acc)[4][4], int k0 = 0,
                                       int k1 = kC) {
#pragma unroll 4
    for (int k = k0; k < k1; ++k) {
        const float4 a = *reinterpret_cast<const float4 *>(X + k * LD + m0);
        const float4 b = *reinterpret_cast<const float4 *>(Y + k * LD + n0);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

__device__ __forceinline__ void zero(float (&acc)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
}

// Products whose operands are both stored with the contraction index contiguous
// (A[m][k], B[n][k]; e.g. W W^T from W alone) use an interleaved thread tile: rows
// ty + 16i, columns tx + 16j, so that the eight lanes of a quarter warp read eight
// consecutive B rows, whose 16-byte pieces fall in distinct bank groups at a row stride of
// 68 floats. acc[i][j] += sum_k A[ty + 16i][k] * B[tx + 16j][k].
__device__ __forceinline__ void mm_rows(const float *__restrict__ A, const float *__restrict__ B,
                                        int ty, int tx, float (&acc)[4][4]) {
#pragma unroll 2
    for (int k = 0; k < kC; k += 4) {
        float4 a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (ty + 16 * i) * LD + k);
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4 *>(B + (tx + 16 * j) * LD + k);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t = acc[i][j];
                t = fmaf(a[i].x, b[j].x, t);
                t = fmaf(a[i].y, b[j].y, t);
                t = fmaf(a[i].z, b[j].z, t);
                acc[i][j] = fmaf(a[i].w, b[j].w, t);
            }
    }
}

// The interleaved tile from k-major operands: acc[i][j] += sum_k X[k][ty + 16i] Y[k][tx + 16j]
__device__ __forceinline__ void mm_kk_il(const float *__restrict__ X, const float *__restrict__ Y,
                                         int ty, int tx, float (&acc)[4][4]) {
#pragma unroll 4
    for (int k = 0; k < kC; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            av[i] = X[k * LD + ty + 16 * i];
            bv[i] = Y[k * LD + tx + 16 * i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

// A row-major, B k-major (standard tile): acc[i][j] += sum_k A[m0 + i][k] * B[k][n0 + j]
__device__ __forceinline__ void mm_rowa(const float *__restrict__ A, const float *__restrict__ B,
                                        int m0, int n0, float (&acc)[4][4]) {
#pragma unroll 2
    for (int k = 0; k < kC; k += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(A + (m0 + i) * LD + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 b = *reinterpret_cast<const float4 *>(B + (k + kk) * LD + n0);
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
            }
        }
    }
}

// Writes an interleaved tile (rows ty + 16i, cols tx + 16j) into buffer Z as Z[m][n].
__device__ __forceinline__ void store_il(float *Z, int ty, int tx, const float (&acc)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Z[(ty + 16 * i) * LD + tx + 16 * j] = acc[i][j];
}

// Writes acc (rows m0.., cols n0..) into buffer Z as Z[m][n].
__device__ __forceinline__ void store_rm(float *Z, int m0, int n0, const float (&acc)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(Z + (m0 + i) * LD + n0) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}

template <typename T>
__device__ __forceinline__ void store_row4(T *dst, const float *v);
template <>
__device__ __forceinline__ void store_row4<float>(float *dst, const float *v) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// T: input element type; TO: element type of q~, k~ and P_b (the backward recomputes them
// in fp32 from bf16 inputs)
template <typename T, typename TO = T>
__global__ void __launch_bounds__(kPrepThreads)
ut_prepare_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ w,
                  const float *__restrict__ beta, const float *__restrict__ log_f, int L,
                  int Lp, int nblk, float scale_log2, TO *__restrict__ qt, TO *__restrict__ kp,
                  float *__restrict__ dg, uint32_t *status) {
    extern __shared__ __align__(16) float sm[];
    float *Wr = sm;            // W[s][c]
    float *Qr = Wr + BUF;      // Q[i][c]
    float *Kr = Qr + BUF;      // K[j][c]
    float *Ar = Kr + BUF;      // A[s][u]
    float *X = Ar + BUF;       // scratch
    float *Y = X + BUF;        // scratch
    float *bs = Y + BUF;       // beta[64]
    float *lc = bs + kC;       // block-local inclusive cumsum of log f [64]

    const int tid = threadIdx.x;
    const int blk = blockIdx.x;
    const int bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t head = (size_t)bh * L;
    if (blk == 0 && bh == 0 && tid == 0 && status) *status = 0u;

    // ---- load W, Q, K (fp32, row-major), beta; padded tokens are zero. Four
    // elements per thread and step, all of a thread's loads issued before the first store.
    {
        constexpr int kIt = kC * kD / 4 / kPrepThreads;
        float wv[kIt][4], qv[kIt][4], kv[kIt][4];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = 4 * (tid + it * kPrepThreads), s = e / kD, c = e % kD;
            const bool in = t0 + s < L;
            const size_t g = (head + t0 + s) * kD + c;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wv[it][j] = in ? Elt<T>::to_f(w[g + j]) : 0.f;
                qv[it][j] = in ? Elt<T>::to_f(q[g + j]) : 0.f;
                kv[it][j] = in ? Elt<T>::to_f(k[g + j]) : 0.f;
            }
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = 4 * (tid + it * kPrepThreads), s = e / kD, c = e % kD;
            *reinterpret_cast<float4 *>(Wr + s * LD + c) = make_float4(wv[it][0], wv[it][1], wv[it][2], wv[it][3]);
            *reinterpret_cast<float4 *>(Qr + s * LD + c) = make_float4(qv[it][0], qv[it][1], qv[it][2], qv[it][3]);
            *reinterpret_cast<float4 *>(Kr + s * LD + c) = make_float4(kv[it][0], kv[it][1], kv[it][2], kv[it][3]);
            *reinterpret_cast<float4 *>(Ar + s * LD + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (tid < kC) {
        const int t = t0 + tid;
        bs[tid] = (t < L) ? beta[head + t] : 0.f;
    }
    if (log_f != nullptr && tid < 32) {
        // inclusive scan of the block's log f values (two per lane)
        const int t_a = t0 + 2 * tid, t_b = t_a + 1;
        float a = (t_a < L) ? log_f[head + t_a] : 0.f;
        float b = (t_b < L) ? log_f[head + t_b] : 0.f;
        b += a;
        float run = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float n = __shfl_up_sync(0xffffffffu, run, o);
            if (tid >= o) run += n;
        }
        const float excl = run - b;
        lc[2 * tid] = excl + a;
        lc[2 * tid + 1] = excl + b;
    }
    __syncthreads();

    const int ty = tid / 16, tx = tid % 16;
    const int m0 = ty * 4, n0 = tx * 4;
    float acc[4][4];

    // ---- G = W W^T -> X (row-major G[s][u])
    zero(acc);
    mm_rows(Wr, Wr, ty, tx, acc);
    store_il(X, ty, tx, acc);
    __syncthreads();

    // ---- A = (I + D N)^{-1} D, one column per group of 4 threads.
    // Column u: A[u][u] = beta_u; for s < u, A[s][u] = -beta_s sum_{v=s+1..u} G[s][v] A[v][u].
    {
        const int u = tid >> 2, part = tid & 3;
        for (int s = kC - 1; s >= 0; --s) {
            float sum = 0.f;
            for (int v = s + 1 + part; v < kC; v += 4) sum = fmaf(X[s * LD + v], Ar[v * LD + u], sum);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (part == 0) {
                float a = 0.f;
                if (s == u) a = bs[u];
                else if (s < u) a = -bs[s] * sum;
                Ar[s * LD + u] = a;
            }
            __syncwarp();
        }
    }
    __syncthreads();

    // ---- Lq^T -> X ([u][i], u <= i), Rk^T -> Y ([s][j], s > j)
    zero(acc);
    mm_rows(Wr, Qr, ty, tx, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (ty + 16 * i > tx + 16 * j) acc[i][j] = 0.f;
    store_il(X, ty, tx, acc);
    zero(acc);
    mm_rows(Wr, Kr, ty, tx, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (ty + 16 * i <= tx + 16 * j) acc[i][j] = 0.f;
    store_il(Y, ty, tx, acc);
    __syncthreads();

    // ---- Qhat^T[s][i] = sum_u A[s][u] Lq^T[u][i]  (in place in X)
    zero(acc);
    mm_rowa(Ar, X, m0, n0, acc);
    __syncthreads();
    store_rm(X, m0, n0, acc);
    __syncthreads();

    const size_t blk_base = (size_t)bh * nblk + blk;

    // ---- diagonal-block logits: Dg[i][j] = scale_log2 * (q_i.k_j - sum_s Qhat[i][s] Rk[j][s])
    // (interleaved tile: rows ty + 16i, columns tx + 16j)
    {
        float qk[4][4], corr[4][4];
        zero(qk);
        zero(corr);
        mm_rows(Qr, Kr, ty, tx, qk);
        mm_kk_il(X, Y, ty, tx, corr);
        float *out = dg + blk_base * kC * kC;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ii = ty + 16 * i;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int jj = tx + 16 * j;
                float x = scale_log2 * (qk[i][j] - corr[i][j]);
                if (log_f != nullptr) x += kLog2e * (lc[ii] - lc[jj]);
                out[ii * kC + jj] = (jj <= ii && t0 + jj < L) ? x : -INFINITY;
            }
        }
    }

    // ---- q~[i][c] = q[i][c] - sum_s Qhat[i][s] W[s][c]
    {
        zero(acc);
        mm_acc(X, Wr, m0, n0, acc);
        TO *out = qt + ((size_t)bh * Lp + t0) * kD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = Qr[(m0 + i) * LD + n0 + j] - acc[i][j];
            store_row4<TO>(out + (m0 + i) * kD + n0, v);
        }
    }
    __syncthreads();

    // ---- Khat^T[u][j] = sum_s A[s][u] Rk^T[s][j]  (in place in Y)
    zero(acc);
    mm_acc(Ar, Y, m0, n0, acc);
    __syncthreads();
    store_rm(Y, m0, n0, acc);
    __syncthreads();

    // ---- k~[j][c] = k[j][c] - sum_u Khat[j][u] W[u][c];  AW = A W -> X
    TO *kp_blk = kp + blk_base * (2 * kC) * kD;
    {
        zero(acc);
        mm_acc(Y, Wr, m0, n0, acc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = Kr[(m0 + i) * LD + n0 + j] - acc[i][j];
            store_row4<TO>(kp_blk + (m0 + i) * kD + n0, v);
        }
        zero(acc);
        mm_rowa(Ar, Wr, m0, n0, acc);
        store_rm(X, m0, n0, acc);
    }
    __syncthreads();

    // ---- P_b[n][c] = delta(n, c) - sum_s W[s][n] (A W)[s][c]
    {
        zero(acc);
        mm_acc(Wr, X, m0, n0, acc);
        TO *out = kp_blk + kC * kD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = ((m0 + i) == (n0 + j) ? 1.f : 0.f) - acc[i][j];
            store_row4<TO>(out + (m0 + i) * kD + n0, v);
        }
    }
}

}  // namespace

size_t ut_prepare_smem_bytes() { return (size_t)(6 * BUF + 2 * kC) * sizeof(float); }

template <typename T>
cudaError_t launch_ut_prepare(const void *q, const void *k, const void *w, const float *beta,
                              const float *log_f, int BH, int L, float scale, void *ws,
                              cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, (int)sizeof(T), log_f != nullptr);
    char *base = static_cast<char *>(ws);
    const size_t smem = ut_prepare_smem_bytes();
    cudaError_t err = cudaFuncSetAttribute(ut_prepare_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(lay.nblk, BH);
    ut_prepare_kernel<T><<<grid, kPrepThreads, smem, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(w), beta,
        log_f, L, lay.Lp, lay.nblk, scale * kLog2e, reinterpret_cast<T *>(base + lay.off_qt),
        reinterpret_cast<T *>(base + lay.off_kp), reinterpret_cast<float *>(base + lay.off_dg),
        reinterpret_cast<uint32_t *>(base));
    return cudaGetLastError();
}

// The per-block factors in fp32 at explicit places, for the backward (log_f: PaTH-FoX
// diagonal logits, else null):
// qt (BH, Lp, 64), kp (BH, nblk, 128, 64) = [k~ rows; P_b rows] per block, dg (BH, nblk, 64,
// 64) diagonal-block logits in log2 units (scale included, -inf above the diagonal and past L).
template <typename T>
cudaError_t launch_ut_prepare_f32out(const void *q, const void *k, const void *w,
                                     const float *beta, const float *log_f, int BH, int L, int Lp,
                                     int nblk, float scale, float *qt, float *kp, float *dg,
                                     uint32_t *status, cudaStream_t stream) {
    const size_t smem = ut_prepare_smem_bytes();
    cudaError_t err = cudaFuncSetAttribute(ut_prepare_kernel<T, float>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(nblk, BH);
    ut_prepare_kernel<T, float><<<grid, kPrepThreads, smem, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(w), beta,
        log_f, L, Lp, nblk, scale * kLog2e, qt, kp, dg, status);
    return cudaGetLastError();
}
template cudaError_t launch_ut_prepare_f32out<float>(const void *, const void *, const void *,
                                                     const float *, const float *, int, int, int,
                                                     int, float, float *, float *, float *,
                                                     uint32_t *, cudaStream_t);
template cudaError_t launch_ut_prepare_f32out<__nv_bfloat16>(
    const void *, const void *, const void *, const float *, const float *, int, int, int, int,
    float, float *, float *, float *, uint32_t *, cudaStream_t);

// PaTH-FoX: log2(e) * inclusive prefix sums of log f per head into the workspace.
template cudaError_t launch_ut_prepare<float>(const void *, const void *, const void *,
                                              const float *, const float *, int, int, float,
                                              void *, cudaStream_t);

}  // namespace path
