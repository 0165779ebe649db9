// Backward pass of PaTH attention (plain PaTH), fp32 on the CUDA cores.
//
// The pages give no backward (review "거리에서 경로로, PaTH Attention" §9 and technical
// summary "技術要約: PaTH Attention" §3 say the block-wise algorithm makes training
// efficient, without the gradient). This is the chain rule applied to the block form of
// the forward. Per head, with 64-token blocks, q~_i, k~_j and the dense block transition
// P_b = H_start(b) ... H_end(b) as in the forward, the logit of query i in block a and key
// j in block b < a is scale * T_ij with
//     T_ab = X_{a,b} K~_b^T,   X_{a,a-1} = Q~_a,   X_{a,b-1} = X_{a,b} P_b^T
// (X_{a,b}: the rows of query block a carried down to key block b). With the softmax
// gradient dS_ij = p_ij (dout_i . v_j - dout_i . out_i) and dT = scale * dS:
//     dv_j    += p_ij dout_i
//     dK~_b   += dT_ab^T X_{a,b}
//     G_b      = G_{b-1} P_b + dT_ab K~_b        (G_b: gradient of X_{a,b}; G_{-1} = 0)
//     dP_b    += G_{b-1}^T X_{a,b}
//     dQ~_a    = G_{a-1}
// The first recursion runs right to left and the second left to right, so the query pass
// (B1) keeps X_{a,b} and dT_ab of its walk in a workspace stash and then runs the gradient
// walk back over it. Within a block, q~, k~, P_b and the diagonal-block logits are
// products of the block's own transitions; the block pass (B2) takes their gradients to
// q, k, w and beta by reverse mode through token-level sweeps:
//     q~_i = H_0 H_1 ... H_i q_i,  k~_j = H_63 ... H_{j+1} k_j,  P_b e_c = H_0 ... H_63 e_c,
//     T_ij = k_j . (H_{j+1} ... H_i q_i)   (j <= i, same block),
// and through each x' = H_s x = x - beta_s w_s (w_s . x), with g the gradient of x':
//     dbeta_s -= (w_s . g)(w_s . x),  dw_s -= beta_s ((w_s . x) g + (w_s . g) x),
//     gradient of x = H_s g.
// Before both passes the fp32 UT preparation kernel recomputes q~, k~, P_b and the diagonal
// logits from the inputs.
#include "common.cuh"

namespace path {

template <typename T>
cudaError_t launch_ut_prepare_f32out(const void *q, const void *k, const void *w,
                                     const float *beta, int BH, int L, int Lp, int nblk,
                                     float scale, float *qt, float *kp, float *dg,
                                     uint32_t *status, cudaStream_t stream);

namespace {

constexpr int LD = 68;          // padded row stride (floats) of a 64 x 64 shared buffer
constexpr int BUF = kC * LD;
constexpr int kThreads = 256;
constexpr int kBlkTile = kC * kD;  // floats in one 64 x 64 tile

// acc[i][j] += sum_k X[k][m0 + i] * Y[k][n0 + j]  (both operands k-major in shared memory)
__device__ __forceinline__ void mm_acc(const float *__restrict__ X, const float *__restrict__ Y,
                                       int m0, int n0, float (&acc)[4][4]) {
#pragma unroll 4
    for (int k = 0; k < kC; ++k) {
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

__device__ __forceinline__ void zero4(float (&a)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[i][j] = 0.f;
}

// 64 x 64 fp32 tile from global (row-major, 64 floats per row) into shared memory, as is
// (dst[r][c]) or transposed (dst[c][r]).
__device__ __forceinline__ void load_tile(float *dst, const float *__restrict__ src, bool transpose) {
    for (int e = threadIdx.x; e < kBlkTile; e += kThreads) {
        const int r = e / kD, c = e % kD;
        const float x = src[e];
        if (transpose) dst[c * LD + r] = x;
        else dst[r * LD + c] = x;
    }
}

// Rows t0 .. t0 + 63 of a (rows, 64) tensor of type T, zero past L, as is and transposed
// (either may be null).
template <typename T>
__device__ __forceinline__ void load_rows(float *dst, float *dst_t, const T *__restrict__ src,
                                          int t0, int L) {
    for (int e = threadIdx.x; e < kBlkTile; e += kThreads) {
        const int r = e / kD, c = e % kD;
        const float x = (t0 + r < L) ? Elt<T>::to_f(src[(size_t)(t0 + r) * kD + c]) : 0.f;
        if (dst) dst[r * LD + c] = x;
        if (dst_t) dst_t[c * LD + r] = x;
    }
}

// ---------------------------------------------------------------- B1: query pass
// One CTA per (query block a, head); a runs from the last block down so that the longest
// walks start first.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
bwd_query_kernel(const T *__restrict__ v, const T *__restrict__ o, const T *__restrict__ dout,
                 const float *__restrict__ lse, const float *__restrict__ qt,
                 const float *__restrict__ kp, const float *__restrict__ dg,
                 float *__restrict__ dqt, float *__restrict__ dkt, float *__restrict__ dP,
                 float *__restrict__ dTd, float *__restrict__ stash, float *__restrict__ dv,
                 int L, int Lp, int nblk, float scale, float scale_log2) {
    extern __shared__ __align__(16) float sm[];
    float *XT = sm;              // pass 1: X^T [c][i]
    float *Xr = XT + BUF;        // X [i][c] (pass 2: from the stash)
    float *KB = Xr + BUF;        // pass 1: K~_b^T [c][j];  pass 2: K~_b [j][c]
    float *PB = KB + BUF;        // pass 1: P_b^T [c][n];   pass 2: P_b [n][c]
    float *B4 = PB + BUF;        // pass 1: V_b^T [c][j];   pass 2: G^T [n][i]
    float *B5 = B4 + BUF;        // pass 1: dout^T [c][i];  pass 2: G [i][n]
    float *dOr = B5 + BUF;       // dout [i][c]
    float *B7 = dOr + BUF;       // pass 1: p [i][j];       pass 2: dT^T [j][i]
    float *dTm = B7 + BUF;       // pass 1: dT [i][j]
    float *lse2 = dTm + BUF;     // per row: lse * log2(e)
    float *Drow = lse2 + kC;     // per row: dout . out

    const int tid = threadIdx.x;
    const int a = nblk - 1 - (int)blockIdx.x;
    const int bh = blockIdx.y;
    const int ty = tid / 16, tx = tid % 16, m0 = ty * 4, n0 = tx * 4;
    const int t0 = a * kC;
    const size_t hL = (size_t)bh * L;

    // ---- per row: lse in log2 units and D_i = dout_i . out_i (4 threads per row)
    {
        const int row = tid >> 2, part = tid & 3;
        float dsum = 0.f;
        if (t0 + row < L) {
            const size_t g = (hL + t0 + row) * kD + part * 16;
#pragma unroll
            for (int c = 0; c < 16; ++c)
                dsum = fmaf(Elt<T>::to_f(dout[g + c]), Elt<T>::to_f(o[g + c]), dsum);
        }
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
        if (part == 0) {
            Drow[row] = dsum;
            lse2[row] = (t0 + row < L) ? lse[hL + t0 + row] * kLog2e : 0.f;
        }
    }
    load_rows<T>(dOr, B5, dout + hL * kD, t0, L);
    load_rows<T>(nullptr, B4, v + hL * kD, t0, L);
    __syncthreads();

    // ---- diagonal block: logits from the table; dT to the block pass, p^T dout to dv
    float pr[4][4], dpm[4][4];
    {
        zero4(dpm);
        mm_acc(B5, B4, m0, n0, dpm);  // dout_i . v_j
        const float *tab = dg + ((size_t)bh * nblk + a) * kBlkTile;
        float *dtd = dTd + ((size_t)bh * nblk + a) * kBlkTile;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = m0 + i;
            const float4 s4 = *reinterpret_cast<const float4 *>(tab + r * kC + n0);
            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
            float dt[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float p = (t0 + r < L) ? exp2f(sv[j] - lse2[r]) : 0.f;
                pr[i][j] = p;
                dt[j] = scale * p * (dpm[i][j] - Drow[r]);
            }
            *reinterpret_cast<float4 *>(dtd + r * kC + n0) = make_float4(dt[0], dt[1], dt[2], dt[3]);
            *reinterpret_cast<float4 *>(B7 + r * LD + n0) = make_float4(pr[i][0], pr[i][1], pr[i][2], pr[i][3]);
        }
    }
    __syncthreads();
    {
        float acc[4][4];
        zero4(acc);
        mm_acc(B7, dOr, m0, n0, acc);  // sum_i p_ij dout_i[c]
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (t0 + m0 + j < L)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    atomicAdd(dv + (hL + t0 + m0 + j) * kD + n0 + c, acc[j][c]);
    }

    // ---- pass 1: right to left over key blocks, X from Q~_a
    const float *qa = qt + ((size_t)bh * Lp + t0) * kD;
    __syncthreads();
    for (int e = tid; e < kBlkTile; e += kThreads) {
        const int r = e / kD, c = e % kD;
        const float x = qa[e];
        XT[c * LD + r] = x;
        Xr[r * LD + c] = x;
    }
    const size_t pair0 = (size_t)bh * ((size_t)nblk * (nblk - 1) / 2) + (size_t)a * (a - 1) / 2;
    for (int b = a - 1; b >= 0; --b) {
        const float *blk = kp + ((size_t)bh * nblk + b) * 2 * kBlkTile;
        __syncthreads();
        load_tile(KB, blk, true);
        load_tile(PB, blk + kBlkTile, true);
        load_rows<T>(nullptr, B4, v + hL * kD, b * kC, L);
        __syncthreads();
        float s[4][4], xn[4][4];
        zero4(s);
        zero4(dpm);
        zero4(xn);
        mm_acc(XT, KB, m0, n0, s);
        mm_acc(B5, B4, m0, n0, dpm);
        if (b > 0) mm_acc(XT, PB, m0, n0, xn);
        float *st = stash + (pair0 + b) * 2 * kBlkTile;  // [X_{a,b} | dT_ab], row-major
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = m0 + i;
            float p4[4], d4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float p = (t0 + r < L) ? exp2f(s[i][j] * scale_log2 - lse2[r]) : 0.f;
                p4[j] = p;
                d4[j] = scale * p * (dpm[i][j] - Drow[r]);
            }
            *reinterpret_cast<float4 *>(B7 + r * LD + n0) = make_float4(p4[0], p4[1], p4[2], p4[3]);
            *reinterpret_cast<float4 *>(dTm + r * LD + n0) = make_float4(d4[0], d4[1], d4[2], d4[3]);
            *reinterpret_cast<float4 *>(st + kBlkTile + r * kC + n0) = make_float4(d4[0], d4[1], d4[2], d4[3]);
            *reinterpret_cast<float4 *>(st + r * kC + n0) =
                *reinterpret_cast<const float4 *>(Xr + r * LD + n0);
        }
        __syncthreads();
        {
            float acc[4][4];
            zero4(acc);
            mm_acc(dTm, Xr, m0, n0, acc);  // dK~_b[j][c] += sum_i dT_ij X_ic
            float *dk = dkt + ((size_t)bh * Lp + (size_t)b * kC) * kD;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) atomicAdd(dk + (m0 + j) * kD + n0 + c, acc[j][c]);
            zero4(acc);
            mm_acc(B7, dOr, m0, n0, acc);  // dv_j += sum_i p_ij dout_i (key block b < a is full)
            float *dvb = dv + (hL + (size_t)b * kC) * kD;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) atomicAdd(dvb + (m0 + j) * kD + n0 + c, acc[j][c]);
        }
        __syncthreads();
        if (b > 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                *reinterpret_cast<float4 *>(Xr + (m0 + i) * LD + n0) =
                    make_float4(xn[i][0], xn[i][1], xn[i][2], xn[i][3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) XT[(n0 + j) * LD + m0 + i] = xn[i][j];
            }
        }
    }

    // ---- pass 2: left to right, G = gradient of X_{a,b}
    float g[4][4];
    zero4(g);
    __syncthreads();
    for (int e = tid; e < BUF; e += kThreads) {
        B4[e] = 0.f;
        B5[e] = 0.f;
    }
    for (int b = 0; b < a; ++b) {
        const float *blk = kp + ((size_t)bh * nblk + b) * 2 * kBlkTile;
        const float *st = stash + (pair0 + b) * 2 * kBlkTile;
        __syncthreads();
        load_tile(Xr, st, false);
        load_tile(B7, st + kBlkTile, true);
        load_tile(KB, blk, false);
        load_tile(PB, blk + kBlkTile, false);
        __syncthreads();
        if (b > 0) {
            float acc[4][4];
            zero4(acc);
            mm_acc(B5, Xr, m0, n0, acc);  // dP_b[n][c] += sum_i G_{b-1}[i][n] X_{a,b}[i][c]
            float *dpb = dP + ((size_t)bh * nblk + b) * kBlkTile;
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) atomicAdd(dpb + (m0 + n) * kC + n0 + c, acc[n][c]);
        }
        zero4(g);
        if (b > 0) mm_acc(B4, PB, m0, n0, g);  // G_{b-1} P_b
        mm_acc(B7, KB, m0, n0, g);             // + dT_ab K~_b
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            *reinterpret_cast<float4 *>(B5 + (m0 + i) * LD + n0) =
                make_float4(g[i][0], g[i][1], g[i][2], g[i][3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) B4[(n0 + j) * LD + m0 + i] = g[i][j];
        }
    }
    // dQ~_a = G_{a-1} (zero for the first block)
    float *dq = dqt + ((size_t)bh * Lp + t0) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(dq + (m0 + i) * kD + n0) = make_float4(g[i][0], g[i][1], g[i][2], g[i][3]);
}

// ---------------------------------------------------------------- B2: block pass
// One CTA per (block, head), 8 warps. Each warp takes sweeps w, w + 8, ... of 192: query
// rows (q~_i and the diagonal logits, i = 0..63), columns of P_b (c = 0..63) and key rows
// (k~_j, j = 0..63). Lane l holds dimensions 2l and 2l + 1 of every vector. A sweep first
// applies its transitions, keeping only w_s . x of each step (64 floats per warp), then
// walks back with the gradient, recovering each step's input by undoing the step: the step
// is x' = x - c w_s with c = beta_s (w_s . x), so x = x' + c w_s, exact up to rounding (no
// H_s is inverted; it is singular at beta_s = 1). dk, dw and dbeta gather in shared memory
// (several sweeps add to one token); dq is written by its query sweep. 68 KB of shared
// memory per CTA, three CTAs per SM.
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_dot(float2 a, float2 b) {
    float s = fmaf(a.x, b.x, a.y * b.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

template <typename T>
__device__ __forceinline__ float2 load2(const T *p) {
    return make_float2(Elt<T>::to_f(p[0]), Elt<T>::to_f(p[1]));
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 3)
bwd_block_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ w,
                 const float *__restrict__ beta, const float *__restrict__ dqt,
                 const float *__restrict__ dkt, const float *__restrict__ dP,
                 const float *__restrict__ dTd, float *__restrict__ dq, float *__restrict__ dk,
                 float *__restrict__ dw, float *__restrict__ dbeta, int L, int Lp, int nblk) {
    extern __shared__ __align__(16) float sm[];
    float2 *Ws = reinterpret_cast<float2 *>(sm);        // w_s, [s][lane]
    float2 *Ks = Ws + kBlkTile / 2;                        // k_j
    float2 *dWs = Ks + kBlkTile / 2;                       // gradient of w_s
    float2 *dKs = dWs + kBlkTile / 2;                      // gradient of k_j
    float *wxs = reinterpret_cast<float *>(dKs + kBlkTile / 2);  // per warp: 64 w.x
    float *bs = wxs + kWarps * kC;                      // beta_s
    float *dBs = bs + kC;                               // gradient of beta_s

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t hL = (size_t)bh * L;
    const int nvalid = min(kC, L - t0);

    // w, k (zero past L: a padded token's transition is the identity), beta
    for (int e = tid; e < kBlkTile / 2; e += kThreads) {
        const int r = e / 32, l = e % 32;
        const bool in = r < nvalid;
        const size_t g = (hL + t0 + r) * kD + 2 * l;
        Ws[e] = in ? load2<T>(w + g) : make_float2(0.f, 0.f);
        Ks[e] = in ? load2<T>(k + g) : make_float2(0.f, 0.f);
        dWs[e] = make_float2(0.f, 0.f);
        dKs[e] = make_float2(0.f, 0.f);
    }
    if (tid < kC) {
        bs[tid] = tid < nvalid ? beta[hL + t0 + tid] : 0.f;
        dBs[tid] = 0.f;
    }
    __syncthreads();

    float *wxw = wxs + warp * kC;
    // gradient through x' = H_s x (x = input, wx = w_s . x); g becomes the gradient of x
    auto back_step = [&](int s, float2 x, float wx, float2 &g) {
        const float2 ws = Ws[s * 32 + lane];
        const float wg = warp_dot(ws, g);
        const float be = bs[s];
        atomicAdd(&dWs[s * 32 + lane].x, -be * fmaf(wx, g.x, wg * x.x));
        atomicAdd(&dWs[s * 32 + lane].y, -be * fmaf(wx, g.y, wg * x.y));
        if (lane == 0) atomicAdd(&dBs[s], -wg * wx);
        g.x = fmaf(-be * wg, ws.x, g.x);
        g.y = fmaf(-be * wg, ws.y, g.y);
    };
    // x <- H_s x, recording w_s . x at wxw[s]
    auto fwd_step = [&](int s, float2 &x) {
        const float2 ws = Ws[s * 32 + lane];
        const float wx = warp_dot(ws, x);
        if (lane == 0) wxw[s] = wx;
        const float a = bs[s] * wx;
        x.x = fmaf(-a, ws.x, x.x);
        x.y = fmaf(-a, ws.y, x.y);
    };
    // x <- the input of step s, from its output x and the recorded w_s . x
    auto undo_step = [&](int s, float wx, float2 &x) {
        const float2 ws = Ws[s * 32 + lane];
        const float a = bs[s] * wx;
        x.x = fmaf(a, ws.x, x.x);
        x.y = fmaf(a, ws.y, x.y);
    };

    const bool has_dp = blk > 0 && blk < nblk - 1;  // P_0 and the last P_b reach no logit
    const bool has_dk = blk < nblk - 1;             // the last block's k~ reach no later query
    for (int task = warp; task < 3 * kC; task += kWarps) {
        const int kind = task / kC, idx = task % kC;
        if (kind == 0) {
            // ---- query row i: x_j = H_{j+1} ... H_i q_i, q~_i = H_0 x_0, T_ij = k_j . x_j
            const int i = idx;
            if (i >= nvalid) continue;
            float2 x = load2<T>(q + (hL + t0 + i) * kD + 2 * lane);
            for (int s = i; s >= 1; --s) fwd_step(s, x);  // wxw[s] = w_s . x_s
            const float wx0 = warp_dot(Ws[lane], x);       // x = x_0
            __syncwarp();
            float2 g = *reinterpret_cast<const float2 *>(dqt + ((size_t)bh * Lp + t0 + i) * kD + 2 * lane);
            const float2 dtr = *reinterpret_cast<const float2 *>(
                dTd + (((size_t)bh * nblk + blk) * kC + i) * kC + 2 * lane);
            back_step(0, x, wx0, g);
            for (int j = 0; j <= i; ++j) {
                const float dtx = __shfl_sync(0xffffffffu, dtr.x, j >> 1);
                const float dty = __shfl_sync(0xffffffffu, dtr.y, j >> 1);
                const float dt = (j & 1) ? dty : dtx;
                const float2 kj = Ks[j * 32 + lane];  // x = x_j here
                g.x = fmaf(dt, kj.x, g.x);
                g.y = fmaf(dt, kj.y, g.y);
                atomicAdd(&dKs[j * 32 + lane].x, dt * x.x);
                atomicAdd(&dKs[j * 32 + lane].y, dt * x.y);
                if (j < i) {
                    const float wx = wxw[j + 1];
                    undo_step(j + 1, wx, x);  // x = x_{j+1}
                    back_step(j + 1, x, wx, g);
                }
            }
            *reinterpret_cast<float2 *>(dq + (hL + t0 + i) * kD + 2 * lane) = g;
        } else if (kind == 1) {
            // ---- column c of P_b = H_0 ... H_63 e_c
            if (!has_dp) continue;
            const int c = idx;
            float2 x = make_float2(2 * lane == c ? 1.f : 0.f, 2 * lane + 1 == c ? 1.f : 0.f);
            for (int s = kC - 1; s >= 1; --s) fwd_step(s, x);
            const float wx0 = warp_dot(Ws[lane], x);
            __syncwarp();
            const float *dpb = dP + ((size_t)bh * nblk + blk) * kBlkTile;
            float2 g = make_float2(dpb[(2 * lane) * kC + c], dpb[(2 * lane + 1) * kC + c]);
            back_step(0, x, wx0, g);
            for (int j = 0; j + 1 < kC; ++j) {
                const float wx = wxw[j + 1];
                undo_step(j + 1, wx, x);
                back_step(j + 1, x, wx, g);
            }
        } else {
            // ---- key row j: k~_j = H_63 ... H_{j+1} k_j
            const int j = idx;
            if (j >= nvalid || !has_dk) continue;
            float2 y = Ks[j * 32 + lane];
            for (int s = j + 1; s < kC; ++s) fwd_step(s, y);  // wxw[s]: w_s . (input of H_s)
            __syncwarp();
            float2 g = *reinterpret_cast<const float2 *>(dkt + ((size_t)bh * Lp + t0 + j) * kD + 2 * lane);
            for (int s = kC - 1; s > j; --s) {
                const float wx = wxw[s];
                undo_step(s, wx, y);  // y = input of H_s
                back_step(s, y, wx, g);
            }
            atomicAdd(&dKs[j * 32 + lane].x, g.x);
            atomicAdd(&dKs[j * 32 + lane].y, g.y);
        }
        __syncwarp();  // the next sweep rewrites wxw
    }
    __syncthreads();
    for (int e = tid; e < nvalid * 32; e += kThreads) {
        const int r = e / 32, l = e % 32;
        const size_t g = (hL + t0 + r) * kD + 2 * l;
        *reinterpret_cast<float2 *>(dk + g) = dKs[e];
        *reinterpret_cast<float2 *>(dw + g) = dWs[e];
    }
    if (tid < nvalid) dbeta[hL + t0 + tid] = dBs[tid];
}

}  // namespace

// Workspace of the backward: 256-byte status header, then fp32 q~ (BH, Lp, 64),
// [k~; P_b] (BH, nblk, 128, 64), diagonal logits (BH, nblk, 64, 64), dq~ and dk~ (BH, Lp,
// 64), dP_b and the diagonal dT (BH, nblk, 64, 64), and the query pass's stash: X_{a,b} and
// dT_ab for every pair b < a (BH, nblk (nblk - 1) / 2, 2, 64, 64).
BwdLayout bwd_layout(int B, int H, int L) {
    BwdLayout y;
    y.BH = B * H;
    y.nblk = (L + kC - 1) / kC;
    y.Lp = y.nblk * kC;
    const size_t bh = (size_t)y.BH, tile = (size_t)kBlkTile * 4;
    const size_t rows = bh * y.Lp * kD * 4, blocks = bh * y.nblk * tile;
    size_t off = 256;
    y.off_qt = off;
    off = align256(off + rows);
    y.off_kp = off;
    off = align256(off + 2 * blocks);
    y.off_dg = off;
    off = align256(off + blocks);
    y.off_dqt = off;
    off = align256(off + rows);
    y.off_dkt = off;
    off = align256(off + rows);
    y.off_dP = off;
    off = align256(off + blocks);
    y.off_dTd = off;
    off = align256(off + blocks);
    y.off_stash = off;
    off = align256(off + bh * ((size_t)y.nblk * (y.nblk - 1) / 2) * 2 * tile);
    y.total = off;
    return y;
}

size_t bwd_query_smem() { return (size_t)(9 * BUF + 2 * kC) * sizeof(float); }
size_t bwd_block_smem() { return (size_t)(4 * kBlkTile + kWarps * kC + 2 * kC) * sizeof(float); }

// dq, dk, dv, dw (B*H, L, 64) and dbeta (B*H, L) fp32. dv gathers by atomics from zero.
template <typename T>
cudaError_t launch_path_bwd(const void *q, const void *k, const void *v, const void *w,
                            const float *beta, const void *o, const float *lse, const void *dout,
                            int B, int H, int L, float scale, float *dq, float *dk, float *dv,
                            float *dw, float *dbeta, void *ws, cudaStream_t stream) {
    const BwdLayout y = bwd_layout(B, H, L);
    char *base = static_cast<char *>(ws);
    float *qt = reinterpret_cast<float *>(base + y.off_qt);
    float *kp = reinterpret_cast<float *>(base + y.off_kp);
    float *dg = reinterpret_cast<float *>(base + y.off_dg);
    float *dqt = reinterpret_cast<float *>(base + y.off_dqt);
    float *dkt = reinterpret_cast<float *>(base + y.off_dkt);
    float *dPb = reinterpret_cast<float *>(base + y.off_dP);
    float *dTd = reinterpret_cast<float *>(base + y.off_dTd);
    float *stash = reinterpret_cast<float *>(base + y.off_stash);
    cudaError_t e;
    if ((e = cudaMemsetAsync(base, 0, 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dkt, 0, (size_t)y.BH * y.Lp * kD * 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dPb, 0, (size_t)y.BH * y.nblk * kBlkTile * 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dv, 0, (size_t)y.BH * L * kD * 4, stream)) != cudaSuccess) return e;
    if ((e = launch_ut_prepare_f32out<T>(q, k, w, beta, y.BH, L, y.Lp, y.nblk, scale, qt, kp, dg,
                                         reinterpret_cast<uint32_t *>(base), stream)) != cudaSuccess)
        return e;
    const size_t s1 = bwd_query_smem(), s2 = bwd_block_smem();
    if ((e = cudaFuncSetAttribute(bwd_query_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)s1)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_block_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)s2)) != cudaSuccess)
        return e;
    const dim3 grid(y.nblk, y.BH);
    bwd_query_kernel<T><<<grid, kThreads, s1, stream>>>(
        static_cast<const T *>(v), static_cast<const T *>(o), static_cast<const T *>(dout), lse,
        qt, kp, dg, dqt, dkt, dPb, dTd, stash, dv, L, y.Lp, y.nblk, scale, scale * kLog2e);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_block_kernel<T><<<grid, kThreads, s2, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(w), beta,
        dqt, dkt, dPb, dTd, dq, dk, dw, dbeta, L, y.Lp, y.nblk);
    return cudaGetLastError();
}

template cudaError_t launch_path_bwd<float>(const void *, const void *, const void *, const void *,
                                            const float *, const void *, const float *,
                                            const void *, int, int, int, float, float *, float *,
                                            float *, float *, float *, void *, cudaStream_t);
template cudaError_t launch_path_bwd<__nv_bfloat16>(const void *, const void *, const void *,
                                                    const void *, const float *, const void *,
                                                    const float *, const void *, int, int, int,
                                                    float, float *, float *, float *, float *,
                                                    float *, void *, cudaStream_t);

}  // namespace path
