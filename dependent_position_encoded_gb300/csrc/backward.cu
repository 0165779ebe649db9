// Backward pass of PaTH attention and PaTH-FoX, fp32 on the CUDA cores.
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
// logits from the inputs. PaTH-FoX adds the bias c_i - c_j (c = cumsum of log f) to every
// logit; it leaves dT unchanged and gives d log f_s = sum over j < s <= i of dS_ij, formed
// from the row and column sums of dS. Every key block is visited (no early exit).
#include "bwd_f32_tiles.cuh"

namespace path {

template <typename T>
cudaError_t launch_ut_prepare_f32out(const void *q, const void *k, const void *w,
                                     const float *beta, const float *log_f, int BH, int L, int Lp,
                                     int nblk, float scale, float *qt, float *kp, float *dg,
                                     uint32_t *status, cudaStream_t stream);

namespace {

using namespace bwd_f32;

// ---------------------------------------------------------------- B1: query pass
// One CTA per (query block a, head), two per SM; a runs from the last block down so that
// the longest walks start first. Five 64 x 64 fp32 buffers, all row-major:
//   pass 1: R0 X [i][c], R1 dout [i][c], R2 K~_b [j][c] then p [i][j], R3 P_b [n][c] then
//           dT [i][j], R4 V_b [j][c]
//   pass 2: R0 X, R1 dT [i][j], R2 K~_b [j][c], R3 P_b [n][c], R4 G [i][n]
// Groups 0 and 1 form the logits and dout V_b^T of their rows (so p and dS stay in their
// registers) and, in pass 2, the new G; groups 2 and 3 carry X to the next key block and,
// in pass 2, add the dP_b terms; in between each group takes half of dk~ or dv.
// PaTH-FoX (FOX): the gate bias c_i - c_j joins every logit, as (C_a - C_b) + loc_i - loc_j
// with C the fp64 sums of log f before each block and loc the block-local inclusive sums;
// the row sums of dS go to rsum and its column sums to csum (atomically), from which the
// gate gradient is formed afterwards.
template <typename T, bool FOX>
__global__ void __launch_bounds__(kThreads, 2)
bwd_query_kernel(const T *__restrict__ v, const T *__restrict__ o, const T *__restrict__ dout,
                 const float *__restrict__ lse, const float *__restrict__ qt,
                 const float *__restrict__ kp, const float *__restrict__ dg,
                 float *__restrict__ dqt, float *__restrict__ dkt, float *__restrict__ dP,
                 float *__restrict__ dTd, float *__restrict__ stash, float *__restrict__ dv,
                 int L, int Lp, int nblk, float scale, float scale_log2,
                 const float *__restrict__ loc, const double *__restrict__ cb,
                 float *__restrict__ rsum, float *__restrict__ csum) {
    extern __shared__ __align__(16) float sm[];
    float *R0 = sm, *R1 = R0 + BUF, *R2 = R1 + BUF, *R3 = R2 + BUF, *R4 = R3 + BUF;
    float *lse2 = R4 + BUF;     // per row: lse * log2(e)
    float *Drow = lse2 + kC;    // per row: dout . out
    float *loci = Drow + kC;    // FoX: block-local gate sums of the query rows
    float *locj = loci + kC;    // FoX: those of the current key block

    const int tid = threadIdx.x;
    const int a = nblk - 1 - (int)blockIdx.x;
    const int bh = blockIdx.y;
    const int grp = tid >> 6, lt = tid & 63, ty = lt >> 3, tx = lt & 7;
    const int rb = (grp & 1) * 32;
    const int r0 = rb + ty, m0 = rb + 4 * ty, c0 = 4 * tx, n0 = tx;
    const bool lead = grp < 2;  // groups 0 and 1: logits, p, dS, G
    const int t0 = a * kC;
    const size_t hL = (size_t)bh * L;
    const T *vh = v + hL * kD;

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
            if (FOX) loci[row] = (t0 + row < L) ? loc[(size_t)bh * Lp + t0 + row] : 0.f;
        }
    }
    // FoX: row sums of dS stay in registers (the eight lanes of a row end with its total);
    // column sums of a tile go out with one atomic per column and warp
    float rs_acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto fox_sums = [&](float (&rp)[4], float (&cp)[8], int kb) {
        fox_tile_sums(rp, cp, rs_acc, csum + (size_t)bh * Lp + (size_t)kb * kC, n0);
    };

    load_rows<T>(R1, nullptr, dout + hL * kD, t0, L);
    load_rows<T>(R4, nullptr, vh, t0, L);
    __syncthreads();

    // ---- diagonal block: logits from the table; dT to the block pass, p^T dout to dv
    if (lead) {
        float dt[4][8], pr[4][8], rp[4] = {0.f, 0.f, 0.f, 0.f};
        float cp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        zero48(dt);
        mmrb48(R1, R4, r0, n0, dt);  // dout_i . v_j
        const float *tab = dg + ((size_t)bh * nblk + a) * kBlkTile;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + 8 * i;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float p = (t0 + r < L) ? exp2f(tab[r * kC + n0 + 8 * j] - lse2[r]) : 0.f;
                const float ds = p * (dt[i][j] - Drow[r]);
                if (FOX) {
                    rp[i] += ds;
                    cp[j] += ds;
                }
                pr[i][j] = p;
                dt[i][j] = scale * ds;
            }
        }
        put_rb(dTd + ((size_t)bh * nblk + a) * kBlkTile, kC, dt, r0, n0);
        if (FOX) fox_sums(rp, cp, a);
        put_rb(R2, LD, pr, r0, n0);  // p [i][j]
    }
    __syncthreads();
    if (!lead) {
        float acc[4][8];
        zero48(acc);
        mmkk48(R2, R1, m0, c0, acc);  // sum_i p_ij dout_i[c]
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (t0 + m0 + i < L)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    atomicAdd(dv + (hL + t0 + m0 + i) * kD + col48(c0, j), acc[i][j]);
    }

    // ---- pass 1: right to left over key blocks, X from Q~_a
    auto kp_block = [&](int b) { return kp + ((size_t)bh * nblk + b) * 2 * kBlkTile; };
    __syncthreads();
    load_tile(R0, qt + ((size_t)bh * Lp + t0) * kD, false);
    const size_t pair0 = (size_t)bh * ((size_t)nblk * (nblk - 1) / 2) + (size_t)a * (a - 1) / 2;
    for (int b = a - 1; b >= 0; --b) {
        __syncthreads();
        load_tile(R2, kp_block(b), false);
        load_tile(R3, kp_block(b) + kBlkTile, false);
        load_rows<T>(R4, nullptr, vh, b * kC, L);
        if (FOX && tid < kC) locj[tid] = loc[(size_t)bh * Lp + (size_t)b * kC + tid];
        __syncthreads();
        // lead groups: acc1 = logits, acc2 = dout V_b^T; the others: acc1 = X P_b^T
        float acc1[4][8], acc2[4][8];
        zero48(acc1);
        zero48(acc2);
        if (lead) {
            mmrb48(R0, R2, r0, n0, acc1);
            mmrb48(R1, R4, r0, n0, acc2);
        } else if (b > 0) {
            mmrb48(R0, R3, r0, n0, acc1);
        }
        float *st = stash + (pair0 + b) * 2 * kBlkTile;  // [X_{a,b} | dT_ab], row-major
#pragma unroll
        for (int it = 0; it < kBlkTile / 4 / kThreads; ++it) {
            const int e = 4 * (tid + it * kThreads), r = e / kD, c = e % kD;
            *reinterpret_cast<float4 *>(st + e) = *reinterpret_cast<const float4 *>(R0 + r * LD + c);
        }
        if (lead) {
            float rp[4] = {0.f, 0.f, 0.f, 0.f}, cp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const float dcb = FOX ? (float)(cb[(size_t)bh * nblk + a] - cb[(size_t)bh * nblk + b]) : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + 8 * i;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float x2 = acc1[i][j] * scale_log2;
                    if (FOX) x2 += kLog2e * ((dcb + loci[r]) - locj[n0 + 8 * j]);
                    const float p = (t0 + r < L) ? exp2f(x2 - lse2[r]) : 0.f;
                    const float ds = p * (acc2[i][j] - Drow[r]);
                    if (FOX) {
                        rp[i] += ds;
                        cp[j] += ds;
                    }
                    acc1[i][j] = p;           // acc1 now holds p
                    acc2[i][j] = scale * ds;  // acc2 now holds dT
                }
            }
            put_rb(st + kBlkTile, kC, acc2, r0, n0);
            if (FOX) fox_sums(rp, cp, b);
        }
        __syncthreads();  // K~_b and P_b are read: their buffers take p and dT
        if (lead) {
            put_rb(R2, LD, acc1, r0, n0);
            put_rb(R3, LD, acc2, r0, n0);
        }
        __syncthreads();
        {
            float acc[4][8];
            zero48(acc);
            if (lead) {  // dK~_b[j][c] += sum_i dT_ij X_ic
                mmkk48(R3, R0, m0, c0, acc);
                red_kk(dkt + ((size_t)bh * Lp + (size_t)b * kC) * kD, acc, m0, c0);
            } else {     // dv_j += sum_i p_ij dout_i (key block b < a is full)
                mmkk48(R2, R1, m0, c0, acc);
                red_kk(dv + (hL + (size_t)b * kC) * kD, acc, m0, c0);
            }
        }
        __syncthreads();
        if (!lead && b > 0) put_rb(R0, LD, acc1, r0, n0);
    }

    // ---- pass 2: left to right, G = gradient of X_{a,b}
    float g[4][8];
    zero48(g);
    __syncthreads();
    for (int e = tid; e < BUF; e += kThreads) R4[e] = 0.f;
    for (int b = 0; b < a; ++b) {
        const float *st = stash + (pair0 + b) * 2 * kBlkTile;
        __syncthreads();
        load_tile(R0, st, false);
        load_tile(R1, st + kBlkTile, false);
        load_tile(R2, kp_block(b), false);
        load_tile(R3, kp_block(b) + kBlkTile, false);
        __syncthreads();
        if (lead) {
            zero48(g);
            if (b > 0) mm48(R4, R3, r0, c0, g);  // G_{b-1} P_b
            mm48(R1, R2, r0, c0, g);             // + dT_ab K~_b
        } else if (b > 0) {                      // dP_b[n][c] += sum_i G_{b-1}[i][n] X_{a,b}[i][c]
            float acc[4][8];
            zero48(acc);
            mmkk48(R4, R0, m0, c0, acc);
            red_kk(dP + ((size_t)bh * nblk + b) * kBlkTile, acc, m0, c0);
        }
        __syncthreads();
        if (lead) put48(R4, g, r0, c0);
    }
    if (lead) {
        // dQ~_a = G_{a-1} (zero for the first block)
        st48(dqt + ((size_t)bh * Lp + t0) * kD, g, r0, c0);
        if (FOX && tx == 0)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + r0 + 8 * i < L) rsum[(size_t)bh * Lp + t0 + r0 + 8 * i] = rs_acc[i];
    }
}

// ---------------------------------------------------------------- B2: block pass
// One CTA per (block, head), 8 warps (two CTAs per SM at d = 64, one at d = 128). Warp w runs
// groups of eight sweeps, each group in lockstep: query rows i = 8w .. 8w + 7 (q~_i and the
// diagonal logits), columns c = (d / 8) w .. (d / 8) w + d / 8 - 1 of P_b (one group at
// d = 64, two at d = 128), and key rows j = 8w .. 8w + 7 (k~_j); short query sweeps meet
// long key sweeps, so the warps' loads match. Lane l holds dimensions NE l .. NE l + NE - 1
// (NE = d / 32) of every vector. A sweep first applies its transitions, recording only
// w_s . x of each step, then walks back with the gradient, recovering each step's input by
// undoing the step: the step is x' = x - c w_s with c = beta_s (w_s . x), so x = x' + c w_s,
// exact up to rounding (no H_s is inverted; it is singular at beta_s = 1). Per step the
// eight sweeps share one read of w_s and beta_s, run eight independent warp reductions,
// and add their summed dw, dk and dbeta terms to shared memory with one atomic per lane
// and dimension. dq is written by its query sweep.
constexpr int kWarps = kThreads / 32;
constexpr int kNS = 8;  // sweeps per warp group

// NE consecutive fp32 values from / to memory (8- or 16-byte aligned)
template <int NE>
__device__ __forceinline__ void ldv(float (&r)[NE], const float *p) {
    static_assert(NE == 2 || NE == 4, "two or four dimensions per lane");
    if constexpr (NE == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        r[0] = t.x;
        r[1] = t.y;
    } else {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        r[0] = t.x;
        r[1] = t.y;
        r[2] = t.z;
        r[3] = t.w;
    }
}
template <int NE>
__device__ __forceinline__ void stv(float *p, const float (&r)[NE]) {
    if constexpr (NE == 2)
        *reinterpret_cast<float2 *>(p) = make_float2(r[0], r[1]);
    else
        *reinterpret_cast<float4 *>(p) = make_float4(r[0], r[1], r[2], r[3]);
}
template <typename T, int NE>
__device__ __forceinline__ void loadv(float (&r)[NE], const T *p) {
#pragma unroll
    for (int e = 0; e < NE; ++e) r[e] = Elt<T>::to_f(p[e]);
}
// NE consecutive values of type T in shared memory as fp32 (one 8- or 16-byte load for
// fp32, 4 or 8 bytes for bf16)
template <int NE>
__device__ __forceinline__ void ldsv(float (&r)[NE], const float *p) { ldv<NE>(r, p); }
template <int NE>
__device__ __forceinline__ void ldsv(float (&r)[NE], const __nv_bfloat16 *p) {
    if constexpr (NE == 2) {
        const float2 t = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(p));
        r[0] = t.x;
        r[1] = t.y;
    } else {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const float2 t0 = unpack_bf16x2(u.x), t1 = unpack_bf16x2(u.y);
        r[0] = t0.x;
        r[1] = t0.y;
        r[2] = t1.x;
        r[3] = t1.y;
    }
}
// NE consecutive values of type T copied from global to shared memory, or zeros
template <typename T, int NE>
__device__ __forceinline__ void copyv(T *dst, const T *src, bool in) {
    if constexpr (sizeof(T) * NE == 8) {
        *reinterpret_cast<uint2 *>(dst) = in ? *reinterpret_cast<const uint2 *>(src) : make_uint2(0u, 0u);
    } else if constexpr (sizeof(T) * NE == 16) {
        *reinterpret_cast<uint4 *>(dst) = in ? *reinterpret_cast<const uint4 *>(src) : make_uint4(0u, 0u, 0u, 0u);
    } else {
        static_assert(sizeof(T) * NE == 4, "4, 8 or 16 bytes per lane");
        *reinterpret_cast<uint32_t *>(dst) = in ? *reinterpret_cast<const uint32_t *>(src) : 0u;
    }
}
template <int NE>
__device__ __forceinline__ void zerov(float (&r)[NE]) {
#pragma unroll
    for (int e = 0; e < NE; ++e) r[e] = 0.f;
}

// out[k] = w . x[k] over the warp, for the eight vectors of a group. A transposed butterfly:
// at xor 16, 8 and 4 each lane keeps half of its partial sums and adds its partner's copy
// of them, so lane l ends with the total of vector 4 bit4(l) + 2 bit3(l) + bit2(l) after
// two more levels; eight shuffles from lanes 4k broadcast the totals (17 shuffles, not 40)
template <int NE>
__device__ __forceinline__ void dot8(const float (&x)[kNS][NE], const float (&w)[NE],
                                     float (&out)[kNS]) {
    constexpr unsigned kAll = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    float p[kNS];
#pragma unroll
    for (int k = 0; k < kNS; ++k) {
        float t = w[NE - 1] * x[k][NE - 1];
#pragma unroll
        for (int e = NE - 2; e >= 0; --e) t = fmaf(w[e], x[k][e], t);
        p[k] = t;
    }
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = (h16 ? p[4 + i] : p[i]) + __shfl_xor_sync(kAll, h16 ? p[i] : p[4 + i], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        b[i] = (h8 ? a[2 + i] : a[i]) + __shfl_xor_sync(kAll, h8 ? a[i] : a[2 + i], 8);
    float c = (h4 ? b[1] : b[0]) + __shfl_xor_sync(kAll, h4 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(kAll, c, 2);
    c += __shfl_xor_sync(kAll, c, 1);
#pragma unroll
    for (int k = 0; k < kNS; ++k) out[k] = __shfl_sync(kAll, c, 4 * k);
}

// Workspace inputs (fp32): dqt, dkt (BH, Lp, D), dP (BH, nblk, D, D), dTd (BH, nblk, 64, 64).
// w and k stay in shared memory in their input type (exact). Built for fp32 inputs; bf16
// inputs take the matrix-form block passes of backward_block_mm.cu.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, (D == 64 || sizeof(T) == 2) ? 2 : 1)
bwd_block_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ w,
                 const float *__restrict__ beta, const float *__restrict__ dqt,
                 const float *__restrict__ dkt, const float *__restrict__ dP,
                 const float *__restrict__ dTd, float *__restrict__ dq, float *__restrict__ dk,
                 float *__restrict__ dw, float *__restrict__ dbeta, int L, int Lp, int nblk) {
    constexpr int NE = D / 32;
    constexpr int kTile = kC * D;  // floats in one 64 x D tile
    extern __shared__ __align__(16) float sm[];
    float *dWs = sm;              // gradient of w_s, [s][dimension]
    float *dKs = dWs + kTile;     // gradient of k_j
    float *wxs = dKs + kTile;     // per warp: [s][sweep] w_s . x
    float *bs = wxs + kWarps * kC * kNS;  // beta_s
    float *dBs = bs + kC;                 // gradient of beta_s
    T *Ws = reinterpret_cast<T *>(dBs + kC);  // w_s (input type)
    T *Ks = Ws + kTile;                       // k_j

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t hL = (size_t)bh * L;
    const int nvalid = min(kC, L - t0);
    const int el = NE * lane;  // this lane's first dimension

    // w, k (zero past L: a padded token's transition is the identity), beta
    for (int e = tid; e < kTile / NE; e += kThreads) {
        const int r = e / 32;
        const size_t g = (hL + t0 + r) * D + NE * (e % 32);
        float z[NE];
        zerov(z);
        copyv<T, NE>(Ws + NE * e, w + g, r < nvalid);
        copyv<T, NE>(Ks + NE * e, k + g, r < nvalid);
        stv<NE>(dWs + NE * e, z);
        stv<NE>(dKs + NE * e, z);
    }
    if (tid < kC) {
        bs[tid] = tid < nvalid ? beta[hL + t0 + tid] : 0.f;
        dBs[tid] = 0.f;
    }
    __syncthreads();

    float *wxw = wxs + warp * kC * kNS;
    const int base = kNS * warp;  // first query / key row of this warp's groups
    float x[kNS][NE], g[kNS][NE];
    float wx[kNS], wg[kNS];

    // x[k] <- H_s x[k] for the sweeps with act(k), recording w_s . x[k] at wxw[s][k]
    auto fwd = [&](int s, auto act) {
        float ws[NE];
        ldsv<NE>(ws, Ws + s * D + el);
        const float be = bs[s];
        dot8<NE>(x, ws, wx);
        if (lane == 0) {
            *reinterpret_cast<float4 *>(wxw + s * kNS) = make_float4(wx[0], wx[1], wx[2], wx[3]);
            *reinterpret_cast<float4 *>(wxw + s * kNS + 4) = make_float4(wx[4], wx[5], wx[6], wx[7]);
        }
#pragma unroll
        for (int kk = 0; kk < kNS; ++kk)
            if (act(kk))
#pragma unroll
                for (int e = 0; e < NE; ++e) x[kk][e] = fmaf(-be * wx[kk], ws[e], x[kk][e]);
    };
    // one step back through H_s for the sweeps with act(k): x[k] <- the step's input (undo),
    // dw_s, dbeta_s gather the terms, g[k] <- H_s g[k]. `undo` false for a step whose input
    // is already in x (the first step back, through H_0, with w_0 . x given in wx).
    auto back = [&](int s, bool undo, auto act) {
        float ws[NE];
        ldsv<NE>(ws, Ws + s * D + el);
        const float be = bs[s];
        if (undo) {
            const float4 a = *reinterpret_cast<const float4 *>(wxw + s * kNS);
            const float4 b = *reinterpret_cast<const float4 *>(wxw + s * kNS + 4);
            wx[0] = a.x; wx[1] = a.y; wx[2] = a.z; wx[3] = a.w;
            wx[4] = b.x; wx[5] = b.y; wx[6] = b.z; wx[7] = b.w;
#pragma unroll
            for (int kk = 0; kk < kNS; ++kk)
                if (act(kk))
#pragma unroll
                    for (int e = 0; e < NE; ++e) x[kk][e] = fmaf(be * wx[kk], ws[e], x[kk][e]);
        }
        dot8<NE>(g, ws, wg);
        float dws[NE];
        zerov(dws);
        float db = 0.f;
#pragma unroll
        for (int kk = 0; kk < kNS; ++kk)
            if (act(kk)) {
#pragma unroll
                for (int e = 0; e < NE; ++e) dws[e] += fmaf(wx[kk], g[kk][e], wg[kk] * x[kk][e]);
                db = fmaf(wg[kk], wx[kk], db);
#pragma unroll
                for (int e = 0; e < NE; ++e) g[kk][e] = fmaf(-be * wg[kk], ws[e], g[kk][e]);
            }
#pragma unroll
        for (int e = 0; e < NE; ++e) atomicAdd(dWs + s * D + el + e, -be * dws[e]);
        if (lane == 0) atomicAdd(&dBs[s], -db);
    };

    const auto all = [](int) { return true; };
    // ---- query rows i = base + k: x_j = H_{j+1} ... H_i q_i, q~_i = H_0 x_0, T_ij = k_j . x_j
    {
        float2 dtr[kNS];
#pragma unroll
        for (int kk = 0; kk < kNS; ++kk) {
            const int i = base + kk;
            if (i < nvalid) {
                loadv<T, NE>(x[kk], q + (hL + t0 + i) * D + el);
                ldv<NE>(g[kk], dqt + ((size_t)bh * Lp + t0 + i) * D + el);
                dtr[kk] = *reinterpret_cast<const float2 *>(
                    dTd + (((size_t)bh * nblk + blk) * kC + i) * kC + 2 * lane);
            } else {
                zerov(x[kk]);
                zerov(g[kk]);
                dtr[kk] = make_float2(0.f, 0.f);
            }
        }
        for (int s = base + kNS - 1; s >= 1; --s) fwd(s, [&](int kk) { return s <= base + kk; });
        __syncwarp();
        {
            float w0[NE];
            ldsv<NE>(w0, Ws + el);
            dot8<NE>(x, w0, wx);  // w_0 . x_0
        }
        back(0, false, all);
        for (int j = 0; j < base + kNS; ++j) {
            float kj[NE], dka[NE];  // x[k] = x_j here
            ldsv<NE>(kj, Ks + j * D + el);
            zerov(dka);
#pragma unroll
            for (int kk = 0; kk < kNS; ++kk)
                if (j <= base + kk) {
                    const float dtx = __shfl_sync(0xffffffffu, dtr[kk].x, j >> 1);
                    const float dty = __shfl_sync(0xffffffffu, dtr[kk].y, j >> 1);
                    const float dt = (j & 1) ? dty : dtx;
#pragma unroll
                    for (int e = 0; e < NE; ++e) {
                        g[kk][e] = fmaf(dt, kj[e], g[kk][e]);
                        dka[e] = fmaf(dt, x[kk][e], dka[e]);
                    }
                }
#pragma unroll
            for (int e = 0; e < NE; ++e) atomicAdd(dKs + j * D + el + e, dka[e]);
            if (j + 1 < base + kNS) back(j + 1, true, [&](int kk) { return j + 1 <= base + kk; });
        }
#pragma unroll
        for (int kk = 0; kk < kNS; ++kk)
            if (base + kk < nvalid) stv<NE>(dq + (hL + t0 + base + kk) * D + el, g[kk]);
    }
    __syncwarp();  // the next group rewrites wxw

    // ---- columns c of P_b = H_0 ... H_63 (P_0 and the last P_b reach no logit)
    if (blk > 0 && blk < nblk - 1) {
        const float *dpb = dP + ((size_t)bh * nblk + blk) * D * D;
        for (int cg = 0; cg < D / 64; ++cg) {
            const int cbase = (D / 8) * warp + kNS * cg;
#pragma unroll
            for (int kk = 0; kk < kNS; ++kk) {
                const int c = cbase + kk;
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    x[kk][e] = el + e == c ? 1.f : 0.f;
                    g[kk][e] = dpb[(el + e) * D + c];
                }
            }
            for (int s = kC - 1; s >= 1; --s) fwd(s, all);
            __syncwarp();
            {
                float w0[NE];
                ldsv<NE>(w0, Ws + el);
                dot8<NE>(x, w0, wx);
            }
            back(0, false, all);
            for (int s = 1; s < kC; ++s) back(s, true, all);
            __syncwarp();
        }
    }

    // ---- key rows j = base + k: k~_j = H_63 ... H_{j+1} k_j (the last block's k~ reach no
    // later query)
    if (blk < nblk - 1) {
#pragma unroll
        for (int kk = 0; kk < kNS; ++kk) {
            const int j = base + kk;
            if (j < nvalid) {
                ldsv<NE>(x[kk], Ks + j * D + el);
                ldv<NE>(g[kk], dkt + ((size_t)bh * Lp + t0 + j) * D + el);
            } else {
                zerov(x[kk]);
                zerov(g[kk]);
            }
        }
        for (int s = base + 1; s < kC; ++s) fwd(s, [&](int kk) { return s > base + kk; });
        __syncwarp();
        for (int s = kC - 1; s > base; --s) back(s, true, [&](int kk) { return s > base + kk; });
#pragma unroll
        for (int kk = 0; kk < kNS; ++kk)
            if (base + kk < nvalid)
#pragma unroll
                for (int e = 0; e < NE; ++e) atomicAdd(dKs + (base + kk) * D + el + e, g[kk][e]);
    }
    __syncthreads();
    for (int e = tid; e < nvalid * 32; e += kThreads) {
        const size_t gi = (hL + t0 + e / 32) * D + NE * (e % 32);
        float a[NE];
        ldv<NE>(a, dKs + NE * e);
        stv<NE>(dk + gi, a);
        ldv<NE>(a, dWs + NE * e);
        stv<NE>(dw + gi, a);
    }
    if (tid < nvalid) dbeta[hL + t0 + tid] = dBs[tid];
}

// ---------------------------------------------------------------- PaTH-FoX gate sums
// Per token the block-local inclusive sums of log f (fp32) and per block the fp64 sum of
// log f over every earlier token of the head, so that c_i - c_j = (C_a - C_b) + loc_i - loc_j
// keeps fp32 accuracy at any length. One CTA per head: a warp per 64-token block, then an
// fp64 exclusive scan of the block totals (a contiguous run of blocks per thread).
__global__ void __launch_bounds__(kThreads)
bwd_fox_sums_kernel(const float *__restrict__ log_f, int L, int Lp, int nblk,
                    float *__restrict__ loc, double *__restrict__ cb) {
    __shared__ double part[kThreads];
    const int bh = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t hL = (size_t)bh * L;
    double *cbh = cb + (size_t)bh * nblk;
    for (int b = warp; b < nblk; b += kThreads / 32) {
        const int ta = b * kC + 2 * lane, tb = ta + 1;
        const float x0 = ta < L ? log_f[hL + ta] : 0.f;
        const float x1 = (tb < L ? log_f[hL + tb] : 0.f) + x0;
        float run = x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, run, o);
            if (lane >= o) run += n;
        }
        loc[(size_t)bh * Lp + ta] = run - x1 + x0;
        loc[(size_t)bh * Lp + tb] = run;
        if (lane == 31) cbh[b] = (double)run;  // the block's total, scanned below
    }
    __syncthreads();
    const int per = (nblk + kThreads - 1) / kThreads;
    const int b0 = min(nblk, tid * per), b1 = min(nblk, b0 + per);
    double sum = 0.0;
    for (int b = b0; b < b1; ++b) sum += cbh[b];
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        double run = 0.0;
        for (int i = 0; i < kThreads; ++i) {
            const double t = part[i];
            part[i] = run;
            run += t;
        }
    }
    __syncthreads();
    double run = part[tid];
    for (int b = b0; b < b1; ++b) {
        const double t = cbh[b];
        cbh[b] = run;
        run += t;
    }
}

// d log f_s = sum over pairs j < s <= i of dS_ij = sum_{t >= s} (rowsum_t - colsum_t) of dS,
// since the bias c_i - c_j moves with c_i on row i and against c_j on column j, and
// c_t = sum_{u <= t} log f_u. One warp per head walks the tokens from the end in fp64.
__global__ void __launch_bounds__(32)
bwd_fox_dlogf_kernel(const float *__restrict__ rsum, const float *__restrict__ csum, int L,
                     int Lp, float *__restrict__ dlogf) {
    const int bh = blockIdx.x, lane = threadIdx.x;
    double acc = 0.0;
    for (int top = L - 1; top >= 0; top -= 32) {
        const int t = top - lane;
        double v = t >= 0 ? (double)rsum[(size_t)bh * Lp + t] - (double)csum[(size_t)bh * Lp + t] : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (t >= 0) dlogf[(size_t)bh * L + t] = (float)(acc + v);
        acc += __shfl_sync(0xffffffffu, v, 31);
    }
}

}  // namespace

// Workspace of the backward: 256-byte status header, then fp32 q~ (BH, Lp, 64),
// [k~; P_b] (BH, nblk, 128, 64), diagonal logits (BH, nblk, 64, 64), dq~ and dk~ (BH, Lp,
// 64), dP_b and the diagonal dT (BH, nblk, 64, 64), and the query pass's stash: X_{a,b} and
// dT_ab for every pair b < a (BH, nblk (nblk - 1) / 2, 2, 64, 64); PaTH-FoX adds the
// block-local gate sums, the row and column sums of dS (BH, Lp) fp32 each, and the per-block
// gate prefixes (BH, nblk) fp64.
BwdLayout bwd_layout(int B, int H, int L, bool fox) {
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
    y.off_loc = y.off_rs = y.off_cs = y.off_cb = off;
    if (fox) {
        const size_t tok = bh * y.Lp * 4;
        y.off_rs = align256(off + tok);
        y.off_cs = align256(y.off_rs + tok);
        y.off_cb = align256(y.off_cs + tok);
        off = align256(y.off_cb + bh * y.nblk * 8);
    }
    y.total = off;
    return y;
}

size_t bwd_query_smem() { return (size_t)(5 * BUF + 4 * kC) * sizeof(float); }

// The token-level block pass (fp32 inputs) at head size D (64 or 128): dq, dk, dw (BH, L, D) and dbeta
// (BH, L) fp32 from dqt, dkt (BH, Lp, D), dP (BH, nblk, D, D) and the diagonal dT
// (BH, nblk, 64, 64).
template <typename T>
cudaError_t launch_bwd_block_sweep(const void *q, const void *k, const void *w, const float *beta,
                                   const float *dqt, const float *dkt, const float *dP,
                                   const float *dTd, float *dq, float *dk, float *dw,
                                   float *dbeta, int BH, int L, int Lp, int nblk, int D,
                                   cudaStream_t stream) {
    auto kern = D == 128 ? bwd_block_kernel<T, 128> : bwd_block_kernel<T, 64>;
    const size_t sm = (size_t)(2 * kC * D + kWarps * kC * kNS + 2 * kC) * sizeof(float) +
                      (size_t)2 * kC * D * sizeof(T);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    kern<<<dim3(nblk, BH), kThreads, sm, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(w), beta, dqt,
        dkt, dP, dTd, dq, dk, dw, dbeta, L, Lp, nblk);
    return cudaGetLastError();
}

// dq, dk, dv, dw (B*H, L, 64) and dbeta (B*H, L) fp32; with log_f (PaTH-FoX) also dlogf
// (B*H, L) fp32. dv gathers by atomics from zero.
template <typename T>
cudaError_t launch_path_bwd(const void *q, const void *k, const void *v, const void *w,
                            const float *beta, const float *log_f, const void *o,
                            const float *lse, const void *dout, int B, int H, int L, float scale,
                            float *dq, float *dk, float *dv, float *dw, float *dbeta, float *dlogf,
                            void *ws, cudaStream_t stream) {
    const bool fox = log_f != nullptr;
    const BwdLayout y = bwd_layout(B, H, L, fox);
    char *base = static_cast<char *>(ws);
    auto at = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    float *qt = at(y.off_qt), *kp = at(y.off_kp), *dg = at(y.off_dg), *dqt = at(y.off_dqt);
    float *dkt = at(y.off_dkt), *dPb = at(y.off_dP), *dTd = at(y.off_dTd), *stash = at(y.off_stash);
    float *loc = at(y.off_loc), *rs = at(y.off_rs), *cs = at(y.off_cs);
    double *cb = reinterpret_cast<double *>(base + y.off_cb);
    const size_t tok = (size_t)y.BH * y.Lp * 4;
    cudaError_t e;
    if ((e = cudaMemsetAsync(base, 0, 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dkt, 0, tok * kD, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dPb, 0, (size_t)y.BH * y.nblk * kBlkTile * 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dv, 0, (size_t)y.BH * L * kD * 4, stream)) != cudaSuccess) return e;
    if (fox) {
        if ((e = cudaMemsetAsync(rs, 0, tok, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(cs, 0, tok, stream)) != cudaSuccess)
            return e;
        bwd_fox_sums_kernel<<<y.BH, kThreads, 0, stream>>>(log_f, L, y.Lp, y.nblk, loc, cb);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = launch_ut_prepare_f32out<T>(q, k, w, beta, log_f, y.BH, L, y.Lp, y.nblk, scale, qt,
                                         kp, dg, reinterpret_cast<uint32_t *>(base), stream)) != cudaSuccess)
        return e;
    auto kq = fox ? bwd_query_kernel<T, true> : bwd_query_kernel<T, false>;
    const size_t s1 = bwd_query_smem();
    if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1)) != cudaSuccess)
        return e;
    const dim3 grid(y.nblk, y.BH);
    kq<<<grid, kThreads, s1, stream>>>(
        static_cast<const T *>(v), static_cast<const T *>(o), static_cast<const T *>(dout), lse,
        qt, kp, dg, dqt, dkt, dPb, dTd, stash, dv, L, y.Lp, y.nblk, scale, scale * kLog2e, loc, cb,
        rs, cs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bwd_block_sweep<T>(q, k, w, beta, dqt, dkt, dPb, dTd, dq, dk, dw, dbeta, y.BH,
                                       L, y.Lp, y.nblk, kD, stream)) != cudaSuccess)
        return e;
    if (fox) {
        bwd_fox_dlogf_kernel<<<y.BH, 32, 0, stream>>>(rs, cs, L, y.Lp, dlogf);
        e = cudaGetLastError();
    }
    return e;
}

// The PaTH-FoX gate sums and d log f on their own, for the tensor-core query pass
// (backward_tc.cu), which keeps its own workspace layout (its block pass for bf16 inputs is
// backward_block_mm.cu).
cudaError_t launch_bwd_fox_sums(const float *log_f, int BH, int L, int Lp, int nblk, float *loc,
                                double *cb, cudaStream_t stream) {
    bwd_fox_sums_kernel<<<BH, kThreads, 0, stream>>>(log_f, L, Lp, nblk, loc, cb);
    return cudaGetLastError();
}

cudaError_t launch_bwd_fox_dlogf(const float *rsum, const float *csum, int BH, int L, int Lp,
                                 float *dlogf, cudaStream_t stream) {
    bwd_fox_dlogf_kernel<<<BH, 32, 0, stream>>>(rsum, csum, L, Lp, dlogf);
    return cudaGetLastError();
}

#define PATH_BWD_INST(T)                                                                        \
    template cudaError_t launch_path_bwd<T>(const void *, const void *, const void *,           \
                                            const void *, const float *, const float *,         \
                                            const void *, const float *, const void *, int, int, \
                                            int, float, float *, float *, float *, float *,     \
                                            float *, float *, void *, cudaStream_t);
PATH_BWD_INST(float)
#undef PATH_BWD_INST
template cudaError_t launch_bwd_block_sweep<float>(const void *, const void *, const void *,
                                                   const float *, const float *, const float *,
                                                   const float *, const float *, float *, float *,
                                                   float *, float *, int, int, int, int, int,
                                                   cudaStream_t);

}  // namespace path
