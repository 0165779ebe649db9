// Backward pass of PaTH attention and PaTH-FoX at head size d = 128 for fp32 inputs, fp32 on
// the CUDA cores (the fp32 bar needs fp32 products; bf16 inputs take the tensor-core query
// pass of backward_tc128.cu).
//
// The pages give no backward (review "거리에서 경로로, PaTH Attention" §9 and technical
// summary "技術要約: PaTH Attention" §3 say the block-wise algorithm makes training
// efficient; §6 of the summary and §9 of the review flag larger heads as costlier). The
// chain rule is that of the d = 64 backward (backward.cu): per head, with q~_i, k~_j and the
// dense block transition P_b of the preparation, the logit of query i in block a and key j
// in block b < a is scale * T_ij with T_ab = X_{a,b} K~_b^T, X_{a,a-1} = Q~_a and
// X_{a,b-1} = X_{a,b} P_b^T; with dT = scale * dS,
//     dv_j += p_ij dout_i,   dK~_b += dT_ab^T X_{a,b},
//     G_b = G_{b-1} P_b + dT_ab K~_b  (G_{-1} = 0),   dP_b += G_{b-1}^T X_{a,b},
//     dQ~_a = G_{a-1}.
// At d = 128 the carried rows X, K~_b, V_b, dout and G are 64 x 128 and P_b is 128 x 128.
// The query pass keeps every 64 x 128 operand as two 64-column halves and P_b as four
// 64 x 64 quadrants, so each product is a sum of the 64 x 64 tile products of
// bwd_f32_tiles.cuh: X K~^T = X0 K0^T + X1 K1^T, the carried rows' column half h of X P^T is
// X0 P_h0^T + X1 P_h1^T, half h of G P is G0 P_0h + G1 P_1h. The preparation is the fp32
// d = 128 forward's (fwd_d128.cu); the block pass is the token-level sweep of backward.cu at
// d = 128 (four dimensions per lane).
#include "bwd_f32_tiles.cuh"

namespace path {

template <typename T>
cudaError_t launch_prep_d128(const void *q, const void *k, const void *w, const float *beta,
                             const float *log_f, int B, int H, int L, float scale, void *ws,
                             cudaStream_t stream);
template <typename T>
cudaError_t launch_bwd_block_sweep(const void *q, const void *k, const void *w, const float *beta,
                                   const float *dqt, const float *dkt, const float *dP,
                                   const float *dTd, float *dq, float *dk, float *dw,
                                   float *dbeta, int BH, int L, int Lp, int nblk, int D,
                                   cudaStream_t stream);
cudaError_t launch_bwd_fox_sums(const float *log_f, int BH, int L, int Lp, int nblk, float *loc,
                                double *cb, cudaStream_t stream);
cudaError_t launch_bwd_fox_dlogf(const float *rsum, const float *csum, int BH, int L, int Lp,
                                 float *dlogf, cudaStream_t stream);

namespace {

using namespace bwd_f32;

constexpr int kD2 = 128;                                  // head size of this file
constexpr size_t kKpRows = (size_t)(kC + kD2) * kD2;      // [k~ (64 rows); P_b (128 rows)]
constexpr size_t kStash = (size_t)kC * kD2 + kC * kC;     // [X_{a,b} (64 x 128) | dT_ab]
constexpr int kBufs = 12;                                 // 64 x 64 fp32 shared buffers

// One CTA of 256 threads per (query block a, head), one per SM; a runs from the last block
// down. Twelve 64 x 64 fp32 buffers (row-major, stride LD):
//   pass 1: X0 X1 (X [i][c], column halves), D0 D1 (dout), K0 K1 (K~_b, then p [i][j] and
//           dT [i][j]), P00 P01 P10 P11 (P_b quadrant [row half][column half]), V0 V1 (V_b)
//   pass 2: X0 X1, dT in D0, K0 K1, the P_b quadrants, G0 G1 (G [i][n]) in V0 V1
// Groups 0 and 1 (lead) form the logits and dout V_b^T of their 32 rows and, in pass 2, the
// new G; groups 2 and 3 carry X to the next key block and, in pass 2, add the dP_b terms; in
// between the lead groups take dk~ and the others dv. PaTH-FoX as at d = 64: the bias
// (C_a - C_b) + loc_i - loc_j joins every logit of an earlier block (the diagonal table
// holds it already), and the row and column sums of dS feed the gate gradient.
template <typename T, bool FOX>
__global__ void __launch_bounds__(kThreads, 1)
bwd_query128_kernel(const T *__restrict__ v, const T *__restrict__ o, const T *__restrict__ dout,
                    const float *__restrict__ lse, const float *__restrict__ qt,
                    const float *__restrict__ kp, const float *__restrict__ dg,
                    float *__restrict__ dqt, float *__restrict__ dkt, float *__restrict__ dP,
                    float *__restrict__ dTd, float *__restrict__ stash, float *__restrict__ dv,
                    int L, int Lp, int nblk, float scale, float scale_log2,
                    const float *__restrict__ loc, const double *__restrict__ cb,
                    float *__restrict__ rsum, float *__restrict__ csum) {
    extern __shared__ __align__(16) float sm[];
    float *X0 = sm, *X1 = X0 + BUF, *D0 = X1 + BUF, *D1 = D0 + BUF, *K0 = D1 + BUF,
          *K1 = K0 + BUF, *P00 = K1 + BUF, *P01 = P00 + BUF, *P10 = P01 + BUF,
          *P11 = P10 + BUF, *V0 = P11 + BUF, *V1 = V0 + BUF;
    float *lse2 = V1 + BUF;     // per row: lse * log2(e)
    float *Drow = lse2 + kC;    // per row: dout . out
    float *loci = Drow + kC;    // FoX: block-local gate sums of the query rows
    float *locj = loci + kC;    // FoX: those of the current key block

    const int tid = threadIdx.x;
    const int a = nblk - 1 - (int)blockIdx.x;
    const int bh = blockIdx.y;
    const int grp = tid >> 6, lt = tid & 63, ty = lt >> 3, tx = lt & 7;
    const int rb = (grp & 1) * 32;
    const int r0 = rb + ty, m0 = rb + 4 * ty, c0 = 4 * tx, n0 = tx;
    const bool lead = grp < 2;
    const int t0 = a * kC;
    const size_t hL = (size_t)bh * L;
    const T *vh = v + hL * kD2;
    const T *douth = dout + hL * kD2;
    auto load_kp = [&](int b) {
        const float *kb = kp + ((size_t)bh * nblk + b) * kKpRows;
        const float *pb = kb + kC * kD2;
        load_tile(K0, kb, false, kD2);
        load_tile(K1, kb + 64, false, kD2);
        load_tile(P00, pb, false, kD2);
        load_tile(P01, pb + 64, false, kD2);
        load_tile(P10, pb + 64 * kD2, false, kD2);
        load_tile(P11, pb + 64 * kD2 + 64, false, kD2);
    };

    // ---- per row: lse in log2 units and D_i = dout_i . out_i (4 threads per row)
    {
        const int row = tid >> 2, part = tid & 3;
        float dsum = 0.f;
        if (t0 + row < L) {
            const size_t g = (hL + t0 + row) * kD2 + part * 32;
#pragma unroll 8
            for (int c = 0; c < 32; ++c)
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
    float rs_acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto fox_sums = [&](float (&rp)[4], float (&cp)[8], int kb) {
        fox_tile_sums(rp, cp, rs_acc, csum + (size_t)bh * Lp + (size_t)kb * kC, n0);
    };

    load_rows<T>(D0, nullptr, douth, t0, L, kD2);
    load_rows<T>(D1, nullptr, douth + 64, t0, L, kD2);
    load_rows<T>(V0, nullptr, vh, t0, L, kD2);
    load_rows<T>(V1, nullptr, vh + 64, t0, L, kD2);
    __syncthreads();

    // ---- diagonal block: logits from the table; dT to the block pass, p^T dout to dv
    if (lead) {
        float dt[4][8], pr[4][8], rp[4] = {0.f, 0.f, 0.f, 0.f};
        float cp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        zero48(dt);
        mmrb48(D0, V0, r0, n0, dt);  // dout_i . v_j
        mmrb48(D1, V1, r0, n0, dt);
        const float *tab = dg + ((size_t)bh * nblk + a) * kC * kC;
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
        put_rb(dTd + ((size_t)bh * nblk + a) * kC * kC, kC, dt, r0, n0);
        if (FOX) fox_sums(rp, cp, a);
        put_rb(K0, LD, pr, r0, n0);  // p [i][j]
    }
    __syncthreads();
    if (!lead) {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            float acc[4][8];
            zero48(acc);
            mmkk48(K0, h ? D1 : D0, m0, c0, acc);  // sum_i p_ij dout_i[c]
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + m0 + i < L)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        atomicAdd(dv + (hL + t0 + m0 + i) * kD2 + 64 * h + col48(c0, j), acc[i][j]);
        }
    }

    // ---- pass 1: right to left over key blocks, X from Q~_a
    __syncthreads();
    load_tile(X0, qt + ((size_t)bh * Lp + t0) * kD2, false, kD2);
    load_tile(X1, qt + ((size_t)bh * Lp + t0) * kD2 + 64, false, kD2);
    const size_t pair0 = (size_t)bh * ((size_t)nblk * (nblk - 1) / 2) + (size_t)a * (a - 1) / 2;
    for (int b = a - 1; b >= 0; --b) {
        __syncthreads();
        load_kp(b);
        load_rows<T>(V0, nullptr, vh, b * kC, L, kD2);
        load_rows<T>(V1, nullptr, vh + 64, b * kC, L, kD2);
        if (FOX && tid < kC) locj[tid] = loc[(size_t)bh * Lp + (size_t)b * kC + tid];
        __syncthreads();
        // lead groups: acc1 = logits, acc2 = dout V_b^T; the others: acc1 / acc2 = column
        // halves 0 / 1 of X P_b^T
        float acc1[4][8], acc2[4][8];
        zero48(acc1);
        zero48(acc2);
        if (lead) {
            mmrb48(X0, K0, r0, n0, acc1);
            mmrb48(X1, K1, r0, n0, acc1);
            mmrb48(D0, V0, r0, n0, acc2);
            mmrb48(D1, V1, r0, n0, acc2);
        } else if (b > 0) {
            mmrb48(X0, P00, r0, n0, acc1);
            mmrb48(X1, P01, r0, n0, acc1);
            mmrb48(X0, P10, r0, n0, acc2);
            mmrb48(X1, P11, r0, n0, acc2);
        }
        float *st = stash + (pair0 + b) * kStash;  // [X_{a,b} | dT_ab], row-major
#pragma unroll 2
        for (int it = 0; it < kC * kD2 / 4 / kThreads; ++it) {
            const int e = 4 * (tid + it * kThreads), r = e / kD2, c = e % kD2;
            const float *src = c < 64 ? X0 + r * LD + c : X1 + r * LD + c - 64;
            *reinterpret_cast<float4 *>(st + e) = *reinterpret_cast<const float4 *>(src);
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
            put_rb(st + kC * kD2, kC, acc2, r0, n0);
            if (FOX) fox_sums(rp, cp, b);
        }
        __syncthreads();  // K~_b and P_b are read: K0, K1 take p and dT
        if (lead) {
            put_rb(K0, LD, acc1, r0, n0);
            put_rb(K1, LD, acc2, r0, n0);
        }
        __syncthreads();
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            float acc[4][8];
            zero48(acc);
            if (lead) {  // dK~_b[j][c] += sum_i dT_ij X_ic
                mmkk48(K1, h ? X1 : X0, m0, c0, acc);
                red_kk(dkt + ((size_t)bh * Lp + (size_t)b * kC) * kD2 + 64 * h, acc, m0, c0, kD2);
            } else {     // dv_j += sum_i p_ij dout_i (key block b < a is full)
                mmkk48(K0, h ? D1 : D0, m0, c0, acc);
                red_kk(dv + (hL + (size_t)b * kC) * kD2 + 64 * h, acc, m0, c0, kD2);
            }
        }
        __syncthreads();
        if (!lead && b > 0) {
            put_rb(X0, LD, acc1, r0, n0);
            put_rb(X1, LD, acc2, r0, n0);
        }
    }

    // ---- pass 2: left to right, G = gradient of X_{a,b}
    float *const dTs = D0, *const G0 = V0, *const G1 = V1;
    float g0[4][8], g1[4][8];
    zero48(g0);
    zero48(g1);
    __syncthreads();
    for (int e = tid; e < BUF; e += kThreads) {
        G0[e] = 0.f;
        G1[e] = 0.f;
    }
    for (int b = 0; b < a; ++b) {
        const float *st = stash + (pair0 + b) * kStash;
        __syncthreads();
        load_tile(X0, st, false, kD2);
        load_tile(X1, st + 64, false, kD2);
        load_tile(dTs, st + kC * kD2, false, kC);
        load_kp(b);
        __syncthreads();
        if (lead) {
            zero48(g0);
            zero48(g1);
            if (b > 0) {  // G_{b-1} P_b, column halves 0 and 1
                mm48(G0, P00, r0, c0, g0);
                mm48(G1, P10, r0, c0, g0);
                mm48(G0, P01, r0, c0, g1);
                mm48(G1, P11, r0, c0, g1);
            }
            mm48(dTs, K0, r0, c0, g0);  // + dT_ab K~_b
            mm48(dTs, K1, r0, c0, g1);
        } else if (b > 0) {  // dP_b[n][c] += sum_i G_{b-1}[i][n] X_{a,b}[i][c], four quadrants
            float *dpb = dP + ((size_t)bh * nblk + b) * kD2 * kD2;
#pragma unroll 1
            for (int qd = 0; qd < 4; ++qd) {
                const int nh = qd >> 1, ch = qd & 1;
                float acc[4][8];
                zero48(acc);
                mmkk48(nh ? G1 : G0, ch ? X1 : X0, m0, c0, acc);
                red_kk(dpb + 64 * nh * kD2 + 64 * ch, acc, m0, c0, kD2);
            }
        }
        __syncthreads();
        if (lead) {
            put48(G0, g0, r0, c0);
            put48(G1, g1, r0, c0);
        }
    }
    if (lead) {
        // dQ~_a = G_{a-1} (zero for the first block)
        float *dq_a = dqt + ((size_t)bh * Lp + t0) * kD2;
        st48(dq_a, g0, r0, c0, kD2);
        st48(dq_a + 64, g1, r0, c0, kD2);
        if (FOX && tx == 0)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + r0 + 8 * i < L) rsum[(size_t)bh * Lp + t0 + r0 + 8 * i] = rs_acc[i];
    }
}

size_t bwd_query128_smem() { return (size_t)(kBufs * BUF + 4 * kC) * sizeof(float); }

// Workspace of the d = 128 backward: first the fp32 d = 128 forward's preparation outputs
// (d128_layout: 256-byte status header, q~, [k~; P_b], diagonal logits and, for PaTH-FoX, its
// gate sums and exit bounds), then dq~ and dk~ (BH, Lp, 128), dP_b (BH, nblk, 128, 128), the
// diagonal dT (BH, nblk, 64, 64) and the query pass's stash: X_{a,b} (64 x 128) and dT_ab
// (64 x 64) for every pair b < a; PaTH-FoX adds the block-local gate sums, the row and
// column sums of dS (BH, Lp) fp32 each and the per-block gate prefixes (BH, nblk) fp64.
struct Bwd128Layout {
    D128Layout f;
    size_t off_dqt, off_dkt, off_dP, off_dTd, off_stash, off_loc, off_rs, off_cs, off_cb, total;
};

Bwd128Layout bwd128_layout(int B, int H, int L, bool fox) {
    Bwd128Layout y;
    y.f = d128_layout(B, H, L, fox);
    const size_t bh = (size_t)y.f.BH, nblk = (size_t)y.f.nblk, Lp = (size_t)y.f.Lp;
    const size_t rows = bh * Lp * kD2 * 4;
    size_t off = y.f.total;
    y.off_dqt = off;
    off = align256(off + rows);
    y.off_dkt = off;
    off = align256(off + rows);
    y.off_dP = off;
    off = align256(off + bh * nblk * kD2 * kD2 * 4);
    y.off_dTd = off;
    off = align256(off + bh * nblk * kC * kC * 4);
    y.off_stash = off;
    off = align256(off + bh * (nblk * (nblk - 1) / 2) * kStash * 4);
    y.off_loc = y.off_rs = y.off_cs = y.off_cb = off;
    if (fox) {
        const size_t tok = bh * Lp * 4;
        y.off_rs = align256(off + tok);
        y.off_cs = align256(y.off_rs + tok);
        y.off_cb = align256(y.off_cs + tok);
        off = align256(y.off_cb + bh * nblk * 8);
    }
    y.total = off;
    return y;
}

}  // namespace

size_t bwd128_ws_bytes(int B, int H, int L, bool fox) { return bwd128_layout(B, H, L, fox).total; }

// dq, dk, dv, dw (B*H, L, 128) and dbeta (B*H, L) fp32; with log_f (PaTH-FoX) also dlogf
// (B*H, L) fp32. dv gathers by atomics from zero.
template <typename T>
cudaError_t launch_path_bwd128(const void *q, const void *k, const void *v, const void *w,
                               const float *beta, const float *log_f, const void *o,
                               const float *lse, const void *dout, int B, int H, int L,
                               float scale, float *dq, float *dk, float *dv, float *dw,
                               float *dbeta, float *dlogf, void *ws, cudaStream_t stream) {
    const bool fox = log_f != nullptr;
    const Bwd128Layout y = bwd128_layout(B, H, L, fox);
    const int BH = y.f.BH, nblk = y.f.nblk, Lp = y.f.Lp;
    char *base = static_cast<char *>(ws);
    auto at = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    const float *qt = at(y.f.off_qt), *kp = at(y.f.off_kp), *dg = at(y.f.off_dg);
    float *dqt = at(y.off_dqt), *dkt = at(y.off_dkt), *dPb = at(y.off_dP), *dTd = at(y.off_dTd);
    float *stash = at(y.off_stash), *loc = at(y.off_loc), *rs = at(y.off_rs), *cs = at(y.off_cs);
    double *cb = reinterpret_cast<double *>(base + y.off_cb);
    const size_t tok = (size_t)BH * Lp * 4;
    cudaError_t e;
    // the preparation clears the status word and writes q~, [k~; P_b] and the diagonal table
    if ((e = launch_prep_d128<T>(q, k, w, beta, log_f, B, H, L, scale, ws, stream)) != cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(dkt, 0, tok * kD2, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dPb, 0, (size_t)BH * nblk * kD2 * kD2 * 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dv, 0, (size_t)BH * L * kD2 * 4, stream)) != cudaSuccess) return e;
    if (fox) {
        if ((e = cudaMemsetAsync(rs, 0, tok, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(cs, 0, tok, stream)) != cudaSuccess ||
            (e = launch_bwd_fox_sums(log_f, BH, L, Lp, nblk, loc, cb, stream)) != cudaSuccess)
            return e;
    }
    auto kq = fox ? bwd_query128_kernel<T, true> : bwd_query128_kernel<T, false>;
    const size_t s1 = bwd_query128_smem();
    if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1)) != cudaSuccess)
        return e;
    kq<<<dim3(nblk, BH), kThreads, s1, stream>>>(
        static_cast<const T *>(v), static_cast<const T *>(o), static_cast<const T *>(dout), lse,
        qt, kp, dg, dqt, dkt, dPb, dTd, stash, dv, L, Lp, nblk, scale, scale * kLog2e, loc, cb, rs,
        cs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bwd_block_sweep<T>(q, k, w, beta, dqt, dkt, dPb, dTd, dq, dk, dw, dbeta, BH, L,
                                       Lp, nblk, kD2, stream)) != cudaSuccess)
        return e;
    if (fox) e = launch_bwd_fox_dlogf(rs, cs, BH, L, Lp, dlogf, stream);
    return e;
}

#define PATH_BWD128_INST(T)                                                                      \
    template cudaError_t launch_path_bwd128<T>(const void *, const void *, const void *,         \
                                               const void *, const float *, const float *,       \
                                               const void *, const float *, const void *, int,   \
                                               int, int, float, float *, float *, float *,       \
                                               float *, float *, float *, void *, cudaStream_t);
PATH_BWD128_INST(float)
#undef PATH_BWD128_INST

}  // namespace path
