// Backward query pass of PaTH attention and PaTH-FoX at head size d = 128 on the tensor
// cores (bf16 inputs): warp-level bf16 MMAs (mma.sync m16n8k16, fp32 accumulation) with
// their operands in padded shared-memory tiles read by ldmatrix.
//
// The pages give no backward (review "거리에서 경로로, PaTH Attention" §9 and technical
// summary "技術要約: PaTH Attention" §3 say the block-wise algorithm makes training
// efficient; §6 of the summary and §9 of the review flag larger heads as costlier). The
// chain rule is that of backward.cu: with X_{a,b} the rows of query block a carried down
// to key block b (X_{a,a-1} = Q~_a, X_{a,b-1} = X_{a,b} P_b^T), T_ab = X_{a,b} K~_b^T,
// dS_ij = p_ij (dout_i . v_j - dout_i . out_i) and dT = scale dS:
//     dv_b += p_ab^T dout_a,   dK~_b += dT_ab^T X_{a,b},
//     G_b = G_{b-1} P_b + dT_ab K~_b  (G_{-1} = 0),   dP_b += G_{b-1}^T X_{a,b},
//     dQ~_a = G_{a-1}.
// The tcgen05 query pass of backward_tc.cu holds a 128-row tile's logits, carried rows and
// gathered products in tensor memory; at d = 128 those need more than its 512 columns, and
// the operand ring more than the shared memory of an SM. Here a CTA owns one 64-row query
// block; X, K~_b, V_b, dout and G (64 x 128) are two 64-column tiles and P_b (128 x 128)
// four quadrants, and every product is a sum of 64 x 64 x 64 warp-tile MMAs.
// Precision follows the d = 64 tensor-core pass: bf16 operands (the bf16 preparation's
// factors, the carried rows rounded to bf16 at every key block and stashed so, p and dT
// rounded to bf16), fp32 accumulation, and G kept in fp32 and fed to its recursion as a bf16
// head and tail (G = G_hi + G_lo, about 16 significant bits). The block pass in matrix form
// (backward_block_mm.cu at d = 128) then takes dq~, dk~, dP_b and the diagonal dT to q, k, w
// and beta.
#include "common.cuh"

namespace path {

cudaError_t launch_ut_prepare_tc128(const void *q, const void *k, const void *w,
                                    const float *beta, const float *log_f, int BH, int L,
                                    float scale, void *ws, uint64_t limit_ns,
                                    cudaStream_t stream);
cudaError_t launch_bwd_block_mm128(const void *q, const void *k, const void *w, const float *beta,
                                   const float *dqt, const float *dkt, const float *dP,
                                   const float *dTd, float *dq, float *dk, float *dw,
                                   float *dbeta, int BH, int L, int Lp, int nblk,
                                   cudaStream_t stream);
cudaError_t launch_bwd_fox_sums(const float *log_f, int BH, int L, int Lp, int nblk, float *loc,
                                double *cb, cudaStream_t stream);
cudaError_t launch_bwd_fox_dlogf(const float *rsum, const float *csum, int BH, int L, int Lp,
                                 float *dlogf, cudaStream_t stream);

namespace {

constexpr int kThr = 256;
constexpr int kD2 = 128;                   // head size of this file
constexpr int SLD = 72;                    // bf16 elements per shared tile row (64 + 8 pad)
constexpr uint32_t kTile = 64 * SLD * 2;   // bytes of one 64 x 64 bf16 tile
// Tile slots. Pass 1: X0 X1 (carried rows), D0 D1 (dout), PT DT (p and dT), and two sets of
// the key block's operands (K0 K1, the P_b quadrants P00 P01 P10 P11, V0 V1), so that the
// next block's loads overlap the current block's MMAs. Pass 2: two sets of the stash's X_b
// (two tiles) and dT_b and the key block's K~_b and P_b; G's bf16 head and tail take D0, D1
// and the V tiles of set 1.
enum : int { X0, X1, D0, D1, PT, DT, SET0, kNumTiles = SET0 + 16 };
enum : int { K0, K1, P00, P01, P10, P11, V0, V1 };  // offsets within a pass-1 set
__host__ __device__ constexpr int s1(int set, int t) { return SET0 + 8 * set + t; }
// pass 2, set 0: X = slots X0, X1, dT = DT, K~_b and P_b = the first six tiles of pass-1 set 0;
// set 1: X = the V tiles of pass-1 set 0, dT = PT, K~_b and P_b = the first six of set 1
__host__ __device__ constexpr int s2x(int set, int h) { return set ? s1(0, V0 + h) : X0 + h; }
__host__ __device__ constexpr int s2dt(int set) { return set ? PT : DT; }
constexpr int G0H = D0, G1H = D1, G0L = s1(1, V0), G1L = s1(1, V1);
constexpr uint32_t kRowsOff = kNumTiles * kTile;  // lse2, Drow, loci, locj: 64 fp32 each
constexpr uint32_t kSmem = kRowsOff + 4 * 64 * 4;
constexpr size_t kKpRows = (size_t)(64 + kD2) * kD2;   // [k~ (64 rows); P_b (128 rows)]
constexpr size_t kStash = (size_t)64 * kD2 + 64 * 64;  // bf16: [X_{a,b} (64 x 128) | dT_ab]

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void red_add_v2(float *p, float a, float b) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(a), "f"(b) : "memory");
}

using Acc = float[4][4];  // a warp's 16 x 32 block: 4 n-tiles of the m16n8 fragment

__device__ __forceinline__ void zero(Acc &a) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[i][j] = 0.f;
}

// acc += A B over k = 0..63 for this warp's block (rows 16 wm .., columns 32 wn ..) of a
// 64 x 64 product: A stored in tile a as [m][k] (AT false) or [k][m] (AT true), B in tile b
// as [n][k] (BT false) or [k][n] (BT true). Fragment element (nt, e) of acc is row
// 16 wm + lane/4 + 8 (e/2), column 32 wn + 8 nt + 2 (lane%4) + e%2.
template <bool AT, bool BT>
__device__ __forceinline__ void wmma64(Acc &acc, uint32_t a, uint32_t b, int wm, int wn,
                                       int lane) {
    const int li = lane & 7, l3 = (lane >> 3) & 1, l4 = lane >> 4;
#pragma unroll
    for (int k0 = 0; k0 < 64; k0 += 16) {
        uint32_t af[4];
        if (!AT)
            ldsm_x4(a + ((16 * wm + (lane & 15)) * SLD + k0 + 8 * l4) * 2, af);
        else
            ldsm_x4_t(a + ((k0 + 8 * l4 + li) * SLD + 16 * wm + 8 * l3) * 2, af);
#pragma unroll
        for (int np = 0; np < 2; ++np) {  // two n-tiles per load
            const int n0 = 32 * wn + 16 * np;
            uint32_t bf[4];
            if (!BT)
                ldsm_x4(b + ((n0 + 8 * l4 + li) * SLD + k0 + 8 * l3) * 2, bf);
            else
                ldsm_x4_t(b + ((k0 + 8 * l3 + li) * SLD + n0 + 8 * l4) * 2, bf);
            mma_bf16(acc[2 * np], af, bf[0], bf[1]);
            mma_bf16(acc[2 * np + 1], af, bf[2], bf[3]);
        }
    }
}

// acc[j] += sum_i A_i B_j over k = 0..63 for this warp's block, NA A tiles and NB B tiles in
// the layouts of wmma64; every fragment is loaded once per k step and used by every product
// that shares it.
template <bool AT, bool BT, int NA, int NB>
__device__ __forceinline__ void wmma64_sum(Acc (&acc)[NB], const uint32_t (&a)[NA],
                                           const uint32_t (&b)[NB], int wm, int wn, int lane) {
    const int li = lane & 7, l3 = (lane >> 3) & 1, l4 = lane >> 4;
#pragma unroll
    for (int k0 = 0; k0 < 64; k0 += 16) {
        uint32_t af[NA][4];
#pragma unroll
        for (int i = 0; i < NA; ++i) {
            if (!AT)
                ldsm_x4(a[i] + ((16 * wm + (lane & 15)) * SLD + k0 + 8 * l4) * 2, af[i]);
            else
                ldsm_x4_t(a[i] + ((k0 + 8 * l4 + li) * SLD + 16 * wm + 8 * l3) * 2, af[i]);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j)
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int n0 = 32 * wn + 16 * np;
                uint32_t bf[4];
                if (!BT)
                    ldsm_x4(b[j] + ((n0 + 8 * l4 + li) * SLD + k0 + 8 * l3) * 2, bf);
                else
                    ldsm_x4_t(b[j] + ((k0 + 8 * l3 + li) * SLD + n0 + 8 * l4) * 2, bf);
#pragma unroll
                for (int i = 0; i < NA; ++i) {
                    mma_bf16(acc[j][2 * np], af[i], bf[0], bf[1]);
                    mma_bf16(acc[j][2 * np + 1], af[i], bf[2], bf[3]);
                }
            }
    }
}

// 64 rows x 64 bf16 from global (row stride ld elements; rows >= nrows read as zero) into a
// tile, asynchronously (16-byte copies; the caller commits them as a group)
__device__ __forceinline__ void cp_tile(uint32_t dst, const __nv_bfloat16 *src, int ld, int nrows) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int e = threadIdx.x + it * kThr, r = e >> 3, c = (e & 7) * 8;
        const bool in = r < nrows;
        const __nv_bfloat16 *g = in ? src + (size_t)r * ld + c : src;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + (r * SLD + c) * 2),
                     "l"(g), "r"(in ? 16 : 0)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// waits until at most N of this thread's committed copy groups are still in flight
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// two bf16 at (r, c), (r, c + 1) of a tile
__device__ __forceinline__ void st_pair(uint8_t *tile, int r, int c, float lo, float hi) {
    *reinterpret_cast<uint32_t *>(tile + (r * SLD + c) * 2) = pack_bf16x2(lo, hi);
}

// this warp's 16 x 32 block of a 64 x 64 result added into a row-major fp32 global tile (ld
// floats per row), rows below nrows
__device__ __forceinline__ void red_block(float *dst, int ld, const Acc &acc, int wm, int wn,
                                          int lane, int nrows) {
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = 16 * wm + g + 8 * hr, c = 32 * wn + 8 * nt + 2 * t4;
            if (r < nrows) red_add_v2(dst + (size_t)r * ld + c, acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        }
}

// FoX: the column sums of this warp's dS values (over its 16 rows) into csum_blk (the key
// block's 64 entries), one atomic per column from the lanes of the first row
__device__ __forceinline__ void fox_col_sums(float (&cs)[4][2], float *csum_blk, int wn, int lane) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v = cs[nt][e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (lane < 4) atomicAdd(csum_blk + 32 * wn + 8 * nt + 2 * lane + e, v);
        }
}

// One CTA of 256 threads (8 warps) per (query block a, head), one per SM; a runs from the
// last block down. Warp w computes rows 16 (w / 2) .. + 15 and columns 32 (w % 2) .. + 31 of
// every 64 x 64 product. Per key block b < a of pass 1 the CTA loads K~_b, P_b and V_b,
// forms the logits, dout V_b^T and (b > 0) X P_b^T, turns the first two into p and dT,
// stashes X_{a,b} and dT_ab, gathers dK~_b and dv_b, and replaces X; pass 2 walks b = 0 ..
// a - 1 over the stash with G.
template <bool FOX>
__global__ void __launch_bounds__(kThr, 1)
bwd_query128_mma_kernel(const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ o,
                        const __nv_bfloat16 *__restrict__ dout, const float *__restrict__ lse,
                        const __nv_bfloat16 *__restrict__ qt, const __nv_bfloat16 *__restrict__ kp,
                        const __half *__restrict__ dg, float *__restrict__ dqt,
                        float *__restrict__ dkt, float *__restrict__ dP, float *__restrict__ dTd,
                        __nv_bfloat16 *__restrict__ stash, float *__restrict__ dv, int L, int Lp,
                        int nb, int nblk_p, int Lp_p, float scale, float scale_log2,
                        const float *__restrict__ loc, const double *__restrict__ cb,
                        float *__restrict__ rsum, float *__restrict__ csum, int heads_fast) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sb = smem_u32(sm);
    auto tile = [&](int t) { return sb + (uint32_t)t * kTile; };
    auto tptr = [&](int t) { return sm + (size_t)t * kTile; };
    float *lse2 = reinterpret_cast<float *>(sm + kRowsOff);  // per row: lse * log2(e)
    float *Drow = lse2 + 64;                                  // per row: dout . out
    float *loci = Drow + 64;  // FoX: block-local gate sums of the query rows
    float *locj = loci + 64;  // FoX: those of the current key block

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 1, wn = warp & 1, g = lane >> 2, t4 = lane & 3;
    // a one-dimensional grid over (query block, head), longest walks first, heads fastest or
    // head by head (heads_fastest)
    const unsigned BH = gridDim.x / (unsigned)nb;
    const int a = nb - 1 - (int)(heads_fast ? blockIdx.x / BH : blockIdx.x % (unsigned)nb);
    const int bh = (int)(heads_fast ? blockIdx.x % BH : blockIdx.x / (unsigned)nb);
    const int t0 = a * 64;
    const int nq = min(64, L - t0);  // query rows of this block below L
    const size_t hL = (size_t)bh * L;
    const __nv_bfloat16 *vh = v + hL * kD2, *douth = dout + hL * kD2;

    // ---- per row: lse in log2 units and D_i = dout_i . out_i (4 threads per row)
    {
        const int row = tid >> 2, part = tid & 3;
        float dsum = 0.f;
        if (row < nq) {
            const size_t gi = (hL + t0 + row) * kD2 + part * 32;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                const uint4 x = *reinterpret_cast<const uint4 *>(dout + gi + c);
                const uint4 y = *reinterpret_cast<const uint4 *>(o + gi + c);
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 p = unpack_bf16x2(xs[e]), q = unpack_bf16x2(ys[e]);
                    dsum = fmaf(p.x, q.x, fmaf(p.y, q.y, dsum));
                }
            }
        }
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
        if (part == 0) {
            Drow[row] = dsum;
            lse2[row] = row < nq ? lse[hL + t0 + row] * kLog2e : 0.f;
            if (FOX) loci[row] = row < nq ? loc[(size_t)bh * Lp + t0 + row] : 0.f;
        }
    }
    float rs[2] = {0.f, 0.f};  // FoX: row sums of dS (rows 16 wm + g, + 8; this warp's columns)

    // pass 1's operands of key block b into set `set`: K~_b, the P_b quadrants, V_b
    auto stage1 = [&](int set, int b) {
        const __nv_bfloat16 *kb = kp + ((size_t)bh * nblk_p + b) * kKpRows;
        cp_tile(tile(s1(set, K0)), kb, kD2, 64);
        cp_tile(tile(s1(set, K1)), kb + 64, kD2, 64);
        cp_tile(tile(s1(set, P00)), kb + 64 * kD2, kD2, 64);
        cp_tile(tile(s1(set, P01)), kb + 64 * kD2 + 64, kD2, 64);
        cp_tile(tile(s1(set, P10)), kb + 128 * kD2, kD2, 64);
        cp_tile(tile(s1(set, P11)), kb + 128 * kD2 + 64, kD2, 64);
        cp_tile(tile(s1(set, V0)), vh + (size_t)b * 64 * kD2, kD2, 64);
        cp_tile(tile(s1(set, V1)), vh + (size_t)b * 64 * kD2 + 64, kD2, 64);
        cp_commit();
    };
    const size_t pair0 = (size_t)bh * ((size_t)nb * (nb - 1) / 2) + (size_t)a * (a - 1) / 2;
    // pass 2's operands of key block b into set `set`: the stashed X_{a,b} and dT_ab, K~_b, P_b
    auto stage2 = [&](int set, int b) {
        const __nv_bfloat16 *st = stash + (pair0 + b) * kStash;
        const __nv_bfloat16 *kb = kp + ((size_t)bh * nblk_p + b) * kKpRows;
        cp_tile(tile(s2x(set, 0)), st, kD2, 64);
        cp_tile(tile(s2x(set, 1)), st + 64, kD2, 64);
        cp_tile(tile(s2dt(set)), st + 64 * kD2, 64, 64);
        cp_tile(tile(s1(set, K0)), kb, kD2, 64);
        cp_tile(tile(s1(set, K1)), kb + 64, kD2, 64);
        cp_tile(tile(s1(set, P00)), kb + 64 * kD2, kD2, 64);
        cp_tile(tile(s1(set, P01)), kb + 64 * kD2 + 64, kD2, 64);
        cp_tile(tile(s1(set, P10)), kb + 128 * kD2, kD2, 64);
        cp_tile(tile(s1(set, P11)), kb + 128 * kD2 + 64, kD2, 64);
        cp_commit();
    };

    // the diagonal block's dout, V (into set 1) and Q~_a; then key block a - 1 into set 0
    const __nv_bfloat16 *qa = qt + ((size_t)bh * Lp_p + t0) * kD2;
    cp_tile(tile(D0), douth + (size_t)t0 * kD2, kD2, nq);
    cp_tile(tile(D1), douth + (size_t)t0 * kD2 + 64, kD2, nq);
    cp_tile(tile(s1(1, V0)), vh + (size_t)t0 * kD2, kD2, nq);
    cp_tile(tile(s1(1, V1)), vh + (size_t)t0 * kD2 + 64, kD2, nq);
    cp_tile(tile(X0), qa, kD2, 64);
    cp_tile(tile(X1), qa + 64, kD2, 64);
    cp_commit();
    if (a > 0) {
        stage1(0, a - 1);
        cp_wait<1>();
    } else {
        cp_wait<0>();
    }
    __syncthreads();

    // ---- diagonal block: logits from the preparation's table; dT to the block pass
    {
        Acc ov;
        zero(ov);
        wmma64<false, false>(ov, tile(D0), tile(s1(1, V0)), wm, wn, lane);  // dout_i . v_j
        wmma64<false, false>(ov, tile(D1), tile(s1(1, V1)), wm, wn, lane);
        const __half *tab = dg + ((size_t)bh * nblk_p + a) * 64 * 64;
        float *dtd = dTd + ((size_t)bh * nb + a) * 64 * 64;
        float cs[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = 16 * wm + g + 8 * hr, c = 32 * wn + 8 * nt + 2 * t4;
                const float2 lg = __half22float2(*reinterpret_cast<const __half2 *>(tab + r * 64 + c));
                float p[2], dt[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pe = r < nq ? exp2f((e ? lg.y : lg.x) - lse2[r]) : 0.f;
                    const float ds = pe * (ov[nt][2 * hr + e] - Drow[r]);
                    if (FOX) {
                        rs[hr] += ds;
                        cs[nt][e] += ds;
                    }
                    p[e] = pe;
                    dt[e] = scale * ds;
                }
                *reinterpret_cast<float2 *>(dtd + r * 64 + c) = make_float2(dt[0], dt[1]);
                st_pair(tptr(PT), r, c, p[0], p[1]);
            }
        if (FOX) fox_col_sums(cs, csum + (size_t)bh * Lp + (size_t)a * 64, wn, lane);
    }
    __syncthreads();
    {  // dv_j += sum_i p_ij dout_i, j in the diagonal block, both column halves
        Acc acc[2];
        zero(acc[0]);
        zero(acc[1]);
        wmma64_sum<true, true, 1, 2>(acc, {tile(PT)}, {tile(D0), tile(D1)}, wm, wn, lane);
        red_block(dv + (hL + t0) * kD2, kD2, acc[0], wm, wn, lane, nq);
        red_block(dv + (hL + t0) * kD2 + 64, kD2, acc[1], wm, wn, lane, nq);
    }

    // ---- pass 1: right to left over key blocks, X from Q~_a; key block b in set (a-1-b) % 2
    for (int b = a - 1; b >= 0; --b) {
        const int set = (a - 1 - b) & 1;
        __syncthreads();  // the previous step's readers of its set, p and dT are done
        if (b > 0) {
            stage1(set ^ 1, b - 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        if (FOX && tid < 64) locj[tid] = loc[(size_t)bh * Lp + (size_t)b * 64 + tid];
        __syncthreads();
        // sx[0]: x_i . k~_j; sx[1], sx[2]: column halves 0 and 1 of X P_b^T (b > 0); each X
        // half's fragments serve all three
        Acc sx[3], ov;
        zero(sx[0]);
        zero(sx[1]);
        zero(sx[2]);
        zero(ov);
        if (b > 0) {
            wmma64_sum<false, false, 1, 3>(sx, {tile(X0)},
                                           {tile(s1(set, K0)), tile(s1(set, P00)), tile(s1(set, P10))},
                                           wm, wn, lane);
            wmma64_sum<false, false, 1, 3>(sx, {tile(X1)},
                                           {tile(s1(set, K1)), tile(s1(set, P01)), tile(s1(set, P11))},
                                           wm, wn, lane);
        } else {
            wmma64<false, false>(sx[0], tile(X0), tile(s1(set, K0)), wm, wn, lane);
            wmma64<false, false>(sx[0], tile(X1), tile(s1(set, K1)), wm, wn, lane);
        }
        wmma64<false, false>(ov, tile(D0), tile(s1(set, V0)), wm, wn, lane);  // dout_i . v_j
        wmma64<false, false>(ov, tile(D1), tile(s1(set, V1)), wm, wn, lane);
        Acc &s = sx[0], &xn0 = sx[1], &xn1 = sx[2];
        {
            const float dcb = FOX ? (float)(cb[(size_t)bh * nb + a] - cb[(size_t)bh * nb + b]) : 0.f;
            float cs[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = 16 * wm + g + 8 * hr, c = 32 * wn + 8 * nt + 2 * t4;
                    float p[2], dt[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float x2 = s[nt][2 * hr + e] * scale_log2;
                        if (FOX) x2 += kLog2e * ((dcb + loci[r]) - locj[c + e]);
                        const float pe = r < nq ? exp2f(x2 - lse2[r]) : 0.f;
                        const float ds = pe * (ov[nt][2 * hr + e] - Drow[r]);
                        if (FOX) {
                            rs[hr] += ds;
                            cs[nt][e] += ds;
                        }
                        p[e] = pe;
                        dt[e] = scale * ds;
                    }
                    st_pair(tptr(PT), r, c, p[0], p[1]);
                    st_pair(tptr(DT), r, c, dt[0], dt[1]);
                }
            if (FOX) fox_col_sums(cs, csum + (size_t)bh * Lp + (size_t)b * 64, wn, lane);
        }
        __syncthreads();  // p and dT complete
        {
            // stash: X_{a,b} (64 x 128) and dT_ab (64 x 64), bf16 row-major
            __nv_bfloat16 *st = stash + (pair0 + b) * kStash;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int e = tid + it * kThr, r = e >> 4, c = (e & 15) * 8;
                const uint8_t *src = tptr(c < 64 ? X0 : X1) + (r * SLD + (c & 63)) * 2;
                *reinterpret_cast<uint4 *>(st + r * kD2 + c) = *reinterpret_cast<const uint4 *>(src);
            }
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int e = tid + it * kThr, r = e >> 3, c = (e & 7) * 8;
                *reinterpret_cast<uint4 *>(st + 64 * kD2 + r * 64 + c) =
                    *reinterpret_cast<const uint4 *>(tptr(DT) + (r * SLD + c) * 2);
            }
        }
        {
            Acc acc[2];
            zero(acc[0]);  // dK~_b[j][c] += sum_i dT_ij X_ic, both column halves
            zero(acc[1]);
            wmma64_sum<true, true, 1, 2>(acc, {tile(DT)}, {tile(X0), tile(X1)}, wm, wn, lane);
            float *dk_b = dkt + ((size_t)bh * Lp + (size_t)b * 64) * kD2;
            red_block(dk_b, kD2, acc[0], wm, wn, lane, 64);
            red_block(dk_b + 64, kD2, acc[1], wm, wn, lane, 64);
            zero(acc[0]);  // dv_j += sum_i p_ij dout_i (key block b < a is full)
            zero(acc[1]);
            wmma64_sum<true, true, 1, 2>(acc, {tile(PT)}, {tile(D0), tile(D1)}, wm, wn, lane);
            float *dv_b = dv + (hL + (size_t)b * 64) * kD2;
            red_block(dv_b, kD2, acc[0], wm, wn, lane, 64);
            red_block(dv_b + 64, kD2, acc[1], wm, wn, lane, 64);
        }
        __syncthreads();  // X is no longer read: it takes X P_b^T
        if (b > 0) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = 16 * wm + g + 8 * hr, c = 32 * wn + 8 * nt + 2 * t4;
                    st_pair(tptr(X0), r, c, xn0[nt][2 * hr], xn0[nt][2 * hr + 1]);
                    st_pair(tptr(X1), r, c, xn1[nt][2 * hr], xn1[nt][2 * hr + 1]);
                }
        }
    }

    // ---- pass 2: left to right, G = gradient of X_{a,b} (fp32 in registers; its bf16 head
    // and tail in shared memory as the MMA operand)
    Acc g0, g1;
    zero(g0);
    zero(g1);
    if (a > 0) {
        __syncthreads();  // pass 1 is done with every tile
        stage2(0, 0);
    }
    for (int b = 0; b < a; ++b) {
        const int set = b & 1;
        __syncthreads();  // the previous step's readers of its set and of G are done
        if (b + 1 < a) {
            stage2(set ^ 1, b + 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        const int xa = s2x(set, 0), xb = s2x(set, 1), dts = s2dt(set);
        Acc nn[2];  // column halves 0 and 1 of G_b
        zero(nn[0]);
        zero(nn[1]);
        if (b > 0) {  // G_{b-1} P_b: each row half of G (head and tail) against its P_b quadrants
            wmma64_sum<false, true, 2, 2>(nn, {tile(G0H), tile(G0L)},
                                          {tile(s1(set, P00)), tile(s1(set, P01))}, wm, wn, lane);
            wmma64_sum<false, true, 2, 2>(nn, {tile(G1H), tile(G1L)},
                                          {tile(s1(set, P10)), tile(s1(set, P11))}, wm, wn, lane);
        }
        // + dT_ab K~_b
        wmma64_sum<false, true, 1, 2>(nn, {tile(dts)}, {tile(s1(set, K0)), tile(s1(set, K1))}, wm,
                                      wn, lane);
        Acc &n0 = nn[0], &n1 = nn[1];
        if (b > 0) {  // dP_b[n][c] += sum_i G_{b-1}[i][n] X_{a,b}[i][c], four quadrants
            float *dpb = dP + ((size_t)bh * nb + b) * kD2 * kD2;
#pragma unroll 1
            for (int nh = 0; nh < 2; ++nh) {  // row half nh of dP_b, both column halves
                Acc acc[2];
                zero(acc[0]);
                zero(acc[1]);
                wmma64_sum<true, true, 2, 2>(acc, {tile(nh ? G1H : G0H), tile(nh ? G1L : G0L)},
                                             {tile(xa), tile(xb)}, wm, wn, lane);
                red_block(dpb + (size_t)64 * nh * kD2, kD2, acc[0], wm, wn, lane, 64);
                red_block(dpb + (size_t)64 * nh * kD2 + 64, kD2, acc[1], wm, wn, lane, 64);
            }
        }
        __syncthreads();  // G_{b-1} is no longer read
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                g0[nt][e] = n0[nt][e];
                g1[nt][e] = n1[nt][e];
            }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = 16 * wm + g + 8 * hr, c = 32 * wn + 8 * nt + 2 * t4;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float x0 = h ? g1[nt][2 * hr] : g0[nt][2 * hr];
                    const float x1 = h ? g1[nt][2 * hr + 1] : g0[nt][2 * hr + 1];
                    const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                    st_pair(tptr(h ? G1H : G0H), r, c, __bfloat162float(h0), __bfloat162float(h1));
                    st_pair(tptr(h ? G1L : G0L), r, c, x0 - __bfloat162float(h0),
                            x1 - __bfloat162float(h1));
                }
            }
    }
    // dQ~_a = G_{a-1} (zero for the first block)
    float *dq_a = dqt + ((size_t)bh * Lp + t0) * kD2;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = 16 * wm + g + 8 * hr, c = 32 * wn + 8 * nt + 2 * t4;
            *reinterpret_cast<float2 *>(dq_a + (size_t)r * kD2 + c) =
                make_float2(g0[nt][2 * hr], g0[nt][2 * hr + 1]);
            *reinterpret_cast<float2 *>(dq_a + (size_t)r * kD2 + 64 + c) =
                make_float2(g1[nt][2 * hr], g1[nt][2 * hr + 1]);
        }
    if (FOX) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float x = rs[hr];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            const int r = 16 * wm + g + 8 * hr;
            if (t4 == 0 && r < nq) atomicAdd(rsum + (size_t)bh * Lp + t0 + r, x);
        }
    }
}

// Workspace of the bf16 d = 128 backward: the tensor-core d = 128 forward's preparation
// workspace first (d128_tc_layout, whose 256-byte header is the status header; blocks
// rounded up to even), then with nb = ceil(L / 64) and Lp = 64 nb: fp32 dq~ and dk~
// (BH, Lp, 128), dP_b (BH, nb, 128, 128) and the diagonal dT (BH, nb, 64, 64), the bf16
// stash of X_{a,b} (64 x 128) and dT_ab (64 x 64) for every pair b < a; PaTH-FoX adds the
// block-local gate sums, the row and column sums of dS (BH, Lp) fp32 each and the per-block
// gate prefixes (BH, nb) fp64.
struct BwdTc128Layout {
    D128TcLayout f;
    int nb, Lp;
    size_t off_dqt, off_dkt, off_dP, off_dTd, off_stash, off_loc, off_rs, off_cs, off_cb, total;
};

BwdTc128Layout bwd_tc128_layout(int B, int H, int L, bool fox) {
    BwdTc128Layout y;
    y.f = d128_tc_layout(B, H, L, fox);
    y.nb = (L + 63) / 64;
    y.Lp = 64 * y.nb;
    const size_t bh = (size_t)y.f.BH, nb = (size_t)y.nb;
    const size_t rows = bh * y.Lp * kD2 * 4;
    size_t off = y.f.total;
    y.off_dqt = off;
    off = align256(off + rows);
    y.off_dkt = off;
    off = align256(off + rows);
    y.off_dP = off;
    off = align256(off + bh * nb * kD2 * kD2 * 4);
    y.off_dTd = off;
    off = align256(off + bh * nb * 64 * 64 * 4);
    y.off_stash = off;
    off = align256(off + bh * (nb * (nb - 1) / 2) * kStash * 2);
    y.off_loc = y.off_rs = y.off_cs = y.off_cb = off;
    if (fox) {
        const size_t tok = bh * y.Lp * 4;
        y.off_rs = align256(off + tok);
        y.off_cs = align256(y.off_rs + tok);
        y.off_cb = align256(y.off_cs + tok);
        off = align256(y.off_cb + bh * nb * 8);
    }
    y.total = off;
    return y;
}

}  // namespace

size_t bwd_tc128_ws_bytes(int B, int H, int L, bool fox) {
    return bwd_tc128_layout(B, H, L, fox).total;
}

// bf16 inputs at d = 128: dq, dk, dv, dw (B*H, L, 128) and dbeta (B*H, L) fp32; with log_f
// (PaTH-FoX) also dlogf (B*H, L) fp32. dv gathers by atomics from zero.
cudaError_t launch_path_bwd128_tc(const void *q, const void *k, const void *v, const void *w,
                                  const float *beta, const float *log_f, const void *o,
                                  const float *lse, const void *dout, int B, int H, int L,
                                  float scale, float *dq, float *dk, float *dv, float *dw,
                                  float *dbeta, float *dlogf, void *ws, uint64_t limit_ns,
                                  cudaStream_t stream) {
    const bool fox = log_f != nullptr;
    const BwdTc128Layout y = bwd_tc128_layout(B, H, L, fox);
    const int BH = y.f.BH, nb = y.nb, Lp = y.Lp;
    char *base = static_cast<char *>(ws);
    auto at = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    float *dqt = at(y.off_dqt), *dkt = at(y.off_dkt), *dPb = at(y.off_dP), *dTd = at(y.off_dTd);
    float *loc = at(y.off_loc), *rs = at(y.off_rs), *cs = at(y.off_cs);
    double *cb = reinterpret_cast<double *>(base + y.off_cb);
    const size_t tok = (size_t)BH * Lp * 4;
    cudaError_t e;
    if ((e = cudaMemsetAsync(base, 0, 4, stream)) != cudaSuccess) return e;
    if ((e = launch_ut_prepare_tc128(q, k, w, beta, log_f, BH, L, scale, ws, limit_ns, stream)) !=
        cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(dkt, 0, tok * kD2, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dPb, 0, (size_t)BH * nb * kD2 * kD2 * 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dv, 0, (size_t)BH * L * kD2 * 4, stream)) != cudaSuccess) return e;
    if (fox) {
        if ((e = cudaMemsetAsync(rs, 0, tok, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(cs, 0, tok, stream)) != cudaSuccess ||
            (e = launch_bwd_fox_sums(log_f, BH, L, Lp, nb, loc, cb, stream)) != cudaSuccess)
            return e;
    }
    auto kq = fox ? bwd_query128_mma_kernel<true> : bwd_query128_mma_kernel<false>;
    if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem)) !=
        cudaSuccess)
        return e;
    if ((size_t)BH * nb > 0x7fffffffu) return cudaErrorInvalidConfiguration;
    // shared per token: [K~_b; P_b] (768 B) and v (256 B)
    const bool hf = heads_fastest((size_t)BH, (size_t)L, 1024);
    kq<<<(unsigned)(BH * nb), kThr, kSmem, stream>>>(
        static_cast<const __nv_bfloat16 *>(v), static_cast<const __nv_bfloat16 *>(o),
        static_cast<const __nv_bfloat16 *>(dout), lse,
        reinterpret_cast<const __nv_bfloat16 *>(base + y.f.off_qt),
        reinterpret_cast<const __nv_bfloat16 *>(base + y.f.off_kp),
        reinterpret_cast<const __half *>(base + y.f.off_dg), dqt, dkt, dPb, dTd,
        reinterpret_cast<__nv_bfloat16 *>(base + y.off_stash), dv, L, Lp, nb, y.f.nblk, y.f.Lp,
        scale, scale * kLog2e, loc, cb, rs, cs, hf ? 1 : 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bwd_block_mm128(q, k, w, beta, dqt, dkt, dPb, dTd, dq, dk, dw, dbeta, BH, L,
                                    Lp, nb, stream)) != cudaSuccess)
        return e;
    if (fox) e = launch_bwd_fox_dlogf(rs, cs, BH, L, Lp, dlogf, stream);
    return e;
}

}  // namespace path
