// K1 (bf16): per-block UT preprocessing of PaTH attention on tcgen05 tensor cores.
//
// Technical summary "技術要約: PaTH Attention" §3 ("UT変換による表現": the product of a
// block's transitions is I - W^T T^{-1} W with T triangular and built from beta; the
// block-wise algorithm precomputes boundary-adjusted queries and keys per block). For one
// block of 64 tokens of one head (W, Q, K rows = w_s, q_i, k_j; D = diag(beta)):
//   G  = W W^T,  E = D strictly-upper(G),  A = (I + E)^{-1} D      (fp32)
//   Lq = lower-incl(Q W^T),  Rk = strictly-upper(K W^T)
//   U  = A^T W,  V' = A W,  Khat = Rk A
//   q~ = Q - Lq U            (rows: (H_0 ... H_i) q_i)
//   k~ = K - Rk V'           (rows: (H_{j+1} ... H_63)^T k_j)
//   P_b = I - W^T V'         (H_0 ... H_63, dense)
//   diag logits (j <= i) = scale * (Q K^T - Lq Khat^T) [+ sum_{s=j+1..i} log f_s]
// Lq U equals (Lq A^T) W and Lq Khat^T equals Lq A^T Rk^T, the leading/trailing partial
// products of the UT form (sub-blocks of A invert the matching sub-blocks of T).
//
// (I + E)^{-1} is formed blockwise (ut_inverse.cuh): the four 16 x 16 diagonal blocks by
// back-substitution, then the 16- and 32-block combine products, each 16 x 8 output tile
// one warp's mma.sync with tf32 operands (these products are too small for tcgen05, and the
// fragment loads keep shared-memory traffic low; A goes on as fp16, so tf32's 10-bit
// significand matches its use).
//
// tcgen05.mma groups, all M = 128, with 64x64 16-bit tiles in 128-byte-swizzled shared
// memory (K-major tiles stacked in M must be adjacent; MN-major atoms use the LBO stride):
//   MMA1 (bf16):  [Q; W] x [W; K]^T          -> Q W^T | (Q K^T)  /  W W^T | W K^T
//   MMA3 (fp16):  [A^T; A] x [W | Rk^T]      -> U | Khat^T       /  V' | (unused)
//   G1 (fp16):    [W^T; Lq] x [U | V']       -> (unused) | W^T V'  /  Lq U | (unused)
//   G2:           [Q; W] x [K; 0]^T (bf16) - [Lq; Rk] x [Khat^T | V'] (fp16), one
//                 accumulator                -> diag logits | 0    /  (unused) | -Rk V'
// The last two groups stack their operands so that every TMEM lane holds a row somebody
// needs (P_b or q~ after G1, the diagonal table or k~ after G2): their epilogues run on all
// eight warps, at the price of MMAs half of whose output is discarded.
// Second-level operands are fp16 (11-bit significand; all bounded, |A_su| <= 4), fp32
// accumulation. One CTA of 256 threads per (block, head): warps w and w + 4 read the same
// 32 TMEM lanes (rows) and split every 64-column epilogue into halves, thread 0 issues
// the TMA loads and the MMAs. 128 TMEM columns, 72 KB of tiles and 80 registers per
// thread, so three CTAs (24 warps) share an SM.
#include "common.cuh"
#include "ut_inverse.cuh"

namespace path {

namespace {

constexpr int kThreads = 256;
constexpr uint32_t kT = 8192;  // one 64 x 64 16-bit tile

// Tile slots (from the 1024-aligned base). Q, W, K adjacent (MMA1 A = [Q; W], B = [W; K]);
// slot 3 stages P_b for its TMA store; Lq^T and Rk^T adjacent (A = [Lq; Rk]), after the last
// group the staging of the diagonal table and k~; AT, A adjacent (MMA3 A). U, KhT, V reuse the
// slots of AT, A and the solve scratch; U's slot stages q~ after G1.
constexpr uint32_t T_Q = 0 * kT, T_W = 1 * kT, T_K = 2 * kT, T_PB = 3 * kT, T_LQ = 4 * kT,
                   T_RKT = 5 * kT, T_AT = 6 * kT, T_A = 7 * kT, T_U = 6 * kT, T_KHT = 7 * kT,
                   T_V = 8 * kT;
constexpr uint32_t SCR = 6 * kT;           // solve scratch (E/X fp32 + Y) overlays slots 6-8
using ut_inverse::XLD;
using ut_inverse::YLD;
using ut_inverse::blocked_unit_upper_inverse;
using ut_inverse::mma_tf32;
using ut_inverse::to_tf32;
using ut_inverse::warp_tile_16x8;
constexpr uint32_t Y_OFF = SCR + 64 * XLD * 4;
constexpr uint32_t BAR_OFF = 9 * kT;       // 2 mbarriers
constexpr uint32_t SLOT_OFF = BAR_OFF + 16;
constexpr uint32_t BETA_OFF = SLOT_OFF + 16;
constexpr uint32_t LC_OFF = BETA_OFF + 256;
constexpr uint32_t kSmemBytes = LC_OFF + 256 + 1024;
constexpr uint32_t kTmemCols = 128;

static_assert(Y_OFF + 32 * YLD * 4 <= 9 * kT, "solve scratch fits in slots 6-8");

// idesc for kind::f16 with both operands bf16 (fmt 1) or fp16 (fmt 0)
__host__ __device__ constexpr uint32_t idesc16(int M, int N, uint32_t fmt, bool a_mn, bool b_mn,
                                               bool neg_a = false) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((neg_a ? 1u : 0u) << 13) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Writes 32 fp32 values as half `hf` (16-bit columns 32hf .. 32hf+31, fp16 or bf16) of
// row `row` of a swizzled tile.
template <bool HALF>
__device__ __forceinline__ void store_half16(uint8_t *tile, int row, int hf, const float *x) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u;
        const float *s = x + 8 * c;
        if (HALF) {
            u.x = pack_h2(s[0], s[1]); u.y = pack_h2(s[2], s[3]);
            u.z = pack_h2(s[4], s[5]); u.w = pack_h2(s[6], s[7]);
        } else {
            u.x = pack_bf16x2(s[0], s[1]); u.y = pack_bf16x2(s[2], s[3]);
            u.z = pack_bf16x2(s[4], s[5]); u.w = pack_bf16x2(s[6], s[7]);
        }
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, 4 * hf + c)) = u;
    }
}

// Reads half `hf` of one bf16 row of a swizzled tile as 32 fp32 values.
__device__ __forceinline__ void load_half_bf16(const uint8_t *tile, int row, int hf, float *x) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tile + sw128_offset(row, 4 * hf + c));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            x[8 * c + 2 * e] = f.x;
            x[8 * c + 2 * e + 1] = f.y;
        }
    }
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_row32(uint32_t taddr, float *x) {
    uint32_t a[32];
    tmem_ld32(taddr, a);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(a[j]);
}

// Thread layout: warp w reads TMEM lanes 32 (w mod 4) .. +31 (the accumulator rows lr) and
// handles the 32-column half hf = w / 4 of every 64-column block of its row, so each row's
// epilogue is split between two warps.
// FOX: the forget-gate bias on the diagonal table, and per query row |q~_i| (qn) and the
// largest entry of its table row (dmax), per key block the largest |k~_j| (bkmax), all from
// the rounded values the workspace holds, and the block's fp64 total of log f (btot) and
// smallest in-block prefix sum (bmin), for the early-exit pass.
template <bool FOX>
__global__ void __launch_bounds__(kThreads, 3)
ut_prepare_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_qt_out,
                     const __grid_constant__ CUtensorMap tm_kp_out,
                     const __grid_constant__ CUtensorMap tm_dg_out, const float *__restrict__ beta,
                     const float *__restrict__ log_f, int L, int Lp, int nblk, float scale_log2,
                     float *__restrict__ qn, float *__restrict__ dmax,
                     float *__restrict__ bkmax, double *__restrict__ btot,
                     double *__restrict__ bmin, uint32_t *status, uint64_t limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    float *const X = reinterpret_cast<float *>(sm + SCR);
    float *const Y = reinterpret_cast<float *>(sm + Y_OFF);
    float *const bs = reinterpret_cast<float *>(sm + BETA_OFF);
    float *const lc = reinterpret_cast<float *>(sm + LC_OFF);
    uint32_t *const slot = reinterpret_cast<uint32_t *>(sm + SLOT_OFF);
    const uint32_t bar_tma = base + BAR_OFF, bar_mma = base + BAR_OFF + 8;

    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const int qd = warp & 3, hf = warp >> 2;
    const int lr = 32 * qd + lane;  // accumulator row (TMEM lane) of this thread
    const int c0 = 32 * hf;         // first column of this thread's half
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t head = (size_t)bh * L;
    if (blk == 0 && bh == 0 && r == 0 && status) *status = 0u;

    __shared__ uint32_t abort_s;
    if (r == 0) {
        abort_s = 0u;
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_w);
        mbar_arrive_expect_tx(bar_tma, 3 * kT);
        tma_load_3d(base + T_Q, &tm_q, bar_tma, 0, t0, bh);
        tma_load_3d(base + T_W, &tm_w, bar_tma, 0, t0, bh);
        tma_load_3d(base + T_K, &tm_k, bar_tma, 0, t0, bh);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // beta is first needed after MMA1: its load overlaps the TMA loads and MMA1
    const float beta_r = (r < kC && t0 + r < L) ? beta[head + t0 + r] : 0.f;
    if (FOX && warp == 1) {
        const int ln = r - 32;
        const int ta = t0 + 2 * ln, tb = ta + 1;
        const float a = (ta < L) ? log_f[head + ta] : 0.f;
        const float b = ((tb < L) ? log_f[head + tb] : 0.f) + a;
        float run = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, run, o);
            if (ln >= o) run += n;
        }
        lc[2 * ln] = run - b + a;
        lc[2 * ln + 1] = run;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t lane_off = (uint32_t)(32 * qd) << 16;

    // bounded wait of the whole CTA: thread 0 polls the barrier and the others wait at
    // __syncthreads (polling by every thread would load the shared-memory pipe that the
    // other CTAs on the SM are using); a timeout skips the remaining work
    auto wait_all = [&](uint32_t bar, uint32_t par) {
        if (r == 0) {
            bool ok = mbar_try_wait(bar, par);
            if (!ok) {
                const uint64_t tstart = cycles_now();
                while (!(ok = mbar_try_wait(bar, par)) &&
                       cycles_now() - tstart < ns_to_cycles(limit_ns)) {
                }
            }
            if (!ok) {
                report_status(status, kStatusTimeout);
                abort_s = 1u;
            }
        }
        __syncthreads();
        return abort_s == 0u;
    };

    // ---- MMA1: [Q; W] x [W; K]^T (bf16) -> cols 0..127
    if (r == 0) {
        const uint64_t t0s = cycles_now();
        bool ok = mbar_try_wait(bar_tma, 0);
        while (!ok && cycles_now() - t0s < ns_to_cycles(limit_ns)) ok = mbar_try_wait(bar_tma, 0);
        if (ok) {
            tc_fence_after();
            const uint64_t a = sdesc_sw128(base + T_Q, 16, 1024);
            const uint64_t b = sdesc_sw128(base + T_W, 16, 1024);
            constexpr uint32_t ID = idesc16(128, 128, 1, false, false);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a + 2 * kk, b + 2 * kk, ID, kk > 0);
        } else {
            report_status(status, kStatusTimeout);
        }
        umma_commit(bar_mma);
    }
    if (r < kC) bs[r] = beta_r;
    bool ok = wait_all(bar_mma, 0);  // (its barrier also publishes bs)
    if (ok) {
        tc_fence_after();
        float x[32];
        if (lr < kC) {
            const int i = lr;
            // row i of Q W^T -> Lq (u <= i), fp16, stored transposed (tile rows u): Lq is
            // an MN-major operand of the last two groups
            tmem_row32(tmem + lane_off + c0, x);
            uint8_t *lqt = sm + T_LQ + 2 * (i & 7);
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<__half *>(lqt + sw128_offset(c0 + u, i >> 3)) =
                    __float2half_rn(c0 + u > i ? 0.f : x[u]);
            // W to fp16 in place (MMA1 has completed; later MMAs take fp16 operands)
            load_half_bf16(sm + T_W, i, hf, x);
            store_half16<true>(sm + T_W, i, hf, x);
        } else {
            const int s = lr - kC;
            // row s of W W^T -> E = beta_s G[s][v] for v > s (fp32 scratch)
            tmem_row32(tmem + lane_off + c0, x);
            const float bsv = bs[s];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                float e[4];
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int v = c0 + 4 * q4 + e4;
                    e[e4] = (v > s) ? bsv * x[4 * q4 + e4] : 0.f;
                }
                *reinterpret_cast<float4 *>(X + s * XLD + c0 + 4 * q4) =
                    make_float4(e[0], e[1], e[2], e[3]);
            }
            // row s of W K^T -> Rk^T (s > j), fp16
            tmem_row32(tmem + lane_off + 64 + c0, x);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (s <= c0 + j) x[j] = 0.f;
            store_half16<true>(sm + T_RKT, s, hf, x);
        }
    }
    __syncthreads();

    // ---- A = (I + E)^{-1} D, then A (rows s) and A^T (rows u) as fp16 tiles
    if (ok) {
        blocked_unit_upper_inverse(X, Y, r);
        float a[32];
        if (lr < kC) {
            const int s = lr;  // row s: A[s][u] = X[s][u] beta_u, u >= s
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const int u = c0 + 4 * u4;
                const float4 xv = *reinterpret_cast<const float4 *>(X + s * XLD + u);
                const float4 bv = *reinterpret_cast<const float4 *>(bs + u);
                a[4 * u4] = (u >= s) ? xv.x * bv.x : 0.f;
                a[4 * u4 + 1] = (u + 1 >= s) ? xv.y * bv.y : 0.f;
                a[4 * u4 + 2] = (u + 2 >= s) ? xv.z * bv.z : 0.f;
                a[4 * u4 + 3] = (u + 3 >= s) ? xv.w * bv.w : 0.f;
            }
        } else {
            const int u = lr - kC;  // column u: A[s][u], s <= u
            const float bu = bs[u];
#pragma unroll
            for (int s2 = 0; s2 < 32; ++s2)
                a[s2] = (c0 + s2 <= u) ? X[(c0 + s2) * XLD + u] * bu : 0.f;
        }
        __syncthreads();  // the scratch overlays the A tiles
        if (lr < kC) store_half16<true>(sm + T_A, lr, hf, a);
        else store_half16<true>(sm + T_AT, lr - kC, hf, a);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA3: [A^T; A] x [W | Rk^T] (fp16, B MN-major, N = 128) -> cols 0..127
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t a = sdesc_sw128(base + T_AT, 16, 1024);
        const uint64_t b = sdesc_sw128(base + T_W, T_RKT - T_W, 1024);
        constexpr uint32_t ID = idesc16(128, 128, 0, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a + 2 * kk, b + 128 * kk, ID, kk > 0);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 1);
    if (ok) {
        tc_fence_after();
        float x[32];
        if (lr < kC) {
            tmem_row32(tmem + lane_off + c0, x);       // U row u
            store_half16<true>(sm + T_U, lr, hf, x);
            tmem_row32(tmem + lane_off + 64 + c0, x);  // Khat^T row u
            store_half16<true>(sm + T_KHT, lr, hf, x);
        } else {
            tmem_row32(tmem + lane_off + c0, x);       // V' row s
            store_half16<true>(sm + T_V, lr - kC, hf, x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- G1: [W^T; Lq] x [U | V'] (fp16, both MN-major, N = 128): rows n (0-63) give
    // W^T V' (columns 64-127), rows 64 + i give Lq U (columns 0-63); the off-diagonal
    // blocks are unused
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t a = sdesc_sw128(base + T_W, T_LQ - T_W, 1024);
        const uint64_t b = sdesc_sw128(base + T_U, T_V - T_U, 1024);
        constexpr uint32_t ID = idesc16(128, 128, 0, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a + 128 * kk, b + 128 * kk, ID, kk > 0);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 0);

    const size_t blk_base = (size_t)bh * nblk + blk;
    float qs = 0.f;  // FoX: this thread's half of |q~_i|^2 (the other half goes through bs)
    if (ok) {
        tc_fence_after();
        float x[32];
        if (lr < kC) {
            // P_b row n = lr: delta - (W^T V')_n
            tmem_row32(tmem + lane_off + 64 + c0, x);
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = (c0 + c == lr ? 1.f : 0.f) - x[c];
            store_half16<false>(sm + T_PB, lr, hf, x);  // written by one TMA store below
        } else {
            // q~_i = q_i - (Lq U)_i
            const int i = lr - kC;
            float y[32];
            load_half_bf16(sm + T_Q, i, hf, y);
            tmem_row32(tmem + lane_off + c0, x);
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] -= x[c];
            store_half16<false>(sm + T_U, i, hf, y);  // q~, written by one TMA store below
            if (FOX) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float r16 = __bfloat162float(__float2bfloat16_rn(y[c]));
                    qs = fmaf(r16, r16, qs);
                }
                if (hf == 1) bs[i] = qs;  // beta is no longer needed
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (r == 0 && ok) {
        tma_store_3d(&tm_kp_out, base + T_PB, 0, 2 * kC * blk + kC, bh);  // P_b
        tma_store_3d(&tm_qt_out, base + T_U, 0, t0, bh);                  // q~
    }
    if (FOX && ok && hf == 0 && lr >= kC)
        qn[(size_t)bh * Lp + t0 + lr - kC] = sqrtf(qs + bs[lr - kC]);

    // ---- G2: [Q; W] x K^T (bf16, N = 64) - [Lq; Rk] x Khat^T into columns 0-63 and
    // -[Lq; Rk] x V' into columns 64-127 (fp16, MN-major, N = 64 each): rows i (0-63) give
    // Q K^T - Lq Khat^T, rows 64 + j give -Rk V'; W is fp16 by now, so the W rows of the first
    // product are unused, like the off-diagonal blocks
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t aq = sdesc_sw128(base + T_Q, 16, 1024);
        const uint64_t bk = sdesc_sw128(base + T_K, 16, 1024);
        constexpr uint32_t IDQK = idesc16(128, 64, 1, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, aq + 2 * kk, bk + 2 * kk, IDQK, kk > 0);
        const uint64_t a = sdesc_sw128(base + T_LQ, T_RKT - T_LQ, 1024);
        const uint64_t bh_ = sdesc_sw128(base + T_KHT, 16, 1024);
        const uint64_t bv = sdesc_sw128(base + T_V, 16, 1024);
        constexpr uint32_t IDN = idesc16(128, 64, 0, true, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a + 128 * kk, bh_ + 128 * kk, IDN, 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + 64, a + 128 * kk, bv + 128 * kk, IDN, kk > 0);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 1);
    // FoX partial maxima and key norms in the Q slot, free once G2 has completed
    float *const part = reinterpret_cast<float *>(sm + T_Q);
    if (ok) {
        tc_fence_after();
        float x[32];
        if (lr < kC) {
            // diagonal logits of row i, log2 units, j <= i
            const int i = lr;
            tmem_row32(tmem + lane_off + c0, x);
            const float lci = FOX ? lc[i] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int jj = c0 + j;
                float v = scale_log2 * x[j];
                if (FOX) v += kLog2e * (lci - lc[jj]);
                x[j] = (jj <= i && t0 + jj < L) ? v : -INFINITY;
            }
            store_half16<true>(sm + T_LQ, i, hf, x);  // the table, written by one TMA store
            if (FOX) {
                float dm = -INFINITY;
#pragma unroll
                for (int j = 0; j < 32; ++j) dm = fmaxf(dm, __half2float(__float2half_rn(x[j])));
                part[i * 2 + hf] = dm;
            }
        } else {
            // k~_j = k_j - (Rk V')_j
            const int j = lr - kC;
            float y[32];
            load_half_bf16(sm + T_K, j, hf, y);
            tmem_row32(tmem + lane_off + 64 + c0, x);
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] += x[c];
            store_half16<false>(sm + T_RKT, j, hf, y);  // k~, written by one TMA store
            if (FOX) {
                float ks = 0.f;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float r16 = __bfloat162float(__float2bfloat16_rn(y[c]));
                    ks = fmaf(r16, r16, ks);
                }
                // rows past L are padding: they take part in no logit
                part[256 + j * 2 + hf] = (t0 + j < L) ? ks : 0.f;
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (r == 0 && ok) {
        tma_store_3d(&tm_dg_out, base + T_LQ, 0, kC * blk, bh);          // diagonal table
        tma_store_3d(&tm_kp_out, base + T_RKT, 0, 2 * kC * blk, bh);     // k~
    }
    if (FOX && ok && hf == 0 && lr < kC) {
        // table row lr: combine the two half-row partials
        dmax[(size_t)bh * Lp + t0 + lr] = fmaxf(part[lr * 2], part[lr * 2 + 1]);
    }
    if (FOX && warp == 1) {
        // for the early-exit bounds, in fp64 (off the block's critical path: fp64 is slow
        // here): the block's total of log f and the smallest of its inclusive prefix sums
        const int ta = t0 + 2 * lane, tb = ta + 1;
        const double da = (ta < L) ? (double)log_f[head + ta] : 0.0;
        const double db = ((tb < L) ? (double)log_f[head + tb] : 0.0) + da;
        double drun = db;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, drun, o);
            if (lane >= o) drun += n;
        }
        double dm = fmin(drun - db + da, drun);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dm = fmin(dm, __shfl_xor_sync(0xffffffffu, dm, o));
        const size_t bb = (size_t)bh * nblk + blk;
        if (lane == 31) btot[bb] = drun;
        if (lane == 0) bmin[bb] = dm;
    }
    if (FOX && ok && warp == 2) {
        // largest |k~_j| of the block: lane l takes rows l and l + 32
        const float *kpart = part + 256;
        float m = fmaxf(sqrtf(kpart[lane * 2] + kpart[lane * 2 + 1]),
                        sqrtf(kpart[(lane + 32) * 2] + kpart[(lane + 32) * 2 + 1]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) bkmax[blk_base] = m;
    }
    if (r == 0) bulk_wait_all();  // the stores have read their tiles and written the outputs
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- head size 128
// The same per-block preprocessing at d = 128 (technical summary "技術要約: PaTH Attention"
// §3; review "거리에서 경로로, PaTH Attention" §9 flags larger heads as costlier): W, Q, K are
// 64 x 128, the UT factor A stays 64 x 64, U = A^T W and V' = A W are 64 x 128 and the dense
// block transition P_b = I - W^T V' is 128 x 128. A 64 x 128 16-bit operand is two 64 x 64
// swizzled atoms (columns 0-63 and 64-127); K-major operands walk the two atoms in their
// k-steps, MN-major ones stack them at a fixed byte stride.
//   MMA1 (bf16, K = 128):  [Q; W] x [W; K]^T                -> Q W^T | (Q K^T) / W W^T | W K^T
//   MMA3 (fp16, N = 192):  [A^T; A] x [W | Rk^T]            -> U | Khat^T / V' | (unused)
//   MMA4x:                 Lq x U (fp16, N = 128) ; Q x K^T (bf16, K = 128) - Lq x Khat^T
//   MMA4y (fp16):          W^T x V' (M = 128, N = 128)      -> I - P_b
//                          Rk x V'                          -> k~ = K - Rk V'
// Outputs: q~ (BH, Lp, 128) bf16; per block [k~ (64 rows); P_b (128 rows)] x 128 bf16; the
// fp16 diagonal table. PaTH-FoX also writes, in log2 units, the rows' in-block inclusive gate
// sums lc2, the keys' tail sums T2_b - lc2_j and the block totals T2_b (fp64).
// 8 KB slots: 0 Q0 1 W0 2 K0 3 Q1 4 W1 5 K1 (bf16 inputs, [Q;W;K] per column half so that
// [Q;W] and [W;K] are contiguous in each half); 6 Wh0 7 Wh1 8 Rk^T (fp16, MMA3's B at an 8 KB
// stride); 9 Lq; 10-12 the solve scratch, then A^T, A; after MMA3: U0 = 10, U1 = 11,
// Khat^T = 12, V'0 = 1, V'1 = 4 (W's bf16 halves are dead after MMA1). The outputs are staged
// in dead slots and written by TMA stores: after MMA4x q~ in 10, 11 and the table in 9; after
// MMA4y P_b in 0, 1 (rows 0-63) and 3, 4 (rows 64-127), k~ in 6, 7 (column halves).
constexpr uint32_t k2Slots = 13;
constexpr uint32_t P2_Q0 = 0 * kT, P2_W0 = 1 * kT, P2_K0 = 2 * kT, P2_Q1 = 3 * kT, P2_W1 = 4 * kT,
                   P2_K1 = 5 * kT, P2_WH0 = 6 * kT, P2_WH1 = 7 * kT, P2_RKT = 8 * kT,
                   P2_LQ = 9 * kT, P2_SCR = 10 * kT, P2_AT = 10 * kT, P2_A = 11 * kT,
                   P2_U0 = 10 * kT, P2_U1 = 11 * kT, P2_KHT = 12 * kT, P2_V0 = 1 * kT,
                   P2_V1 = 4 * kT;
constexpr uint32_t P2_OQ0 = 10 * kT, P2_OQ1 = 11 * kT, P2_ODG = 9 * kT, P2_OP00 = 0 * kT,
                   P2_OP01 = 1 * kT, P2_OP10 = 3 * kT, P2_OP11 = 4 * kT, P2_OK0 = 6 * kT,
                   P2_OK1 = 7 * kT;
constexpr uint32_t P2_Y = P2_SCR + 64 * XLD * 4;
constexpr uint32_t P2_BAR = k2Slots * kT, P2_SLOT = P2_BAR + 16, P2_BETA = P2_SLOT + 16,
                   P2_LC = P2_BETA + 256;
// PaTH-FoX: per row and column half the partial |q~|^2, table maximum and |k~|^2
constexpr uint32_t P2_PART = P2_LC + 256;
constexpr uint32_t k2SmemBytes = P2_PART + 3 * 128 * 4 + 1024;
static_assert(P2_Y + 32 * YLD * 4 <= 13 * kT, "d = 128 solve scratch fits in slots 10-12");

// 64 consecutive 16-bit values (one swizzled atom row) as fp32
__device__ __forceinline__ void load_row_bf16(const uint8_t *tile, int row, float *x) {
    load_half_bf16(tile, row, 0, x);
    load_half_bf16(tile, row, 1, x + 32);
}

template <bool FOX>
__global__ void __launch_bounds__(kThreads, 2)
ut_prepare_tc128_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_qt_out,
                        const __grid_constant__ CUtensorMap tm_kp_out,
                        const __grid_constant__ CUtensorMap tm_dg_out, const float *__restrict__ beta,
                        const float *__restrict__ log_f, int L, int Lp, int nblk,
                        float scale_log2, float *__restrict__ lc2, float *__restrict__ tail2,
                        double *__restrict__ tot2, float *__restrict__ qn,
                        float *__restrict__ dmax, float *__restrict__ bkmax,
                        double *__restrict__ btot, double *__restrict__ bmin, uint32_t *status,
                        uint64_t limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    float *const X = reinterpret_cast<float *>(sm + P2_SCR);
    float *const Y = reinterpret_cast<float *>(sm + P2_Y);
    float *const bs = reinterpret_cast<float *>(sm + P2_BETA);
    float *const lc = reinterpret_cast<float *>(sm + P2_LC);
    float *const part = reinterpret_cast<float *>(sm + P2_PART);  // [3][64 rows][2 halves]
    uint32_t *const slot = reinterpret_cast<uint32_t *>(sm + P2_SLOT);
    const uint32_t bar_tma = base + P2_BAR, bar_mma = base + P2_BAR + 8;

    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const int qd = warp & 3, hf = warp >> 2;
    const int lr = 32 * qd + lane;
    const int c0 = 32 * hf;
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int t0 = blk * kC;
    const size_t head = (size_t)bh * L;
    if (blk == 0 && bh == 0 && r == 0 && status) *status = 0u;

    __shared__ uint32_t abort_s;
    if (r == 0) {
        abort_s = 0u;
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_w);
        mbar_arrive_expect_tx(bar_tma, 6 * kT);
        tma_load_3d(base + P2_Q0, &tm_q, bar_tma, 0, t0, bh);
        tma_load_3d(base + P2_Q1, &tm_q, bar_tma, 64, t0, bh);
        tma_load_3d(base + P2_W0, &tm_w, bar_tma, 0, t0, bh);
        tma_load_3d(base + P2_W1, &tm_w, bar_tma, 64, t0, bh);
        tma_load_3d(base + P2_K0, &tm_k, bar_tma, 0, t0, bh);
        tma_load_3d(base + P2_K1, &tm_k, bar_tma, 64, t0, bh);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), 256);
        tmem_relinquish();
        tc_fence_before();
    }
    const float beta_r = (r < kC && t0 + r < L) ? beta[head + t0 + r] : 0.f;
    if (FOX && warp == 1) {
        const int ln = r - 32;
        const int ta = t0 + 2 * ln, tb = ta + 1;
        const float a = (ta < L) ? log_f[head + ta] : 0.f;
        const float b = ((tb < L) ? log_f[head + tb] : 0.f) + a;
        float run = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, run, o);
            if (ln >= o) run += n;
        }
        const float la = run - b + a, lb = run;
        lc[2 * ln] = la;
        lc[2 * ln + 1] = lb;
        const float tot = __shfl_sync(0xffffffffu, run, 31);
        const size_t row = (size_t)bh * Lp + t0 + 2 * ln;
        lc2[row] = kLog2e * la;
        lc2[row + 1] = kLog2e * lb;
        tail2[row] = kLog2e * (tot - la);
        tail2[row + 1] = kLog2e * (tot - lb);
        if (ln == 0) tot2[(size_t)bh * nblk + blk] = kLog2eD * (double)tot;
        // for the early-exit bounds, in fp64: the block's total of log f and the smallest of
        // its inclusive prefix sums
        const double da = (ta < L) ? (double)log_f[head + ta] : 0.0;
        const double db = ((tb < L) ? (double)log_f[head + tb] : 0.0) + da;
        double drun = db;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, drun, o);
            if (ln >= o) drun += n;
        }
        double dm = fmin(drun - db + da, drun);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dm = fmin(dm, __shfl_xor_sync(0xffffffffu, dm, o));
        if (ln == 31) btot[(size_t)bh * nblk + blk] = drun;
        if (ln == 0) bmin[(size_t)bh * nblk + blk] = dm;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t lane_off = (uint32_t)(32 * qd) << 16;

    auto wait_all = [&](uint32_t bar, uint32_t par) {
        if (r == 0) {
            bool ok = mbar_try_wait(bar, par);
            if (!ok) {
                const uint64_t tstart = cycles_now();
                while (!(ok = mbar_try_wait(bar, par)) &&
                       cycles_now() - tstart < ns_to_cycles(limit_ns)) {
                }
            }
            if (!ok) {
                report_status(status, kStatusTimeout);
                abort_s = 1u;
            }
        }
        __syncthreads();
        return abort_s == 0u;
    };

    // ---- MMA1: [Q; W] x [W; K]^T (bf16, K = 128: atoms at slot 0 / 3 and 1 / 4)
    if (r == 0) {
        const uint64_t t0s = cycles_now();
        bool ok = mbar_try_wait(bar_tma, 0);
        while (!ok && cycles_now() - t0s < ns_to_cycles(limit_ns)) ok = mbar_try_wait(bar_tma, 0);
        if (ok) {
            tc_fence_after();
            constexpr uint32_t ID = idesc16(128, 128, 1, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ha = kk < 4 ? P2_Q0 : P2_Q1, hb = kk < 4 ? P2_W0 : P2_W1;
                umma_bf16(tmem, sdesc_sw128(base + ha, 16, 1024) + 2 * (kk & 3),
                          sdesc_sw128(base + hb, 16, 1024) + 2 * (kk & 3), ID, kk > 0);
            }
        } else {
            report_status(status, kStatusTimeout);
        }
        umma_commit(bar_mma);
    }
    if (r < kC) bs[r] = beta_r;
    bool ok = wait_all(bar_mma, 0);
    if (ok) {
        tc_fence_after();
        float x[64];
        if (lr < kC) {
            const int i = lr;
            tmem_row32(tmem + lane_off + c0, x);
#pragma unroll
            for (int u = 0; u < 32; ++u)
                if (c0 + u > i) x[u] = 0.f;
            store_half16<true>(sm + P2_LQ, i, hf, x);
            // W row i, column half hf, to fp16 (MMA3 and MMA4y take fp16 operands)
            load_row_bf16(sm + (hf ? P2_W1 : P2_W0), i, x);
            store_half16<true>(sm + (hf ? P2_WH1 : P2_WH0), i, 0, x);
            store_half16<true>(sm + (hf ? P2_WH1 : P2_WH0), i, 1, x + 32);
        } else {
            const int s = lr - kC;
            tmem_row32(tmem + lane_off + c0, x);
            const float bsv = bs[s];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                float e[4];
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int v = c0 + 4 * q4 + e4;
                    e[e4] = (v > s) ? bsv * x[4 * q4 + e4] : 0.f;
                }
                *reinterpret_cast<float4 *>(X + s * XLD + c0 + 4 * q4) =
                    make_float4(e[0], e[1], e[2], e[3]);
            }
            tmem_row32(tmem + lane_off + 64 + c0, x);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (s <= c0 + j) x[j] = 0.f;
            store_half16<true>(sm + P2_RKT, s, hf, x);
        }
    }
    __syncthreads();

    // ---- A = (I + E)^{-1} D as A (rows s) and A^T (rows u), fp16
    if (ok) {
        blocked_unit_upper_inverse(X, Y, r);
        float a[32];
        if (lr < kC) {
            const int s = lr;
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const int u = c0 + 4 * u4;
                const float4 xv = *reinterpret_cast<const float4 *>(X + s * XLD + u);
                const float4 bv = *reinterpret_cast<const float4 *>(bs + u);
                a[4 * u4] = (u >= s) ? xv.x * bv.x : 0.f;
                a[4 * u4 + 1] = (u + 1 >= s) ? xv.y * bv.y : 0.f;
                a[4 * u4 + 2] = (u + 2 >= s) ? xv.z * bv.z : 0.f;
                a[4 * u4 + 3] = (u + 3 >= s) ? xv.w * bv.w : 0.f;
            }
        } else {
            const int u = lr - kC;
            const float bu = bs[u];
#pragma unroll
            for (int s2 = 0; s2 < 32; ++s2)
                a[s2] = (c0 + s2 <= u) ? X[(c0 + s2) * XLD + u] * bu : 0.f;
        }
        __syncthreads();  // the scratch overlays the A tiles
        if (lr < kC) store_half16<true>(sm + P2_A, lr, hf, a);
        else store_half16<true>(sm + P2_AT, lr - kC, hf, a);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA3: [A^T; A] x [Wh0 | Wh1 | Rk^T] (fp16, B MN-major at an 8 KB stride, N = 192)
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t a = sdesc_sw128(base + P2_AT, 16, 1024);
        const uint64_t b = sdesc_sw128(base + P2_WH0, kT, 1024);
        constexpr uint32_t ID = idesc16(128, 192, 0, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a + 2 * kk, b + 128 * kk, ID, kk > 0);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 1);
    if (ok) {
        tc_fence_after();
        float x[32];
        if (lr < kC) {
            // U row u, column half hf (64 values), and Khat^T row u, half hf (32 values)
            uint8_t *ut = sm + (hf ? P2_U1 : P2_U0);
            tmem_row32(tmem + lane_off + 64 * hf, x);
            store_half16<true>(ut, lr, 0, x);
            tmem_row32(tmem + lane_off + 64 * hf + 32, x);
            store_half16<true>(ut, lr, 1, x);
            tmem_row32(tmem + lane_off + 128 + c0, x);
            store_half16<true>(sm + P2_KHT, lr, hf, x);
        } else {
            uint8_t *vt = sm + (hf ? P2_V1 : P2_V0);
            tmem_row32(tmem + lane_off + 64 * hf, x);
            store_half16<true>(vt, lr - kC, 0, x);
            tmem_row32(tmem + lane_off + 64 * hf + 32, x);
            store_half16<true>(vt, lr - kC, 1, x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA4x: Lq U -> cols 0..127;  Q K^T - Lq Khat^T -> cols 128..191
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t a1 = sdesc_sw128(base + P2_LQ, 16, 1024);
        const uint64_t b1 = sdesc_sw128(base + P2_U0, kT, 1024);
        constexpr uint32_t ID1 = idesc16(128, 128, 0, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a1 + 2 * kk, b1 + 128 * kk, ID1, kk > 0);
        constexpr uint32_t IDQK = idesc16(128, 64, 1, false, false);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ha = kk < 4 ? P2_Q0 : P2_Q1, hb = kk < 4 ? P2_K0 : P2_K1;
            umma_bf16(tmem + 128, sdesc_sw128(base + ha, 16, 1024) + 2 * (kk & 3),
                      sdesc_sw128(base + hb, 16, 1024) + 2 * (kk & 3), IDQK, kk > 0);
        }
        const uint64_t bh2 = sdesc_sw128(base + P2_KHT, 1024, 1024);
        constexpr uint32_t IDC = idesc16(128, 64, 0, false, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + 128, a1 + 2 * kk, bh2 + 128 * kk, IDC, 1);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 0);

    const size_t blk_base = (size_t)bh * nblk + blk;
    const int kp_row = (kC + 128) * blk;  // first [k~; P_b] row of the block in its head
    if (ok && lr < kC) {
        tc_fence_after();
        const int i = lr;
        float x[32], y[32];
        // q~_i = q_i - (Lq U)_i, column half hf
        const uint8_t *qtile = sm + (hf ? P2_Q1 : P2_Q0);
        float qs = 0.f;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
            load_half_bf16(qtile, i, h2, y);
            tmem_row32(tmem + lane_off + 64 * hf + 32 * h2, x);
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] -= x[c];
            store_half16<false>(sm + (hf ? P2_OQ1 : P2_OQ0), i, h2, y);
            if (FOX) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float r16 = __bfloat162float(__float2bfloat16_rn(y[c]));
                    qs = fmaf(r16, r16, qs);
                }
            }
        }
        if (FOX) part[i * 2 + hf] = qs;
        // diagonal logits, log2 units, j <= i
        tmem_row32(tmem + lane_off + 128 + c0, x);
        const float lci = FOX ? lc[i] : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int jj = c0 + j;
            float v = scale_log2 * x[j];
            if (FOX) v += kLog2e * (lci - lc[jj]);
            x[j] = (jj <= i && t0 + jj < L) ? v : -INFINITY;
        }
        store_half16<true>(sm + P2_ODG, i, hf, x);
        if (FOX) {
            float dm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) dm = fmaxf(dm, __half2float(__float2half_rn(x[j])));
            part[128 + i * 2 + hf] = dm;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (r == 0 && ok) {
        tma_store_3d(&tm_qt_out, base + P2_OQ0, 0, t0, bh);
        tma_store_3d(&tm_qt_out, base + P2_OQ1, 64, t0, bh);
        tma_store_3d(&tm_dg_out, base + P2_ODG, 0, kC * blk, bh);
    }
    if (FOX && ok && hf == 0 && lr < kC) {
        // (q~, table) row lr: combine the two half-row partials
        const size_t row = (size_t)bh * Lp + t0 + lr;
        qn[row] = sqrtf(part[lr * 2] + part[lr * 2 + 1]);
        dmax[row] = fmaxf(part[128 + lr * 2], part[128 + lr * 2 + 1]);
    }

    // ---- MMA4y: W^T V' -> cols 0..127 (rows n of P_b); Rk V' -> cols 128..255 (rows j)
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t bv = sdesc_sw128(base + P2_V0, P2_V1 - P2_V0, 1024);
        const uint64_t aw = sdesc_sw128(base + P2_WH0, kT, 1024);
        constexpr uint32_t IDP = idesc16(128, 128, 0, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, aw + 128 * kk, bv + 128 * kk, IDP, kk > 0);
        const uint64_t ar = sdesc_sw128(base + P2_RKT, kT, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + 128, ar + 128 * kk, bv + 128 * kk, IDP, kk > 0);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 1);
    if (ok) {
        tc_fence_after();
        float x[32];
        // P_b row n = lr, column half hf: delta - (W^T V')_n
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
            const int cb = 64 * hf + 32 * h2;
            tmem_row32(tmem + lane_off + cb, x);
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = (cb + c == lr ? 1.f : 0.f) - x[c];
            uint8_t *pt = sm + (lr < kC ? (hf ? P2_OP01 : P2_OP00) : (hf ? P2_OP11 : P2_OP10));
            store_half16<false>(pt, lr & (kC - 1), h2, x);
        }
        if (lr < kC) {
            // k~_j = k_j - (Rk V')_j
            const int j = lr;
            float y[32];
            const uint8_t *ktile = sm + (hf ? P2_K1 : P2_K0);
            float ks = 0.f;
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {
                load_half_bf16(ktile, j, h2, y);
                tmem_row32(tmem + lane_off + 128 + 64 * hf + 32 * h2, x);
#pragma unroll
                for (int c = 0; c < 32; ++c) y[c] -= x[c];
                store_half16<false>(sm + (hf ? P2_OK1 : P2_OK0), j, h2, y);
                if (FOX) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float r16 = __bfloat162float(__float2bfloat16_rn(y[c]));
                        ks = fmaf(r16, r16, ks);
                    }
                }
            }
            // rows past L are padding: they take part in no logit
            if (FOX) part[256 + j * 2 + hf] = (t0 + j < L) ? ks : 0.f;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (r == 0 && ok) {
        tma_store_3d(&tm_kp_out, base + P2_OK0, 0, kp_row, bh);
        tma_store_3d(&tm_kp_out, base + P2_OK1, 64, kp_row, bh);
        tma_store_3d(&tm_kp_out, base + P2_OP00, 0, kp_row + kC, bh);
        tma_store_3d(&tm_kp_out, base + P2_OP01, 64, kp_row + kC, bh);
        tma_store_3d(&tm_kp_out, base + P2_OP10, 0, kp_row + 2 * kC, bh);
        tma_store_3d(&tm_kp_out, base + P2_OP11, 64, kp_row + 2 * kC, bh);
    }
    if (FOX && ok && warp == 2) {
        // largest |k~_j| of the block: lane l takes rows l and l + 32
        const float *kpart = part + 256;
        float m = fmaxf(sqrtf(kpart[lane * 2] + kpart[lane * 2 + 1]),
                        sqrtf(kpart[(lane + 32) * 2] + kpart[(lane + 32) * 2 + 1]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) bkmax[blk_base] = m;
    }
    if (r == 0) bulk_wait_all();  // the stores have read their tiles and written the outputs
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// (heads, L rows, 64 columns) bf16 input, 64-row boxes, 128-byte swizzle; rows past L
// read as zero.
bool make_input_map(CUtensorMap *m, const void *ptr, int L, int heads) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)L * kD * 2};
    cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kC, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (heads, L rows, 128 columns) bf16, (64 columns, 64 rows) boxes, 128-byte swizzle (the
// inputs, and q~ and [k~; P_b] with their row counts in place of L).
bool make_input_map128(CUtensorMap *m, const void *ptr, int L, int heads) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)L, (cuuint64_t)heads};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)L * 128 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Head size 128, bf16 inputs: the tensor-core preparation into the d128_tc_layout workspace.
cudaError_t launch_ut_prepare_tc128(const void *q, const void *k, const void *w,
                                    const float *beta, const float *log_f, int BH, int L,
                                    float scale, void *ws, uint64_t limit_ns,
                                    cudaStream_t stream) {
    const bool fox = log_f != nullptr;
    const D128TcLayout lay = d128_tc_layout(1, BH, L, fox);
    char *basep = static_cast<char *>(ws);
    CUtensorMap tq, tk, tw, tqto, tkpo, tdgo;
    if (!make_input_map128(&tq, q, L, BH) || !make_input_map128(&tk, k, L, BH) ||
        !make_input_map128(&tw, w, L, BH) ||
        !make_input_map128(&tqto, basep + lay.off_qt, lay.Lp, BH) ||
        !make_input_map128(&tkpo, basep + lay.off_kp, lay.nblk * (kC + 128), BH) ||
        !make_map_f16(&tdgo, basep + lay.off_dg, lay.nblk * kC, BH, kC))
        return cudaErrorInvalidValue;
    auto kern = fox ? ut_prepare_tc128_kernel<true> : ut_prepare_tc128_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)k2SmemBytes);
    if (err != cudaSuccess) return err;
    kern<<<dim3(lay.nblk, BH), kThreads, k2SmemBytes, stream>>>(
        tq, tk, tw, tqto, tkpo, tdgo, beta, log_f, L, lay.Lp, lay.nblk, scale * kLog2e,
        fox ? reinterpret_cast<float *>(basep + lay.off_lc2) : nullptr,
        fox ? reinterpret_cast<float *>(basep + lay.off_tail2) : nullptr,
        fox ? reinterpret_cast<double *>(basep + lay.off_tot2) : nullptr,
        fox ? reinterpret_cast<float *>(basep + lay.off_qn) : nullptr,
        fox ? reinterpret_cast<float *>(basep + lay.off_dmax) : nullptr,
        fox ? reinterpret_cast<float *>(basep + lay.off_bkmax) : nullptr,
        fox ? reinterpret_cast<double *>(basep + lay.off_btot) : nullptr,
        fox ? reinterpret_cast<double *>(basep + lay.off_bmin) : nullptr,
        reinterpret_cast<uint32_t *>(basep), limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_ut_prepare_tc(const void *q, const void *k, const void *w, const float *beta,
                                 const float *log_f, int BH, int L, float scale, void *ws,
                                 uint64_t limit_ns, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 2, log_f != nullptr);
    char *basep = static_cast<char *>(ws);
    CUtensorMap tq, tk, tw;
    if (!make_input_map(&tq, q, L, BH) || !make_input_map(&tk, k, L, BH) ||
        !make_input_map(&tw, w, L, BH))
        return cudaErrorInvalidValue;
    const bool fox = log_f != nullptr;
    CUtensorMap tqto, tkpo, tdgo;  // outputs: q~, [k~; P_b] rows and the fp16 table (64-row boxes)
    if (!make_map_bf16(&tqto, basep + lay.off_qt, lay.Lp, BH, kC) ||
        !make_map_bf16(&tkpo, basep + lay.off_kp, lay.nblk * 2 * kC, BH, kC) ||
        !make_map_f16(&tdgo, basep + lay.off_dg, lay.nblk * kC, BH, kC))
        return cudaErrorInvalidValue;
    auto kern = fox ? ut_prepare_tc_kernel<true> : ut_prepare_tc_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    dim3 grid(lay.nblk, BH);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(
        tq, tk, tw, tqto, tkpo, tdgo, beta, log_f, L, lay.Lp, lay.nblk, scale * kLog2e,
        fox ? reinterpret_cast<float *>(basep + lay.off_qn) : nullptr,
        fox ? reinterpret_cast<float *>(basep + lay.off_dmax) : nullptr,
        fox ? reinterpret_cast<float *>(basep + lay.off_bkmax) : nullptr,
        fox ? reinterpret_cast<double *>(basep + lay.off_btot) : nullptr,
        fox ? reinterpret_cast<double *>(basep + lay.off_bmin) : nullptr,
        reinterpret_cast<uint32_t *>(basep), limit_ns);
    return cudaGetLastError();
}

}  // namespace path
