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
// (I + E)^{-1} is formed blockwise: the four 16 x 16 diagonal blocks by back-substitution,
// then X12 = -X11 E12 X22 for the 16-blocks and for the 32-blocks (fp32). Every factor is
// bounded (X_su = A_su / beta_u), so no intermediate grows.
//
// tcgen05.mma groups, all M = 128, with 64x64 16-bit tiles in 128-byte-swizzled shared
// memory (K-major tiles stacked in M must be adjacent; MN-major atoms use the LBO stride):
//   MMA1 (bf16):  [Q; W] x [W; K]^T          -> Q W^T | (Q K^T)  /  W W^T | W K^T
//   MMA3 (fp16):  [A^T; A] x [W | Rk^T]      -> U | Khat^T       /  V' | (unused)
//   MMA4x:        Lq x U (fp16)              -> Lq U
//                 Q x K^T (bf16) - Lq x Khat^T (fp16), one accumulator -> diag logits
//   MMA4y (fp16): [W^T; Rk] x V'             -> W^T V'          /  Rk V'
// Second-level operands are fp16 (11-bit significand; all bounded, |A_su| <= 4), fp32
// accumulation. One CTA of 128 threads per (block, head), thread r owns TMEM lane r,
// thread 0 issues the TMA loads and the MMAs. 128 TMEM columns and 64 KB of tiles, so
// three CTAs share an SM.
#include "common.cuh"

namespace path {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kT = 8192;  // one 64 x 64 16-bit tile

// Tile slots (from the 1024-aligned base). Q, W, K adjacent (MMA1 A = [Q; W], B = [W; K]);
// AT, A adjacent (MMA3 A). U, KhT, V reuse the slots of AT, A and the solve scratch.
constexpr uint32_t T_Q = 0 * kT, T_W = 1 * kT, T_K = 2 * kT, T_RKT = 3 * kT, T_LQ = 4 * kT,
                   T_AT = 5 * kT, T_A = 6 * kT, T_U = 5 * kT, T_KHT = 6 * kT, T_V = 7 * kT;
constexpr uint32_t SCR = 5 * kT;           // solve scratch (E/X fp32 + Y) overlays slots 5-7
constexpr int XLD = 68;
constexpr uint32_t Y_OFF = SCR + 64 * XLD * 4;
constexpr int YLD = 36;
constexpr uint32_t BAR_OFF = 8 * kT;       // 2 mbarriers
constexpr uint32_t SLOT_OFF = BAR_OFF + 16;
constexpr uint32_t BETA_OFF = SLOT_OFF + 16;
constexpr uint32_t LC_OFF = BETA_OFF + 256;
constexpr uint32_t kSmemBytes = LC_OFF + 256 + 1024;
constexpr uint32_t kTmemCols = 128;

static_assert(Y_OFF + 32 * YLD * 4 <= 8 * kT, "solve scratch fits in slots 5-7");

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

// Writes 64 fp32 values as one 16-bit row (fp16 or bf16) of a swizzled tile.
template <bool HALF>
__device__ __forceinline__ void store_row16(uint8_t *tile, int row, const float *x) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 u;
        const float *s = x + 8 * c;
        if (HALF) {
            u.x = pack_h2(s[0], s[1]); u.y = pack_h2(s[2], s[3]);
            u.z = pack_h2(s[4], s[5]); u.w = pack_h2(s[6], s[7]);
        } else {
            u.x = pack_bf16x2(s[0], s[1]); u.y = pack_bf16x2(s[2], s[3]);
            u.z = pack_bf16x2(s[4], s[5]); u.w = pack_bf16x2(s[6], s[7]);
        }
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, c)) = u;
    }
}

// Reads one bf16 row of a swizzled tile as 64 fp32 values.
__device__ __forceinline__ void load_row_bf16(const uint8_t *tile, int row, float *x) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tile + sw128_offset(row, c));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            x[8 * c + 2 * e] = f.x;
            x[8 * c + 2 * e + 1] = f.y;
        }
    }
}

// 64 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_row64(uint32_t taddr, float *x) {
    uint32_t a[32], b[32];
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        x[j] = __uint_as_float(a[j]);
        x[32 + j] = __uint_as_float(b[j]);
    }
}

__device__ __forceinline__ void store_global_row(__nv_bfloat16 *dst, const float *y) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        d[c] = make_uint4(pack_bf16x2(y[8 * c], y[8 * c + 1]), pack_bf16x2(y[8 * c + 2], y[8 * c + 3]),
                          pack_bf16x2(y[8 * c + 4], y[8 * c + 5]),
                          pack_bf16x2(y[8 * c + 6], y[8 * c + 7]));
}

// (I + E)^{-1} in place over E (upper triangle; E is zero on and below the diagonal),
// all 128 threads. On return X[s][u] (s <= u) holds the inverse.
__device__ __forceinline__ void blocked_unit_upper_inverse(float *X, float *Y, int r) {
    // level 0: the four 16 x 16 diagonal blocks, one column per thread
    float x[16];
    const int u = r & 63, b0 = (u >> 4) << 4, lu = u & 15;
    if (r < 64) {
#pragma unroll
        for (int l = 15; l >= 0; --l) {
            float acc = 0.f;
#pragma unroll
            for (int m = l + 1; m < 16; ++m) acc = fmaf(X[(b0 + l) * XLD + b0 + m], x[m], acc);
            x[l] = (l == lu) ? 1.f : ((l < lu) ? -acc : 0.f);
        }
    }
    __syncthreads();
    if (r < 64) {
#pragma unroll
        for (int l = 0; l < 16; ++l) X[(b0 + l) * XLD + u] = x[l];
    }
    __syncthreads();
    // level 1: X[16p', 16p'+16..] = -X11 E12 X22 for the two 32-blocks p
    {
        const int p = r >> 6, q = r & 63, i = q >> 2, c0 = (q & 3) * 4;
        const int o = 32 * p;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float e = X[(o + i) * XLD + o + 16 + m];
            const float4 xr = *reinterpret_cast<const float4 *>(X + (o + 16 + m) * XLD + o + 16 + c0);
            y[0] = fmaf(e, xr.x, y[0]); y[1] = fmaf(e, xr.y, y[1]);
            y[2] = fmaf(e, xr.z, y[2]); y[3] = fmaf(e, xr.w, y[3]);
        }
        *reinterpret_cast<float4 *>(Y + (16 * p + i) * YLD + c0) = make_float4(y[0], y[1], y[2], y[3]);
        __syncthreads();
        float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float xv = X[(o + i) * XLD + o + m];
            const float4 yr = *reinterpret_cast<const float4 *>(Y + (16 * p + m) * YLD + c0);
            z[0] = fmaf(xv, yr.x, z[0]); z[1] = fmaf(xv, yr.y, z[1]);
            z[2] = fmaf(xv, yr.z, z[2]); z[3] = fmaf(xv, yr.w, z[3]);
        }
        *reinterpret_cast<float4 *>(X + (o + i) * XLD + o + 16 + c0) =
            make_float4(-z[0], -z[1], -z[2], -z[3]);
    }
    __syncthreads();
    // level 2: X[0:32, 32:64] = -X[0:32, 0:32] E[0:32, 32:64] X[32:64, 32:64]
    {
        const int i = r >> 2, c0 = (r & 3) * 8;
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 8
        for (int m = 0; m < 32; ++m) {
            const float e = X[i * XLD + 32 + m];
            const float4 a = *reinterpret_cast<const float4 *>(X + (32 + m) * XLD + 32 + c0);
            const float4 b = *reinterpret_cast<const float4 *>(X + (32 + m) * XLD + 36 + c0);
            y[0] = fmaf(e, a.x, y[0]); y[1] = fmaf(e, a.y, y[1]);
            y[2] = fmaf(e, a.z, y[2]); y[3] = fmaf(e, a.w, y[3]);
            y[4] = fmaf(e, b.x, y[4]); y[5] = fmaf(e, b.y, y[5]);
            y[6] = fmaf(e, b.z, y[6]); y[7] = fmaf(e, b.w, y[7]);
        }
        *reinterpret_cast<float4 *>(Y + i * YLD + c0) = make_float4(y[0], y[1], y[2], y[3]);
        *reinterpret_cast<float4 *>(Y + i * YLD + c0 + 4) = make_float4(y[4], y[5], y[6], y[7]);
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 8
        for (int m = 0; m < 32; ++m) {
            const float xv = X[i * XLD + m];
            const float4 a = *reinterpret_cast<const float4 *>(Y + m * YLD + c0);
            const float4 b = *reinterpret_cast<const float4 *>(Y + m * YLD + c0 + 4);
            y[0] = fmaf(xv, a.x, y[0]); y[1] = fmaf(xv, a.y, y[1]);
            y[2] = fmaf(xv, a.z, y[2]); y[3] = fmaf(xv, a.w, y[3]);
            y[4] = fmaf(xv, b.x, y[4]); y[5] = fmaf(xv, b.y, y[5]);
            y[6] = fmaf(xv, b.z, y[6]); y[7] = fmaf(xv, b.w, y[7]);
        }
        *reinterpret_cast<float4 *>(X + i * XLD + 32 + c0) = make_float4(-y[0], -y[1], -y[2], -y[3]);
        *reinterpret_cast<float4 *>(X + i * XLD + 36 + c0) = make_float4(-y[4], -y[5], -y[6], -y[7]);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 3)
ut_prepare_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_w, const float *__restrict__ beta,
                     const float *__restrict__ log_f, int L, int Lp, int nblk, float scale_log2,
                     __nv_bfloat16 *__restrict__ qt, __nv_bfloat16 *__restrict__ kp,
                     __half *__restrict__ dg, uint32_t *status, uint64_t limit_ns) {
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

    const int r = threadIdx.x, warp = r >> 5;
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
    if (log_f != nullptr && warp == 1) {
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
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    // bounded wait used by every thread; a timeout skips the remaining work
    auto wait_all = [&](uint32_t bar, uint32_t par) {
        bool ok = mbar_try_wait(bar, par);
        if (!ok) {
            const uint64_t tstart = cycles_now();
            while (!(ok = mbar_try_wait(bar, par)) && cycles_now() - tstart < ns_to_cycles(limit_ns)) {
            }
        }
        if (!ok) {
            report_status(status, kStatusTimeout);
            abort_s = 1u;
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
        float x[64];
        if (r < kC) {
            // row i of Q W^T -> Lq (u <= i), fp16
            tmem_row64(tmem + lane_off, x);
#pragma unroll
            for (int u = 0; u < 64; ++u)
                if (u > r) x[u] = 0.f;
            store_row16<true>(sm + T_LQ, r, x);
        } else {
            const int s = r - kC;
            // row s of W W^T -> E = beta_s G[s][v] for v > s (fp32 scratch)
            tmem_row64(tmem + lane_off, x);
            const float bsv = bs[s];
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
                float e[4];
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int v = 4 * q4 + e4;
                    e[e4] = (v > s) ? bsv * x[v] : 0.f;
                }
                *reinterpret_cast<float4 *>(X + s * XLD + 4 * q4) = make_float4(e[0], e[1], e[2], e[3]);
            }
            // row s of W K^T -> Rk^T (s > j), fp16
            tmem_row64(tmem + lane_off + 64, x);
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (s <= j) x[j] = 0.f;
            store_row16<true>(sm + T_RKT, s, x);
            // W to fp16 in place (MMA1 has completed; later MMAs take fp16 operands)
            load_row_bf16(sm + T_W, s, x);
            store_row16<true>(sm + T_W, s, x);
        }
    }
    __syncthreads();

    // ---- A = (I + E)^{-1} D, then A (rows s) and A^T (rows u) as fp16 tiles
    if (ok) {
        blocked_unit_upper_inverse(X, Y, r);
        float a[64];
        if (r < kC) {
            const int s = r;   // row s: A[s][u] = X[s][u] beta_u, u >= s
#pragma unroll
            for (int u4 = 0; u4 < 16; ++u4) {
                const float4 xv = *reinterpret_cast<const float4 *>(X + s * XLD + 4 * u4);
                const float4 bv = *reinterpret_cast<const float4 *>(bs + 4 * u4);
                const int u = 4 * u4;
                a[u] = (u >= s) ? xv.x * bv.x : 0.f;
                a[u + 1] = (u + 1 >= s) ? xv.y * bv.y : 0.f;
                a[u + 2] = (u + 2 >= s) ? xv.z * bv.z : 0.f;
                a[u + 3] = (u + 3 >= s) ? xv.w * bv.w : 0.f;
            }
        } else {
            const int u = r - kC;  // column u: A[s][u], s <= u
            const float bu = bs[u];
#pragma unroll
            for (int s2 = 0; s2 < 64; ++s2) a[s2] = (s2 <= u) ? X[s2 * XLD + u] * bu : 0.f;
        }
        __syncthreads();  // the scratch overlays the A tiles
        if (r < kC) store_row16<true>(sm + T_A, r, a);
        else store_row16<true>(sm + T_AT, r - kC, a);
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
        float x[64];
        if (r < kC) {
            tmem_row64(tmem + lane_off, x);       // U row u
            store_row16<true>(sm + T_U, r, x);
            tmem_row64(tmem + lane_off + 64, x);  // Khat^T row u
            store_row16<true>(sm + T_KHT, r, x);
        } else {
            tmem_row64(tmem + lane_off, x);       // V' row s
            store_row16<true>(sm + T_V, r - kC, x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA4x: Lq U -> cols 0..63;  Q K^T - Lq Khat^T -> cols 64..127
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t a1 = sdesc_sw128(base + T_LQ, 16, 1024);
        const uint64_t b1 = sdesc_sw128(base + T_U, 1024, 1024);
        constexpr uint32_t ID1 = idesc16(128, 64, 0, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a1 + 2 * kk, b1 + 128 * kk, ID1, kk > 0);
        const uint64_t aq = sdesc_sw128(base + T_Q, 16, 1024);
        const uint64_t bk = sdesc_sw128(base + T_K, 16, 1024);
        constexpr uint32_t IDQK = idesc16(128, 64, 1, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + 64, aq + 2 * kk, bk + 2 * kk, IDQK, kk > 0);
        const uint64_t bh2 = sdesc_sw128(base + T_KHT, 1024, 1024);
        constexpr uint32_t IDC = idesc16(128, 64, 0, false, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + 64, a1 + 2 * kk, bh2 + 128 * kk, IDC, 1);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 0);

    const size_t blk_base = (size_t)bh * nblk + blk;
    __nv_bfloat16 *kp_blk = kp + blk_base * (2 * kC) * kD;
    if (ok && r < kC) {
        tc_fence_after();
        const int i = r;
        float x[64], y[64];
        // q~_i = q_i - (Lq U)_i
        load_row_bf16(sm + T_Q, i, y);
        tmem_row64(tmem + lane_off, x);
#pragma unroll
        for (int c = 0; c < 64; ++c) y[c] -= x[c];
        store_global_row(qt + ((size_t)bh * Lp + t0 + i) * kD, y);
        // diagonal logits, log2 units, j <= i
        tmem_row64(tmem + lane_off + 64, x);
        const float lci = (log_f != nullptr) ? lc[i] : 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            float v = scale_log2 * x[j];
            if (log_f != nullptr) v += kLog2e * (lci - lc[j]);
            x[j] = (j <= i && t0 + j < L) ? v : -INFINITY;
        }
        uint4 *dd = reinterpret_cast<uint4 *>(dg + (blk_base * kC + i) * kC);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            dd[c] = make_uint4(pack_h2(x[8 * c], x[8 * c + 1]), pack_h2(x[8 * c + 2], x[8 * c + 3]),
                               pack_h2(x[8 * c + 4], x[8 * c + 5]), pack_h2(x[8 * c + 6], x[8 * c + 7]));
    } else if (ok && warp >= 2) {
        // warps 2-3: the lanes of MMA4x rows 64..127 hold nothing; keep the warp collective
    }
    tc_fence_before();
    __syncthreads();

    // ---- MMA4y: [W^T; Rk] x V' (fp16, A and B MN-major) -> cols 0..63
    if (r == 0 && ok) {
        tc_fence_after();
        const uint64_t a2 = sdesc_sw128(base + T_W, T_RKT - T_W, 1024);
        const uint64_t b2 = sdesc_sw128(base + T_V, 1024, 1024);
        constexpr uint32_t ID2 = idesc16(128, 64, 0, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a2 + 128 * kk, b2 + 128 * kk, ID2, kk > 0);
    }
    if (r == 0) umma_commit(bar_mma);
    if (ok) ok = wait_all(bar_mma, 1);
    if (ok) {
        tc_fence_after();
        float x[64];
        tmem_row64(tmem + lane_off, x);
        if (r < kC) {
            // P_b row n = r: delta - (W^T V')_n
#pragma unroll
            for (int c = 0; c < 64; ++c) x[c] = (c == r ? 1.f : 0.f) - x[c];
            store_global_row(kp_blk + (kC + r) * kD, x);
        } else {
            // k~_j = k_j - (Rk V')_j
            const int j = r - kC;
            float y[64];
            load_row_bf16(sm + T_K, j, y);
#pragma unroll
            for (int c = 0; c < 64; ++c) y[c] -= x[c];
            store_global_row(kp_blk + j * kD, y);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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

}  // namespace

cudaError_t launch_ut_prepare_tc(const void *q, const void *k, const void *w, const float *beta,
                                 const float *log_f, int BH, int L, float scale, void *ws,
                                 uint64_t limit_ns, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 2, log_f != nullptr);
    char *basep = static_cast<char *>(ws);
    CUtensorMap tq, tk, tw;
    if (!make_input_map(&tq, q, L, BH) || !make_input_map(&tk, k, L, BH) ||
        !make_input_map(&tw, w, L, BH))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(ut_prepare_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    dim3 grid(lay.nblk, BH);
    ut_prepare_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(
        tq, tk, tw, beta, log_f, L, lay.Lp, lay.nblk, scale * kLog2e,
        reinterpret_cast<__nv_bfloat16 *>(basep + lay.off_qt),
        reinterpret_cast<__nv_bfloat16 *>(basep + lay.off_kp),
        reinterpret_cast<__half *>(basep + lay.off_dg), reinterpret_cast<uint32_t *>(basep),
        limit_ns);
    return cudaGetLastError();
}

}  // namespace path
