// Backward query pass of PaTH attention and PaTH-FoX on tcgen05 tensor cores (bf16 inputs).
//
// The pages give no backward (review "거리에서 경로로, PaTH Attention" §9 and technical
// summary "技術要約: PaTH Attention" §3 say the block-wise algorithm is what makes training
// efficient). The gradient is the chain rule through the block form of the forward, as in
// backward.cu: with X_{a,b} the rows of query block a carried down to key block b
// (X_{a,a-1} = Q~_a, X_{a,b-1} = X_{a,b} P_b^T), T_ab = X_{a,b} K~_b^T,
// dS_ij = p_ij (dout_i . v_j - dout_i . out_i) and dT = scale dS:
//     dv_b  += p_ab^T dout_a            dK~_b += dT_ab^T X_{a,b}
//     G_b    = G_{b-1} P_b + dT_ab K~_b  (G_{-1} = 0)      dP_b += G_{b-1}^T X_{a,b}
//     dQ~_a  = G_{a-1}
// The carried rows run right to left and their gradient left to right, and P_b can be
// singular (beta = 1), so the walk keeps X_{a,b} and dT_ab in a workspace stash (bf16,
// the operands the tensor cores read) and walks back over it.
//
// A CTA owns the 128-row tile of query blocks A0 = 2t and A1 = 2t + 1 of one head (the
// forward's tile). Pass 1 visits key blocks b = 2t+1, 2t, ..., 0:
//   b = 2t+1: A1's diagonal block (logits from the forward preparation's table);
//   b = 2t:   A0's diagonal block and A1's first off-diagonal block;
//   b < 2t:   both query blocks off-diagonal.
// Per step, M = 128 MMAs with bf16 operands in 128-byte-swizzled shared memory and fp32
// accumulators in TMEM:
//   [S | X'] = X [K~_b; P_b]^T   (N = 128: logits and the carried rows for the next block)
//   O_v      = dout V_b^T        (N = 64)
//   D_kv     = [p^T; dT^T] [X | dout]   (M = 128, N = 128, K = 128 tile rows: the
//              off-diagonal blocks of D_kv are dv_b's and dK~_b's contributions; the
//              diagonal ones are unused)
// Pass 2 visits b = 0 .. 2t with G split into a bf16 head and tail (G = G_hi + G_lo,
// so the recursion keeps about 16 significant bits):
//   G'  = G_hi P_b + G_lo P_b + dT_b K~_b          (N = 64, K = 64 each)
//   D_p = [G_hi^T; G_lo^T] X_b                      (M = 128, K = 128: the two 64-row halves
//                                                    sum to dP_b's contribution)
// dK~, dv and dP_b gather by fp32 vector atomics; dq~ and the diagonal dT are written by
// their owners. The block pass of backward.cu then takes dq~, dk~, dP_b and the diagonal
// dT to q, k, w and beta.
//
// Warp roles (416 threads): warps 0-7 read the TMEM lanes of their rows after each MMA1
// (softmax gradient, p, dT, the carried rows) and after each pass-2 MMA (G), two warps per
// lane quadrant, each on one 32-column half of every row; warps 8-11 drain D_kv / D_p into
// the gathered gradients; warp 12 allocates TMEM and its lane 0 issues
// every TMA load and MMA. Every wait is bounded; on a timeout the CTA records
// PATH_ERR_TIMEOUT in the workspace status word, every role leaves its loop, the issuing
// lane waits for its copies and MMAs in flight, and TMEM is freed.
#include "common.cuh"

namespace path {

cudaError_t launch_ut_prepare_tc(const void *q, const void *k, const void *w, const float *beta,
                                 const float *log_f, int BH, int L, float scale, void *ws,
                                 uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_bwd_block_mm(const void *q, const void *k, const void *w, const float *beta,
                                const float *dqt, const float *dkt, const float *dP,
                                const float *dTd, float *dq, float *dk, float *dw,
                                float *dbeta, int BH, int L, int Lp, int nblk,
                                cudaStream_t stream);
cudaError_t launch_bwd_fox_sums(const float *log_f, int BH, int L, int Lp, int nblk, float *loc,
                                double *cb, cudaStream_t stream);
cudaError_t launch_bwd_fox_dlogf(const float *rsum, const float *csum, int BH, int L, int Lp,
                                 float *dlogf, cudaStream_t stream);

namespace {

constexpr int kThr = 416;
constexpr uint32_t kT128 = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kT64 = 64 * 128;    // 64 rows x 64 bf16
constexpr int NS1 = 4, NS2 = 3;
constexpr uint32_t kStage1 = kT128 + kT64;  // [K~_b; P_b] and V_b
constexpr uint32_t kStage2 = 3 * kT128;     // [K~_b; P_b], stash X_b, stash dT_b
constexpr int kCsLd = 129;                  // FoX: transposed dS buffer stride (floats)

// byte offsets from the 1024-aligned base
constexpr uint32_t S_XB0 = 0, S_XB1 = kT128, S_DO = 2 * kT128, S_PT = 3 * kT128,
                   S_DT = 4 * kT128, S_STG1 = 5 * kT128;
constexpr uint32_t S_STG2 = S_DO;  // pass 2: dout, p, dT and the pass-1 ring are free
constexpr uint32_t S_END = S_STG1 + NS1 * kStage1;
static_assert(S_STG2 + NS2 * kStage2 <= S_END, "pass-2 ring fits");
constexpr uint32_t S_CS = S_END;  // FoX only
constexpr uint32_t kCsBytes = 64 * kCsLd * 4;
// FoX: a constant K-major B operand of 16 rows x 128 columns whose row 0 is all ones;
// [p^T; dS^T] times it gives in column 0 the column sums of dS over the tile's rows
constexpr uint32_t S_ONES = (S_CS + kCsBytes + 1023u) & ~1023u;
constexpr uint32_t kOnesBytes = 16 * 128 * 2;
template <bool FOX>
__host__ __device__ constexpr uint32_t bwd_tc_smem_end() { return FOX ? S_ONES + kOnesBytes : S_END; }

// barrier indices
constexpr int B_FULL1 = 0, B_FULL2 = B_FULL1 + NS1, B_LD0 = B_FULL2 + NS2, B_M1 = B_LD0 + 1,
              B_EPI = B_M1 + 1, B_M2 = B_EPI + 1, B_KVF = B_M2 + 2, B_M1B = B_KVF + 2,
              B_EPIB = B_M1B + 1, B_M2B = B_EPIB + 1, B_DPF = B_M2B + 2, B_FIN = B_DPF + 2,
              B_CSA = B_FIN + 1, B_CSB = B_CSA + 1, NBAR = B_CSB + 1;

// TMEM columns
constexpr uint32_t C_SX = 0, C_OV = 128, C_KV0 = 256, C_KV1 = 384;  // pass 1
constexpr uint32_t C_CS0 = 192, C_CS1 = 208;                        // pass 1, FoX: dS column sums
constexpr uint32_t C_G = 0, C_DP0 = 256, C_DP1 = 384;                // pass 2

template <bool FOX>
constexpr uint32_t bwd_tc_smem() {
    return 1024 + bwd_tc_smem_end<FOX>() + NBAR * 8 + 16;
}

__host__ __device__ constexpr uint32_t idesc_b16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Wait {
    volatile uint32_t *abort;
    uint32_t *status;
    uint64_t limit_ns;
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = cycles_now(), lim = ns_to_cycles(limit_ns);
        for (;;) {
            if (mbar_try_wait(bar, parity)) return true;
            if (*abort) return false;
            if (cycles_now() - t0 > lim) {
                report_status(status, kStatusTimeout);
                *abort = 1u;
                return false;
            }
        }
    }
};

// Registers per thread after the split (launch: 128 for all 416 threads, the share of a
// sub-partition holding four warps); rows 8 x 152 + drains 4 x 80 + issuer 104 <= 13 x 128.
constexpr int kRegRow = 152, kRegDrain = 80, kRegIssue = 104;
static_assert(8 * kRegRow + 4 * kRegDrain + kRegIssue <= 13 * 128, "register split");
template <int N>
__device__ __forceinline__ void reg_alloc_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// 32 TMEM columns of this thread's lane as floats (waits for the load).
__device__ __forceinline__ void tld32(uint32_t taddr, float *x) {
    uint32_t u[32];
    tmem_ld32(taddr, u);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(u[j]);
}

// 32 values as bf16 into half h (columns 32h .. 32h + 31) of row r of a swizzled tile.
__device__ __forceinline__ void st_row_half(uint8_t *tile, int r, int h, const float *x) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float *s = x + 8 * c;
        *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 4 * h + c)) =
            make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]),
                       pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
    }
}

// One CTA per (tile t of query blocks 2t, 2t+1; head). nblk: real blocks of the head;
// nbe: blocks rounded up to even (the forward preparation's layout); Lp = 64 nblk.
template <bool FOX>
__global__ void __launch_bounds__(kThr, 1)
bwd_query_tc_kernel(const __grid_constant__ CUtensorMap tm_qt,
                    const __grid_constant__ CUtensorMap tm_kp,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_st,
                    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                    const float *__restrict__ lse, const __half *__restrict__ dg,
                    __nv_bfloat16 *__restrict__ stash, float *__restrict__ dqt,
                    float *__restrict__ dkt, float *__restrict__ dP, float *__restrict__ dTd,
                    float *__restrict__ dv, const float *__restrict__ loc,
                    const double *__restrict__ cb, float *__restrict__ rsum,
                    float *__restrict__ csum, int L, int Lp, int nblk, int nbe, float scale,
                    float scale_log2, uint32_t *status, uint64_t limit_ns, int heads_fast) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    constexpr uint32_t S_BAR = bwd_tc_smem_end<FOX>();
    auto bar = [&](int i) { return base + S_BAR + 8u * (uint32_t)i; };
    uint32_t *const tslot = reinterpret_cast<uint32_t *>(sm + S_BAR + 8 * NBAR);
    volatile uint32_t *const abort_f = tslot + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int npair = nbe >> 1;
    // longest walks first, heads fastest or head by head (heads_fastest)
    const int t = npair - 1 - (int)(heads_fast ? blockIdx.y : blockIdx.x);
    const int bh = heads_fast ? blockIdx.x : blockIdx.y;
    const int steps1 = 2 * t + 2, steps2 = 2 * t + 1;
    const size_t rec0 = (size_t)t * t;  // first stash record of this tile within the head
    const Wait wait{abort_f, status, limit_ns};
    // in the warp-collective roles every lane takes the same branch after a wait (the TMEM
    // loads that follow are warp-wide), even if a limit expires between two lanes' polls
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait(b, parity)) != 0;
    };

    if (tid == 0) {
        *abort_f = 0u;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == B_EPI || i == B_EPIB || i == B_CSA || i == B_CSB)
                cnt = 8;  // the row warps
            if (i == B_KVF || i == B_KVF + 1 || i == B_DPF || i == B_DPF + 1)
                cnt = 4;  // the gather drains
            mbar_init(bar(i), cnt);
        }
        fence_mbar_init();
    }
    if (warp == 12) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    if (FOX && tid < (int)(kOnesBytes / 16)) {
        // row 0 of each 64-column half: 128 bytes of bf16 ones (the swizzle moves chunks
        // only within a row); every other row zero
        const uint32_t off = 16u * (uint32_t)tid;
        const uint32_t one2 = 0x3F803F80u;
        *reinterpret_cast<uint4 *>(sm + S_ONES + off) =
            (off % 2048u) < 128u ? make_uint4(one2, one2, one2, one2) : make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 12) {
        // ================================================================ issuer
        reg_alloc_dec<kRegIssue>();
        if (lane == 0) {
            tma_prefetch_desc(&tm_qt);
            tma_prefetch_desc(&tm_kp);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_st);
            uint32_t issued1 = 0, done1 = 0, issued2 = 0, done2 = 0;  // ring loads
            bool ok = true;
            mbar_arrive_expect_tx(bar(B_LD0), 2 * kT128);
            tma_load_3d(base + S_XB0, &tm_qt, bar(B_LD0), 0, 128 * t, bh);
            tma_load_3d(base + S_DO, &tm_do, bar(B_LD0), 0, 128 * t, bh);
            auto load1 = [&](int s) {  // pass-1 step s: key block 2t + 1 - s
                const int b = 2 * t + 1 - s, st = s % NS1;
                const uint32_t dst = base + S_STG1 + (uint32_t)st * kStage1;
                mbar_arrive_expect_tx(bar(B_FULL1 + st), kStage1);
                tma_load_3d(dst, &tm_kp, bar(B_FULL1 + st), 0, 128 * b, bh);
                tma_load_3d(dst + kT128, &tm_v, bar(B_FULL1 + st), 0, 64 * b, bh);
                ++issued1;
            };
            auto load2 = [&](int b) {  // pass-2 step b
                const int st = b % NS2;
                const uint32_t dst = base + S_STG2 + (uint32_t)st * kStage2;
                const int row = (int)((rec0 + (size_t)b) * 256);
                mbar_arrive_expect_tx(bar(B_FULL2 + st), kStage2);
                tma_load_3d(dst, &tm_kp, bar(B_FULL2 + st), 0, 128 * b, bh);
                tma_load_3d(dst + kT128, &tm_st, bar(B_FULL2 + st), 0, row, bh);
                tma_load_3d(dst + 2 * kT128, &tm_st, bar(B_FULL2 + st), 0, row + 128, bh);
                ++issued2;
            };
            for (int s = 0; s < steps1 && s < NS1; ++s) load1(s);
            ok = wait(bar(B_LD0), 0);
            // MMA2 of pass-1 step s: D_kv[s % 2] = [p^T; dT^T] [X_s | dout] (the p tile sits
            // below the dT tile, so both M halves are addressed upward from it)
            uint32_t kv_uses[2] = {0, 0}, kvf_waits[2] = {0, 0};
            // the stash records of pass-1 step s (s >= 1), by TMA from the tiles the row
            // epilogue left: dS of key block b (rows 128-255 of record b) and the carried rows
            // for key block b - 1 (rows 0-127 of record b - 1); record 2t is written at step 0
            // by the row epilogue
            auto stash_stores = [&](int s) {
                const int b = 2 * t + 1 - s;
                if (s < 1) return;
                tma_store_3d(&tm_st, base + S_DT, 0, (int)((rec0 + (size_t)b) * 256 + 128), bh);
                if (b > 0)
                    tma_store_3d(&tm_st, base + ((s & 1) ? S_XB1 : S_XB0), 0,
                                 (int)((rec0 + (size_t)(b - 1)) * 256), bh);
            };
            auto mma2 = [&](int s) -> bool {
                const int i = s & 1;
                bulk_wait_read();  // the stash stores have read the tiles this MMA's successors rewrite
                if (kv_uses[i] > 0) {  // the drain of step s - 2 has read this accumulator
                    if (!wait(bar(B_KVF + i), kvf_waits[i] & 1)) return false;
                    ++kvf_waits[i];
                }
                ++kv_uses[i];
                tc_fence_after();
                const uint32_t xs = (s >= 1) ? ((s - 1) & 1 ? S_XB1 : S_XB0) : S_XB0;
                const uint64_t a = sdesc_sw128(base + S_PT, S_DT - S_PT, 1024);
                const uint64_t b = sdesc_sw128(base + xs, S_DO - xs, 1024);
                constexpr uint32_t ID = idesc_b16(128, 128, true, true);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16(tmem + (i ? C_KV1 : C_KV0), a + 128 * kk, b + 128 * kk, ID, kk > 0);
                if (FOX) {
                    // [p^T; dS^T] x ones: rows 64 + j of column 0 hold sum_i dS_ij (K-major
                    // operand: 32 bytes per k-step, the second 64 columns 2 KB on)
                    constexpr uint32_t IDC = idesc_b16(128, 16, true, false);
                    const uint64_t bo = sdesc_sw128(base + S_ONES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16(tmem + (i ? C_CS1 : C_CS0), a + 128 * kk,
                                  bo + (uint64_t)(128 * (kk >> 2) + 2 * (kk & 3)), IDC, kk > 0);
                }
                umma_commit(bar(B_M2 + i));
                return true;
            };
            for (int s = 0; ok && s < steps1; ++s) {
                const int st = s % NS1;
                if (!(ok = wait(bar(B_FULL1 + st), (done1 / NS1) & 1))) break;
                ++done1;
                if (s > 0 && !(ok = wait(bar(B_EPI), (s - 1) & 1))) break;
                if (s > 0) stash_stores(s - 1);
                tc_fence_after();
                const uint32_t stg = base + S_STG1 + (uint32_t)st * kStage1;
                if (s > 0) {
                    const uint32_t xs = (s - 1) & 1 ? S_XB1 : S_XB0;
                    const uint64_t a = sdesc_sw128(base + xs, 16, 1024);
                    const uint64_t b = sdesc_sw128(stg, 16, 1024);
                    constexpr uint32_t ID = idesc_b16(128, 128, false, false);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + C_SX, a + 2 * kk, b + 2 * kk, ID, kk > 0);
                }
                {
                    const uint64_t a = sdesc_sw128(base + S_DO, 16, 1024);
                    const uint64_t b = sdesc_sw128(stg + kT128, 16, 1024);
                    constexpr uint32_t ID = idesc_b16(128, 64, false, false);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + C_OV, a + 2 * kk, b + 2 * kk, ID, kk > 0);
                }
                umma_commit(bar(B_M1));
                // then step s - 1's gradient gather (off the critical path: the row epilogue of
                // step s waits for it only before it overwrites that MMA's operands)
                if (s > 0) {
                    if (!(ok = mma2(s - 1))) break;
                    // the stage of step s - 1 is free (its MMA1 completed before that epilogue)
                    if (s - 1 + NS1 < steps1) load1(s - 1 + NS1);
                }
            }
            if (ok) ok = wait(bar(B_EPI), (steps1 - 1) & 1);
            if (ok) stash_stores(steps1 - 1);
            if (ok) ok = mma2(steps1 - 1);
            bulk_wait_all();  // pass 2 reads the stash back (and rewrites the X tiles)
            // pass 2 starts once both D_kv drains are done (their TMEM columns become D_p,
            // and the last MMA2, which read dout, p and dT, has completed)
            for (int i = 0; ok && i < 2; ++i)
                if (kv_uses[i] > kvf_waits[i]) {
                    ok = wait(bar(B_KVF + i), kvf_waits[i] & 1);
                    ++kvf_waits[i];
                }
            uint32_t dp_uses[2] = {0, 0}, dpf_waits[2] = {0, 0};
            if (ok)
                for (int b = 0; b < steps2 && b < NS2; ++b) load2(b);
            for (int b = 0; ok && b < steps2; ++b) {
                const int st = b % NS2;
                if (!(ok = wait(bar(B_FULL2 + st), (done2 / NS2) & 1))) break;
                ++done2;
                if (b > 0) {
                    if (!(ok = wait(bar(B_EPIB), (b - 1) & 1))) break;
                    if (b - 1 + NS2 < steps2) load2(b - 1 + NS2);
                }
                const int i = b & 1;
                if (b > 0 && dp_uses[i] > 0) {
                    if (!(ok = wait(bar(B_DPF + i), dpf_waits[i] & 1))) break;
                    ++dpf_waits[i];
                }
                tc_fence_after();
                const uint32_t stg = base + S_STG2 + (uint32_t)st * kStage2;
                // G' = G_hi P_b + G_lo P_b + dT_b K~_b   (B operands MN-major: rows = K index)
                constexpr uint32_t IDG = idesc_b16(128, 64, false, true);
                const uint64_t bp = sdesc_sw128(stg + kT64, 1024, 1024);  // P_b [n][c]
                const uint64_t bk = sdesc_sw128(stg, 1024, 1024);         // K~_b [j][c]
                if (b > 0) {
                    const uint64_t ah = sdesc_sw128(base + S_XB0, 16, 1024);
                    const uint64_t al = sdesc_sw128(base + S_XB1, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + C_G, ah + 2 * kk, bp + 128 * kk, IDG, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + C_G, al + 2 * kk, bp + 128 * kk, IDG, 1);
                }
                {
                    const uint64_t ad = sdesc_sw128(stg + 2 * kT128, 16, 1024);  // dT_b [i][j]
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + C_G, ad + 2 * kk, bk + 128 * kk, IDG, (b > 0 || kk > 0));
                }
                umma_commit(bar(B_M1B));
                if (b > 0) {
                    ++dp_uses[i];
                    // [G_hi^T; G_lo^T] X_b: A MN-major over the two G tiles, K = 128 rows
                    const uint64_t a = sdesc_sw128(base + S_XB0, S_XB1 - S_XB0, 1024);
                    const uint64_t bx = sdesc_sw128(stg + kT128, 1024, 1024);  // X_b [i][c]
                    constexpr uint32_t IDP = idesc_b16(128, 64, true, true);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16(tmem + (i ? C_DP1 : C_DP0), a + 128 * kk, bx + 128 * kk, IDP,
                                  kk > 0);
                }
                // the row epilogue overwrites the G tiles that the dP_b MMAs read: it waits for
                // this commit before it writes them
                if (b > 0) umma_commit(bar(B_M2B + i));
            }
            // wait for every MMA issued and every copy in flight before TMEM is freed
            umma_commit(bar(B_FIN));
            mbar_wait(bar(B_FIN), 0, limit_ns);
            while (done1 < issued1) {
                mbar_wait(bar(B_FULL1 + done1 % NS1), (done1 / NS1) & 1, limit_ns);
                ++done1;
            }
            while (done2 < issued2) {
                mbar_wait(bar(B_FULL2 + done2 % NS2), (done2 / NS2) & 1, limit_ns);
                ++done2;
            }
            if (!ok) {
                report_status(status, kStatusTimeout);
                *abort_f = 1u;
            }
        }
    } else if (warp < 8) {
        // ================================================================ row epilogue
        reg_alloc_inc<kRegRow>();
        // two warps per TMEM lane quadrant: warp w takes columns 32 hw .. 32 hw + 31 of every
        // 64-column block of its rows (hw = w / 4)
        const int hw = warp >> 2;
        const int r = 32 * (warp & 3) + lane;  // tile row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const int tok = 128 * t + r;
        const bool valid = tok < L;
        const int blk_row = 2 * t + (r >> 6);  // the row's query block
        const size_t hL = (size_t)bh * L;
        float Drow = 0.f, lse2 = 0.f;
        if (valid) {
            const uint4 *po = reinterpret_cast<const uint4 *>(o + (hL + tok) * kD);
            const uint4 *pd = reinterpret_cast<const uint4 *>(dout + (hL + tok) * kD);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 a = __ldg(po + c), d = __ldg(pd + c);
                const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wd[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fa = unpack_bf16x2(wa[e]), fd = unpack_bf16x2(wd[e]);
                    Drow = fmaf(fa.x, fd.x, fmaf(fa.y, fd.y, Drow));
                }
            }
            lse2 = lse[hL + tok] * kLog2e;
        }
        double ca = 0.0;
        float loci = 0.f, rs_acc = 0.f;
        if (FOX && valid) {
            ca = cb[(size_t)bh * nblk + blk_row];
            loci = loc[(size_t)bh * Lp + tok];
        }
        float *const csb = reinterpret_cast<float *>(sm + S_CS);
        bool ok = wait_warp(bar(B_LD0), 0);
        // ---------------- pass 1
        for (int s = 0; ok && s < steps1; ++s) {
            const int b = 2 * t + 1 - s;
            if (!(ok = wait_warp(bar(B_M1), s & 1))) break;
            tc_fence_after();
            const bool diag = (s == 0) ? (r >= 64) : (s == 1 && r < 64);  // warp-uniform
            const bool offd = (s >= 2) || (s == 1 && r >= 64);
            const __half *tab = dg + (((size_t)bh * nbe + b) * kC + (r & 63)) * kC;
            float dcb = 0.f;
            if (FOX && offd && valid) dcb = (float)(ca - cb[(size_t)bh * nblk + b]);
#pragma unroll 1
            for (int h = hw; h < hw + 1; ++h) {
                float ov[32], x[32];
                {
                    // both loads of the half in flight before one wait
                    uint32_t u1[32], u2[32];
                    tmem_ld32(tmem + lane_off + C_OV + 32 * h, u1);
                    if (offd) tmem_ld32(tmem + lane_off + C_SX + 32 * h, u2);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        ov[j] = __uint_as_float(u1[j]);
                        x[j] = __uint_as_float(u2[j]);
                    }
                }
                if (diag) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(tab + 32 * h);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const uint4 c = __ldg(src + q8);
                        const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f =
                                __half22float2(*reinterpret_cast<const __half2 *>(&w4[e]));
                            x[8 * q8 + 2 * e] = f.x;
                            x[8 * q8 + 2 * e + 1] = f.y;
                        }
                    }
                }
                float p[32], dd[32];  // p and dS of the half row
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float l2 = x[j];
                    if (offd) {
                        l2 = x[j] * scale_log2;
                        if (FOX)
                            l2 += kLog2e * ((dcb + loci) -
                                            __ldg(loc + (size_t)bh * Lp + (size_t)b * kC + 32 * h + j));
                    }
                    const float pj = (valid && (diag || offd)) ? ex2_approx(l2 - lse2) : 0.f;
                    const float ds = pj * (ov[j] - Drow);
                    p[j] = pj;
                    dd[j] = ds;
                    if (FOX) {
                        rs_acc += ds;
                        // the MMA sums the off-diagonal columns; the diagonal blocks (steps 0
                        // and 1) go through the transposed buffer
                        if (s <= 1) csb[(32 * h + j) * kCsLd + r] = diag ? ds : 0.f;
                    }
                }
                // the p, dT and carried-row tiles are operands of the previous step's gather
                // MMA, which runs while this step's loads and exponentials are done
                if (s >= 1 && !(ok = wait_warp(bar(B_M2 + ((s - 1) & 1)), ((s - 1) >> 1) & 1)))
                    break;
                st_row_half(sm + S_PT, r, h, p);
                if (diag && b < nblk) {  // the diagonal dT, fp32, for the block pass
                    float4 *d4 = reinterpret_cast<float4 *>(
                        dTd + (((size_t)bh * nblk + b) * kC + (r & 63)) * kC + 32 * h);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        d4[c] = make_float4(scale * dd[4 * c], scale * dd[4 * c + 1],
                                            scale * dd[4 * c + 2], scale * dd[4 * c + 3]);
                }
                // the dS operand tile (p's registers, now free), off-diagonal rows only and
                // unscaled (the products that use it are scaled on output, so PaTH-FoX's
                // column sums come out of the MMA for any scale); the issuer stores the tile
                // as the step's stash record of dS by TMA
                float *tv = p;
#pragma unroll
                for (int j = 0; j < 32; ++j) tv[j] = offd ? dd[j] : 0.f;
                st_row_half(sm + S_DT, r, h, tv);
            }
            if (!ok) break;
            // the carried rows for the next key block (and their stash record)
            if (s == 0) {
                // stash record 2t holds the state at key block 2t: zero for block 2t's rows
                // (their walk starts below it), q~ for block 2t+1's rows
                __nv_bfloat16 *dst =
                    stash + ((((size_t)bh * npair * npair) + rec0 + (size_t)(2 * t)) * 256 + r) * kD;
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int c = 4 * hw; c < 4 * hw + 4; ++c)
                    d4[c] = (r < 64) ? make_uint4(0u, 0u, 0u, 0u)
                                     : *reinterpret_cast<const uint4 *>(sm + S_XB0 + sw128_offset(r, c));
            } else if (b > 0) {
                // the carried rows for key block b - 1 (the issuer stores the tile as its stash
                // record by TMA)
                uint8_t *xn = sm + ((s & 1) ? S_XB1 : S_XB0);
                if (s == 1 && r < 64) {
                    // block 2t's rows keep q~ (their walk starts at key block 2t - 1)
#pragma unroll
                    for (int c = 4 * hw; c < 4 * hw + 4; ++c)
                        *reinterpret_cast<uint4 *>(xn + sw128_offset(r, c)) =
                            *reinterpret_cast<const uint4 *>(sm + S_XB0 + sw128_offset(r, c));
                } else {
                    float x[32];
                    tld32(tmem + lane_off + C_SX + 64 + 32 * hw, x);
                    st_row_half(xn, r, hw, x);
                }
            }
            fence_proxy_async_smem();
            // the stash record written above at step 0 is read back by TMA in pass 2, which
            // starts after this pass's last step
            if (s == steps1 - 1) fence_proxy_async_global();
            tc_fence_before();
            mbar_arrive_warp(bar(B_EPI));
            if (FOX && s <= 1) {
                // column sums of the diagonal blocks' dS over the tile's 128 rows: each thread
                // sums a quarter column once all eight warps have written theirs (B_CSA), and the
                // buffer is rewritten only after every thread has read it (B_CSB)
                mbar_arrive_warp(bar(B_CSA));
                if (!(ok = wait_warp(bar(B_CSA), s & 1))) break;
                const int rt = 128 * hw + r, j = rt & 63, quarter = rt >> 6;
                const float *col = csb + j * kCsLd + 32 * quarter;
                float acc = 0.f;
#pragma unroll 8
                for (int i = 0; i < 32; ++i) acc += col[i];
                if (64 * b + j < L) atomicAdd(csum + (size_t)bh * Lp + 64 * b + j, acc);
                mbar_arrive_warp(bar(B_CSB));
                if (!(ok = wait_warp(bar(B_CSB), s & 1))) break;
            }
        }
        if (FOX && valid) atomicAdd(rsum + (size_t)bh * Lp + tok, rs_acc);  // two halves per row
        // ---------------- pass 2
        if (ok && t == 0 && r < 64 && 0 < nblk) {
            // block 0 carries nothing: dq~ = 0
            float4 *dq4 = reinterpret_cast<float4 *>(dqt + ((size_t)bh * Lp + r) * kD);
#pragma unroll
            for (int c = 8 * hw; c < 8 * hw + 8; ++c) dq4[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int b = 0; ok && b < steps2; ++b) {
            if (!(ok = wait_warp(bar(B_M1B), b & 1))) break;
            tc_fence_after();
            float g[32];  // this warp's half of the row of G
            tld32(tmem + lane_off + C_G + 32 * hw, g);
            const bool last_a0 = (b == 2 * t - 1) && r < 64 && 2 * t < nblk;
            const bool last_a1 = (b == 2 * t) && r >= 64 && 2 * t + 1 < nblk;
            if (last_a0 || last_a1) {
                // the recursion runs on G / scale (its dS operand is unscaled)
                float4 *dq4 = reinterpret_cast<float4 *>(dqt + ((size_t)bh * Lp + tok) * kD);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dq4[8 * hw + c] = make_float4(scale * g[4 * c], scale * g[4 * c + 1],
                                                  scale * g[4 * c + 2], scale * g[4 * c + 3]);
            }
            if (b < 2 * t) {
                // the dP_b MMA of this step reads the G tiles being replaced
                if (b > 0 && !(ok = wait_warp(bar(B_M2B + (b & 1)), ((b - 1) >> 1) & 1))) break;
                float lo[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) lo[j] = g[j] - __bfloat162float(__float2bfloat16_rn(g[j]));
                st_row_half(sm + S_XB0, r, hw, g);
                st_row_half(sm + S_XB1, r, hw, lo);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive_warp(bar(B_EPIB));
            }
        }
    } else {
        // ================================================================ gather drains
        reg_alloc_dec<kRegDrain>();
        const int m = tid - 256;  // TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp - 8)) << 16;
        const size_t hL = (size_t)bh * L;
        bool ok = true;
        for (int s = 0; ok && s < steps1; ++s) {
            const int b = 2 * t + 1 - s, i = s & 1;
            if (!(ok = wait_warp(bar(B_M2 + i), (s >> 1) & 1))) break;
            tc_fence_after();
            const uint32_t acc = tmem + lane_off + (i ? C_KV1 : C_KV0);
            if (m >= 64) {
                // dK~_b row m - 64 (nothing at the first step: block 2t+1 is only a diagonal
                // block)
                if (s >= 1 && b < nblk) {
                    float *dst = dkt + ((size_t)bh * Lp + 64 * b + (m - 64)) * kD;
                    const float ks = scale;  // the tile held dS
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        float x[32];
                        tld32(acc + 32 * h, x);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            red_add_v4(dst + 32 * h + 4 * c, ks * x[4 * c], ks * x[4 * c + 1],
                                       ks * x[4 * c + 2], ks * x[4 * c + 3]);
                    }
                }
                if (FOX && s >= 1) {
                    // sum over the tile's rows of dS_ij, j = m - 64 of key block b
                    float x[32];
                    tld32(tmem + lane_off + (i ? C_CS1 : C_CS0), x);
                    const int j = 64 * b + (m - 64);
                    if (j < L) atomicAdd(csum + (size_t)bh * Lp + j, x[0]);
                }
            } else {
                // dv row j: p^T dout. The TMEM loads are warp-collective, so every lane loads
                // and only the rows inside the sequence are added.
                const int j = 64 * b + m;
                float *dst = dv + (hL + j) * kD;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tld32(acc + 64 + 32 * h, x);
                    if (j < L) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            red_add_v4(dst + 32 * h + 4 * c, x[4 * c], x[4 * c + 1], x[4 * c + 2],
                                       x[4 * c + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_warp(bar(B_KVF + i));
        }
        for (int b = 1; ok && b < steps2; ++b) {
            const int i = b & 1;
            // uses of D_p[i] so far: b = 2, 4, ... for i = 0 and 1, 3, ... for i = 1
            const uint32_t use = (uint32_t)((b - 1) >> 1);
            if (!(ok = wait_warp(bar(B_M2B + i), use & 1))) break;
            tc_fence_after();
            const uint32_t acc = tmem + lane_off + (i ? C_DP1 : C_DP0);
            // the block pass reads dP_b only for 0 < b < nblk - 1
            if (b < nblk - 1) {
                float *dst = dP + (((size_t)bh * nblk + b) * kC + (m & 63)) * kC;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    float x[32];
                    tld32(acc + 32 * h, x);
                    // G / scale in the recursion: scale on output
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        red_add_v4(dst + 32 * h + 4 * c, scale * x[4 * c], scale * x[4 * c + 1],
                                   scale * x[4 * c + 2], scale * x[4 * c + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive_warp(bar(B_DPF + i));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Workspace of the tensor-core backward (bf16 inputs, d = 64): the forward's bf16
// preparation layout first (its 256-byte header is the status header), then fp32 dq~ and dk~
// (BH, Lp, 64), dP_b and the diagonal dT (BH, nblk, 64, 64), the bf16 stash (per head and
// tile t, records b = 0 .. 2t of the carried rows X_b and dT_b, 128 x 64 each), and for
// PaTH-FoX the block-local gate sums, row and column sums of dS (BH, Lp) fp32 and the block
// gate prefixes (BH, nblk) fp64. nblk = ceil(L / 64), Lp = 64 nblk.
struct BwdTcLayout {
    int BH, nblk, nbe, Lp;
    size_t off_dqt, off_dkt, off_dP, off_dTd, off_stash, off_loc, off_rs, off_cs, off_cb, total;
    size_t stash_rows_per_head;
};

BwdTcLayout bwd_tc_layout(int B, int H, int L, bool fox) {
    BwdTcLayout y;
    const FwdLayout f = fwd_layout(B, H, L, 2, fox);
    y.BH = B * H;
    y.nblk = (L + kC - 1) / kC;
    y.nbe = f.nblk;
    y.Lp = y.nblk * kC;
    const size_t bh = (size_t)y.BH, npair = (size_t)y.nbe / 2;
    const size_t rows = bh * y.Lp * kD * 4, blocks = bh * y.nblk * (size_t)kC * kC * 4;
    size_t off = f.total;
    y.off_dqt = off;
    off = align256(off + rows);
    y.off_dkt = off;
    off = align256(off + rows);
    y.off_dP = off;
    off = align256(off + blocks);
    y.off_dTd = off;
    off = align256(off + blocks);
    y.off_stash = off;
    y.stash_rows_per_head = npair * npair * 256;
    off = align256(off + bh * y.stash_rows_per_head * kD * 2);
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

size_t bwd_tc_ws_bytes(int B, int H, int L, bool fox) { return bwd_tc_layout(B, H, L, fox).total; }

// The bf16 backward: preparation (the forward's tensor-core kernel), tensor-core query
// pass, block pass; PaTH-FoX adds the gate sums before and d log f after.
cudaError_t launch_path_bwd_tc(const void *q, const void *k, const void *v, const void *w,
                               const float *beta, const float *log_f, const void *o,
                               const float *lse, const void *dout, int B, int H, int L,
                               float scale, float *dq, float *dk, float *dv, float *dw,
                               float *dbeta, float *dlogf, void *ws, uint64_t limit_ns,
                               cudaStream_t stream) {
    const bool fox = log_f != nullptr;
    const BwdTcLayout y = bwd_tc_layout(B, H, L, fox);
    const FwdLayout f = fwd_layout(B, H, L, 2, fox);
    if (y.stash_rows_per_head >= (size_t)1 << 31) return cudaErrorInvalidValue;
    char *base = static_cast<char *>(ws);
    auto at = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    float *dqt = at(y.off_dqt), *dkt = at(y.off_dkt), *dPb = at(y.off_dP), *dTd = at(y.off_dTd);
    float *loc = at(y.off_loc), *rs = at(y.off_rs), *cs = at(y.off_cs);
    double *cb = reinterpret_cast<double *>(base + y.off_cb);
    __nv_bfloat16 *stash = reinterpret_cast<__nv_bfloat16 *>(base + y.off_stash);
    const size_t tok = (size_t)y.BH * y.Lp * 4;
    cudaError_t e;
    if ((e = cudaMemsetAsync(base, 0, 4, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dkt, 0, tok * kD, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dPb, 0, (size_t)y.BH * y.nblk * kC * kC * 4, stream)) != cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(dv, 0, (size_t)y.BH * L * kD * 4, stream)) != cudaSuccess) return e;
    if (fox) {
        if ((e = cudaMemsetAsync(cs, 0, tok, stream)) != cudaSuccess ||
            (e = cudaMemsetAsync(rs, 0, tok, stream)) != cudaSuccess)
            return e;
        if ((e = launch_bwd_fox_sums(log_f, y.BH, L, y.Lp, y.nblk, loc, cb, stream)) != cudaSuccess)
            return e;
    }
    if ((e = launch_ut_prepare_tc(q, k, w, beta, log_f, y.BH, L, scale, ws, limit_ns, stream)) !=
        cudaSuccess)
        return e;
    CUtensorMap tqt, tkp, tv, tdo, tst;
    if (!make_map_bf16(&tqt, base + f.off_qt, f.Lp, y.BH, 128) ||
        !make_map_bf16(&tkp, base + f.off_kp, f.nblk * 2 * kC, y.BH, 128) ||
        !make_map_bf16(&tv, v, L, y.BH, 64) || !make_map_bf16(&tdo, dout, L, y.BH, 128) ||
        !make_map_bf16(&tst, stash, (int)y.stash_rows_per_head, y.BH, 128))
        return cudaErrorInvalidValue;
    auto kern = fox ? bwd_query_tc_kernel<true> : bwd_query_tc_kernel<false>;
    const uint32_t smem = fox ? bwd_tc_smem<true>() : bwd_tc_smem<false>();
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    // shared per token: [K~_b; P_b] (256 B) and v (128 B)
    const bool hf = heads_fastest((size_t)y.BH, (size_t)L, 384);
    const dim3 grid = hf ? dim3(y.BH, y.nbe / 2) : dim3(y.nbe / 2, y.BH);
    kern<<<grid, kThr, smem, stream>>>(
        tqt, tkp, tv, tdo, tst, static_cast<const __nv_bfloat16 *>(o),
        static_cast<const __nv_bfloat16 *>(dout), lse,
        reinterpret_cast<const __half *>(base + f.off_dg), stash, dqt, dkt, dPb, dTd, dv, loc, cb,
        rs, cs, L, y.Lp, y.nblk, y.nbe, scale, scale * kLog2e, reinterpret_cast<uint32_t *>(base),
        limit_ns, hf ? 1 : 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bwd_block_mm(q, k, w, beta, dqt, dkt, dPb, dTd, dq, dk, dw, dbeta, y.BH, L,
                                 y.Lp, y.nblk, stream)) != cudaSuccess)
        return e;
    if (fox) e = launch_bwd_fox_dlogf(rs, cs, y.BH, L, y.Lp, dlogf, stream);
    return e;
}

}  // namespace path
