// K2 (bf16): the right-to-left block scan of PaTH attention on tcgen05 tensor cores,
// two key blocks per step (the PaTH-FoX forward has its own scan, scan_tc_fox.cu).
//
// Technical summary "技術要約: PaTH Attention" §3 (FlashAttention-style algorithm: per-block
// boundary-adjusted queries and keys, a right-to-left scan over key/value blocks that
// accumulates the Householder product, online softmax, nothing L x L in memory); review
// "거리에서 경로로, PaTH Attention" §9 (the same scheme, blockwise preprocessing and
// blockwise updates of the accumulated transform and softmax statistics).
//
// A tile is 128 query rows = the pair of 64-token blocks (2t, 2t+1) of one head. With q~
// the boundary-adjusted queries, k~ the boundary-adjusted keys and P_b the dense block
// transition, a state row x_i starts as q~_i and the tile visits key-block pairs
// u = t, t-1, ..., 0 (step s visits pair t - s). For an earlier pair the row scores block
// 2u+1 as x . k~_j and block 2u as x . K^_j with K^_j = P_{2u+1}^T k~_j, then leaves as
// Pi_u x with Pi_u = P_{2u} P_{2u+1} (the pair products come from pair_combine.cu). In
// row form one MMA with N = 192 gives both logit blocks and the new state:
//     [S_lo | S_hi | X'] = X [K^_{2u}; K~_{2u+1}; Pi_u]^T,
// followed by O += P [V_{2u}; V_{2u+1}] (K = 128). Step 0 is the tile's own pair: rows of
// block 2t take the diagonal-block table for block 2t and nothing of block 2t+1; rows of
// block 2t+1 take the table for block 2t+1 and the MMA logits x . k~_j against block 2t
// from X [K~_{2t}; P_{2t}]^T (N = 128), which also gives their new state P_{2t} q~_i;
// rows of block 2t keep q~_i.
//
// One CTA owns the tiles A = 2p and B = 2p + 1 of one head and streams the key-block pairs
// 2p+1, 2p, ..., 0 once, so each pair serves both tiles, through two TMA rings: one of
// [K^_{2u}; K~_{2u+1}; Pi_u] (released as soon as both S|state MMAs on it have completed)
// and one of [V_{2u}; V_{2u+1}] (released after the P.V MMAs, which run a softmax later).
// Step 0's operand [K~_{2t}; P_{2t}] is staged in the tile's P buffer, which the softmax
// overwrites only after that MMA.
// TMEM per tile (256 columns): S [0,128) (block 2u in [0,64), 2u+1 in [64,128)), the new
// state [128,192) (at [64,128) on step 0), O [192,256); tile B's columns at +256.
// Warp roles (512 threads; registers moved to the softmax warpgroups with setmaxnreg):
//   warps 0-3 / 4-7  softmax of tile A / B, one row per thread (= TMEM lane): load all
//                    128 logits of the step at once and release S, online softmax with
//                    lazy rescaling, P tile;
//   warps 8-11       the state recurrence of both tiles (one per TMEM lane quadrant):
//                    fp32 -> bf16 conversion of each new state into a swizzled A tile;
//   warps 12 / 13    issue tile A's / B's S|state MMAs (they need the converted state and
//                    the released S of the previous step);
//   warps 14 / 15    issue tile A's / B's P.V MMAs and release the stages; warp 14 also
//                    feeds the TMA ring (both duties poll, neither blocks the other);
//   warp 12 also owns TMEM.
// Each MMA stream has its own issuing thread because the streams wait on different
// conditions (a thread blocked on one would hold back the others); throughput is not the
// reason: one thread issuing back to back keeps the SM's tensor pipe at its math rate for
// N >= 128 (about 65 / 97 / 129 cycles per K = 16 MMA at N = 128 / 192 / 256), N = 64 costs
// about 48 cycles against 32 of math, and more issuers do not raise an SM's rate.
// The state tile and the P tile are single-buffered:
// the state is rewritten once the S|state MMA that read it has completed, P once the
// tile's previous P.V has completed.
#include "common.cuh"

namespace path {

namespace {

constexpr int kScanThreads = 512;
constexpr int NR = 3;                          // TMA stages of [K^; K~; Pi] (S|state operand)
constexpr int NV = 3;                          // TMA stages of [V; V] (P.V operand)
constexpr uint32_t kQBytes = 128 * 128;        // 128 rows x 64 bf16
constexpr uint32_t kRBytes = 192 * 128;        // [K^_{2u}; K~_{2u+1}; Pi_u]
constexpr uint32_t kV2Bytes = 128 * 128;       // [V_{2u}; V_{2u+1}]
constexpr uint32_t kPBytes = 2 * 128 * 128;    // P: 128 x 128 bf16 as two 64-column halves
constexpr float kRescaleThreshold = 8.f;       // lazy rescale: keep the old max within 2^8

// Registers per thread after the split (launch: 128 for all 512 threads).
constexpr int kRegSoftmax = 184, kRegState = 88, kRegIssue = 56;
constexpr int kRegTotal = 256 * kRegSoftmax + 128 * kRegState + 128 * kRegIssue;
static_assert(kRegTotal <= 65536, "register split exceeds the register file");

struct ScanSmem {
    // byte offsets from the 1024-aligned base
    __host__ __device__ static constexpr uint32_t q_st(int t) { return (uint32_t)t * kQBytes; }
    __host__ __device__ static constexpr uint32_t p_buf(int t) { return 2 * kQBytes + (uint32_t)t * kPBytes; }
    static constexpr uint32_t stage_r = 2 * kQBytes + 2 * kPBytes;
    static constexpr uint32_t stage_v = stage_r + NR * kRBytes;
    static constexpr uint32_t bars = stage_v + NV * kV2Bytes;
    // barrier indices: the two rings, then eight per tile, then one
    static constexpr int FULL_R = 0, EMPTY_R = NR, FULL_V = 2 * NR, EMPTY_V = 2 * NR + NV,
                         TILE0 = 2 * NR + 2 * NV;
    static constexpr int QFULL = 0, BAR_SX = 1, BAR_O = 2, QREADY = 3, SFREE = 4, PREADY = 5,
                         FINAL_SX = 6, FINAL_PV = 7;
    __host__ __device__ static constexpr int per_tile(int t, int which) { return TILE0 + 8 * t + which; }
    static constexpr int NEVER = TILE0 + 16, NBARS = TILE0 + 17;
    static constexpr uint32_t tmem_slot = bars + NBARS * 8;
    static constexpr uint32_t abort_flag = tmem_slot + 4;
    static constexpr uint32_t bytes = abort_flag + 4;
};

constexpr uint32_t kScanSmemBytes = ScanSmem::bytes + 1024;  // + alignment slack
static_assert(kScanSmemBytes <= 227u * 1024u, "scan shared memory exceeds the per-CTA limit");

struct Waiter {
    volatile uint32_t *abort;
    uint32_t *status;
    uint64_t limit_ns;
    // Bounded wait; on timeout records the status and raises the CTA abort flag.
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

template <int N>
__device__ __forceinline__ void reg_alloc_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}

// 64 fp16 entries of a diagonal-block table row, in log2 units.
__device__ __forceinline__ void load_diag_row(const __half *row, float *v) {
    const uint4 *src = reinterpret_cast<const uint4 *>(row);
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) {
        const uint4 c = __ldg(src + q8);
        const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w4[e]));
            v[8 * q8 + 2 * e] = f.x;
            v[8 * q8 + 2 * e + 1] = f.y;
        }
    }
}

// RAW: a positive scale, applied inside the exponent's FFMA.
template <bool RAW>
__global__ void __launch_bounds__(kScanThreads, 1)
path_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_qt,
                    const __grid_constant__ CUtensorMap tm_kp128,
                    const __grid_constant__ CUtensorMap tm_kp64,
                    const __grid_constant__ CUtensorMap tm_pr64,
                    const __grid_constant__ CUtensorMap tm_v128,
                    const __half *__restrict__ dg, __nv_bfloat16 *__restrict__ out,
                    float *__restrict__ lse, int L, int nblk, float scale_log2,
                    uint32_t *status, uint64_t limit_ns, int force_timeout, int heads_fast) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = nblk >> 1;                   // tiles = key-block pairs
    const int ncta = (ntile + 1) >> 1;
    // the heaviest tile pairs first, heads fastest or head by head (heads_fastest)
    const int pair = ncta - 1 - (int)(heads_fast ? blockIdx.y : blockIdx.x);
    const int bh = heads_fast ? blockIdx.x : blockIdx.y;
    const bool hasB = 2 * pair + 1 < ntile;
    const int top = hasB ? 2 * pair + 1 : 2 * pair;  // first key-block pair of the stream
    const int nstream = top + 1;
    // tile t (0 = A, 1 = B): tile index, its step count, and stream position of its step 0
    auto tile_of = [&](int t) { return 2 * pair + t; };
    auto nsteps_of = [&](int t) { return tile_of(t) + 1; };
    auto off_of = [&](int t) { return top - tile_of(t); };
    // whether tile t reads stream position n (its values), and the S|state operand of
    // position n (every step but the tile's first); the operand ring skips position 0,
    // which only the top tile's own pair occupies
    auto reads = [&](int t, int n) {
        return (t == 0 || hasB) && n >= off_of(t) && n < off_of(t) + nsteps_of(t);
    };
    auto reads_r = [&](int t, int n) { return reads(t, n) && n > off_of(t); };

    auto bar = [&](int i) { return base + ScanSmem::bars + 8u * (uint32_t)i; };
    auto tbar = [&](int t, int which) { return bar(ScanSmem::per_tile(t, which)); };
    volatile uint32_t *abort_flag =
        reinterpret_cast<volatile uint32_t *>(gbase + ScanSmem::abort_flag);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + ScanSmem::tmem_slot);
    const Waiter wait{abort_flag, status, limit_ns};

    if (threadIdx.x == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(bar(ScanSmem::FULL_R + i), 1);
            mbar_init(bar(ScanSmem::EMPTY_R + i), 2);  // two arrivals per use (see issuers)
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(bar(ScanSmem::FULL_V + i), 1);
            mbar_init(bar(ScanSmem::EMPTY_V + i), 2);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(tbar(t, ScanSmem::QFULL), 1);
            mbar_init(tbar(t, ScanSmem::BAR_SX), 1);
            mbar_init(tbar(t, ScanSmem::BAR_O), 1);
            mbar_init(tbar(t, ScanSmem::QREADY), 4);  // one arrival per warp
            mbar_init(tbar(t, ScanSmem::SFREE), 4);
            mbar_init(tbar(t, ScanSmem::PREADY), 4);
            mbar_init(tbar(t, ScanSmem::FINAL_SX), 1);
            mbar_init(tbar(t, ScanSmem::FINAL_PV), 1);
        }
        mbar_init(bar(ScanSmem::NEVER), 1);
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 12) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // per tile: S [0,128), new state [128,192) ([64,128) on step 0), O [192,256)
    auto t_base = [&](int t) { return tmem + 256u * (uint32_t)t; };
    auto t_o = [&](int t) { return t_base(t) + 192u; };
    auto stage_r = [&](int i) { return base + ScanSmem::stage_r + (uint32_t)i * kRBytes; };
    auto stage_v = [&](int i) { return base + ScanSmem::stage_v + (uint32_t)i * kV2Bytes; };

    // Registers move to the softmax warpgroups (a step's 128 logits per thread); each
    // warpgroup executes its setmaxnreg once, at the head of its role.
    if (warp >= 12) {
      reg_alloc_dec<kRegIssue>();
      if (warp <= 13) {
        // ------------------------------------------------------------ S|state issuers
        const int t = warp - 12;
        if (lane == 0 && (t == 0 || hasB)) {
            constexpr uint32_t ID_DIAG = idesc_bf16(128, 128, false);
            constexpr uint32_t ID_SX = idesc_bf16(128, 192, false);
            const int nst = nsteps_of(t), off = off_of(t);
            bool ok = true;
            if (force_timeout && t == 0) ok = wait(bar(ScanSmem::NEVER), 0);  // nothing arrives here
            const uint64_t a_q = sdesc_sw128(base + ScanSmem::q_st(t), 16, 1024);
            for (int s = 0; ok && s < nst; ++s) {
                if (s == 0) {
                    // q~ and [K~_{2t}; P_{2t}] of the tile's own pair
                    if (!(ok = wait(tbar(t, ScanSmem::QFULL), 0))) break;
                    tc_fence_after();
                    const uint64_t b = sdesc_sw128(base + ScanSmem::p_buf(t), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(t_base(t), a_q + 2 * kk, b + 2 * kk, ID_DIAG, kk > 0);
                } else {
                    const int n = s + off, m = n - 1, st = m % NR;  // operand ring index m
                    if (!(ok = wait(bar(ScanSmem::FULL_R + st), (m / NR) & 1))) break;
                    // the state of step s, converted after the MMA of step s - 1
                    if (!(ok = wait(tbar(t, ScanSmem::QREADY), (s - 1) & 1))) break;
                    // S of step s - 1 has been read by the softmax
                    if (!(ok = wait(tbar(t, ScanSmem::SFREE), (s - 1) & 1))) break;
                    tc_fence_after();
                    const uint64_t b = sdesc_sw128(stage_r(st), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(t_base(t), a_q + 2 * kk, b + 2 * kk, ID_SX, kk > 0);
                    // the operand stage is free once both tiles' MMAs on it have completed
                    // (a stage read by one tile only gets both arrivals from that tile)
                    umma_commit(bar(ScanSmem::EMPTY_R + st));
                    if (!reads_r(1 - t, n)) umma_commit(bar(ScanSmem::EMPTY_R + st));
                }
                umma_commit(tbar(t, ScanSmem::BAR_SX));
            }
            umma_commit(tbar(t, ScanSmem::FINAL_SX));
            const uint64_t t0 = cycles_now();
            while (!mbar_try_wait(tbar(t, ScanSmem::FINAL_SX), 0) &&
                   cycles_now() - t0 < ns_to_cycles(limit_ns)) {
            }
        }
      } else {
        // ------------------------------------------------------------ P.V issuers (+ TMA)
        // Tile A's thread also feeds the TMA ring; both duties poll, neither blocks the other.
        const int t = warp - 14;
        const bool producer = (t == 0);
        if (lane == 0 && (t == 0 || hasB)) {
            constexpr uint32_t ID_PV = idesc_bf16(128, 64, true);
            const int nst = nsteps_of(t), off = off_of(t);
            if (producer) {
                tma_prefetch_desc(&tm_qt);
                tma_prefetch_desc(&tm_kp128);
                tma_prefetch_desc(&tm_kp64);
                tma_prefetch_desc(&tm_pr64);
                tma_prefetch_desc(&tm_v128);
                for (int tt = 0; tt < (hasB ? 2 : 1); ++tt) {
                    const int tile = tile_of(tt);
                    mbar_arrive_expect_tx(tbar(tt, ScanSmem::QFULL), 2 * kQBytes);
                    tma_load_3d(base + ScanSmem::q_st(tt), &tm_qt, tbar(tt, ScanSmem::QFULL), 0,
                                tile * kTile, bh);
                    tma_load_3d(base + ScanSmem::p_buf(tt), &tm_kp128, tbar(tt, ScanSmem::QFULL), 0,
                                2 * tile * 2 * kC, bh);
                }
            }
            const uint64_t a_p = sdesc_sw128(base + ScanSmem::p_buf(t), 16, 1024);
            // next stream position to load into the value ring / operand ring index (the
            // operand of position n goes to index n - 1)
            const int nr_total = nstream - 1;
            int nv_fill = producer ? 0 : nstream, nr_fill = producer ? 0 : nr_total;
            int s = 0;                            // next P.V step
            bool ok = true;
            uint64_t t_last = cycles_now();
            while (ok && (s < nst || nv_fill < nstream || nr_fill < nr_total)) {
                bool progress = false;
                if (nr_fill < nr_total &&
                    (nr_fill < NR ||
                     mbar_test_wait(bar(ScanSmem::EMPTY_R + nr_fill % NR), ((nr_fill / NR) - 1) & 1))) {
                    const int st = nr_fill % NR, u = top - (nr_fill + 1);
                    const uint32_t full = bar(ScanSmem::FULL_R + st);
                    mbar_arrive_expect_tx(full, kRBytes);
                    tma_load_3d(stage_r(st), &tm_pr64, full, 0, u * 2 * kC, bh);
                    tma_load_3d(stage_r(st) + 64 * 128, &tm_kp64, full, 0, (2 * u + 1) * 2 * kC, bh);
                    tma_load_3d(stage_r(st) + 128 * 128, &tm_pr64, full, 0, u * 2 * kC + kC, bh);
                    ++nr_fill;
                    progress = true;
                }
                if (nv_fill < nstream &&
                    (nv_fill < NV ||
                     mbar_test_wait(bar(ScanSmem::EMPTY_V + nv_fill % NV), ((nv_fill / NV) - 1) & 1))) {
                    const int st = nv_fill % NV, u = top - nv_fill;
                    const uint32_t full = bar(ScanSmem::FULL_V + st);
                    mbar_arrive_expect_tx(full, kV2Bytes);
                    tma_load_3d(stage_v(st), &tm_v128, full, 0, u * kTile, bh);
                    ++nv_fill;
                    progress = true;
                }
                if (s < nst) {
                    const int n = s + off, st = n % NV;
                    const bool in_ready = mbar_test_wait(bar(ScanSmem::FULL_V + st), (n / NV) & 1);
                    if (in_ready && mbar_test_wait(tbar(t, ScanSmem::PREADY), s & 1)) {
                        tc_fence_after();
                        const uint64_t b_v = sdesc_sw128(stage_v(st), 1024, 1024);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_bf16(t_o(t), a_p + (uint64_t)((kk >> 2) * (kQBytes >> 4) + 2 * (kk & 3)),
                                      b_v + 128 * kk, ID_PV, (s > 0 || kk > 0));
                        umma_commit(tbar(t, ScanSmem::BAR_O));
                        // two arrivals per value stage (a stage read by one tile only gets
                        // both from that tile)
                        umma_commit(bar(ScanSmem::EMPTY_V + st));
                        if (!reads(1 - t, n)) umma_commit(bar(ScanSmem::EMPTY_V + st));
                        ++s;
                        progress = true;
                    }
                }
                if (progress) {
                    t_last = cycles_now();
                } else if (*abort_flag) {
                    ok = false;
                } else if (cycles_now() - t_last > ns_to_cycles(limit_ns)) {
                    report_status(status, kStatusTimeout);
                    *abort_flag = 1u;
                    ok = false;
                }
            }
            if (producer) {
                // drain: every issued copy has landed before the CTA may exit
                for (int n = (nv_fill > NV ? nv_fill - NV : 0); n < nv_fill; ++n) {
                    const uint32_t bfull = bar(ScanSmem::FULL_V + n % NV);
                    const uint64_t t0 = cycles_now();
                    while (!mbar_try_wait(bfull, (n / NV) & 1) &&
                           cycles_now() - t0 < ns_to_cycles(limit_ns)) {
                    }
                }
                for (int m = (nr_fill > NR ? nr_fill - NR : 0); m < nr_fill; ++m) {
                    const uint32_t bfull = bar(ScanSmem::FULL_R + m % NR);
                    const uint64_t t0 = cycles_now();
                    while (!mbar_try_wait(bfull, (m / NR) & 1) &&
                           cycles_now() - t0 < ns_to_cycles(limit_ns)) {
                    }
                }
                for (int tt = 0; tt < (hasB ? 2 : 1); ++tt) {
                    const uint64_t t0 = cycles_now();
                    while (!mbar_try_wait(tbar(tt, ScanSmem::QFULL), 0) &&
                           cycles_now() - t0 < ns_to_cycles(limit_ns)) {
                    }
                }
            }
            umma_commit(tbar(t, ScanSmem::FINAL_PV));
            const uint64_t t0 = cycles_now();
            while (!mbar_try_wait(tbar(t, ScanSmem::FINAL_PV), 0) &&
                   cycles_now() - t0 < ns_to_cycles(limit_ns)) {
            }
        }
      }
    } else if (warp >= 8) {
        reg_alloc_dec<kRegState>();
        // ------------------------------------------------------------ state warps
        const int quad = warp - 8;
        const int r = quad * 32 + lane;          // row of both tiles = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        bool ok = true;
        // each tile needs a new state after every step but its last; convert whichever tile's
        // S|state MMA completes first (the two tiles' recurrences are independent)
        int next[2] = {0, 0};
        const int need[2] = {nsteps_of(0) - 1, hasB ? nsteps_of(1) - 1 : 0};
        uint64_t t_last = cycles_now();
        while (ok && (next[0] < need[0] || next[1] < need[1])) {
            int t = -1;
            if (lane == 0) {
                for (int c = 1; c >= 0 && t < 0; --c)
                    if (next[c] < need[c] && mbar_test_wait(tbar(c, ScanSmem::BAR_SX), next[c] & 1)) t = c;
            }
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t < 0) {
                // nothing ready: back off briefly so the softmax warps keep the issue slots
                int stop = 0;
                if (lane == 0) {
                    if (*abort_flag) {
                        stop = 1;
                    } else if (cycles_now() - t_last > ns_to_cycles(limit_ns)) {
                        report_status(status, kStatusTimeout);
                        *abort_flag = 1u;
                        stop = 1;
                    }
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) ok = false;
                else __nanosleep(32);
                continue;
            }
            const int s = next[t]++;
            t_last = cycles_now();
            tc_fence_after();
            // the state of step s + 1 replaces that of step s, whose only reader (the
            // S|state MMA of step s) has completed; rows of block 2t keep q~ after step 0
            if (s >= 1 || quad >= 2) {
                uint8_t *row = gbase + ScanSmem::q_st(t);
                const uint32_t src = t_base(t) + (s == 0 ? 64u : 128u) + lane_base;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t x[32];
                    tmem_ld32(src + 32 * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t *e = &x[8 * c];
                        *reinterpret_cast<uint4 *>(row + sw128_offset(r, 4 * h + c)) =
                            make_uint4(pack_bf16x2(__uint_as_float(e[0]), __uint_as_float(e[1])),
                                       pack_bf16x2(__uint_as_float(e[2]), __uint_as_float(e[3])),
                                       pack_bf16x2(__uint_as_float(e[4]), __uint_as_float(e[5])),
                                       pack_bf16x2(__uint_as_float(e[6]), __uint_as_float(e[7])));
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive_warp(tbar(t, ScanSmem::QREADY));
        }
        tc_fence_before();
    } else {
      reg_alloc_inc<kRegSoftmax>();
      if (warp < 4 || hasB) {
        // ------------------------------------------------------------ softmax warps
        const int t = warp >> 2;                 // 0 = tile A, 1 = tile B
        const int r = threadIdx.x - 128 * t;     // tile row = TMEM lane
        const int q = warp & 3;                  // lane quadrant
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int tile = tile_of(t);
        const int nsteps = nsteps_of(t);
        const int i = tile * kTile + r;          // query index
        const size_t head = (size_t)bh;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        // every lane of a warp leaves together: tcgen05.ld/st are warp-collective
        auto wwait = [&](uint32_t b_, uint32_t par) {
            return __all_sync(0xffffffffu, wait(b_, par)) != 0;
        };
        const uint32_t T_S = t_base(t) + lane_base;
        const uint32_t T_O = t_o(t) + lane_base;

        for (int s = 0; s < nsteps && ok; ++s) {
            if (!(ok = wwait(tbar(t, ScanSmem::BAR_SX), s & 1))) break;
            tc_fence_after();
            // the step's 128 logits: column c is key 128 u + c (block 2u, then 2u+1)
            float v[128];
            bool raw_s = RAW;
            if (s == 0) {
                // own pair: table rows for the diagonal blocks, MMA logits of block 2t for the
                // rows of block 2t+1, block 2t+1 masked for the rows of block 2t; all in log2
                // units
                raw_s = false;
                if (q < 2) {
                    load_diag_row(dg + ((head * nblk + 2 * tile) * kC + r) * kC, v);
#pragma unroll
                    for (int j = 64; j < 128; ++j) v[j] = -INFINITY;
                } else {
                    uint32_t a[32], b[32];
                    tmem_ld32(T_S, a);
                    tmem_ld32(T_S + 32, b);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        v[j] = __uint_as_float(a[j]) * scale_log2;
                        v[32 + j] = __uint_as_float(b[j]) * scale_log2;
                    }
                    load_diag_row(dg + ((head * nblk + 2 * tile + 1) * kC + (r - 64)) * kC, v + 64);
                }
            } else {
                uint32_t a[32], b[32], c[32], d[32];
                tmem_ld32(T_S, a);
                tmem_ld32(T_S + 32, b);
                tmem_ld32(T_S + 64, c);
                tmem_ld32(T_S + 96, d);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = __uint_as_float(a[j]);
                    v[32 + j] = __uint_as_float(b[j]);
                    v[64 + j] = __uint_as_float(c[j]);
                    v[96 + j] = __uint_as_float(d[j]);
                }
                if (!RAW) {
                    const float2 sl2 = make_float2(scale_log2, scale_log2);
                    const float2 z2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float2 w = ffma2(make_float2(v[2 * j], v[2 * j + 1]), sl2, z2);
                        v[2 * j] = w.x;
                        v[2 * j + 1] = w.y;
                    }
                }
            }
            // S is in registers: its TMEM columns may be rewritten by the next step's MMA
            tc_fence_before();
            if (s + 1 < nsteps) mbar_arrive_warp(tbar(t, ScanSmem::SFREE));

            // ---- online softmax with lazy rescaling: the running max is raised only when
            // the step's max exceeds it by more than 2^8; then the row sum and O are rescaled
            float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
            for (int j = 4; j < 124; j += 8)
#pragma unroll
                for (int e = 0; e < 4; ++e) m4[e] = fmax3(m4[e], v[j + 2 * e], v[j + 2 * e + 1]);
            float mx = fmax3(fmax3(m4[0], m4[1], v[124]), fmax3(m4[2], m4[3], v[125]),
                             fmaxf(v[126], v[127]));
            if (raw_s) mx *= scale_log2;
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_run + kRescaleThreshold) {
                if (m_run != -INFINITY) {
                    alpha = ex2_approx(m_run - mx);
                    rescale = true;
                    l_run *= alpha;
                }
                m_run = mx;
            }
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
            const float cs = raw_s ? scale_log2 : 1.f;
            const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(neg_m, neg_m);
            float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            uint32_t pk[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float2 x = ffma2(make_float2(v[2 * j], v[2 * j + 1]), cs2, nm2);
                const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                ls[j & 3] = fadd2(ls[j & 3], p);
                pk[j] = pack_bf16x2(p.x, p.y);
            }
            const float2 l01 = fadd2(ls[0], ls[1]), l23 = fadd2(ls[2], ls[3]);
            const float2 l4 = fadd2(l01, l23);
            l_run += l4.x + l4.y;
            // the P tile was last read by this tile's P.V MMA of step s - 1 (on step 0 it held
            // [K~_{2t}; P_{2t}], read by the MMA that produced this step's S); that P.V also
            // has to be complete before O is rescaled
            if (s >= 1 && !(ok = wwait(tbar(t, ScanSmem::BAR_O), (s - 1) & 1))) break;
            uint8_t *prow = gbase + ScanSmem::p_buf(t);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(prow + h * kQBytes + sw128_offset(r, c)) =
                        make_uint4(pk[32 * h + 4 * c], pk[32 * h + 4 * c + 1],
                                   pk[32 * h + 4 * c + 2], pk[32 * h + 4 * c + 3]);
            if (s >= 1 && __any_sync(0xffffffffu, rescale)) {
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t oa[32];
                    tmem_ld32(T_O + 32 * h, oa);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) oa[j] = __float_as_uint(__uint_as_float(oa[j]) * alpha);
                    tmem_st32(T_O + 32 * h, oa);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive_warp(tbar(t, ScanSmem::PREADY));
        }

        // ---- epilogue: O / l, LSE
        if (ok) ok = wwait(tbar(t, ScanSmem::BAR_O), (nsteps - 1) & 1);
        if (ok) {
            tc_fence_after();
            uint32_t oa[32], ob[32];
            tmem_ld32(T_O, oa);
            tmem_ld32(T_O + 32, ob);
            tmem_ld_wait();
            if (i < L) {
                const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(out + (head * L + i) * kD);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t *src = (c < 4) ? &oa[8 * c] : &ob[8 * (c - 4)];
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
                    dst[c] = w;
                }
                if (lse != nullptr) lse[head * L + i] = (m_run + log2f(l_run)) * 0.69314718055994531f;
            }
        }
        tc_fence_before();
      }
    }

    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Returns cudaErrorInvalidValue if the tensor maps cannot be encoded, and
// cudaErrorInvalidConfiguration if the compiled kernel was given fewer registers than the
// warpgroup split redistributes (its setmaxnreg.inc could then never be satisfied).
cudaError_t launch_scan_tc(const void *v, void *out, float *lse, int BH, int L, float scale,
                           void *ws, uint64_t limit_ns, int force_timeout, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 2, false);
    char *basep = static_cast<char *>(ws);
    CUtensorMap tm_qt, tm_kp128, tm_kp64, tm_pr64, tm_v128;
    const int nrows_kp = lay.nblk * 2 * kC, nrows_pr = (lay.nblk / 2) * 2 * kC;
    if (!make_map_bf16(&tm_qt, basep + lay.off_qt, lay.Lp, BH, kTile) ||
        !make_map_bf16(&tm_kp128, basep + lay.off_kp, nrows_kp, BH, 2 * kC) ||
        !make_map_bf16(&tm_kp64, basep + lay.off_kp, nrows_kp, BH, kC) ||
        !make_map_bf16(&tm_pr64, basep + lay.off_pr, nrows_pr, BH, kC) ||
        !make_map_bf16(&tm_v128, v, L, BH, kTile))
        return cudaErrorInvalidValue;
    auto kern = scale > 0.f ? path_scan_tc_kernel<true> : path_scan_tc_kernel<false>;
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.numRegs * kScanThreads < kRegTotal) return cudaErrorInvalidConfiguration;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kScanSmemBytes);
    if (err != cudaSuccess) return err;
    const int ntile = lay.nblk / 2;
    // shared per token: [K^; K~; Pi] (192 B) and v (128 B)
    const bool hf = heads_fastest((size_t)BH, (size_t)L, 320);
    const dim3 grid = hf ? dim3(BH, (ntile + 1) / 2) : dim3((ntile + 1) / 2, BH);
    kern<<<grid, kScanThreads, kScanSmemBytes, stream>>>(
        tm_qt, tm_kp128, tm_kp64, tm_pr64, tm_v128,
        reinterpret_cast<const __half *>(basep + lay.off_dg), static_cast<__nv_bfloat16 *>(out),
        lse, L, lay.nblk, scale * kLog2e,
        reinterpret_cast<uint32_t *>(basep), limit_ns, force_timeout, hf ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace path
