// K2 (bf16): the right-to-left block scan of PaTH attention on tcgen05 tensor cores.
//
// Technical summary "技術要約: PaTH Attention" §3 (FlashAttention-style algorithm: per-block
// boundary-adjusted queries and keys, a right-to-left scan over key/value blocks that
// accumulates the Householder product, online softmax, nothing L x L in memory); review
// "거리에서 경로로, PaTH Attention" §9 (the same scheme, blockwise preprocessing and
// blockwise updates of the accumulated transform and softmax statistics).
//
// A tile is 128 query rows = two 64-token blocks ib0 = 2t, ib1 = 2t + 1 of one head. With
// q~ the boundary-adjusted queries, k~ the boundary-adjusted keys and P_b = H_start(b) ...
// H_end(b) the dense block transition (all from the preprocessing kernel), the logit of
// row i against key j of an earlier block b is
//     scale * k~_j^T P_{b+1} ... P_{ib-1} q~_i,
// so a state row x_i = q~_i is scored against block ib-1, then x_i <- P_{ib-1} x_i, and so
// on down to block 0. In row form a tile advances as X <- X P_b^T, one 128 x 64 x 64 MMA
// per block, next to S = X K~_b^T and O += P V_b. Steps s = 0 .. ib1 visit block ib1 - s:
//   s = 0 : block ib1; rows 64-127 take their diagonal-block logits, rows 0-63 are masked.
//   s = 1 : block ib0; rows 0-63 take their diagonal-block logits, rows 64-127 the MMA
//           logits of block ib0, and only rows 64-127 advance their state by P_{ib0}.
//   s >= 2: block ib1 - s for every row.
//
// One CTA owns a pair of tiles of one head, A = 2p and B = 2p + 1, and streams the key
// blocks 4p+3, 4p+2, ..., 0 (PaTH-FoX: down to the lower of the two tiles' early-exit
// extents from fox_exit.cu) once through an NS-stage TMA ring: B consumes every block,
// A every block from 4p+1 down, so each stage is loaded once for both tiles. A stage holds
// [K~_b; P_b; K~_b] (K~_b loaded twice) and V_b. Per tile and step, S = X K~_b^T and the
// new state X P_b^T come from ONE MMA with N = 128: B = [K~_b; P_b] on even steps (S lands
// in TMEM columns [0,64), the state in [64,128)) and B = [P_b; K~_b] on odd steps (state in
// [64,128), S in [128,192)), so S is double-buffered while the state accumulator is not.
// O += P V_b follows (N = 64, columns [192,256)). Tile B's columns are at +256.
// Warp roles (512 threads):
//   warps 0-3 / 4-7  softmax of tile A / B, one row per thread (= TMEM lane): load S,
//                    release its buffer, online softmax with lazy rescaling, P tile;
//   warps 8-11       the state recurrence of both tiles (one per TMEM lane quadrant):
//                    fp32 -> bf16 conversion of each new state into a swizzled A tile;
//   warps 12 / 13    issue tile A's / B's S|state MMAs (the recurrence: needs the
//                    converted state and a free S buffer, never the softmax of this step);
//   warps 14 / 15    issue tile A's / B's P.V MMAs and release the stages; warp 14
//                    also feeds the TMA ring (both duties poll, neither blocks the other);
//   warp 12 also owns TMEM.
// Each issuing thread is its own in-order MMA stream: one thread issuing back to back
// cannot keep the tensor core busy with N <= 128 instructions, four can.
// The bf16 state tile and the P tile are single-buffered: the state is rewritten once the
// S|state MMA that read it has completed, P once the tile's previous P.V has completed.
#include "common.cuh"

namespace path {

namespace {

constexpr int kScanThreads = 512;
constexpr int NS = 5;                       // TMA stages ([K~|P|K~] and V of one block each)
constexpr uint32_t kTileBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kVBytes = 64 * 128;      // 64 rows x 64 bf16
constexpr uint32_t kKdupBytes = 64 * 128;   // second copy of K~_b after P_b
constexpr uint32_t kStageBytes = kTileBytes + kKdupBytes + kVBytes;
constexpr float kRescaleThreshold = 8.f;    // lazy rescale: keep the old max within 2^8

struct ScanSmem {
    // byte offsets from the 1024-aligned base
    __host__ __device__ static constexpr uint32_t q_st(int t) { return (uint32_t)t * kTileBytes; }
    __host__ __device__ static constexpr uint32_t p_buf(int t) { return (uint32_t)(2 + t) * kTileBytes; }
    static constexpr uint32_t stage = 4 * kTileBytes;
    static constexpr uint32_t bars = stage + NS * kStageBytes;
    // barrier indices: the ring, then ten per tile (S buffers have their own), then one
    static constexpr int FULL = 0, EMPTY = NS, TILE0 = 2 * NS;
    static constexpr int QFULL = 0, BAR_SX = 1 /* 2 */, BAR_O = 3, QREADY = 4,
                         SFREE = 5 /* 2 */, PREADY = 7, FINAL_SX = 8, FINAL_PV = 9;
    __host__ __device__ static constexpr int per_tile(int t, int which) { return TILE0 + 10 * t + which; }
    static constexpr int NEVER = TILE0 + 20, NBARS = TILE0 + 21;
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

// RAW: no bias and a positive scale, so the scale is applied inside the exponent's FFMA.
template <bool FOX, bool RAW>
__global__ void __launch_bounds__(kScanThreads, 1)
path_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_qt,
                    const __grid_constant__ CUtensorMap tm_kp,
                    const __grid_constant__ CUtensorMap tm_k64,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __nv_bfloat16 *__restrict__ qt, const __half *__restrict__ dg,
                    const float *__restrict__ c2, const int *__restrict__ first_blk,
                    __nv_bfloat16 *__restrict__ out,
                    float *__restrict__ lse, int L, int Lp, int nblk, float scale_log2,
                    uint32_t *status, uint64_t limit_ns, int force_timeout) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = nblk >> 1;
    const int npair = (ntile + 1) >> 1;
    const int pair = npair - 1 - (int)blockIdx.x;  // heaviest pairs first
    const int bh = blockIdx.y;
    const bool hasB = 2 * pair + 1 < ntile;
    const int top = hasB ? 4 * pair + 3 : 4 * pair + 1;  // first key block of the stream
    // lowest key block each tile visits: 0, or for PaTH-FoX the early-exit extent of its
    // two query blocks (never above the tile's own first block)
    int fb[2] = {0, 0};
    if (FOX) {
        for (int t = 0; t < (hasB ? 2 : 1); ++t) {
            const int *f = first_blk + (size_t)blockIdx.y * nblk + 4 * pair + 2 * t;
            fb[t] = min(min(__ldg(f), __ldg(f + 1)), 4 * pair + 2 * t);
        }
    }
    const int nstream = top + 1 - (hasB ? min(fb[0], fb[1]) : fb[0]);
    // tile t (0 = A, 1 = B): tile index, its step count, and stream position of its step 0
    auto tile_of = [&](int t) { return 2 * pair + t; };
    auto nsteps_of = [&](int t) { return 2 * tile_of(t) + 2 - fb[t]; };
    auto off_of = [&](int t) { return top - (2 * tile_of(t) + 1); };
    // whether tile t reads stream position n
    auto reads = [&](int t, int n) {
        return (t == 0 || hasB) && n >= off_of(t) && n < off_of(t) + nsteps_of(t);
    };

    auto bar = [&](int i) { return base + ScanSmem::bars + 8u * (uint32_t)i; };
    auto tbar = [&](int t, int which) { return bar(ScanSmem::per_tile(t, which)); };
    volatile uint32_t *abort_flag =
        reinterpret_cast<volatile uint32_t *>(gbase + ScanSmem::abort_flag);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + ScanSmem::tmem_slot);
    const Waiter wait{abort_flag, status, limit_ns};

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bar(ScanSmem::FULL + i), 1);
            mbar_init(bar(ScanSmem::EMPTY + i), 2);  // two arrivals per use (see issuers)
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(tbar(t, ScanSmem::QFULL), 1);
            mbar_init(tbar(t, ScanSmem::BAR_SX), 1);
            mbar_init(tbar(t, ScanSmem::BAR_SX + 1), 1);
            mbar_init(tbar(t, ScanSmem::BAR_O), 1);
            mbar_init(tbar(t, ScanSmem::QREADY), 4);  // one arrival per warp
            mbar_init(tbar(t, ScanSmem::SFREE), 4);
            mbar_init(tbar(t, ScanSmem::SFREE + 1), 4);
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
    // per tile: S of even steps [0,64), new state [64,128), S of odd steps [128,192), O
    auto t_state = [&](int t) { return tmem + 256u * (uint32_t)t + 64u; };
    auto t_s = [&](int t, int s) { return tmem + 256u * (uint32_t)t + ((s & 1) ? 128u : 0u); };
    auto t_sxd = [&](int t, int s) { return tmem + 256u * (uint32_t)t + ((s & 1) ? 64u : 0u); };
    auto t_o = [&](int t) { return tmem + 256u * (uint32_t)t + 192u; };
    auto stage_kp = [&](int i) { return base + ScanSmem::stage + (uint32_t)i * kStageBytes; };
    auto stage_v = [&](int i) { return stage_kp(i) + kTileBytes + kKdupBytes; };

    if (warp >= 12 && warp <= 13) {
        // ------------------------------------------------------------ S|state issuers
        const int t = warp - 12;
        if (lane == 0 && (t == 0 || hasB)) {
            constexpr uint32_t ID_SX = idesc_bf16(128, 128, false);
            const int nst = nsteps_of(t), off = off_of(t);
            bool ok = true;
            if (force_timeout && t == 0) ok = wait(bar(ScanSmem::NEVER), 0);  // nothing arrives here
            for (int s = 1; ok && s < nst; ++s) {
                const int n = s + off, st = n % NS;
                if (!(ok = wait(bar(ScanSmem::FULL + st), (n / NS) & 1))) break;
                // the state of step s: q~ (step 1) or the converted new state of step s - 1
                if (s == 1) {
                    if (!(ok = wait(tbar(t, ScanSmem::QFULL), 0))) break;
                } else if (!(ok = wait(tbar(t, ScanSmem::QREADY), (s - 2) & 1))) {
                    break;
                }
                // S buffer s & 1 was last read by the softmax of step s - 2
                if (s >= 3 && !(ok = wait(tbar(t, ScanSmem::SFREE + (s & 1)), ((s - 3) >> 1) & 1)))
                    break;
                tc_fence_after();
                const uint64_t a_q = sdesc_sw128(base + ScanSmem::q_st(t), 16, 1024);
                const uint64_t b_kp =
                    sdesc_sw128(stage_kp(st) + ((s & 1) ? 64u * 128u : 0u), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(t_sxd(t, s), a_q + 2 * kk, b_kp + 2 * kk, ID_SX, kk > 0);
                umma_commit(tbar(t, ScanSmem::BAR_SX + (s & 1)));
            }
            umma_commit(tbar(t, ScanSmem::FINAL_SX));
            const uint64_t t0 = cycles_now();
            while (!mbar_try_wait(tbar(t, ScanSmem::FINAL_SX), 0) &&
                   cycles_now() - t0 < ns_to_cycles(limit_ns)) {
            }
        }
    } else if (warp >= 14 && warp <= 15) {
        // ------------------------------------------------------------ P.V issuers (+ TMA)
        // Tile A's thread also feeds the TMA ring; both duties poll without blocking.
        const int t = warp - 14;
        const bool producer = (t == 0);
        if (lane == 0 && (t == 0 || hasB)) {
            constexpr uint32_t ID_PV = idesc_bf16(128, 64, true);
            const int nst = nsteps_of(t), off = off_of(t);
            if (producer) {
                tma_prefetch_desc(&tm_qt);
                tma_prefetch_desc(&tm_kp);
                tma_prefetch_desc(&tm_k64);
                tma_prefetch_desc(&tm_v);
                for (int tt = 0; tt < (hasB ? 2 : 1); ++tt) {
                    mbar_arrive_expect_tx(tbar(tt, ScanSmem::QFULL), kTileBytes);
                    tma_load_3d(base + ScanSmem::q_st(tt), &tm_qt, tbar(tt, ScanSmem::QFULL), 0,
                                tile_of(tt) * kTile, bh);
                }
            }
            int n_fill = producer ? 0 : nstream;  // next stream position to load
            int s = 0;                            // next P.V step
            bool ok = true;
            uint64_t t_last = cycles_now();
            while (ok && (s < nst || n_fill < nstream)) {
                bool progress = false;
                if (n_fill < nstream &&
                    (n_fill < NS ||
                     mbar_test_wait(bar(ScanSmem::EMPTY + n_fill % NS), ((n_fill / NS) - 1) & 1))) {
                    const int st = n_fill % NS, b = top - n_fill;
                    if (n_fill == 0) {  // the top tile's own diagonal block: values only
                        mbar_arrive_expect_tx(bar(ScanSmem::FULL + st), kVBytes);
                    } else {
                        mbar_arrive_expect_tx(bar(ScanSmem::FULL + st), kStageBytes);
                        tma_load_3d(stage_kp(st), &tm_kp, bar(ScanSmem::FULL + st), 0, b * 2 * kC, bh);
                        tma_load_3d(stage_kp(st) + kTileBytes, &tm_k64, bar(ScanSmem::FULL + st), 0,
                                    b * 2 * kC, bh);
                    }
                    tma_load_3d(stage_v(st), &tm_v, bar(ScanSmem::FULL + st), 0, b * kC, bh);
                    ++n_fill;
                    progress = true;
                }
                if (s < nst) {
                    const int n = s + off, st = n % NS;
                    const bool in_ready = (s > 0) || mbar_test_wait(bar(ScanSmem::FULL + st), (n / NS) & 1);
                    if (in_ready && mbar_test_wait(tbar(t, ScanSmem::PREADY), s & 1)) {
                        tc_fence_after();
                        const uint64_t a_p = sdesc_sw128(base + ScanSmem::p_buf(t), 16, 1024);
                        const uint64_t b_v = sdesc_sw128(stage_v(st), 1024, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(t_o(t), a_p + 2 * kk, b_v + 128 * kk, ID_PV, (s > 0 || kk > 0));
                        umma_commit(tbar(t, ScanSmem::BAR_O));
                        // this step's S|state MMA completed before its softmax finished, so
                        // this commit covers every read of the stage by tile t; two arrivals
                        // per stage (a stage read by one tile only gets both from that tile)
                        umma_commit(bar(ScanSmem::EMPTY + st));
                        if (!reads(1 - t, n)) umma_commit(bar(ScanSmem::EMPTY + st));
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
                for (int n = (n_fill > NS ? n_fill - NS : 0); n < n_fill; ++n) {
                    const uint32_t bfull = bar(ScanSmem::FULL + n % NS);
                    const uint64_t t0 = cycles_now();
                    while (!mbar_try_wait(bfull, (n / NS) & 1) &&
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
    } else if (warp >= 8) {
        // ------------------------------------------------------------ state warps
        const int quad = warp - 8;
        const int r = quad * 32 + lane;          // row of both tiles = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const size_t head = (size_t)bh;
        bool ok = true;
        auto wwait = [&](uint32_t b_, uint32_t par) {
            return __all_sync(0xffffffffu, wait(b_, par)) != 0;
        };
        const int smax = hasB ? max(nsteps_of(0), nsteps_of(1)) : nsteps_of(0);
        for (int s = 1; s < smax && ok; ++s) {
            for (int t = hasB ? 1 : 0; t >= 0; --t) {
                if (s >= nsteps_of(t) - 1) continue;  // the last step needs no new state
                if (!(ok = wwait(tbar(t, ScanSmem::BAR_SX + (s & 1)), ((s - 1) >> 1) & 1))) break;
                tc_fence_after();
                // the state of step s + 1 replaces that of step s, whose only reader (the
                // S|state MMA of step s) has completed
                uint8_t *row = gbase + ScanSmem::q_st(t);
                if (s >= 2 || quad >= 2) {
                    uint32_t qa[32], qb[32];
                    tmem_ld32(t_state(t) + lane_base, qa);
                    tmem_ld32(t_state(t) + 32 + lane_base, qb);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t *src = (c < 4) ? &qa[8 * c] : &qb[8 * (c - 4)];
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1]));
                        u.y = pack_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3]));
                        u.z = pack_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5]));
                        u.w = pack_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7]));
                        *reinterpret_cast<uint4 *>(row + sw128_offset(r, c)) = u;
                    }
                } else {
                    // rows of block ib0 keep q~ through step 1: copy it from the workspace
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        qt + (head * Lp + (size_t)tile_of(t) * kTile + r) * kD);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(row + sw128_offset(r, c)) = __ldg(src + c);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive_warp(tbar(t, ScanSmem::QREADY));
            }
        }
        tc_fence_before();
    } else if (warp < 4 || hasB) {
        // ------------------------------------------------------------ softmax warps
        const int t = warp >> 2;                 // 0 = tile A, 1 = tile B
        const int r = threadIdx.x - 128 * t;     // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int tile = tile_of(t);
        const int ib0 = 2 * tile, ib1 = 2 * tile + 1;
        const int nsteps = nsteps_of(t);
        const int i = tile * kTile + r;          // query index
        const size_t head = (size_t)bh;
        float m_run = -INFINITY, l_run = 0.f;
        const float c2_i = FOX ? c2[head * Lp + i] : 0.f;
        bool ok = true;
        // every lane of a warp leaves together: tcgen05.ld/st are warp-collective
        auto wwait = [&](uint32_t b_, uint32_t par) {
            return __all_sync(0xffffffffu, wait(b_, par)) != 0;
        };
        const uint32_t T_O = t_o(t);

        for (int s = 0; s < nsteps && ok; ++s) {
            const int b = ib1 - s;
            // logits of this row come from the diagonal-block table (step 0, and step 1 for
            // rows 0-63) or from S in TMEM; they are read twice, in 32-column chunks (row
            // max, then exponentials), which keeps the live register set small
            bool from_diag = false;
            int diag_blk = 0, diag_row = 0;
            if (s == 0) {
                from_diag = true;
                diag_blk = ib1;
                diag_row = r - 64;
            } else {
                if (!(ok = wwait(tbar(t, ScanSmem::BAR_SX + (s & 1)), ((s - 1) >> 1) & 1))) break;
                tc_fence_after();
                if (s == 1 && (warp & 3) < 2) {
                    from_diag = true;
                    diag_blk = ib0;
                    diag_row = r;
                }
            }
            const uint32_t ts = t_s(t, s) + lane_base;
            const __half *drow = dg + (((head * nblk + diag_blk) * kC) + (diag_row < 0 ? 0 : diag_row)) * kC;
            const bool raw_s = RAW && !from_diag;
            // 32 logits of chunk h (log2 units, or raw scores when raw_s)
            auto load_chunk = [&](int h, float (&v)[32]) {
                if (from_diag) {
                    if (diag_row >= 0) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(drow + 32 * h);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            const uint4 c = __ldg(src + q8);
                            const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f =
                                    __half22float2(*reinterpret_cast<const __half2 *>(&w4[e]));
                                v[8 * q8 + 2 * e] = f.x;
                                v[8 * q8 + 2 * e + 1] = f.y;
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = -INFINITY;
                    }
                } else {
                    uint32_t u[32];
                    tmem_ld32(ts + 32 * h, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = RAW ? __uint_as_float(u[j]) : __uint_as_float(u[j]) * scale_log2;
                    if (FOX) {
                        const float4 *cj =
                            reinterpret_cast<const float4 *>(c2 + head * Lp + b * kC + 32 * h);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            const float4 c = __ldg(cj + q4);
                            v[4 * q4 + 0] += c2_i - c.x;
                            v[4 * q4 + 1] += c2_i - c.y;
                            v[4 * q4 + 2] += c2_i - c.z;
                            v[4 * q4 + 3] += c2_i - c.w;
                        }
                    }
                }
            };

            // ---- one pass over two 32-column chunks: online max with lazy rescaling (a
            // chunk raises the running max only if it exceeds it by more than 2^8; then the
            // row sum, O and the chunk already packed are rescaled), exponentials, row sum
            float alpha = 1.f;   // accumulated rescale factor of O for this step
            bool rescale = false;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[32];
                load_chunk(h, v);
                float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
                for (int j = 4; j < 32; j += 4) {
                    m4[0] = fmaxf(m4[0], v[j]);
                    m4[1] = fmaxf(m4[1], v[j + 1]);
                    m4[2] = fmaxf(m4[2], v[j + 2]);
                    m4[3] = fmaxf(m4[3], v[j + 3]);
                }
                float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                if (raw_s) mx *= scale_log2;
                if (mx > m_run + kRescaleThreshold) {
                    if (m_run != -INFINITY) {
                        const float a = ex2_approx(m_run - mx);
                        alpha *= a;
                        rescale = true;
                        l_run *= a;
                        ls[0] *= a; ls[1] *= a; ls[2] *= a; ls[3] *= a;
                        if (h == 1) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float2 f = unpack_bf16x2(pk[j]);
                                pk[j] = pack_bf16x2(f.x * a, f.y * a);
                            }
                        }
                    }
                    m_run = mx;
                }
                const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
                const float cs = raw_s ? scale_log2 : 1.f;
                const float neg_m = -m_use;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p0 = ex2_approx(fmaf(v[2 * j], cs, neg_m));
                    const float p1 = ex2_approx(fmaf(v[2 * j + 1], cs, neg_m));
                    ls[(2 * j) & 3] += p0;
                    ls[(2 * j + 1) & 3] += p1;
                    pk[16 * h + j] = pack_bf16x2(p0, p1);
                }
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // the P tile was last read by this tile's P.V MMA of step s - 1, which also has
            // to be complete before O is rescaled
            if (s >= 1 && !(ok = wwait(tbar(t, ScanSmem::BAR_O), (s - 1) & 1))) break;
            uint8_t *prow = gbase + ScanSmem::p_buf(t);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(prow + sw128_offset(r, c)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            if (s >= 1) {
                // S has been read for the last time: its buffer may be rewritten
                tc_fence_before();
                mbar_arrive_warp(tbar(t, ScanSmem::SFREE + (s & 1)));
            }
            if (s >= 1 && __any_sync(0xffffffffu, rescale)) {
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t oa[32];
                    tmem_ld32(T_O + lane_base + 32 * h, oa);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) oa[j] = __float_as_uint(__uint_as_float(oa[j]) * alpha);
                    tmem_st32(T_O + lane_base + 32 * h, oa);
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
            tmem_ld32(T_O + lane_base, oa);
            tmem_ld32(T_O + lane_base + 32, ob);
            tmem_ld_wait();
            if (i < L) {
                const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(out + (head * L + i) * kD);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t *src = (c < 4) ? &oa[8 * c] : &ob[8 * (c - 4)];
                    uint4 u;
                    u.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
                    u.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
                    u.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
                    u.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
                    dst[c] = u;
                }
                if (lse != nullptr) lse[head * L + i] = (m_run + log2f(l_run)) * 0.69314718055994531f;
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled get_encode_tiled() {
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

// 3-D bf16 map over (heads, rows, 64 columns) with a (1, box_rows, 64) box, 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *ptr, int rows, int heads, int box_rows) {
    EncodeTiled enc = get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)rows * kD * 2};
    cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Returns cudaErrorInvalidValue if the tensor maps cannot be encoded.
cudaError_t launch_scan_tc(const void *v, void *out, float *lse, bool fox, int BH, int L,
                           float scale, void *ws, uint64_t limit_ns, int force_timeout,
                           cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 2, fox);
    char *basep = static_cast<char *>(ws);
    CUtensorMap tm_qt, tm_kp, tm_v;
    CUtensorMap tm_k64;
    if (!make_map(&tm_qt, basep + lay.off_qt, lay.Lp, BH, kTile) ||
        !make_map(&tm_kp, basep + lay.off_kp, lay.nblk * 2 * kC, BH, kTile) ||
        !make_map(&tm_k64, basep + lay.off_kp, lay.nblk * 2 * kC, BH, kC) ||
        !make_map(&tm_v, v, L, BH, kC))
        return cudaErrorInvalidValue;
    auto kern = fox ? path_scan_tc_kernel<true, false>
                    : (scale > 0.f ? path_scan_tc_kernel<false, true>
                                   : path_scan_tc_kernel<false, false>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kScanSmemBytes);
    if (err != cudaSuccess) return err;
    const int ntile = lay.nblk / 2;
    dim3 grid((ntile + 1) / 2, BH);
    kern<<<grid, kScanThreads, kScanSmemBytes, stream>>>(
        tm_qt, tm_kp, tm_k64, tm_v, reinterpret_cast<const __nv_bfloat16 *>(basep + lay.off_qt),
        reinterpret_cast<const __half *>(basep + lay.off_dg),
        fox ? reinterpret_cast<const float *>(basep + lay.off_c2) : nullptr,
        fox ? reinterpret_cast<const int *>(basep + lay.off_fb) : nullptr,
        static_cast<__nv_bfloat16 *>(out), lse, L, lay.Lp, lay.nblk, scale * kLog2e,
        reinterpret_cast<uint32_t *>(basep), limit_ns, force_timeout);
    return cudaGetLastError();
}

}  // namespace path
