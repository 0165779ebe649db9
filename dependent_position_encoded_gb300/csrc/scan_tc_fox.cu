// K2 for PaTH-FoX (bf16): the right-to-left block scan with the forget-gate bias and the
// early exit, one key block per step, on tcgen05 tensor cores.
//
// Technical summary "技術要約: PaTH Attention" §3 (FlashAttention-style algorithm: per-block
// boundary-adjusted queries and keys, a right-to-left scan over key/value blocks that
// accumulates the Householder product, online softmax, nothing L x L in memory); review
// "거리에서 경로로, PaTH Attention" §9 (the same scheme, blockwise preprocessing and
// blockwise updates of the accumulated transform and softmax statistics).
//
// A tile is 128 query rows = the 64-token blocks (2T, 2T+1) of one head. With q~ the
// boundary-adjusted queries, k~ the boundary-adjusted keys and P_b the dense block
// transition, a state row x_i starts as q~_i and scores an earlier key block b as x . k~_j,
// then leaves as P_b x. In row form one MMA with N = 128 gives the logits and the new state:
//     [S | X'] = X [K~_b; P_b]^T,
// followed by O += P V_b (K = 64); every logit takes the gate bias c_i - c_j (review "거리에서
// 경로로, PaTH Attention" §4; technical summary §2 "拡張: PaTH-FoX"). The tile visits key
// blocks 2T+1, 2T, ..., down to the lower of its two query blocks' early-exit extents from
// fox_exit.cu (one key block per step: the exit acts at block granularity). Step 0
// (block 2T+1) is the diagonal-block table for the rows of block 2T+1 and nothing for the
// rows of block 2T; step 1 (block 2T) is the table for the rows of block 2T, which keep q~
// as their state, and the MMA for the rows of block 2T+1; from step 2 on every row takes the
// MMA.
//
// (The plain forward's scan, scan_tc.cu, takes two key blocks per step through block-pair
// products, which pays off over long unskipped walks; with the exit a tile visits a few
// blocks and the pair products would cost more than they save.)
// Everything the recurrence carries stays in tensor memory: the logits and the new state
// come out of the MMA into TMEM, the bf16 state goes back into TMEM and is the next MMA's A
// operand, and the softmax writes P into TMEM as the A operand of P.V. Shared memory holds
// only the streamed B operands ([K~_b; P_b] and V_b, which the preprocessing writes block by
// block) and the tiles' q~, so the loop issues no shared-memory stores and no proxy fences,
// and the tensor cores read only B from shared memory.
//
// A work item is the tiles A = 2p and B = 2p + 1 of one head; it streams the key blocks
// 4p+3, 4p+2, ... down to the lower extent once (each block serves both tiles) through two
// TMA rings: [K~_b; P_b] (released when both S|state MMAs on it have completed) and V_b
// (released after both P.V MMAs). Tile B's step s and tile A's step s - 2 read the same
// stream position. The kernel is persistent, one CTA per SM looping over the items: with the
// exit an item is only a few key blocks long, so barriers, TMEM and the rings are set up
// once, every barrier phase and ring slot continues from one item to the next, and the next
// item's q~ tiles and operands stream in while the current item runs.
// TMEM per tile (256 columns, tile B at +256): S [0,64) and X' [64,128) (one N = 128 MMA),
// O [128,192), P [192,224) and the carried state [224,256) as bf16 pairs.
// Warp roles (512 threads; registers moved to the row warps with setmaxnreg):
//   warps 0-3 / 4-7  tile A / B, one row per thread (= TMEM lane): once the step's MMA has
//                    completed, load S and X', write X' back as the bf16 state of the next
//                    step (so the recurrence waits for nothing else), then the online
//                    softmax of the 64 logits with lazy rescaling and P into TMEM;
//   warps 8 / 9      issue tile A's / B's S|state MMAs (they need the previous step's S and
//                    X' read and the new state written); warp 8 also owns TMEM;
//   warps 10 / 11    issue tile A's / B's P.V MMAs and release the value stages;
//   warp 12          loads the items' q~ tiles and feeds the two TMA rings (warps 13-15 have
//                    no role).
// P and the carried state are single-buffered: P is rewritten once the tile's previous P.V
// has completed, the state once the S|state MMA that read it has completed.
#include "common.cuh"

namespace path {

namespace {

constexpr int kScanThreads = 512;
constexpr int NR = 6;                          // TMA stages of [K~_b; P_b] (S|state operand)
constexpr int NV = 6;                          // TMA stages of V_b (P.V operand)
constexpr uint32_t kQBytes = 128 * 128;        // 128 rows x 64 bf16
constexpr uint32_t kRBytes = 128 * 128;        // [K~_b; P_b]
constexpr uint32_t kVBytes = 64 * 128;         // V_b
constexpr float kRescaleThreshold = 8.f;       // lazy rescale: keep the old max within 2^8
// Registers per thread after the split (launch: 128 for all 512 threads). Each SM
// sub-partition holds two row warps and two of the others, whose sum fits its 16384.
constexpr int kRegRow = 168, kRegOther = 88;
static_assert(256 * kRegRow + 256 * kRegOther <= 65536, "register split exceeds the register file");
// TMEM columns within a tile's 256
constexpr uint32_t TC_S = 0, TC_X = 64, TC_O = 128, TC_P = 192, TC_XB = 224;


struct ScanSmem {
    // byte offsets from the 1024-aligned base
    __host__ __device__ static constexpr uint32_t q_st(int t) { return (uint32_t)t * kQBytes; }
    static constexpr uint32_t stage_r = 2 * kQBytes;
    static constexpr uint32_t stage_v = stage_r + NR * kRBytes;
    static constexpr uint32_t bars = stage_v + NV * kVBytes;
    // barrier indices: the two rings, then eight per tile, then one
    static constexpr int FULL_R = 0, EMPTY_R = NR, FULL_V = 2 * NR, EMPTY_V = 2 * NR + NV,
                         TILE0 = 2 * NR + 2 * NV;
    // NEXT: the tile's S and X' of the last MMA have been read and the state of the next
    // step written (first phase of an item: q~ written); QFREE: the row warps have taken the
    // item's q~ tile, which the next item's may replace
    static constexpr int QFULL = 0, QFREE = 1, SX_DONE = 2, O_DONE = 3, NEXT = 4, PREADY = 5,
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
    // Bounded wait; on timeout records the status and raises the CTA abort flag. Between
    // checks of the clock and the abort flag the thread sleeps on the barrier (up to 20 us).
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = cycles_now(), lim = ns_to_cycles(limit_ns);
        for (;;) {
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
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

// tcgen05.mma kind::f16 with the A operand in tensor memory (M = 128: lane = row, each 32-bit
// column two consecutive K elements, eight columns per K = 16 instruction).
__device__ __forceinline__ void umma_bf16_tA(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
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

// One work item: a pair of tiles (A = 2p, B = 2p + 1) of one head. Every role derives the
// same item sequence, so the rings' and the per-tile barriers' phases continue across items
// from counters each role keeps for itself.
struct Item {
    int bh, pair, top, nstream, nr_total;
    bool hasB, hole2;
    int nst0, nst1, off1;  // steps of tiles A and B, and stream position of B's step 0
    __device__ __forceinline__ int tile(int t) const { return 2 * pair + t; }
    __device__ __forceinline__ bool has(int t) const { return t == 0 || hasB; }
    __device__ __forceinline__ int nsteps(int t) const { return t ? nst1 : nst0; }
    // stream position of tile t's step 0 (tile A's is 2 when tile B exists)
    __device__ __forceinline__ int off(int t) const { return t ? off1 : (hasB ? 2 : 0); }
    // whether tile t reads stream position n (its values), and the S|state operand of
    // position n (every step but the tile's first)
    __device__ __forceinline__ bool reads(int t, int n) const {
        return has(t) && n >= off(t) && n < off(t) + nsteps(t);
    }
    __device__ __forceinline__ bool reads_r(int t, int n) const { return reads(t, n) && n > off(t); }
    // The operand ring skips position 0 (only the top tile's diagonal step) and, when tile
    // B's extent ends at its own lower block, position 2 (tile A's diagonal step), which no
    // S|state MMA reads either: the ring index of position n within the item.
    __device__ __forceinline__ int ring_r(int n) const { return n - 1 - ((hole2 && n > 2) ? 1 : 0); }
};

// Item idx of ncta tile pairs per head: head idx / ncta, its tile pairs heaviest first.
__device__ __forceinline__ Item make_item(int idx, int ncta, int ntile, int nblk,
                                          const int *__restrict__ first_blk) {
    Item it;
    it.bh = idx / ncta;
    it.pair = ncta - 1 - idx % ncta;
    it.hasB = 2 * it.pair + 1 < ntile;
    it.top = 2 * (it.hasB ? 2 * it.pair + 1 : 2 * it.pair) + 1;  // first key block of the stream
    // lowest key block a tile visits: the lower early-exit extent of its two query blocks
    // (never above the tile's lower block)
    auto lowest = [&](int tile) {
        const int *f = first_blk + (size_t)it.bh * nblk + 2 * tile;
        return min(min(__ldg(f), __ldg(f + 1)), 2 * tile);
    };
    const int tA = 2 * it.pair, loA = lowest(tA);
    const int loB = it.hasB ? lowest(tA + 1) : loA;
    it.nst0 = 2 * tA + 2 - loA;
    it.nst1 = it.hasB ? 2 * (tA + 1) + 2 - loB : 0;
    it.off1 = 0;
    it.nstream = it.top + 1 - min(loA, loB);
    it.hole2 = it.hasB && it.nst1 == 2;
    it.nr_total = it.nstream - 1 - (it.hole2 ? 1 : 0);
    return it;
}

// Persistent: CTA c takes items c, c + gridDim.x, ... (one CTA per SM), so the barriers, TMEM
// and the TMA rings are set up once and the next item's q~ and operands stream in while the
// current item runs.
__global__ void __launch_bounds__(kScanThreads, 1)
path_scan_tc_fox_kernel(const __grid_constant__ CUtensorMap tm_qt,
                        const __grid_constant__ CUtensorMap tm_kp128,
                        const __grid_constant__ CUtensorMap tm_v64,
                        const __half *__restrict__ dg, const float *__restrict__ c2,
                        const float *__restrict__ pbase, const int *__restrict__ first_blk,
                        __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, int L, int Lp,
                        int nblk, int nitems, float scale_log2, uint32_t *status,
                        uint64_t limit_ns, int force_timeout) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = nblk >> 1;                   // 128-row tiles per head
    const int ncta = (ntile + 1) >> 1;             // tile pairs per head

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
            mbar_init(tbar(t, ScanSmem::QFREE), 4);  // one arrival per warp
            mbar_init(tbar(t, ScanSmem::SX_DONE), 1);
            mbar_init(tbar(t, ScanSmem::O_DONE), 1);
            mbar_init(tbar(t, ScanSmem::NEXT), 4);
            mbar_init(tbar(t, ScanSmem::PREADY), 4);
            mbar_init(tbar(t, ScanSmem::FINAL_SX), 1);
            mbar_init(tbar(t, ScanSmem::FINAL_PV), 1);
        }
        mbar_init(bar(ScanSmem::NEVER), 1);
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto t_base = [&](int t) { return tmem + 256u * (uint32_t)t; };
    auto stage_r = [&](int i) { return base + ScanSmem::stage_r + (uint32_t)i * kRBytes; };
    auto stage_v = [&](int i) { return base + ScanSmem::stage_v + (uint32_t)i * kVBytes; };

    // Registers move to the row warps; each warpgroup executes its setmaxnreg once, at the
    // head of its roles.
    if (warp >= 8) {
      reg_alloc_dec<kRegOther>();
      if (warp == 8 || warp == 9) {
        // ------------------------------------------------------------ S|state issuers
        const int t = warp - 8;
        if (lane == 0) {
            constexpr uint32_t ID_SX = idesc_bf16(128, 128, false);
            bool ok = true;
            if (force_timeout && t == 0) ok = wait(bar(ScanSmem::NEVER), 0);  // nothing arrives here
            const uint32_t a_x = t_base(t) + TC_XB;
            int rb = 0, sxb = 0;  // operands consumed and MMAs issued in earlier items
            for (int idx = blockIdx.x; ok && idx < nitems; idx += gridDim.x) {
                const Item it = make_item(idx, ncta, ntile, nblk, first_blk);
                if (it.has(t)) {
                    const int nst = it.nsteps(t);
                    for (int s = 1; ok && s < nst; ++s) {
                        const int n = s + it.off(t), m = rb + it.ring_r(n), st = m % NR;
                        if (!(ok = wait(bar(ScanSmem::FULL_R + st), (m / NR) & 1))) break;
                        // the carried state of step s written (q~ for s = 1), S and X' of
                        // step s - 1 read
                        if (!(ok = wait(tbar(t, ScanSmem::NEXT), (sxb + s - 1) & 1))) break;
                        tc_fence_after();
                        const uint64_t b = sdesc_sw128(stage_r(st), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16_tA(t_base(t) + TC_S, a_x + 8 * kk, b + 2 * kk, ID_SX, kk > 0);
                        // the operand stage is free once both tiles' MMAs on it have
                        // completed (a stage read by one tile only gets both arrivals from it)
                        umma_commit(bar(ScanSmem::EMPTY_R + st));
                        if (!it.reads_r(1 - t, n)) umma_commit(bar(ScanSmem::EMPTY_R + st));
                        umma_commit(tbar(t, ScanSmem::SX_DONE));
                    }
                    sxb += nst - 1;
                }
                rb += it.nr_total;
            }
            umma_commit(tbar(t, ScanSmem::FINAL_SX));
            const uint64_t t0 = cycles_now();
            while (!mbar_try_wait(tbar(t, ScanSmem::FINAL_SX), 0) &&
                   cycles_now() - t0 < ns_to_cycles(limit_ns)) {
            }
        }
      } else if (warp == 10 || warp == 11) {
        // ------------------------------------------------------------ P.V issuers
        const int t = warp - 10;
        if (lane == 0) {
            constexpr uint32_t ID_PV = idesc_bf16(128, 64, true);
            const uint32_t a_p = t_base(t) + TC_P;
            bool ok = true;
            int vb = 0, pvb = 0;  // values consumed and MMAs issued in earlier items
            for (int idx = blockIdx.x; ok && idx < nitems; idx += gridDim.x) {
                const Item it = make_item(idx, ncta, ntile, nblk, first_blk);
                if (it.has(t)) {
                    const int nst = it.nsteps(t);
                    for (int s = 0; ok && s < nst; ++s) {
                        const int n = s + it.off(t), v = vb + n, st = v % NV;
                        if (!(ok = wait(bar(ScanSmem::FULL_V + st), (v / NV) & 1))) break;
                        if (!(ok = wait(tbar(t, ScanSmem::PREADY), (pvb + s) & 1))) break;
                        tc_fence_after();
                        const uint64_t b_v = sdesc_sw128(stage_v(st), 1024, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16_tA(t_base(t) + TC_O, a_p + 8 * kk, b_v + 128 * kk, ID_PV,
                                         (s > 0 || kk > 0));
                        umma_commit(tbar(t, ScanSmem::O_DONE));
                        // two arrivals per value stage (a stage read by one tile only gets
                        // both from that tile)
                        umma_commit(bar(ScanSmem::EMPTY_V + st));
                        if (!it.reads(1 - t, n)) umma_commit(bar(ScanSmem::EMPTY_V + st));
                    }
                    pvb += nst;
                }
                vb += it.nstream;
            }
            umma_commit(tbar(t, ScanSmem::FINAL_PV));
            const uint64_t t0 = cycles_now();
            while (!mbar_try_wait(tbar(t, ScanSmem::FINAL_PV), 0) &&
                   cycles_now() - t0 < ns_to_cycles(limit_ns)) {
            }
        }
      } else if (warp == 12) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_qt);
            tma_prefetch_desc(&tm_kp128);
            tma_prefetch_desc(&tm_v64);
            int rfill = 0, vfill = 0;  // operands and values loaded so far (all items)
            int qc[2] = {0, 0};        // q~ tiles loaded so far per tile slot
            bool ok = true;
            for (int idx = blockIdx.x; ok && idx < nitems; idx += gridDim.x) {
                const Item it = make_item(idx, ncta, ntile, nblk, first_blk);
                // q~ of the item's tiles, once the row warps have taken the previous one
                for (int tt = 0; ok && tt < (it.hasB ? 2 : 1); ++tt) {
                    if (qc[tt] > 0 && !(ok = wait(tbar(tt, ScanSmem::QFREE), (qc[tt] - 1) & 1)))
                        break;
                    mbar_arrive_expect_tx(tbar(tt, ScanSmem::QFULL), kQBytes);
                    tma_load_3d(base + ScanSmem::q_st(tt), &tm_qt, tbar(tt, ScanSmem::QFULL), 0,
                                it.tile(tt) * kTile, it.bh);
                    ++qc[tt];
                }
                int nr = 0, nv = 0;
                uint64_t t_last = cycles_now();
                while (ok && (nr < it.nr_total || nv < it.nstream)) {
                    bool progress = false;
                    if (nr < it.nr_total &&
                        (rfill < NR ||
                         mbar_test_wait(bar(ScanSmem::EMPTY_R + rfill % NR), ((rfill / NR) - 1) & 1))) {
                        const int st = rfill % NR;
                        const int b = it.top - (nr + 1 + ((it.hole2 && nr >= 1) ? 1 : 0));
                        const uint32_t full = bar(ScanSmem::FULL_R + st);
                        mbar_arrive_expect_tx(full, kRBytes);
                        tma_load_3d(stage_r(st), &tm_kp128, full, 0, b * 2 * kC, it.bh);
                        ++nr;
                        ++rfill;
                        progress = true;
                    }
                    if (nv < it.nstream &&
                        (vfill < NV ||
                         mbar_test_wait(bar(ScanSmem::EMPTY_V + vfill % NV), ((vfill / NV) - 1) & 1))) {
                        const int st = vfill % NV, b = it.top - nv;
                        const uint32_t full = bar(ScanSmem::FULL_V + st);
                        mbar_arrive_expect_tx(full, kVBytes);
                        tma_load_3d(stage_v(st), &tm_v64, full, 0, b * kC, it.bh);
                        ++nv;
                        ++vfill;
                        progress = true;
                    }
                    if (progress) {
                        t_last = cycles_now();
                    } else if (*abort_flag) {
                        ok = false;
                    } else if (cycles_now() - t_last > ns_to_cycles(limit_ns)) {
                        report_status(status, kStatusTimeout);
                        *abort_flag = 1u;
                        ok = false;
                    } else {
                        __nanosleep(64);
                    }
                }
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int n = (vfill > NV ? vfill - NV : 0); n < vfill; ++n) {
                const uint32_t bfull = bar(ScanSmem::FULL_V + n % NV);
                const uint64_t t0 = cycles_now();
                while (!mbar_try_wait(bfull, (n / NV) & 1) &&
                       cycles_now() - t0 < ns_to_cycles(limit_ns)) {
                }
            }
            for (int m = (rfill > NR ? rfill - NR : 0); m < rfill; ++m) {
                const uint32_t bfull = bar(ScanSmem::FULL_R + m % NR);
                const uint64_t t0 = cycles_now();
                while (!mbar_try_wait(bfull, (m / NR) & 1) &&
                       cycles_now() - t0 < ns_to_cycles(limit_ns)) {
                }
            }
            for (int tt = 0; tt < 2; ++tt) {
                if (qc[tt] == 0) continue;
                const uint64_t t0 = cycles_now();
                while (!mbar_try_wait(tbar(tt, ScanSmem::QFULL), (qc[tt] - 1) & 1) &&
                       cycles_now() - t0 < ns_to_cycles(limit_ns)) {
                }
            }
        }
      }
    } else {
      reg_alloc_inc<kRegRow>();
      {
        // ------------------------------------------------------------ row warps
        const int t = warp >> 2;                 // 0 = tile A, 1 = tile B
        const int r = threadIdx.x - 128 * t;     // tile row = TMEM lane
        const int q = warp & 3;                  // lane quadrant
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        // every lane of a warp leaves together: tcgen05.ld/st are warp-collective
        auto wwait = [&](uint32_t b_, uint32_t par) {
            return __all_sync(0xffffffffu, wait(b_, par)) != 0;
        };
        const uint32_t T_S = t_base(t) + TC_S + lane_base;
        const uint32_t T_X = t_base(t) + TC_X + lane_base;
        const uint32_t T_XB = t_base(t) + TC_XB + lane_base;
        const uint32_t T_O = t_base(t) + TC_O + lane_base;
        const uint32_t T_P = t_base(t) + TC_P + lane_base;
        bool ok = true;
        int sxb = 0, pvb = 0, qc = 0;  // MMAs and q~ tiles of this tile slot in earlier items
        for (int idx = blockIdx.x; ok && idx < nitems; idx += gridDim.x) {
            const Item it = make_item(idx, ncta, ntile, nblk, first_blk);
            if (!it.has(t)) continue;
            const int tile = it.tile(t);
            const int nsteps = it.nsteps(t);
            const int i = tile * kTile + r;          // query index
            const size_t head = (size_t)it.bh;
            float m_run = -INFINITY, l_run = 0.f;
            // gate sums relative to the base of their pair of blocks; per step the row's
            // offset against the pair u of the key block is (base_tile - base_u) in fp32-pair
            // arithmetic + rel_i
            const float rel_i = c2[head * Lp + i];
            const float2 base_own = *reinterpret_cast<const float2 *>(pbase + (head * ntile + tile) * 2);
            auto row_offset = [&](int u) {
                const float2 bu = *reinterpret_cast<const float2 *>(pbase + (head * ntile + u) * 2);
                return ((base_own.x - bu.x) + (base_own.y - bu.y)) + rel_i;
            };

            // the carried state of step 1 is q~: the row goes from the TMA tile into TMEM
            // (the previous item's MMAs, which read the old state, have all completed)
            if (!(ok = wwait(tbar(t, ScanSmem::QFULL), qc & 1))) break;
            {
                const uint8_t *row = gbase + ScanSmem::q_st(t);
                uint32_t x[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(row + sw128_offset(r, c));
                    x[4 * c] = u.x; x[4 * c + 1] = u.y; x[4 * c + 2] = u.z; x[4 * c + 3] = u.w;
                }
                tmem_st32(T_XB, x);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive_warp(tbar(t, ScanSmem::QFREE));
                mbar_arrive_warp(tbar(t, ScanSmem::NEXT));
                ++qc;
            }

            for (int s = 0; s < nsteps && ok; ++s) {
                const int b = 2 * tile + 1 - s;      // key block of this step
                // the step's 64 logits (column c is key 64 b + c), in log2 units
                float v[64];
                if (s == 0) {
                    // rows of block 2T+1: their diagonal-block table; rows of block 2T see no
                    // key of block 2T+1
                    if (q >= 2) {
                        load_diag_row(dg + ((head * nblk + b) * kC + (r - 64)) * kC, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 64; ++j) v[j] = -INFINITY;
                    }
                } else {
                    // every warp waits for each MMA of its tile (a skipped phase would read
                    // as done)
                    if (!(ok = wwait(tbar(t, ScanSmem::SX_DONE), (sxb + s - 1) & 1))) break;
                    tc_fence_after();
                    const bool diag = (s == 1 && q < 2);      // rows of block 2T at step 1
                    // the next state: X' for rows past their diagonal step; rows of block 2T
                    // keep q~ after step 1
                    const bool carry = (s + 1 < nsteps) && !diag;
                    uint32_t a[32], c[32];
                    if (!diag) {
                        tmem_ld32(T_S, a);
                        tmem_ld32(T_S + 32, c);
                    }
                    if (carry) {
                        uint32_t xa[32], xp[32];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            tmem_ld32(T_X + 32 * h, xa);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                xp[16 * h + j] = pack_bf16x2(__uint_as_float(xa[2 * j]), __uint_as_float(xa[2 * j + 1]));
                        }
                        tmem_st32(T_XB, xp);
                        tmem_st_wait();
                    } else {
                        tmem_ld_wait();
                    }
                    // S and X' are in registers and the new state is written: the next MMA
                    // may go
                    tc_fence_before();
                    if (s + 1 < nsteps) mbar_arrive_warp(tbar(t, ScanSmem::NEXT));
                    if (diag) {
                        load_diag_row(dg + ((head * nblk + b) * kC + r) * kC, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            v[j] = __uint_as_float(a[j]);
                            v[32 + j] = __uint_as_float(c[j]);
                        }
                        // v = scale log2(e) S + c2_i - c2_j, two columns per instruction
                        const float4 *cj = reinterpret_cast<const float4 *>(c2 + head * Lp + b * kC);
                        const float2 sl2 = make_float2(scale_log2, scale_log2);
                        const float ci = row_offset(b >> 1);
                        const float2 ci2 = make_float2(ci, ci);
                        const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
                        for (int q4 = 0; q4 < 16; ++q4) {
                            const float4 cc = __ldg(cj + q4);
                            const float2 b0 = ffma2(make_float2(cc.x, cc.y), neg1, ci2);
                            const float2 b1 = ffma2(make_float2(cc.z, cc.w), neg1, ci2);
                            const float2 w0 = ffma2(make_float2(v[4 * q4], v[4 * q4 + 1]), sl2, b0);
                            const float2 w1 = ffma2(make_float2(v[4 * q4 + 2], v[4 * q4 + 3]), sl2, b1);
                            v[4 * q4] = w0.x; v[4 * q4 + 1] = w0.y;
                            v[4 * q4 + 2] = w1.x; v[4 * q4 + 3] = w1.y;
                        }
                    }
                }
                // ---- online softmax with lazy rescaling: the running max is raised only when
                // the step's max exceeds it by more than 2^8; then the row sum and O are
                // rescaled
                float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
                for (int j = 4; j < 60; j += 8)
#pragma unroll
                    for (int e = 0; e < 4; ++e) m4[e] = fmax3(m4[e], v[j + 2 * e], v[j + 2 * e + 1]);
                const float mx = fmax3(fmax3(m4[0], m4[1], v[60]), fmax3(m4[2], m4[3], v[61]),
                                       fmaxf(v[62], v[63]));
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
                const float2 one2 = make_float2(1.f, 1.f), nm2 = make_float2(neg_m, neg_m);
                float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float2 x = ffma2(make_float2(v[2 * j], v[2 * j + 1]), one2, nm2);
                    const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    ls[j & 3] = fadd2(ls[j & 3], p);
                    pk[j] = pack_bf16x2(p.x, p.y);
                }
                const float2 l01 = fadd2(ls[0], ls[1]), l23 = fadd2(ls[2], ls[3]);
                const float2 l4 = fadd2(l01, l23);
                l_run += l4.x + l4.y;
                // P was last read by this tile's P.V MMA of step s - 1 (at step 0: of the
                // previous item, complete before its epilogue), which also has to be complete
                // before O is rescaled
                if (s >= 1 && !(ok = wwait(tbar(t, ScanSmem::O_DONE), (pvb + s - 1) & 1))) break;
                tc_fence_after();
                tmem_st32(T_P, pk);
                if (s >= 1 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t oa[32];
                        tmem_ld32(T_O + 32 * h, oa);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) oa[j] = __float_as_uint(__uint_as_float(oa[j]) * alpha);
                        tmem_st32(T_O + 32 * h, oa);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive_warp(tbar(t, ScanSmem::PREADY));
            }

            // ---- epilogue: O / l, LSE (the next item's first P.V overwrites O only after
            // this warp's next P arrival)
            if (ok) ok = wwait(tbar(t, ScanSmem::O_DONE), (pvb + nsteps - 1) & 1);
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
                tc_fence_before();
            }
            sxb += nsteps - 1;
            pvb += nsteps;
        }
        tc_fence_before();
      }
    }

    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Returns cudaErrorInvalidValue if the tensor maps cannot be encoded, and
// cudaErrorInvalidConfiguration if the compiled kernel was given fewer registers than the
// warpgroup split redistributes (its setmaxnreg.inc could then never be satisfied).
cudaError_t launch_scan_tc_fox(const void *v, void *out, float *lse, int BH, int L, float scale,
                               void *ws, uint64_t limit_ns, int force_timeout,
                               cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 2, true);
    char *basep = static_cast<char *>(ws);
    CUtensorMap tm_qt, tm_kp128, tm_v64;
    const int nrows_kp = lay.nblk * 2 * kC;
    if (!make_map_bf16(&tm_qt, basep + lay.off_qt, lay.Lp, BH, kTile) ||
        !make_map_bf16(&tm_kp128, basep + lay.off_kp, nrows_kp, BH, 2 * kC) ||
        !make_map_bf16(&tm_v64, v, L, BH, kC))
        return cudaErrorInvalidValue;
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, path_scan_tc_fox_kernel);
    if (err != cudaSuccess) return err;
    if (fa.numRegs * kScanThreads < 256 * kRegRow + 256 * kRegOther)
        return cudaErrorInvalidConfiguration;
    err = cudaFuncSetAttribute(path_scan_tc_fox_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmemBytes);
    if (err != cudaSuccess) return err;
    int dev = 0, nsm = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    const int ntile = lay.nblk / 2;
    const int nitems = ((ntile + 1) / 2) * BH;  // tile pairs of every head
    const int grid = nitems < nsm ? nitems : nsm;
    path_scan_tc_fox_kernel<<<grid, kScanThreads, kScanSmemBytes, stream>>>(
        tm_qt, tm_kp128, tm_v64, reinterpret_cast<const __half *>(basep + lay.off_dg),
        reinterpret_cast<const float *>(basep + lay.off_c2),
        reinterpret_cast<const float *>(basep + lay.off_pbase),
        reinterpret_cast<const int *>(basep + lay.off_fb), static_cast<__nv_bfloat16 *>(out), lse,
        L, lay.Lp, lay.nblk, nitems, scale * kLog2e, reinterpret_cast<uint32_t *>(basep),
        limit_ns, force_timeout);
    return cudaGetLastError();
}

}  // namespace path
