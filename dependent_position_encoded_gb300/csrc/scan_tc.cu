// K2 (bf16): the right-to-left block scan of PaTH attention on tcgen05 tensor cores.
//
// Technical summary "技術要約: PaTH Attention" §3 (FlashAttention-style algorithm: per-block
// boundary-adjusted queries and keys, a right-to-left scan over key/value blocks that
// accumulates the Householder product, online softmax, nothing L x L in memory); review
// "거리에서 경로로, PaTH Attention" §9 (the same scheme, blockwise preprocessing and
// blockwise updates of the accumulated transform and softmax statistics).
//
// One CTA owns a tile of 128 query rows = two 64-token blocks ib0 = 2t, ib1 = 2t + 1 of
// one head. With q~ the boundary-adjusted queries, k~ the boundary-adjusted keys and
// P_b = H_start(b) ... H_end(b) the dense block transition (all from the preprocessing
// kernel), the logit of row i against key j of an earlier block b is
//     scale * k~_j^T P_{b+1} ... P_{ib-1} q~_i,
// so a state row x_i = q~_i is scored against block ib-1, then x_i <- P_{ib-1} x_i, and
// so on down to block 0. In row form the whole tile advances as X <- X P_b^T, one
// 128 x 64 x 64 MMA per block, next to S = X K~_b^T and O += P V_b.
// Steps s = 0 .. ib1 visit key block b = ib1 - s:
//   s = 0 : block ib1; rows 64-127 take their diagonal-block logits, rows 0-63 are masked.
//   s = 1 : block ib0; rows 0-63 take their diagonal-block logits, rows 64-127 the MMA
//           logits of block ib0, and only rows 64-127 advance their state by P_{ib0}.
//   s >= 2: block ib1 - s for every row.
//
// Warp roles (192 threads): warps 0-3 own one query row per thread (TMEM lane = row):
// online softmax with lazy rescaling, fp32 -> bf16 conversion of the new state into the
// swizzled A-operand tile. Warp 4 allocates TMEM and one lane issues every MMA. Warp 5
// (one lane) streams K~|P_b and V_b tiles by TMA through an NS-stage ring.
// The bf16 state tile is double-buffered (step s reads buffer s & 1 while the new state
// of step s + 1 is written into the other one: the S MMA of step s may still be reading
// its operand when the state MMA that precedes it has completed). The probability tile
// is single-buffered: it is rewritten only after the previous P.V MMA has completed.
// TMEM columns: [0,64) new state, [64,128) and [128,192) S (double buffer), [192,256) O.
#include "common.cuh"

namespace path {

namespace {

constexpr int kScanThreads = 192;
constexpr int NS = 2;                       // TMA stages (K~|P and V of one block each)
constexpr uint32_t kTileBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kVBytes = 64 * 128;      // 64 rows x 64 bf16
constexpr uint32_t kStageBytes = kTileBytes + kVBytes;
constexpr float kRescaleThreshold = 8.f;    // lazy rescale: keep the old max within 2^8

struct ScanSmem {
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t q_st = 0;                         // two 16 KB state tiles
    static constexpr uint32_t p_buf = 2 * kTileBytes;           // one 16 KB tile
    static constexpr uint32_t stage = p_buf + kTileBytes;       // NS stages
    static constexpr uint32_t bars = stage + NS * kStageBytes;
    // barrier indices
    static constexpr int FULL = 0, EMPTY = NS, QFULL = 2 * NS, BAR_QN = 2 * NS + 1,
                         BAR_S = 2 * NS + 2, BAR_O = 2 * NS + 3, QREADY = 2 * NS + 4,
                         PREADY = 2 * NS + 5, FINAL = 2 * NS + 6, NEVER = 2 * NS + 7,
                         NBARS = 2 * NS + 8;
    static constexpr uint32_t tmem_slot = bars + NBARS * 8;
    static constexpr uint32_t abort_flag = tmem_slot + 4;
    static constexpr uint32_t bytes = abort_flag + 4;
};

constexpr uint32_t kScanSmemBytes = ScanSmem::bytes + 1024;  // + alignment slack

struct Waiter {
    volatile uint32_t *abort;
    uint32_t *status;
    uint64_t limit_ns;
    // Bounded wait; on timeout records the status and raises the CTA abort flag.
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            for (int i = 0; i < 32; ++i)
                if (mbar_try_wait(bar, parity)) return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                report_status(status, kStatusTimeout);
                *abort = 1u;
                return false;
            }
        }
    }
};

template <bool FOX>
__global__ void __launch_bounds__(kScanThreads, 2)
path_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_qt,
                    const __grid_constant__ CUtensorMap tm_kp,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __nv_bfloat16 *__restrict__ qt, const __half *__restrict__ dg,
                    const float *__restrict__ c2, __nv_bfloat16 *__restrict__ out,
                    float *__restrict__ lse, int L, int Lp, int nblk, float scale_log2,
                    uint32_t *status, uint64_t limit_ns, int force_timeout) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = nblk >> 1;
    const int tile = ntile - 1 - (int)blockIdx.x;  // longest tiles first
    const int bh = blockIdx.y;
    const int ib0 = 2 * tile, ib1 = 2 * tile + 1;
    const int nsteps = ib1 + 1;

    auto bar = [&](int i) { return base + ScanSmem::bars + 8u * (uint32_t)i; };
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + ScanSmem::abort_flag);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + ScanSmem::tmem_slot);
    const Waiter wait{abort_flag, status, limit_ns};

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bar(ScanSmem::FULL + i), 1);
            mbar_init(bar(ScanSmem::EMPTY + i), 1);
        }
        mbar_init(bar(ScanSmem::QFULL), 1);
        mbar_init(bar(ScanSmem::BAR_QN), 1);
        mbar_init(bar(ScanSmem::BAR_S), 1);
        mbar_init(bar(ScanSmem::BAR_O), 1);
        mbar_init(bar(ScanSmem::QREADY), 128);
        mbar_init(bar(ScanSmem::PREADY), 128);
        mbar_init(bar(ScanSmem::FINAL), 1);
        mbar_init(bar(ScanSmem::NEVER), 1);
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t T_QN = tmem + 0, T_S0 = tmem + 64, T_O = tmem + 192;

    auto q_st = [&](int i) { return base + ScanSmem::q_st + (uint32_t)i * kTileBytes; };
    const uint32_t p_buf = base + ScanSmem::p_buf;
    auto stage_kp = [&](int i) { return base + ScanSmem::stage + (uint32_t)i * kStageBytes; };
    auto stage_v = [&](int i) { return stage_kp(i) + kTileBytes; };

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_qt);
            tma_prefetch_desc(&tm_kp);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(bar(ScanSmem::QFULL), kTileBytes);
            tma_load_3d(q_st(1), &tm_qt, bar(ScanSmem::QFULL), 0, tile * kTile, bh);
            int issued = 0;
            for (int s = 0; s < nsteps; ++s) {
                const int st = s % NS;
                if (s >= NS && !wait(bar(ScanSmem::EMPTY + st), ((s / NS) - 1) & 1)) break;
                const int b = ib1 - s;
                if (s == 0) {
                    mbar_arrive_expect_tx(bar(ScanSmem::FULL + st), kVBytes);
                } else {
                    mbar_arrive_expect_tx(bar(ScanSmem::FULL + st), kStageBytes);
                    tma_load_3d(stage_kp(st), &tm_kp, bar(ScanSmem::FULL + st), 0, b * 2 * kC, bh);
                }
                tma_load_3d(stage_v(st), &tm_v, bar(ScanSmem::FULL + st), 0, b * kC, bh);
                issued = s + 1;
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int s = (issued > NS ? issued - NS : 0); s < issued; ++s) {
                const uint32_t bfull = bar(ScanSmem::FULL + s % NS);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bfull, (s / NS) & 1) && globaltimer_ns() - t0 < limit_ns) {
                }
            }
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(ScanSmem::QFULL), 0) && globaltimer_ns() - t0 < limit_ns) {
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_KMAJ = idesc_bf16(128, 64, false);
            constexpr uint32_t ID_PV = idesc_bf16(128, 64, true);
            bool ok = true;
            if (force_timeout) ok = wait(bar(ScanSmem::NEVER), 0);  // nothing arrives here
            auto issue_sq = [&](int s) -> bool {
                const int st = s % NS;
                if (!wait(bar(ScanSmem::FULL + st), (s / NS) & 1)) return false;
                if (s >= 2 && !wait(bar(ScanSmem::QREADY), (s - 2) & 1)) return false;
                tc_fence_after();
                const uint64_t a_q = sdesc_sw128(q_st(s & 1), 16, 1024);
                const uint64_t b_k = sdesc_sw128(stage_kp(st), 16, 1024);
                const uint64_t b_p = sdesc_sw128(stage_kp(st) + 64 * 128, 16, 1024);
                if (s < nsteps - 1) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(T_QN, a_q + 2 * kk, b_p + 2 * kk, ID_KMAJ, kk > 0);
                    umma_commit(bar(ScanSmem::BAR_QN));
                }
                const uint32_t t_s = T_S0 + 64u * (uint32_t)(s & 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(t_s, a_q + 2 * kk, b_k + 2 * kk, ID_KMAJ, kk > 0);
                umma_commit(bar(ScanSmem::BAR_S));
                return true;
            };
            if (ok) ok = wait(bar(ScanSmem::QFULL), 0);
            if (ok && nsteps >= 2) ok = issue_sq(1);
            for (int s = 0; ok && s < nsteps; ++s) {
                if (s + 1 >= 2 && s + 1 <= nsteps - 1 && !(ok = issue_sq(s + 1))) break;
                const int st = s % NS;
                if (s == 0 && !(ok = wait(bar(ScanSmem::FULL + st), 0))) break;
                if (!(ok = wait(bar(ScanSmem::PREADY), s & 1))) break;
                tc_fence_after();
                const uint64_t a_p = sdesc_sw128(p_buf, 16, 1024);
                const uint64_t b_v = sdesc_sw128(stage_v(st), 1024, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(T_O, a_p + 2 * kk, b_v + 128 * kk, ID_PV, (s > 0 || kk > 0));
                umma_commit(bar(ScanSmem::BAR_O));
                umma_commit(bar(ScanSmem::EMPTY + st));
            }
            // every MMA issued above has completed before TMEM is released
            umma_commit(bar(ScanSmem::FINAL));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(ScanSmem::FINAL), 0) && globaltimer_ns() - t0 < limit_ns) {
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int r = threadIdx.x;             // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int i = tile * kTile + r;        // query index
        const size_t head = (size_t)bh;
        float m_run = -INFINITY, l_run = 0.f;
        const float c2_i = FOX ? c2[head * Lp + i] : 0.f;
        bool ok = true;
        // every lane of a warp leaves together: tcgen05.ld/st are warp-collective
        auto wwait = [&](uint32_t b_, uint32_t par) {
            return __all_sync(0xffffffffu, wait(b_, par)) != 0;
        };

        for (int s = 0; s < nsteps && ok; ++s) {
            const int b = ib1 - s;
            float x[64];
            bool from_diag = false;
            int diag_blk = 0, diag_row = 0;
            if (s == 0) {
                from_diag = true;
                diag_blk = ib1;
                diag_row = r - 64;
            } else {
                if (s < nsteps - 1) {
                    if (!(ok = wwait(bar(ScanSmem::BAR_QN), (s - 1) & 1))) break;
                    tc_fence_after();
                    // the state of step s + 1 goes to buffer (s + 1) & 1
                    uint8_t *row = gbase + ScanSmem::q_st + (uint32_t)((s + 1) & 1) * kTileBytes;
                    if (s >= 2 || warp >= 2) {
                        uint32_t qa[32], qb[32];
                        tmem_ld32(T_QN + lane_base, qa);
                        tmem_ld32(T_QN + lane_base + 32, qb);
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
                            qt + (head * Lp + (size_t)tile * kTile + r) * kD);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(row + sw128_offset(r, c)) = __ldg(src + c);
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(ScanSmem::QREADY));
                }
                if (!(ok = wwait(bar(ScanSmem::BAR_S), (s - 1) & 1))) break;
                tc_fence_after();
                if (s == 1 && warp < 2) {
                    from_diag = true;
                    diag_blk = ib0;
                    diag_row = r;
                } else {
                    uint32_t sa[32], sb[32];
                    const uint32_t t_s = T_S0 + 64u * (uint32_t)(s & 1) + lane_base;
                    tmem_ld32(t_s, sa);
                    tmem_ld32(t_s + 32, sb);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        x[j] = __uint_as_float(sa[j]) * scale_log2;
                        x[j + 32] = __uint_as_float(sb[j]) * scale_log2;
                    }
                    if (FOX) {
                        const float4 *cj = reinterpret_cast<const float4 *>(c2 + head * Lp + b * kC);
#pragma unroll
                        for (int q4 = 0; q4 < 16; ++q4) {
                            const float4 c = __ldg(cj + q4);
                            x[4 * q4 + 0] += c2_i - c.x;
                            x[4 * q4 + 1] += c2_i - c.y;
                            x[4 * q4 + 2] += c2_i - c.z;
                            x[4 * q4 + 3] += c2_i - c.w;
                        }
                    }
                }
            }
            if (from_diag) {
                if (diag_row >= 0) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        dg + (((head * nblk + diag_blk) * kC) + diag_row) * kC);
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
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
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) x[j] = -INFINITY;
                }
            }

            // ---- online softmax (base 2), lazy rescaling of O
            float mx = x[0];
#pragma unroll
            for (int j = 1; j < 64; ++j) mx = fmaxf(mx, x[j]);
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_run + kRescaleThreshold) {
                if (m_run != -INFINITY) {
                    alpha = exp2f(m_run - mx);
                    rescale = true;
                }
                m_run = mx;
                l_run *= alpha;
            }
            if (s >= 1 && __any_sync(0xffffffffu, rescale)) {
                // O must be complete up to step s - 1 before it is rewritten
                if (!(ok = wwait(bar(ScanSmem::BAR_O), (s - 1) & 1))) break;
                tc_fence_after();
                uint32_t oa[32], ob[32];
                tmem_ld32(T_O + lane_base, oa);
                tmem_ld32(T_O + lane_base + 32, ob);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    oa[j] = __float_as_uint(__uint_as_float(oa[j]) * alpha);
                    ob[j] = __float_as_uint(__uint_as_float(ob[j]) * alpha);
                }
                tmem_st32(T_O + lane_base, oa);
                tmem_st32(T_O + lane_base + 32, ob);
                tmem_st_wait();
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            float lsum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = exp2f(x[2 * j] - m_use);
                const float p1 = exp2f(x[2 * j + 1] - m_use);
                lsum += p0 + p1;
                pk[j] = pack_bf16x2(p0, p1);
            }
            l_run += lsum;
            // the P tile was last read by the P.V MMA of step s - 1
            if (s >= 1 && !(ok = wwait(bar(ScanSmem::BAR_O), (s - 1) & 1))) break;
            uint8_t *prow = gbase + ScanSmem::p_buf;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 u = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                *reinterpret_cast<uint4 *>(prow + sw128_offset(r, c)) = u;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(ScanSmem::PREADY));
        }

        // ---- epilogue: O / l, LSE
        if (ok) ok = wwait(bar(ScanSmem::BAR_O), (nsteps - 1) & 1);
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
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
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
    if (!make_map(&tm_qt, basep + lay.off_qt, lay.Lp, BH, kTile) ||
        !make_map(&tm_kp, basep + lay.off_kp, lay.nblk * 2 * kC, BH, kTile) ||
        !make_map(&tm_v, v, L, BH, kC))
        return cudaErrorInvalidValue;
    auto kern = fox ? path_scan_tc_kernel<true> : path_scan_tc_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kScanSmemBytes);
    if (err != cudaSuccess) return err;
    dim3 grid(lay.nblk / 2, BH);
    kern<<<grid, kScanThreads, kScanSmemBytes, stream>>>(
        tm_qt, tm_kp, tm_v, reinterpret_cast<const __nv_bfloat16 *>(basep + lay.off_qt),
        reinterpret_cast<const __half *>(basep + lay.off_dg),
        fox ? reinterpret_cast<const float *>(basep + lay.off_c2) : nullptr,
        static_cast<__nv_bfloat16 *>(out), lse, L, lay.Lp, lay.nblk, scale * kLog2e,
        reinterpret_cast<uint32_t *>(basep), limit_ns, force_timeout);
    return cudaGetLastError();
}

}  // namespace path
