// The right-to-left block scan of PaTH attention at head size 128 on tcgen05 tensor cores
// (bf16 inputs), PaTH and PaTH-FoX.
//
// Technical summary "技術要約: PaTH Attention" §3 (per-block boundary-adjusted queries and
// keys, a right-to-left scan over key/value blocks that carries the accumulated Householder
// product, online softmax, nothing L x L in memory); review "거리에서 경로로, PaTH
// Attention" §9 (larger heads cost more). A tile is the 128 query rows of the blocks
// A0 = 2t and A1 = 2t + 1 of one head. With X the tile's carried rows (starting as q~) the
// tile visits key blocks b = 2t+1, 2t, ..., 0:
//   b = 2t+1: A1's diagonal block (the preparation's table); A0 has no key there;
//   b = 2t:   A0's diagonal block (table); A1's logits x . k~_j from the MMA below, after
//             which A1's rows are carried through block 2t;
//   b < 2t:   both blocks from the MMA.
// Per key block, M = 128 MMAs with bf16 operands in 128-byte-swizzled shared memory and
// fp32 accumulators in TMEM:
//   [S | X'] = X [K~_b; P_b]^T    N = 192 (64 logits, 128 carried columns), K = 128
//   O       += P V_b               N = 128, K = 64
// At d = 128 a tile needs S 64 + X' 128 + O 128 TMEM columns, so a CTA holds one tile.
// PaTH-FoX: the bias c_i - c_j of a key in an earlier block is formed, in log2 units, as
// (lc2_i + sum of the block totals strictly between the two blocks, an fp64 running sum per
// row) + (T2_b - lc2_j), so no difference of two long prefix sums is taken; the tile stops
// at the lower of its two query blocks' early-exit extents (fox_exit.cu, from the bounds
// the preparation wrote), below which every key weighs less than e^-40 of the row maximum.
//
// Warp roles (288 threads): warps 0-3 softmax, one row per thread (logits or the table
// row, lazy rescaling of O when the running maximum rises by more than 2^8, the P tile),
// and the final O / l; warps 4-7 convert each carried row from TMEM to the bf16 X tile;
// warp 8 allocates TMEM and its lane 0 issues the TMA loads (three stages of [K~_b; P_b],
// two of V_b) and the MMAs. Every wait is bounded; on a timeout the CTA records
// PATH_ERR_TIMEOUT in the workspace status word, every role leaves its loop, the issuing
// lane waits for its copies and MMAs in flight, and TMEM is freed.
#include "common.cuh"

namespace path {

namespace {

constexpr int kThr = 288;
constexpr int NR = 3, NV = 2;
constexpr uint32_t kXBytes = 2 * 128 * 128;      // 128 rows x 128 bf16 (two atoms)
constexpr uint32_t kPBytes = 128 * 128;          // 128 rows x 64 bf16
constexpr uint32_t kRAtom = 192 * 128;           // 192 rows x 64 bf16
constexpr uint32_t kRBytes = 2 * kRAtom;         // [K~_b; P_b] x 128 columns
constexpr uint32_t kVAtom = 64 * 128;
constexpr uint32_t kVBytes = 2 * kVAtom;         // V_b: 64 rows x 128 columns
constexpr uint32_t S_X = 0, S_P = kXBytes, S_R = S_P + kPBytes, S_V = S_R + NR * kRBytes,
                   S_BAR = S_V + NV * kVBytes;
constexpr int B_LD0 = 0, B_RF = 1, B_RE = B_RF + NR, B_VF = B_RE + NR, B_VE = B_VF + NV,
              B_SX = B_VE + NV, B_PV = B_SX + 1, B_XR = B_PV + 1, B_SF = B_XR + 1,
              B_PR = B_SF + 1, B_FIN = B_PR + 1, NBAR = B_FIN + 1;
constexpr uint32_t kSmem = 1024 + S_BAR + NBAR * 8 + 16;
static_assert(kSmem <= 227u * 1024u, "d = 128 scan shared memory");
constexpr uint32_t C_S = 0, C_X = 64, C_O = 256;
constexpr float kRescale = 8.f;

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

__device__ __forceinline__ void tld32(uint32_t taddr, float *x) {
    uint32_t u[32];
    tmem_ld32(taddr, u);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(u[j]);
}

// 32 values as bf16 into 16-byte chunks c0 .. c0 + 3 of row r of a swizzled atom
__device__ __forceinline__ void st_chunks(uint8_t *atom, int r, int c0, const float *x) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float *s = x + 8 * c;
        *reinterpret_cast<uint4 *>(atom + sw128_offset(r, c0 + c)) =
            make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]),
                       pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
    }
}

// (heads, rows, 128 columns) bf16 with (64 columns, box_rows) boxes, 128-byte swizzle
bool make_map128(CUtensorMap *m, const void *ptr, int rows, int heads, int box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)rows * 128 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One CTA per (tile t, head). nblk: blocks rounded up to even; Lp = 64 nblk.
template <bool FOX>
__global__ void __launch_bounds__(kThr, 1)
scan_tc128_kernel(const __grid_constant__ CUtensorMap tm_qt,
                  const __grid_constant__ CUtensorMap tm_kp,
                  const __grid_constant__ CUtensorMap tm_v, const __half *__restrict__ dg,
                  const float *__restrict__ lc2, const float *__restrict__ tail2,
                  const double *__restrict__ tot2, const int *__restrict__ first_blk,
                  __nv_bfloat16 *__restrict__ out,
                  float *__restrict__ lse, int L, int Lp, int nblk, float scale_log2,
                  uint32_t *status, uint64_t limit_ns, int heads_fast) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    auto bar = [&](int i) { return base + S_BAR + 8u * (uint32_t)i; };
    uint32_t *const tslot = reinterpret_cast<uint32_t *>(sm + S_BAR + 8 * NBAR);
    volatile uint32_t *const abort_f = tslot + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int npair = nblk >> 1;
    // longest walks first, heads fastest or head by head (heads_fastest)
    const int t = npair - 1 - (int)(heads_fast ? blockIdx.y : blockIdx.x);
    const int bh = heads_fast ? blockIdx.x : blockIdx.y;
    // key blocks 2t+1 down to 0, or for PaTH-FoX down to the lower early-exit extent of the
    // tile's two query blocks (never above block 2t, its own lower diagonal block)
    int lo = 0;
    if (FOX) {
        const int *f = first_blk + (size_t)bh * nblk + 2 * t;
        lo = min(min(__ldg(f), __ldg(f + 1)), 2 * t);
    }
    const int steps = 2 * t + 2 - lo;
    const Wait wait{abort_f, status, limit_ns};
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait(b, parity)) != 0;
    };

    if (tid == 0) {
        *abort_f = 0u;
        for (int i = 0; i < NBAR; ++i)
            mbar_init(bar(i), (i == B_XR || i == B_SF || i == B_PR) ? 4u : 1u);
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 8) {
        // ================================================================ issuer
        if (lane == 0) {
            tma_prefetch_desc(&tm_qt);
            tma_prefetch_desc(&tm_kp);
            tma_prefetch_desc(&tm_v);
            uint32_t r_iss = 0, r_done = 0, v_iss = 0, v_done = 0;
            mbar_arrive_expect_tx(bar(B_LD0), kXBytes);
            tma_load_3d(base + S_X, &tm_qt, bar(B_LD0), 0, 128 * t, bh);
            tma_load_3d(base + S_X + kXBytes / 2, &tm_qt, bar(B_LD0), 64, 128 * t, bh);
            auto load_r = [&](int s) {  // step s >= 1: [K~_b; P_b], b = 2t + 1 - s
                const int b = 2 * t + 1 - s, st = (s - 1) % NR;
                const uint32_t dst = base + S_R + (uint32_t)st * kRBytes;
                mbar_arrive_expect_tx(bar(B_RF + st), kRBytes);
                tma_load_3d(dst, &tm_kp, bar(B_RF + st), 0, 192 * b, bh);
                tma_load_3d(dst + kRAtom, &tm_kp, bar(B_RF + st), 64, 192 * b, bh);
                ++r_iss;
            };
            auto load_v = [&](int s) {
                const int b = 2 * t + 1 - s, st = s % NV;
                const uint32_t dst = base + S_V + (uint32_t)st * kVBytes;
                mbar_arrive_expect_tx(bar(B_VF + st), kVBytes);
                tma_load_3d(dst, &tm_v, bar(B_VF + st), 0, 64 * b, bh);
                tma_load_3d(dst + kVAtom, &tm_v, bar(B_VF + st), 64, 64 * b, bh);
                ++v_iss;
            };
            for (int s = 1; s < steps && s <= NR; ++s) load_r(s);
            for (int s = 0; s < steps && s < NV; ++s) load_v(s);
            bool ok = true;
            auto issue_pv = [&](int s) -> bool {
                const int vs = s % NV;
                if (!wait(bar(B_VF + vs), (s / NV) & 1)) return false;
                ++v_done;
                if (!wait(bar(B_PR), s & 1)) return false;
                tc_fence_after();
                const uint64_t a = sdesc_sw128(base + S_P, 16, 1024);
                const uint64_t bv = sdesc_sw128(base + S_V + (uint32_t)vs * kVBytes, kVAtom, 1024);
                constexpr uint32_t ID = idesc_b16(128, 128, false, true);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + C_O, a + 2 * kk, bv + 128 * kk, ID, (s > 0 || kk > 0));
                umma_commit(bar(B_PV));
                umma_commit(bar(B_VE + vs));
                // the V stage of step s - 1 refills with step s + 1
                if (s >= 1 && s + 1 < steps && s + 1 >= NV) {
                    const int pvs = (s - 1) % NV;
                    if (!wait(bar(B_VE + pvs), ((s - 1) / NV) & 1)) return false;
                    load_v(s + 1);
                }
                return true;
            };
            for (int s = 0; ok && s < steps; ++s) {
                if (s >= 1) {
                    const int st = (s - 1) % NR;
                    if (!(ok = wait(bar(B_RF + st), ((s - 1) / NR) & 1))) break;
                    ++r_done;
                    if (s == 1) {
                        if (!(ok = wait(bar(B_LD0), 0))) break;
                    } else {
                        // step s - 1's carried rows converted and its logits read
                        if (!(ok = wait(bar(B_XR), (s - 2) & 1))) break;
                        if (!(ok = wait(bar(B_SF), (s - 2) & 1))) break;
                    }
                    tc_fence_after();
                    const uint32_t rs = base + S_R + (uint32_t)st * kRBytes;
                    constexpr uint32_t ID = idesc_b16(128, 192, false, false);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = kk < 4 ? 0u : 1u;
                        umma_bf16(tmem + C_S,
                                  sdesc_sw128(base + S_X + off * (kXBytes / 2), 16, 1024) + 2 * (kk & 3),
                                  sdesc_sw128(rs + off * kRAtom, 16, 1024) + 2 * (kk & 3), ID, kk > 0);
                    }
                    umma_commit(bar(B_SX));
                    umma_commit(bar(B_RE + st));
                    // the stage of step s - 1 refills with step s + 2
                    if (s >= 2 && s + 2 < steps) {
                        const int pst = (s - 2) % NR;
                        if (!(ok = wait(bar(B_RE + pst), ((s - 2) / NR) & 1))) break;
                        load_r(s + 2);
                    }
                }
                // P.V of the previous step after this step's logits MMA, so that the softmax
                // stays off the chain of carried rows
                if (s >= 1 && !(ok = issue_pv(s - 1))) break;
            }
            if (ok) ok = issue_pv(steps - 1);
            umma_commit(bar(B_FIN));
            mbar_wait(bar(B_FIN), 0, limit_ns);
            while (r_done < r_iss) {
                const int s = (int)r_done + 1;
                mbar_wait(bar(B_RF + (s - 1) % NR), ((s - 1) / NR) & 1, limit_ns);
                ++r_done;
            }
            while (v_done < v_iss) {
                const int s = (int)v_done;
                mbar_wait(bar(B_VF + s % NV), (s / NV) & 1, limit_ns);
                ++v_done;
            }
            if (!ok) {
                report_status(status, kStatusTimeout);
                *abort_f = 1u;
            }
        }
    } else if (warp < 4) {
        // ================================================================ softmax
        const int r = tid;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        const int tok = 128 * t + r;
        const bool valid = tok < L;
        const size_t hLp = (size_t)bh * Lp;
        float m_run = -INFINITY, l_run = 0.f;
        double between = 0.0;
        const float lci = (FOX && valid) ? lc2[hLp + tok] : 0.f;
        bool ok = true;
        for (int s = 0; ok && s < steps; ++s) {
            const int b = 2 * t + 1 - s;
            const bool diag = (s == 0) ? (r >= 64) : (s == 1 && r < 64);  // warp-uniform
            const bool offd = (s >= 2) || (s == 1 && r >= 64);
            float x[64];
            if (s >= 1) {
                if (!(ok = wait_warp(bar(B_SX), (s - 1) & 1))) break;
                tc_fence_after();
                if (offd) {
                    tld32(tmem + lane_off + C_S, x);
                    tld32(tmem + lane_off + C_S + 32, x + 32);
                }
                tc_fence_before();
                mbar_arrive_warp(bar(B_SF));
            }
            if (diag) {
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(dg + (((size_t)bh * nblk + b) * kC + (r & 63)) * kC);
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const uint4 c = __ldg(src + q8);
                    const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w4[e]));
                        x[8 * q8 + 2 * e] = f.x;
                        x[8 * q8 + 2 * e + 1] = f.y;
                    }
                }
            } else if (offd) {
                const float rb = FOX ? (float)((double)lci + between) : 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    float v = x[j] * scale_log2;
                    if (FOX) v += rb + __ldg(tail2 + hLp + (size_t)b * kC + j);
                    x[j] = v;
                }
                if (FOX) between += tot2[(size_t)bh * nblk + b];
            }
            const bool live = valid && (diag || offd);
            float mx = -INFINITY;
            if (live) {
#pragma unroll
                for (int j = 0; j < 64; j += 2) mx = fmax3(mx, x[j], x[j + 1]);
            }
            // P and O are free once the previous P.V has completed
            if (s >= 1) {
                if (!(ok = wait_warp(bar(B_PV), (s - 1) & 1))) break;
                tc_fence_after();
            }
            float alpha = 1.f;
            if (mx > m_run + kRescale || (m_run == -INFINITY && mx > -INFINITY)) {
                alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mx);
                m_run = mx;
            }
            // rows whose O already holds weighted values and whose maximum rose: rescale O
            // (the loads and stores are warp-wide; other lanes multiply by 1)
            const bool resc = (alpha != 1.f) && (l_run > 0.f);
            if (__any_sync(0xffffffffu, resc)) {
                const float f = resc ? alpha : 1.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_off + C_O + 32 * c, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * f);
                    tmem_st32(tmem + lane_off + C_O + 32 * c, u);
                }
                tmem_st_wait();
            }
            l_run *= alpha;
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            float p[64];
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                p[j] = live ? ex2_approx(x[j] - m_use) : 0.f;
                sum += p[j];
            }
            l_run += sum;
            st_chunks(sm + S_P, r, 0, p);
            st_chunks(sm + S_P, r, 4, p + 32);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive_warp(bar(B_PR));
        }
        if (ok) ok = wait_warp(bar(B_PV), (steps - 1) & 1);
        if (ok) {
            tc_fence_after();
            const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
            if (valid) {
                if (lse != nullptr)
                    lse[(size_t)bh * L + tok] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
            }
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tld32(tmem + lane_off + C_O + 32 * c, o);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)bh * L + tok) * 128 + 32 * c);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                                            pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                            pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                            pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
                }
            }
        }
    } else {
        // ================================================================ carried rows
        const int r = tid - 128;
        const uint32_t lane_off = (uint32_t)(32 * (warp - 4)) << 16;
        bool ok = true;
        for (int s = 1; ok && s < steps; ++s) {
            if (s == steps - 1) break;  // the last key block carries nothing further
            if (!(ok = wait_warp(bar(B_SX), (s - 1) & 1))) break;
            tc_fence_after();
            // block 2t's rows keep q~ past their own (diagonal) block
            if (!(s == 1 && r < 64)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float x[32];
                    tld32(tmem + lane_off + C_X + 32 * c, x);
                    st_chunks(sm + S_X + (uint32_t)(c >> 1) * (kXBytes / 2), r, 4 * (c & 1), x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive_warp(bar(B_XR));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Head size 128, bf16 inputs: the scan over the d128_tc_layout workspace.
cudaError_t launch_scan_tc128(const void *v, void *out, float *lse, bool fox, int BH, int L,
                              float scale, void *ws, uint64_t limit_ns, cudaStream_t stream) {
    const D128TcLayout y = d128_tc_layout(1, BH, L, fox);
    char *base = static_cast<char *>(ws);
    CUtensorMap tq, tk, tv;
    if (!make_map128(&tq, base + y.off_qt, y.Lp, BH, 128) ||
        !make_map128(&tk, base + y.off_kp, y.nblk * 192, BH, 192) ||
        !make_map128(&tv, v, L, BH, 64))
        return cudaErrorInvalidValue;
    auto kern = fox ? scan_tc128_kernel<true> : scan_tc128_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmem);
    if (e != cudaSuccess) return e;
    // shared per token: [K~_b; P_b] (768 B) and v (256 B)
    const bool hf = heads_fastest((size_t)BH, (size_t)L, 1024);
    kern<<<hf ? dim3(BH, y.nblk / 2) : dim3(y.nblk / 2, BH), kThr, kSmem, stream>>>(
        tq, tk, tv, reinterpret_cast<const __half *>(base + y.off_dg),
        fox ? reinterpret_cast<const float *>(base + y.off_lc2) : nullptr,
        fox ? reinterpret_cast<const float *>(base + y.off_tail2) : nullptr,
        fox ? reinterpret_cast<const double *>(base + y.off_tot2) : nullptr,
        fox ? reinterpret_cast<const int *>(base + y.off_first) : nullptr,
        static_cast<__nv_bfloat16 *>(out), lse, L, y.Lp, y.nblk, scale * kLog2e,
        reinterpret_cast<uint32_t *>(base), limit_ns, hf ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace path
