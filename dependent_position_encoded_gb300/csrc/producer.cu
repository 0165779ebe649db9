// The w / beta producer: per token, the Householder direction w and strength beta that
// PaTH attention consumes.
//
// Review "거리에서 경로로, PaTH Attention" §3: w comes from a low-dimensional linear
// projection and a short convolution of size 3 and is then L2-normalised; beta is twice a
// sigmoid. Technical summary "技術要約: PaTH Attention" §2: beta_s = 2 sigmoid(u^T x_s + b);
// §6: beta is clipped for bf16. Per token t of sequence b and head h:
//   z_t   = W_down x_t                                    (R)
//   y_t   = W_up z_t                                      (H*d)
//   y'_t  = conv[:,2] * y_t + conv[:,1] * y_{t-1} + conv[:,0] * y_{t-2}   (zero before t = 0)
//   w_t,h = y'_t,h / max(|y'_t,h|, 1e-12),   beta_t,h = min(2 sigmoid(u_h . x_t + b_h), beta_max)
//
// Three launches:
//   P0 forms the tap-scaled up-projections W'_k = diag(conv[:,k]) W_up (bf16), so that the
//      convolution becomes part of the second contraction: y'_t = sum_k W'_k z_{t-2+k};
//   P1 (tcgen05): [z | beta logits] = x [W_down; u]^T for 128-token tiles, streaming x
//      through a TMA ring (six stages and one CTA per SM where they fit, else three stages);
//      the epilogue writes z (bf16) and beta;
//   P2 (tcgen05): persistent over (128-token tile, two-head chunk) units, each CTA an equal
//      contiguous run of them; per unit three accumulating contractions of
//      z tiles loaded at rows t0, t0-1, t0-2 (a negative start row reads zeros: the causal
//      zero history) with W'_2, W'_1, W'_0, two heads (N = 128) per TMEM buffer, double
//      buffered; the epilogue normalises each head row into a 128-byte-swizzled shared tile
//      that one TMA tensor store writes to w in the (B, H, L, d) layout the attention
//      takes (rows past L are clipped by the store).
// x is read once and w written once: the pair is bound by HBM bandwidth.
#include <algorithm>

#include "common.cuh"

namespace path {

namespace {

constexpr uint32_t kRowTile = 128 * 128;  // 128 rows x 64 bf16, 128-byte swizzled

__host__ __device__ constexpr uint32_t idesc_bf16_kk(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// Named barrier over the four epilogue warps (ids 1..; 0 is __syncthreads).
__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Bounded wait by one thread; false (and the status word set) after limit_ns.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t par, uint64_t limit_ns,
                                             uint32_t *status) {
    if (mbar_wait(bar, par, limit_ns)) return true;
    report_status(status, kStatusTimeout);
    return false;
}

// ---------------------------------------------------------------- P0: tap-scaled W_up
__global__ void producer_scale_kernel(const __nv_bfloat16 *__restrict__ w_up,
                                      const float *__restrict__ conv, int C, int R,
                                      __nv_bfloat16 *__restrict__ wk) {
    const size_t n = (size_t)C * R;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i / R);
        const float v = __bfloat162float(w_up[i]);
#pragma unroll
        for (int k = 0; k < 3; ++k) wk[(size_t)k * n + i] = __float2bfloat16_rn(conv[c * 3 + k] * v);
    }
}

// ---------------------------------------------------------------- P1: z and beta
constexpr int kP1StagesMax = 6;  // ring depth when it fits (else 3)
constexpr int kP1Threads = 192;  // warps 0-3: epilogue (TMEM lanes 0-127); 4: TMA; 5: MMA

// Persistent: CTA c takes the 128-token tiles c, c + grid, ... The TMA ring runs across
// tile boundaries and the accumulator is double-buffered in TMEM (acc_cols columns each),
// so one tile's epilogue overlaps the next tile's loads and MMAs.
template <int kP1Stages>
__global__ void __launch_bounds__(kP1Threads, 1)
producer_down_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_wd,
                     const __grid_constant__ CUtensorMap tm_u, const float *__restrict__ bias,
                     float beta_max, int BL, int L, int D, int R, int H, int Hp, int acc_cols,
                     __nv_bfloat16 *__restrict__ z, float *__restrict__ beta_out,
                     uint32_t *status, uint64_t limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    const int NB = R + Hp;
    const uint32_t stage_bytes = kRowTile + (uint32_t)NB * 128;
    const uint32_t bar0 = base + kP1Stages * stage_bytes;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kP1Stages + s); };
    auto acc_full = [&](int i) { return bar0 + 8u * (2 * kP1Stages + i); };
    auto acc_empty = [&](int i) { return bar0 + 8u * (2 * kP1Stages + 2 + i); };
    uint32_t *const slot = reinterpret_cast<uint32_t *>(sm + (bar0 - base) + 8 * (2 * kP1Stages + 4));
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = D / 64;
    const int ntiles = (BL + 127) / 128;
    const int nmine = blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        abort_s = 0u;
        for (int s = 0; s < kP1Stages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), (uint32_t)(2 * acc_cols));
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;

    if (warp == 4 && lane == 0) {
        // ---- TMA producer: x chunk (128 tokens x 64) and [W_down; u] chunk (NB x 64)
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_wd);
        tma_prefetch_desc(&tm_u);
        int i = 0;
        bool ok = true;
        for (int j = 0; j < nmine && ok; ++j) {
            const int row0 = (blockIdx.x + j * gridDim.x) * 128;
            for (int kc = 0; kc < nk; ++kc, ++i) {
                const int s = i % kP1Stages;
                if (i >= kP1Stages &&
                    !wait_bounded(empty(s), ((i / kP1Stages) - 1) & 1, limit_ns, status)) {
                    abort_s = 1u;
                    ok = false;
                    break;
                }
                const uint32_t a = base + s * stage_bytes, b = a + kRowTile;
                mbar_arrive_expect_tx(full(s), stage_bytes);
                tma_load_2d(a, &tm_x, full(s), kc * 64, row0);
                tma_load_2d(b, &tm_wd, full(s), kc * 64, 0);
                tma_load_2d(b + (uint32_t)R * 128, &tm_u, full(s), kc * 64, 0);
            }
        }
        // drain: every issued copy has landed before the CTA may exit
        for (int q = (i > kP1Stages ? i - kP1Stages : 0); q < i; ++q)
            mbar_wait(full(q % kP1Stages), (q / kP1Stages) & 1, limit_ns);
    } else if (warp == 5 && lane == 0) {
        // ---- MMA issuer: acc[j & 1] (128 x NB) = x_tile [W_down; u]^T
        const uint32_t idesc = idesc_bf16_kk(128, NB);
        bool ok = true;
        int i = 0;
        for (int j = 0; j < nmine && ok; ++j) {
            const int buf = j & 1;
            if (j >= 2 && !wait_bounded(acc_empty(buf), ((j >> 1) - 1) & 1, limit_ns, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kc = 0; kc < nk; ++kc, ++i) {
                const int s = i % kP1Stages;
                if (!wait_bounded(full(s), (i / kP1Stages) & 1, limit_ns, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(base + s * stage_bytes, 16, 1024);
                const uint64_t bd = sdesc_sw128(base + s * stage_bytes + kRowTile, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + (uint32_t)(buf * acc_cols), ad + 2 * kk, bd + 2 * kk, idesc,
                              (kc > 0 || kk > 0) ? 1u : 0u);
                umma_commit(empty(s));
            }
            if (ok) umma_commit(acc_full(buf));
        }
        if (!ok) {
            abort_s = 1u;
            // release the epilogue, which waits on accumulators it has not seen yet
            umma_commit(acc_full(0));
            umma_commit(acc_full(1));
        }
    } else if (warp < 4) {
        // ---- epilogue: row = token row0 + 32 warp + lane
        const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
        uint32_t v[32];
        for (int j = 0; j < nmine; ++j) {
            const int buf = j & 1;
            if (threadIdx.x == 0 && !wait_bounded(acc_full(buf), (j >> 1) & 1, limit_ns, status))
                abort_s = 1u;
            epi_sync();
            if (abort_s != 0u) break;
            tc_fence_after();
            const uint32_t tb = tl + (uint32_t)(buf * acc_cols);
            const int tok = (blockIdx.x + j * gridDim.x) * 128 + 32 * warp + lane;
            for (int c0 = 0; c0 < R; c0 += 32) {
                tmem_ld32(tb + c0, v);
                tmem_ld_wait();
                if (tok < BL) {
                    uint4 *dst = reinterpret_cast<uint4 *>(z + (size_t)tok * R + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                            pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                            pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                            pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                }
            }
            const int bq = tok / L, t = tok - bq * L;
            for (int h0 = 0; h0 < H; h0 += 32) {
                tmem_ld32(tb + R + h0, v);
                tmem_ld_wait();
                if (tok < BL) {
#pragma unroll 4
                    for (int q = 0; q < 32; ++q) {
                        const int h = h0 + q;
                        if (h >= H) break;
                        const float a = __uint_as_float(v[q]) + bias[h];
                        const float be = 2.f / (1.f + expf(-a));
                        beta_out[((size_t)bq * H + h) * L + t] = fminf(be, beta_max);
                    }
                }
            }
            tc_fence_before();
            epi_sync();
            if (threadIdx.x == 0) mbar_arrive(acc_empty(buf));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)(2 * acc_cols));
    }
}

// ---------------------------------------------------------------- P2: w
constexpr int kP2Stages = 3;
constexpr int kP2Threads = 192;  // warps 0-3: epilogue; 4: TMA; 5: MMA
constexpr int kP2Cols = 256;     // two 128-column (two-head) accumulators
// One z tile per 64-wide K chunk: rows t0-2 .. t0+133 (136 loaded, slot of 144 rows so that
// the next chunk starts on a 1024-byte boundary). The MMA of tap k reads rows k .. k+127,
// i.e. tokens t - 2 + k: its descriptor starts k rows (k * 128 bytes) into the tile. The
// 128-byte swizzle follows the absolute shared-memory address bits, as the TMA wrote it.
constexpr int kZRows = 136;
constexpr uint32_t kZSlot = 144 * 128;

__global__ void __launch_bounds__(kP2Threads, 1)
producer_up_kernel(const __grid_constant__ CUtensorMap tm_z,
                   const __grid_constant__ CUtensorMap tm_wk,
                   const __grid_constant__ CUtensorMap tm_w, int nseq, int L, int R, int H,
                   uint32_t *status, uint64_t limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    const int nkc = R / 64;                       // 64-wide K chunks of z
    const uint32_t a_base = base;                      // z tiles, one per K chunk
    const uint32_t b_base = base + (uint32_t)nkc * kZSlot;  // W' ring
    const uint32_t c_base = b_base + kP2Stages * kRowTile;  // two staging tiles of w
    const uint32_t bar0 = c_base + 2 * kRowTile;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kP2Stages + s); };
    const uint32_t a_full = bar0 + 8u * (2 * kP2Stages);
    auto acc_full = [&](int i) { return bar0 + 8u * (2 * kP2Stages + 1 + i); };
    auto acc_empty = [&](int i) { return bar0 + 8u * (2 * kP2Stages + 3 + i); };
    const uint32_t a_empty = bar0 + 8u * (2 * kP2Stages + 5);
    uint32_t *const slot = reinterpret_cast<uint32_t *>(sm + (bar0 - base) + 8 * (2 * kP2Stages + 6));
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nchunk = (H + 1) / 2;                // two heads per accumulator
    const int ntps = (L + 127) / 128;              // 128-token tiles per sequence
    const int nitems = ntps * nseq;                // work items (tile, sequence)
    // units (item, chunk) in item-major order; CTA c takes the contiguous range [u0, u1), so
    // every CTA gets the same number of two-head chunks within one and reloads z only where
    // its range crosses into the next item
    const long long nunits = (long long)nitems * nchunk;
    const int u0 = (int)(nunits * blockIdx.x / gridDim.x);
    const int u1 = (int)(nunits * (blockIdx.x + 1) / gridDim.x);
    const int it0 = u0 / nchunk, it1 = u1 > u0 ? (u1 - 1) / nchunk + 1 : it0;  // items [it0, it1)
    if (threadIdx.x == 0) {
        abort_s = 0u;
        for (int s = 0; s < kP2Stages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), kP2Cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;

    if (warp == 4 && lane == 0) {
        // ---- TMA: per work item the three shifted z tiles (once the previous item's MMAs
        // have read them), then W'_tap chunks in consumption order (chunk, tap, K chunk)
        tma_prefetch_desc(&tm_z);
        tma_prefetch_desc(&tm_wk);
        int i = 0, j = 0;
        bool ok = true;
        for (int item = it0; item < it1 && ok; ++item, ++j) {
            const int t0 = (item % ntps) * 128, bq = item / ntps;
            const int c0 = max(u0 - item * nchunk, 0), c1 = min(u1 - item * nchunk, nchunk);
            if (j >= 1 && !wait_bounded(a_empty, (j - 1) & 1, limit_ns, status)) {
                abort_s = 1u;
                break;
            }
            mbar_arrive_expect_tx(a_full, (uint32_t)nkc * kZRows * 128);
            for (int kc = 0; kc < nkc; ++kc)
                tma_load_3d(a_base + (uint32_t)kc * kZSlot, &tm_z, a_full, kc * 64, t0 - 2, bq);
            for (int step = c0 * 3 * nkc; step < c1 * 3 * nkc; ++step, ++i) {
                const int s = i % kP2Stages;
                if (i >= kP2Stages &&
                    !wait_bounded(empty(s), ((i / kP2Stages) - 1) & 1, limit_ns, status)) {
                    abort_s = 1u;
                    ok = false;
                    break;
                }
                const int kc = step % nkc, tap = (step / nkc) % 3, chunk = step / (3 * nkc);
                mbar_arrive_expect_tx(full(s), kRowTile);
                tma_load_3d(b_base + (uint32_t)s * kRowTile, &tm_wk, full(s), kc * 64, 128 * chunk,
                            tap);
            }
        }
        // drain: every issued copy has landed before the CTA may exit
        for (int q = (i > kP2Stages ? i - kP2Stages : 0); q < i; ++q)
            mbar_wait(full(q % kP2Stages), (q / kP2Stages) & 1, limit_ns);
        if (j > 0) mbar_wait(a_full, (j - 1) & 1, limit_ns);
    } else if (warp == 5 && lane == 0) {
        // ---- MMA: acc[g & 1] (g counts chunks over all items) = sum over taps and K chunks
        // of z_tap W'_tap^T (N = 128)
        const uint32_t idesc = idesc_bf16_kk(128, 128);
        bool ok = true;
        int i = 0, g = 0, j = 0;
        for (int item = it0; item < it1 && ok; ++item, ++j) {
            const int c0 = max(u0 - item * nchunk, 0), c1 = min(u1 - item * nchunk, nchunk);
            if (!wait_bounded(a_full, j & 1, limit_ns, status)) {
                ok = false;
                break;
            }
            for (int chunk = c0; chunk < c1 && ok; ++chunk, ++g) {
                const int buf = g & 1;
                if (g >= 2 && !wait_bounded(acc_empty(buf), ((g >> 1) - 1) & 1, limit_ns, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int tap = 0; tap < 3 && ok; ++tap) {
                    for (int kc = 0; kc < nkc; ++kc, ++i) {
                        const int s = i % kP2Stages;
                        if (!wait_bounded(full(s), (i / kP2Stages) & 1, limit_ns, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad =
                            sdesc_sw128(a_base + (uint32_t)kc * kZSlot + 128u * tap, 16, 1024);
                        const uint64_t bd = sdesc_sw128(b_base + (uint32_t)s * kRowTile, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(tmem + 128u * buf, ad + 2 * kk, bd + 2 * kk, idesc,
                                      (tap > 0 || kc > 0 || kk > 0) ? 1u : 0u);
                        umma_commit(empty(s));
                    }
                }
                if (ok) umma_commit(acc_full(buf));
            }
            if (ok) umma_commit(a_empty);  // the item's z tiles may be replaced
        }
        if (!ok) {
            abort_s = 1u;
            // release the epilogue: it waits on the accumulators it has not yet seen
            for (int i2 = 0; i2 < 2; ++i2) umma_commit(acc_full(i2));
        }
    } else if (warp < 4) {
        // ---- epilogue: row = token t0 + 32 warp + lane; two heads per accumulator. Each
        // head row is normalised into staging tile hn & 1 (hn counts heads), which one TMA
        // tensor store writes out (rows past L are clipped by the store). One barrier per
        // head: before it, thread 0 waits until the previous head's store has read its
        // tile, which is the tile the next head fills.
        const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
        const int r = 32 * warp + lane;
        int g = 0, hn = 0;
        for (int u = u0; u < u1; ++u, ++g) {
            const int item = u / nchunk, chunk = u % nchunk;
            const int t0 = (item % ntps) * 128, bq = item / ntps;
            const int buf = g & 1;
            if (threadIdx.x == 0 &&
                !wait_bounded(acc_full(buf), (g >> 1) & 1, limit_ns, status))
                abort_s = 1u;
            epi_sync();
            if (abort_s != 0u) break;
            tc_fence_after();
            const int nh = min(2, H - 2 * chunk);
            for (int hh = 0; hh < nh; ++hh, ++hn) {
                const int h = 2 * chunk + hh;
                uint32_t a[32], b[32];
                tmem_ld32(tl + 128u * buf + 64u * hh, a);
                tmem_ld32(tl + 128u * buf + 64u * hh + 32u, b);
                tmem_ld_wait();
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float p = __uint_as_float(a[j]), q = __uint_as_float(b[j]);
                    ss = fmaf(p, p, fmaf(q, q, ss));
                }
                const float inv = rsqrtf(fmaxf(ss, 1e-24f));  // 1 / max(|y'|, 1e-12)
                // row r, 128-byte swizzled (conflict-free: the eight lanes of a store phase
                // hold eight consecutive rows and land in eight distinct chunks)
                uint8_t *const tile = sm + (c_base - base) + (hn & 1) * kRowTile;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, q4)) = make_uint4(
                        pack_bf16x2(__uint_as_float(a[8 * q4]) * inv, __uint_as_float(a[8 * q4 + 1]) * inv),
                        pack_bf16x2(__uint_as_float(a[8 * q4 + 2]) * inv, __uint_as_float(a[8 * q4 + 3]) * inv),
                        pack_bf16x2(__uint_as_float(a[8 * q4 + 4]) * inv, __uint_as_float(a[8 * q4 + 5]) * inv),
                        pack_bf16x2(__uint_as_float(a[8 * q4 + 6]) * inv, __uint_as_float(a[8 * q4 + 7]) * inv));
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 4 + q4)) = make_uint4(
                        pack_bf16x2(__uint_as_float(b[8 * q4]) * inv, __uint_as_float(b[8 * q4 + 1]) * inv),
                        pack_bf16x2(__uint_as_float(b[8 * q4 + 2]) * inv, __uint_as_float(b[8 * q4 + 3]) * inv),
                        pack_bf16x2(__uint_as_float(b[8 * q4 + 4]) * inv, __uint_as_float(b[8 * q4 + 5]) * inv),
                        pack_bf16x2(__uint_as_float(b[8 * q4 + 6]) * inv, __uint_as_float(b[8 * q4 + 7]) * inv));
                fence_proxy_async_smem();
                if (hh == nh - 1) tc_fence_before();  // the chunk's TMEM reads are done
                if (threadIdx.x == 0) bulk_wait_read();
                epi_sync();
                if (threadIdx.x == 0) {
                    tma_store_3d(&tm_w, c_base + (uint32_t)(hn & 1) * kRowTile, 0, t0, bq * H + h);
                    if (hh == nh - 1) mbar_arrive(acc_empty(buf));
                }
            }
        }
    }
    if (threadIdx.x == 0) bulk_wait_all();  // the last tiles have been written
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kP2Cols);
    }
}

// 2-D bf16 map (rows x cols, cols contiguous), box (64 cols, box_rows), 128-byte swizzle.
bool map2d(CUtensorMap *m, const void *ptr, int cols, long long rows, int box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map (d2, d1, d0 = cols contiguous), box (64, box_rows, 1), 128-byte swizzle.
bool map3d(CUtensorMap *m, const void *ptr, int cols, int d1, int d2, int box_rows = 128) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * d1};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Workspace of the producer: 256-byte status header, z (B*L, R) bf16, W'_0..2 (3, H*d, R) bf16.
size_t producer_ws_bytes(int B, int L, int R, int H) {
    return 256 + align256((size_t)B * L * R * 2) + align256((size_t)3 * H * kD * R * 2);
}

size_t producer_down_smem(int R, int Hp, int stages) {
    return (size_t)stages * (kRowTile + (size_t)(R + Hp) * 128) + 8 * (2 * stages + 5) + 1024;
}
size_t producer_up_smem(int R) {
    return (size_t)(R / 64) * kZSlot + (size_t)(kP2Stages + 2) * kRowTile +
           8 * (2 * kP2Stages + 7) + 1024;
}

// The caller has checked the sizes (d = 64, D and R multiples of 64, R + round16(H) <= 256).
cudaError_t launch_producer(const void *x, const void *w_down, const void *w_up, const float *conv,
                            const void *u, const float *bias, float beta_max, void *w_out,
                            float *beta_out, int B, int L, int D, int R, int H, void *ws,
                            uint64_t limit_ns, cudaStream_t stream) {
    char *wsb = static_cast<char *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(wsb);
    __nv_bfloat16 *z = reinterpret_cast<__nv_bfloat16 *>(wsb + 256);
    __nv_bfloat16 *wk = reinterpret_cast<__nv_bfloat16 *>(wsb + 256 + align256((size_t)B * L * R * 2));
    const int C = H * kD;
    const long long BL = (long long)B * L;
    const int Hp = (H + 15) & ~15;
    const int acc_cols = (R + Hp) <= 128 ? 128 : 256;  // per accumulator (two of them)
    int dev = 0, nsm = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    if ((err = cudaMemsetAsync(status, 0, 4, stream)) != cudaSuccess) return err;
    producer_scale_kernel<<<(unsigned)std::min<size_t>(((size_t)C * R + 255) / 256, 4096), 256, 0,
                            stream>>>(static_cast<const __nv_bfloat16 *>(w_up), conv, C, R, wk);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    CUtensorMap tx, twd, tu, tz, twk, tw;
    if (!map2d(&tx, x, D, BL, 128) || !map2d(&twd, w_down, D, R, R) || !map2d(&tu, u, D, H, Hp) ||
        !map3d(&tz, z, R, L, B, kZRows) || !map3d(&twk, wk, R, C, 3) || !map3d(&tw, w_out, kD, L, B * H))
        return cudaErrorInvalidValue;
    // one CTA per SM with a deep ring (kP1StagesMax stages) when it fits in shared memory,
    // else three stages; with 256-column accumulators (2 x 256 = all of TMEM) a second CTA
    // on the SM would block in its TMEM allocation: ask for enough shared memory to keep it off
    const bool deep = producer_down_smem(R, Hp, kP1StagesMax) <= 227 * 1024;
    const size_t s1n = producer_down_smem(R, Hp, deep ? kP1StagesMax : 3);
    const size_t s1 = (acc_cols == 128 || deep) ? s1n : std::max<size_t>(s1n, 120 * 1024);
    const size_t s2 = producer_up_smem(R);
    auto k1 = deep ? producer_down_kernel<kP1StagesMax> : producer_down_kernel<3>;
    if ((err = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1)) !=
        cudaSuccess)
        return err;
    if ((err = cudaFuncSetAttribute(producer_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)s2)) != cudaSuccess)
        return err;
    // two CTAs per SM while both fit (TMEM 2 x 2 x 128 columns, shared memory), else one
    const long long tiles1 = (BL + 127) / 128;
    const int per_sm1 = (acc_cols == 128 && 2 * (s1 + 1024) <= 228 * 1024) ? 2 : 1;
    const unsigned g1 = (unsigned)std::min<long long>(tiles1, (long long)per_sm1 * nsm);
    k1<<<g1, kP1Threads, s1, stream>>>(
        tx, twd, tu, bias, beta_max, (int)BL, L, D, R, H, Hp, acc_cols, z, beta_out, status,
        limit_ns);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const long long units2 = (long long)((L + 127) / 128) * B * ((H + 1) / 2);
    const int per_sm2 = 2 * (s2 + 1024) <= 228 * 1024 ? 2 : 1;  // TMEM: 2 x 256 columns fit
    const unsigned g2 = (unsigned)std::min<long long>(units2, (long long)per_sm2 * nsm);
    producer_up_kernel<<<g2, kP2Threads, s2, stream>>>(tz, twk, tw, B, L, R, H, status, limit_ns);
    return cudaGetLastError();
}

}  // namespace path
