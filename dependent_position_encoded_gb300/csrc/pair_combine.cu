// Pair products of the block transitions, for the scan's two-block steps (bf16 inputs).
//
// Technical summary "技術要約: PaTH Attention" §3 and review "거리에서 경로로, PaTH
// Attention" §9: the scan carries each query's accumulated transition product from block
// to block. For a pair of blocks u = (2u, 2u+1), visited upper block first, a state row x
// scores the upper block's keys as x . k~_j, is carried to P_{2u+1} x, scores the lower
// block's keys, and leaves as P_{2u} P_{2u+1} x. So one step over the pair needs, besides
// the upper keys k~_j (j in 2u+1),
//     K^_j = P_{2u+1}^T k~_j   (j in 2u)    and    Pi_u = P_{2u} P_{2u+1},
// i.e. the row blocks of [K~_{2u}; P_{2u}] P_{2u+1}: one 128 x 64 x 64 MMA per pair.
// The bf16 operands are the preprocessing outputs; fp32 accumulation in TMEM; the results
// are rounded to bf16 like every other scan operand.
#include "common.cuh"

namespace path {

namespace {

constexpr uint32_t kPcA = 128 * 128;  // [K~_{2u}; P_{2u}]: 128 rows x 64 bf16
constexpr uint32_t kPcB = 64 * 128;   // P_{2u+1}: 64 rows x 64 bf16
constexpr uint32_t kPcBar = kPcA + kPcB;
// 26 KB per CTA: at most eight CTAs per SM, so their 64 TMEM columns each never exceed 512
constexpr uint32_t kPcSmem = 26 * 1024;
static_assert(kPcBar + 64 + 1024 <= kPcSmem, "pair-combine shared memory");

__global__ void __launch_bounds__(128)
pair_combine_kernel(const __grid_constant__ CUtensorMap tm_kp128,
                    const __grid_constant__ CUtensorMap tm_kp64, __nv_bfloat16 *__restrict__ pr,
                    int npair, uint32_t *status, uint64_t limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t bar_tma = base + kPcBar, bar_mma = base + kPcBar + 8;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(gbase + kPcBar + 16);
    const int u = blockIdx.x, bh = blockIdx.y, r = threadIdx.x, warp = r >> 5;

    if (r == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, kPcA + kPcB);
        tma_load_3d(base, &tm_kp128, bar_tma, 0, (2 * u) * 2 * kC, bh);
        tma_load_3d(base + kPcA, &tm_kp64, bar_tma, 0, (2 * u + 1) * 2 * kC + kC, bh);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), 64);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    bool ok = true;
    if (r == 0) {
        ok = mbar_wait(bar_tma, 0, limit_ns);
        if (ok) {
            tc_fence_after();
            // D = A B with B = P_{2u+1} stored row-major (rows = the contraction index), i.e.
            // an MN-major operand: 16 rows (2048 bytes) per K = 16 step
            constexpr uint32_t ID = idesc_bf16(128, 64, true);
            const uint64_t a = sdesc_sw128(base, 16, 1024);
            const uint64_t b = sdesc_sw128(base + kPcA, 1024, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem, a + 2 * kk, b + 128 * kk, ID, kk > 0);
        }
        umma_commit(bar_mma);  // also covers the no-MMA case: the barrier still completes
        if (!ok) report_status(status, kStatusTimeout);
    }
    const bool done = __all_sync(0xffffffffu, mbar_wait(bar_mma, 0, limit_ns));
    if (done) {
        tc_fence_after();
        uint32_t x[32], y[32];
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        tmem_ld32(tmem + lane_base, x);
        tmem_ld32(tmem + lane_base + 32, y);
        tmem_ld_wait();
        uint4 *dst = reinterpret_cast<uint4 *>(pr + (((size_t)bh * npair + u) * 2 * kC + r) * kD);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t *s = (c < 4) ? &x[8 * c] : &y[8 * (c - 4)];
            dst[c] = make_uint4(pack_bf16x2(__uint_as_float(s[0]), __uint_as_float(s[1])),
                                pack_bf16x2(__uint_as_float(s[2]), __uint_as_float(s[3])),
                                pack_bf16x2(__uint_as_float(s[4]), __uint_as_float(s[5])),
                                pack_bf16x2(__uint_as_float(s[6]), __uint_as_float(s[7])));
        }
    } else if (r == 0) {
        report_status(status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

}  // namespace

cudaError_t launch_pair_combine(int BH, int L, void *ws, uint64_t limit_ns, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 2, false);
    char *basep = static_cast<char *>(ws);
    const int npair = lay.nblk / 2;
    CUtensorMap tm128, tm64;
    if (!make_map_bf16(&tm128, basep + lay.off_kp, lay.nblk * 2 * kC, BH, 2 * kC) ||
        !make_map_bf16(&tm64, basep + lay.off_kp, lay.nblk * 2 * kC, BH, kC))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(pair_combine_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kPcSmem);
    if (err != cudaSuccess) return err;
    pair_combine_kernel<<<dim3(npair, BH), 128, kPcSmem, stream>>>(
        tm128, tm64, reinterpret_cast<__nv_bfloat16 *>(basep + lay.off_pr), npair,
        reinterpret_cast<uint32_t *>(basep), limit_ns);
    return cudaGetLastError();
}

}  // namespace path
