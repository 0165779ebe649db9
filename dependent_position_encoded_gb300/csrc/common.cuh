// Shared definitions of the PaTH attention kernels for sm_103a: the workspace
// layout, bf16 helpers and inline-PTX wrappers for mbarriers, TMA and tcgen05.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace path {

constexpr int kD = 64;      // head size (the only one supported)
constexpr int kC = 64;      // tokens per UT block
constexpr int kTile = 128;  // query rows per tensor-core tile (two UT blocks)
constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLog2eD = 1.4426950408889634;

// Status word codes written by kernels into the workspace header.
constexpr uint32_t kStatusTimeout = 7u;

// ---------------------------------------------------------------- workspace
// All regions start on 256-byte boundaries. Per head (bh) and block b:
//   qt  : (BH, Lp, 64)        boundary-adjusted queries  q~_i = (H_start ... H_i) q_i
//   kp  : (BH, nblk, 128, 64) rows 0-63 keys k~_j = H_end ... H_{j+1} k_j,
//                             rows 64-127 the dense block transition P_b (row-major)
//   dg  : (BH, nblk, 64, 64)  diagonal-block logits in log2 units (masked -inf): fp16 for
//                             bf16 inputs, fp32 for fp32 inputs
//   pr  : (BH, nblk/2, 128, 64) bf16 inputs only: per pair of blocks u = (2u, 2u+1),
//                             rows 0-63 K^_j = P_{2u+1}^T k~_j (keys of block 2u carried
//                             through block 2u+1), rows 64-127 Pi_u = P_{2u} P_{2u+1}
//   c2  : (BH, Lp)            fp32 log2(e) * cumsum(log f) relative to the base of the
//                             token's pair of blocks, with the pair bases as fp32 pairs
//                             (PaTH-FoX only)
// nblk is rounded up to an even count so that 128-row tiles are complete;
// padded tokens carry identity transitions and zero queries and keys.
struct FwdLayout {
    int BH, L, nblk, Lp, elt;
    size_t off_qt, off_kp, off_dg, off_pr, off_c2, off_pbase, off_mpre, off_kpre, off_fb;
    size_t off_btot, off_bmin, off_boff, off_bkmax, off_qn, off_dmax, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Launch order of the kernels whose CTAs walk key blocks for longer the later their query
// tile (every such grid lists each head's tiles longest walk first). When the operands that
// a head's CTAs share (shared_bytes_per_token for every token of every head) fit in about
// three quarters of L2, heads go fastest, so that the longest walks of all heads start first and
// the end of the launch is made of short walks. Otherwise CTAs run head by head, so that
// the CTAs resident together share their key blocks in L2.
inline bool heads_fastest(size_t BH, size_t L, size_t shared_bytes_per_token) {
    return BH * L * shared_bytes_per_token <= ((size_t)96 << 20);
}

// Workspace of the d = 128 forward (defined in fwd_d128.cu).
struct D128Layout {
    int BH, nblk, Lp;
    size_t off_qt, off_kp, off_dg;
    size_t off_lc, off_tail, off_tot;  // PaTH-FoX only (else all equal to total)
    size_t off_mlc, off_kmax, off_cst, off_mpre, off_kpre, total;  // PaTH-FoX early exit
};
D128Layout d128_layout(int B, int H, int L, bool fox);

// Workspace of the tensor-core d = 128 forward (bf16 inputs). nblk = ceil(L / 64) rounded up
// to even, Lp = 64 nblk:
//   qt  : (BH, Lp, 128) bf16 boundary-adjusted queries
//   kp  : (BH, nblk, 192, 128) bf16: rows 0-63 k~_j, rows 64-191 the block transition P_b
//   dg  : (BH, nblk, 64, 64) fp16 diagonal-block logits, log2 units, -inf where masked
//   PaTH-FoX: lc2, tail2 (BH, Lp) fp32 in-block inclusive gate sums and the keys' tail sums
//   T2_b - lc2_j, tot2 (BH, nblk) fp64 block totals, all in log2 units; for the early exit
//   per query row |q~_i| and the diagonal-table row maximum qn, dmax (BH, Lp) fp32, per key
//   block the fp64 total and in-block minimum of the gate prefix sums btot, bmin (natural
//   log), the largest |k~_j| bkmax, the block offsets boff (fp64), the prefix bounds mpre,
//   kpre (fp32) and per query block the first key block it needs (int32), all (BH, nblk)
struct D128TcLayout {
    int BH, nblk, Lp;
    size_t off_qt, off_kp, off_dg, off_lc2, off_tail2, off_tot2;
    size_t off_qn, off_dmax, off_btot, off_bmin, off_bkmax, off_boff, off_mpre, off_kpre,
        off_first, total;
};
inline D128TcLayout d128_tc_layout(int B, int H, int L, bool fox) {
    D128TcLayout y;
    y.BH = B * H;
    const int nb = (L + kC - 1) / kC;
    y.nblk = (nb + 1) & ~1;
    y.Lp = y.nblk * kC;
    const size_t bh = (size_t)y.BH;
    size_t off = 256;
    y.off_qt = off;
    off = align256(off + bh * y.Lp * 128 * 2);
    y.off_kp = off;
    off = align256(off + bh * y.nblk * 192 * 128 * 2);
    y.off_dg = off;
    off = align256(off + bh * y.nblk * kC * kC * 2);
    y.off_lc2 = y.off_tail2 = y.off_tot2 = off;
    y.off_qn = y.off_dmax = y.off_btot = y.off_bmin = y.off_bkmax = y.off_boff = off;
    y.off_mpre = y.off_kpre = y.off_first = off;
    if (fox) {
        const size_t rows = bh * y.Lp, blocks = bh * y.nblk;
        off = align256(off + rows * 4);
        y.off_tail2 = off;
        off = align256(off + rows * 4);
        y.off_tot2 = off;
        off = align256(off + blocks * 8);
        y.off_qn = off;
        off = align256(off + rows * 4);
        y.off_dmax = off;
        off = align256(off + rows * 4);
        y.off_btot = off;
        off = align256(off + blocks * 8);
        y.off_bmin = off;
        off = align256(off + blocks * 8);
        y.off_boff = off;
        off = align256(off + blocks * 8);
        y.off_bkmax = off;
        off = align256(off + blocks * 4);
        y.off_mpre = off;
        off = align256(off + blocks * 4);
        y.off_kpre = off;
        off = align256(off + blocks * 4);
        y.off_first = off;
        off = align256(off + blocks * 4);
    }
    y.total = off;
    return y;
}

// Workspace of the backward pass (defined in backward.cu).
struct BwdLayout {
    int BH, nblk, Lp;
    size_t off_qt, off_kp, off_dg, off_dqt, off_dkt, off_dP, off_dTd, off_stash;
    size_t off_loc, off_rs, off_cs, off_cb, total;  // PaTH-FoX only (else all equal to total)
};
BwdLayout bwd_layout(int B, int H, int L, bool fox);

inline FwdLayout fwd_layout(int B, int H, int L, int elt_bytes, bool fox) {
    FwdLayout lay;
    lay.BH = B * H;
    lay.L = L;
    int nb = (L + kC - 1) / kC;
    lay.nblk = (nb + 1) & ~1;
    lay.Lp = lay.nblk * kC;
    lay.elt = elt_bytes;
    size_t bh = (size_t)lay.BH;
    size_t off = 256;  // status header
    lay.off_qt = off;
    off = align256(off + bh * lay.Lp * kD * elt_bytes);
    lay.off_kp = off;
    off = align256(off + bh * lay.nblk * 2 * kC * kD * elt_bytes);
    lay.off_dg = off;
    off = align256(off + bh * lay.nblk * kC * kC * (elt_bytes == 2 ? 2 : 4));
    // bf16 PaTH: the block-pair products of the two-block scan steps (the PaTH-FoX scan takes
    // one block per step and needs none)
    lay.off_pr = off;
    if (elt_bytes == 2 && !fox) off = align256(off + bh * (lay.nblk / 2) * 2 * kC * kD * 2);
    // PaTH-FoX only, with c2 = log2(e) * cumsum(log f): c2 relative to the base of its
    // pair of blocks, c2_t - c2_base(t / 128) (BH, Lp) fp32, and the pair bases as fp32 pairs
    // hi + lo (BH, nblk / 2, 2); per key block the prefix minimum of c2 and prefix maximum
    // of |k~| (BH, nblk) fp32; per query block the first key block the scan visits
    // (BH, nblk) int32; and the per-block fp64 totals, in-block minima, offsets and fp32
    // key-norm maxima they come from
    lay.off_c2 = lay.off_pbase = lay.off_mpre = lay.off_kpre = lay.off_fb = off;
    lay.off_btot = lay.off_bmin = lay.off_boff = lay.off_bkmax = off;
    lay.off_qn = lay.off_dmax = off;
    if (fox) {
        const size_t nb = bh * lay.nblk;
        off = align256(off + bh * lay.Lp * sizeof(float));
        lay.off_pbase = off;
        off = align256(off + nb * sizeof(float));  // (nblk / 2) pairs x (hi, lo)
        lay.off_mpre = off;
        off = align256(off + nb * sizeof(float));
        lay.off_kpre = off;
        off = align256(off + nb * sizeof(float));
        lay.off_fb = off;
        off = align256(off + nb * sizeof(int));
        lay.off_btot = off;
        off = align256(off + nb * sizeof(double));
        lay.off_bmin = off;
        off = align256(off + nb * sizeof(double));
        lay.off_boff = off;
        off = align256(off + nb * sizeof(double));
        lay.off_bkmax = off;
        off = align256(off + nb * sizeof(float));
        // per query row: |q~_i| and the largest entry of its diagonal-table row (written by
        // the bf16 preprocessing so that the early-exit pass need not re-read the rows)
        lay.off_qn = off;
        off = align256(off + bh * lay.Lp * sizeof(float));
        lay.off_dmax = off;
        off = align256(off + bh * lay.Lp * sizeof(float));
    }
    lay.total = off;
    return lay;
}

// Decode: per head and split, (m, l, o[d]) partial results (d = 64 or 128).
constexpr int kDecodeChunk = 1024;  // cached keys per split
inline int decode_splits(int cap) { return (cap + kDecodeChunk - 1) / kDecodeChunk; }
inline size_t decode_ws_bytes(int B, int H, int cap, int d = kD) {
    return 256 + align256((size_t)B * H * decode_splits(cap) * (d + 2) * sizeof(float));
}

// ---------------------------------------------------------------- conversions
template <typename T> struct Elt;
template <> struct Elt<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elt<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// SM cycle counter: cheap enough to read inside polling loops. Wait limits are given
// in nanoseconds and converted at 2 cycles per ns, so at clocks up to 2 GHz a limit never
// expires early (it may expire somewhat later at lower clocks).
__device__ __forceinline__ uint64_t cycles_now() { return (uint64_t)clock64(); }
__host__ __device__ constexpr uint64_t ns_to_cycles(uint64_t ns) { return 2 * ns; }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// One arrival per warp: every lane's prior writes (and fences) are ordered before lane 0's
// release by the warp barrier, so an mbarrier counts warps instead of threads.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` nanoseconds for the phase to
// complete (it wakes when the phase completes), so a waiting warp takes no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase (for polling loops that watch several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns false after about `limit_ns` nanoseconds without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = cycles_now(), lim = ns_to_cycles(limit_ns);
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (cycles_now() - t0 > lim) return false;
    }
}

// Packed fp32 pairs (sm_100 and later): one instruction for two lanes of work.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// max of three (sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 2^x on the SFU (approximate, subnormal results flushed to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B bf16,
// A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4)                           // D format: f32
           | (1u << 7)                         // A format: bf16
           | (1u << 10)                        // B format: bf16
           | ((b_mn_major ? 1u : 0u) << 16)    // B major-ness
           | ((uint32_t)(N >> 3) << 17)        // N / 8
           | ((uint32_t)(M >> 4) << 24);       // M / 16
}

// Tensor store of a 128-byte-swizzled shared tile (box of the map) at (c0, c1, c2); one
// bulk group per store.
__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 version field = 1).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t of the warp gets its lane's columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile
// whose rows are 128 bytes (64 bf16) long.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Records the first error code in the workspace status word.
__device__ __forceinline__ void report_status(uint32_t *status, uint32_t code) {
    if (status) atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------- host: TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 3-D 16-bit (bf16 or fp16) map over (heads, rows, 64 columns) with a (1, box_rows, 64) box and 128-byte
// swizzle (the layout every tcgen05 operand tile here uses). Rows beyond `rows` read 0.
inline bool make_map_16bit(CUtensorMap *m, CUtensorMapDataType type, const void *ptr, int rows,
                           int heads, int box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)rows * kD * 2};
    cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, type, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool make_map_bf16(CUtensorMap *m, const void *ptr, int rows, int heads, int box_rows) {
    return make_map_16bit(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rows, heads, box_rows);
}

inline bool make_map_f16(CUtensorMap *m, const void *ptr, int rows, int heads, int box_rows) {
    return make_map_16bit(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ptr, rows, heads, box_rows);
}

}  // namespace path
