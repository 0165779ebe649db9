// K2 (fp32 dtype): the right-to-left block scan of PaTH attention in fp32 FFMA.
//
// Same algorithm as the tensor-core scan (technical summary "技術要約: PaTH Attention" §3;
// review "거리에서 경로로, PaTH Attention" §9), for fp32 inputs whose tolerance rules out
// bf16 operands: one CTA per 64-row query block of one head holds the state
// X = (q~_i)_i in shared memory and, for key block b = ib, ib-1, ..., 0, forms the
// logits (diagonal block: precomputed; earlier blocks: X K~_b^T), updates the online
// softmax, accumulates O += P V_b and advances X <- X P_b^T.
#include "common.cuh"

namespace path {

namespace {

constexpr int LD = 68;
constexpr int BUF = kC * LD;
constexpr int kThreads = 256;

__device__ __forceinline__ void mm_acc(const float *__restrict__ X, const float *__restrict__ Y,
                                       int m0, int n0, float (&acc)[4][4]) {
#pragma unroll 4
    for (int k = 0; k < kC; ++k) {
        const float4 a = *reinterpret_cast<const float4 *>(X + k * LD + m0);
        const float4 b = *reinterpret_cast<const float4 *>(Y + k * LD + n0);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

template <bool FOX>
__global__ void __launch_bounds__(kThreads)
path_scan_f32_kernel(const float *__restrict__ v, const float *__restrict__ qt,
                     const float *__restrict__ kp, const float *__restrict__ dg,
                     const float *__restrict__ c2, const float *__restrict__ pbase,
                     const int *__restrict__ first_blk,
                     float *__restrict__ out, float *__restrict__ lse, int L, int Lp, int nblk,
                     float scale_log2) {
    extern __shared__ __align__(16) float sm[];
    float *XT = sm;          // state, transposed: XT[c][i]
    float *KT = XT + BUF;    // k~_b transposed: KT[c][j]
    float *PT = KT + BUF;    // P_b transposed: PT[c][n] = P_b[n][c]
    float *Vs = PT + BUF;    // V_b[j][c]
    float *Ss = Vs + BUF;    // logits S[i][j] (log2 units)
    float *PsT = Ss + BUF;   // probabilities, transposed: PsT[j][i]
    float *alpha_s = PsT + BUF;
    float *c2k = alpha_s + kC;

    const int tid = threadIdx.x;
    const int ib = blockIdx.x;
    const int bh = blockIdx.y;
    if (ib * kC >= L) return;
    const size_t head = (size_t)bh;
    const int ty = tid / 16, tx = tid % 16, m0 = ty * 4, n0 = tx * 4;
    const int row = tid >> 2, part = tid & 3;  // softmax: 4 threads per row
    float m_run = -INFINITY, l_run = 0.f;
    // gate sums relative to the base of their pair of blocks; per key block the row's
    // offset against pair b / 2 is (base_own - base) in fp32-pair arithmetic + rel_row
    const float rel_row = FOX ? c2[head * Lp + ib * kC + row] : 0.f;
    const int npair = nblk >> 1;
    const float2 base_own = FOX ? *reinterpret_cast<const float2 *>(pbase + (head * npair + (ib >> 1)) * 2)
                                : make_float2(0.f, 0.f);

    for (int e = tid; e < kC * kD; e += kThreads) {
        const int i = e / kD, c = e % kD;
        XT[c * LD + i] = qt[(head * Lp + (size_t)ib * kC + i) * kD + c];
    }
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    // PaTH-FoX stops above the blocks whose keys all weigh below e^-40 (see fox_exit.cu)
    const int b_last = FOX ? first_blk[head * nblk + ib] : 0;
    for (int b = ib; b >= b_last; --b) {
        __syncthreads();
        for (int e = tid; e < kC * kD; e += kThreads) {
            const int j = e / kD, c = e % kD;
            const int t = b * kC + j;
            Vs[j * LD + c] = (t < L) ? v[(head * L + t) * kD + c] : 0.f;
            if (b < ib) {
                const float *blk = kp + ((head * nblk + b) * 2 * kC) * kD;
                KT[c * LD + j] = blk[j * kD + c];
                PT[c * LD + j] = blk[(kC + j) * kD + c];
            } else {
                Ss[j * LD + c] = dg[((head * nblk + b) * kC + j) * kC + c];
            }
        }
        if (FOX && b < ib && tid < kC) c2k[tid] = c2[head * Lp + b * kC + tid];
        float c2_row = 0.f;
        if (FOX && b < ib) {
            const float2 bb = *reinterpret_cast<const float2 *>(pbase + (head * npair + (b >> 1)) * 2);
            c2_row = ((base_own.x - bb.x) + (base_own.y - bb.y)) + rel_row;
        }
        __syncthreads();
        if (b < ib) {
            float s[4][4], xn[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = xn[i][j] = 0.f;
            mm_acc(XT, KT, m0, n0, s);
            mm_acc(XT, PT, m0, n0, xn);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4 *>(Ss + (m0 + i) * LD + n0) =
                    make_float4(s[i][0] * scale_log2, s[i][1] * scale_log2, s[i][2] * scale_log2,
                                s[i][3] * scale_log2);
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) XT[(n0 + j) * LD + m0 + i] = xn[i][j];
        }
        __syncthreads();
        // ---- online softmax, 4 threads per row, 16 columns each
        {
            float x[16];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                x[j] = Ss[row * LD + part * 16 + j];
                if (FOX && b < ib) x[j] += c2_row - c2k[part * 16 + j];
                mx = fmaxf(mx, x[j]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float p = exp2f(x[j] - m_use);
                sum += p;
                PsT[(part * 16 + j) * LD + row] = p;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            l_run = l_run * alpha + sum;
            m_run = m_new;
            if (part == 0) alpha_s[row] = alpha;
        }
        __syncthreads();
        {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = alpha_s[m0 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] *= a[i];
            mm_acc(PsT, Vs, m0, n0, acc);
        }
    }
    __syncthreads();
    if (part == 0) alpha_s[row] = (l_run > 0.f) ? 1.f / l_run : 0.f;
    if (lse != nullptr && part == 0 && ib * kC + row < L)
        lse[head * L + ib * kC + row] = (m_run + log2f(l_run)) * 0.69314718055994531f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = ib * kC + m0 + i;
        if (t < L) {
            const float inv = alpha_s[m0 + i];
            *reinterpret_cast<float4 *>(out + (head * L + t) * kD + n0) =
                make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
        }
    }
}

}  // namespace

cudaError_t launch_scan_f32(const void *v, void *out, float *lse, bool fox, int BH, int L,
                            float scale, void *ws, cudaStream_t stream) {
    const FwdLayout lay = fwd_layout(1, BH, L, 4, fox);
    char *basep = static_cast<char *>(ws);
    const size_t smem = (size_t)(6 * BUF + 2 * kC) * sizeof(float);
    auto kern = fox ? path_scan_f32_kernel<true> : path_scan_f32_kernel<false>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((L + kC - 1) / kC, BH);
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const float *>(v), reinterpret_cast<const float *>(basep + lay.off_qt),
        reinterpret_cast<const float *>(basep + lay.off_kp),
        reinterpret_cast<const float *>(basep + lay.off_dg),
        fox ? reinterpret_cast<const float *>(basep + lay.off_c2) : nullptr,
        fox ? reinterpret_cast<const float *>(basep + lay.off_pbase) : nullptr,
        fox ? reinterpret_cast<const int *>(basep + lay.off_fb) : nullptr,
        static_cast<float *>(out), lse, L, lay.Lp, lay.nblk, scale * kLog2e);
    return cudaGetLastError();
}

}  // namespace path
