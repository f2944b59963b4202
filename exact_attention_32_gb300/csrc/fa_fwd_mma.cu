// Exact attention forward with warp-level tensor-core MMAs (mma.sync m16n8k16).
//
// One CTA owns one 128-row query tile of one (batch, head) slice and streams
// the admitted 64-row K/V tiles through shared memory (cp.async, two stages).
// Per K/V tile it follows the per-tile steps of "6.1 FlashAttention V1 in
// detail", section 5.1 (scores, tile row max, new running max, correction
// factor and exp-sum, output update), but keeps the unnormalised numerator u
// and divides by l once at the end ("FlashAttention: IO-Aware Tiling, ...",
// section "FlashAttention-2": rescaling optimisation; the (m, l, u) form of
// "FlashAttention: optimize data movement before counting FLOPs", section 02).
// The query-outer loop order with the grid over query tiles is the
// FlashAttention-2 inversion described on the same llms.blog page.
//
// Exponentials are base 2 with scale*log2(e) folded into one FMA per score;
// the running max is kept in unscaled dot-product units (scale > 0).
// Scores past N and, when causal, keys after the query are set to -inf before
// the max, so they add nothing to l or u ("6.1 ...", section 8.3, the K/V
// out-of-range mask).
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"

namespace {

constexpr int kBr = 128;  // query rows per CTA, 16 per warp
constexpr int kBc = 64;   // keys per K/V tile
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk c of row r in a row-major tile with CH chunks
// per row; the low three chunk bits are XORed with the row so that the eight
// rows an ldmatrix phase touches fall into distinct banks.
template <int CH>
__device__ __forceinline__ uint32_t swz(int r, int c)
{
    return static_cast<uint32_t>(r * CH + ((c & ~7) | ((c ^ r) & 7))) * 16u;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_mma_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                  const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ o,
                  float *__restrict__ lse, int N, int64_t BH, int n_qtiles, float scale,
                  float scale_log2)
{
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sQ = smem_addr(smem);
    const uint32_t sK = sQ + kBr * D * 2;
    const uint32_t sV = sK + 2 * kBc * D * 2;

    // heaviest (last) query tiles first so causal work finishes evenly
    const int64_t unit = blockIdx.x;
    const int qt = n_qtiles - 1 - static_cast<int>(unit / BH);
    const int64_t bh = unit % BH;
    const int64_t base = bh * static_cast<int64_t>(N) * D;
    const __nv_bfloat16 *qh = q + base, *kh = k + base, *vh = v + base;
    const int q0 = qt * kBr;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int row_w = warp * 16;

    for (int c = tid; c < kBr * CH; c += kThreads) {
        const int r = c / CH, ch = c % CH, gr = q0 + r;
        const bool ok = gr < N;
        cp_async16(sQ + swz<CH>(r, ch), qh + static_cast<int64_t>(ok ? gr : 0) * D + ch * 8, ok);
    }
    const int kv_end = CAUSAL ? min(N, q0 + kBr) : N;
    const int n_kv = (kv_end + kBc - 1) / kBc;
    auto load_kv = [&](int j, int stage) {
        const uint32_t dk = sK + stage * kBc * D * 2, dv = sV + stage * kBc * D * 2;
        for (int c = tid; c < kBc * CH; c += kThreads) {
            const int r = c / CH, ch = c % CH, gr = j * kBc + r;
            const bool ok = gr < N;
            const int64_t off = static_cast<int64_t>(ok ? gr : 0) * D + ch * 8;
            cp_async16(dk + swz<CH>(r, ch), kh + off, ok);
            cp_async16(dv + swz<CH>(r, ch), vh + off, ok);
        }
    };
    load_kv(0, 0);
    cp_commit();

    float m_r[2] = {-INFINITY, -INFINITY};  // running max, unscaled units
    float l_r[2] = {0.f, 0.f};              // this thread's share of the exp-sum (fp32 terms; LSE)
    float lq_r[2] = {0.f, 0.f};             // the same over the bf16-rounded terms (normalises O)
    float acc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    for (int j = 0; j < n_kv; ++j) {
        if (j + 1 < n_kv) load_kv(j + 1, (j + 1) & 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const uint32_t kS = sK + (j & 1) * kBc * D * 2, vS = sV + (j & 1) * kBc * D * 2;

        // S = Q K^T for this warp's 16 rows x 64 keys
        float s[kBc / 8][4];
#pragma unroll
        for (int i = 0; i < kBc / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sQ + swz<CH>(row_w + (lane & 7) + ((lane >> 3) & 1) * 8, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
            for (int nn = 0; nn < kBc / 16; ++nn) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kS + swz<CH>(nn * 16 + (lane & 7) + (lane >> 4) * 8, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
                mma16816(s[2 * nn], a0, a1, a2, a3, b0, b1);
                mma16816(s[2 * nn + 1], a0, a1, a2, a3, b2, b3);
            }
        }

        // masks: keys past N, and causal keys after the query row
        const int k0 = j * kBc;
        const bool need_mask = (k0 + kBc > N) || (CAUSAL && k0 + kBc - 1 > q0 + row_w);
        if (need_mask) {
#pragma unroll
            for (int n = 0; n < kBc / 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = k0 + n * 8 + 2 * t + (e & 1);
                    const int row = q0 + row_w + g + (e >> 1) * 8;
                    if (key >= N || (CAUSAL && key > row)) s[n][e] = -INFINITY;
                }
        }

        // online softmax: new running max, correction factor alpha, exp-sum
        float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
        for (int n = 0; n < kBc / 8; ++n) {
            mx[0] = fmaxf(mx[0], fmaxf(s[n][0], s[n][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[n][2], s[n][3]));
        }
        float ms[2], alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            // a row with every key so far masked keeps m = -inf; use 0 as its reference
            const float ref = (mx[r] == -INFINITY) ? 0.f : mx[r];
            alpha[r] = ex2((m_r[r] - ref) * scale_log2);
            ms[r] = ref * scale_log2;
            m_r[r] = mx[r];
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < kBc / 8; ++n) {
            s[n][0] = ex2(fmaf(s[n][0], scale_log2, -ms[0]));
            s[n][1] = ex2(fmaf(s[n][1], scale_log2, -ms[0]));
            s[n][2] = ex2(fmaf(s[n][2], scale_log2, -ms[1]));
            s[n][3] = ex2(fmaf(s[n][3], scale_log2, -ms[1]));
            rs[0] += s[n][0] + s[n][1];
            rs[1] += s[n][2] + s[n][3];
        }
        l_r[0] = l_r[0] * alpha[0] + rs[0];
        l_r[1] = l_r[1] * alpha[1] + rs[1];
        lq_r[0] *= alpha[0];
        lq_r[1] *= alpha[1];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            acc[i][0] *= alpha[0];
            acc[i][1] *= alpha[0];
            acc[i][2] *= alpha[1];
            acc[i][3] *= alpha[1];
        }

        // u += P V, with P rounded to bf16; the S accumulator layout of two
        // adjacent 8-key blocks is the A-operand layout of one 16-key step
#pragma unroll
        for (int kk = 0; kk < kBc / 16; ++kk) {
            const uint32_t a0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            const uint32_t a1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            const uint32_t a2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            const uint32_t a3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            lq_r[0] += bf16_lo(a0) + bf16_hi(a0) + bf16_lo(a2) + bf16_hi(a2);
            lq_r[1] += bf16_lo(a1) + bf16_hi(a1) + bf16_lo(a3) + bf16_hi(a3);
#pragma unroll
            for (int nd = 0; nd < D / 16; ++nd) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vS + swz<CH>(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, nd * 2 + (lane >> 4)), b0, b1, b2, b3);
                mma16816(acc[2 * nd], a0, a1, a2, a3, b0, b1);
                mma16816(acc[2 * nd + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();  // this stage is refilled two iterations later
    }

    // epilogue: O = u / l (bf16), LSE = m * scale + ln(l).  u was accumulated
    // from bf16-rounded P, so it is divided by the sum of those rounded terms.
    float inv[2], lrow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float l = l_r[r], lq = lq_r[r];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        lq += __shfl_xor_sync(0xffffffffu, lq, 1);
        lq += __shfl_xor_sync(0xffffffffu, lq, 2);
        lrow[r] = l;
        inv[r] = 1.f / lq;
    }
    const int gr0 = q0 + row_w + g, gr1 = gr0 + 8;
    __nv_bfloat16 *oh = o + base;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + 2 * t;
        if (gr0 < N)
            *reinterpret_cast<uint32_t *>(oh + static_cast<int64_t>(gr0) * D + col) =
                pack_bf16(acc[i][0] * inv[0], acc[i][1] * inv[0]);
        if (gr1 < N)
            *reinterpret_cast<uint32_t *>(oh + static_cast<int64_t>(gr1) * D + col) =
                pack_bf16(acc[i][2] * inv[1], acc[i][3] * inv[1]);
    }
    if (t == 0) {
        float *lh = lse + bh * N;
        if (gr0 < N) lh[gr0] = m_r[0] * scale + logf(lrow[0]);
        if (gr1 < N) lh[gr1] = m_r[1] * scale + logf(lrow[1]);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch(const FaProblem &p, cudaStream_t stream)
{
    const int smem = (kBr + 4 * kBc) * D * 2;
    auto kern = fa_fwd_mma_kernel<D, CAUSAL>;
    cudaError_t e = set_max_dynamic_smem<fa_fwd_mma_kernel<D, CAUSAL>>(smem);
    if (e != cudaSuccess) return e;
    const int n_qtiles = static_cast<int>((p.N + kBr - 1) / kBr);
    const int64_t BH = p.B * p.H;
    const int64_t blocks = BH * n_qtiles;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    kern<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
        static_cast<const __nv_bfloat16 *>(p.v), static_cast<__nv_bfloat16 *>(p.o), p.lse,
        static_cast<int>(p.N), BH, n_qtiles, p.scale, scale_log2);
    return cudaGetLastError();
}

}  // namespace

cudaError_t fa_launch_mma(const FaProblem &p, cudaStream_t stream)
{
    if (p.d == 64) return p.causal ? launch<64, true>(p, stream) : launch<64, false>(p, stream);
    return p.causal ? launch<128, true>(p, stream) : launch<128, false>(p, stream);
}
