// Merge of partial attention results over disjoint key ranges.
//
// Each part s holds, per row, an output O_s normalised over its own keys and
// LSE_s = m_s + ln(l_s).  Folding the parts with the two-block merge of
// "FlashAttention: IO-Aware Tiling, Online Softmax Mathematics, ...", section
// "Online Softmax Mathematics" (m = max(m1, m2), l = e^(m1-m) l1 + e^(m2-m) l2,
// O = (l1 e^(m1-m) / l) O1 + (l2 e^(m2-m) / l) O2), taken over all parts at once,
// gives
//     LSE = M + ln(sum_s e^(LSE_s - M)),   M = max_s LSE_s,
//     O   = sum_s e^(LSE_s - LSE) O_s.
// A part with LSE_s = -inf (no admitted key) has weight 0.  A row with no key
// in any part gets O = 0, LSE = -inf.
//
// Memory-bound: one warp per row, lane s holds LSE_s (S <= 32 parts), each
// lane owns d/32 consecutive output columns, read as one 16- or 8-byte vector
// per part (a warp reads a 256- or 512-byte contiguous row), written as bf16.
// The O vectors of up to 8 parts are loaded together, the first 8 alongside
// the LSE load, so a row costs about one memory latency instead of two.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "fa_internal.h"

namespace {

constexpr int kWarpsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
fa_combine_kernel(const float *__restrict__ o_parts, const float *__restrict__ lse_parts, int S, int64_t rows,
                  __nv_bfloat16 *__restrict__ o, float *__restrict__ lse)
{
    constexpr int PER = D / 32;  // output columns per lane
    constexpr int kBatch = 8;    // parts whose O vectors are in flight together
    using Vec = typename std::conditional<PER == 4, float4, float2>::type;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp0; r < rows; r += n_warps) {
        // the O vectors of the first parts do not depend on the weights: their
        // loads go out together with the LSE load, before the reductions
        const float ls = lane < S ? lse_parts[lane * rows + r] : -INFINITY;
        Vec x[kBatch];
#pragma unroll
        for (int s = 0; s < kBatch; ++s)
            if (s < S) x[s] = *reinterpret_cast<const Vec *>(o_parts + (static_cast<int64_t>(s) * rows + r) * D + lane * PER);
        float m = ls;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float w = (m == -INFINITY) ? 0.f : expf(ls - m);
        float z = w;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        const float inv_z = z > 0.f ? 1.f / z : 0.f;
        float acc[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = 0.f;
        for (int s0 = 0; s0 < S; s0 += kBatch) {
            if (s0 > 0) {
#pragma unroll
                for (int s = 0; s < kBatch; ++s)
                    if (s0 + s < S)
                        x[s] = *reinterpret_cast<const Vec *>(o_parts + (static_cast<int64_t>(s0 + s) * rows + r) * D +
                                                              lane * PER);
            }
#pragma unroll
            for (int s = 0; s < kBatch; ++s) {
                const float ws = __shfl_sync(0xffffffffu, w, (s0 + s) & 31) * inv_z;
                if (s0 + s < S) {
                    if constexpr (PER == 4) {
                        acc[0] = fmaf(ws, x[s].x, acc[0]);
                        acc[1] = fmaf(ws, x[s].y, acc[1]);
                        acc[2] = fmaf(ws, x[s].z, acc[2]);
                        acc[3] = fmaf(ws, x[s].w, acc[3]);
                    } else {
                        acc[0] = fmaf(ws, x[s].x, acc[0]);
                        acc[1] = fmaf(ws, x[s].y, acc[1]);
                    }
                }
            }
        }
        __nv_bfloat16 *dst = o + r * D + lane * PER;
        if constexpr (PER == 4) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0], acc[1]);
            const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2], acc[3]);
            uint2 v;
            v.x = *reinterpret_cast<const uint32_t *>(&a);
            v.y = *reinterpret_cast<const uint32_t *>(&b);
            *reinterpret_cast<uint2 *>(dst) = v;
        } else {
            const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0], acc[1]);
            *reinterpret_cast<__nv_bfloat162 *>(dst) = a;
        }
        if (lane == 0) lse[r] = z > 0.f ? m + logf(z) : -INFINITY;
    }
}

}  // namespace

cudaError_t fa_launch_combine(const float *o_parts, const float *lse_parts, int n_parts, int64_t rows, int d,
                              void *o, float *lse, int sm_count, cudaStream_t stream)
{
    const int64_t want = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(sm_count) * 16;  // grid-stride beyond 16 blocks per SM
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (d == 64)
        fa_combine_kernel<64><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
            o_parts, lse_parts, n_parts, rows, static_cast<__nv_bfloat16 *>(o), lse);
    else
        fa_combine_kernel<128><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
            o_parts, lse_parts, n_parts, rows, static_cast<__nv_bfloat16 *>(o), lse);
    return cudaGetLastError();
}
