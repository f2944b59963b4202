// Test-only check of the tcgen05 operand layouts the attention kernel relies on.
//
// One CTA of 128 threads:
//   1. Q, K, V (128 x D bf16, row-major in global memory) are written into
//      shared memory in the 128-byte-swizzled layout a TMA tile load with
//      128-byte swizzle produces: D/64 column blocks of [128 rows][128 bytes],
//      16-byte chunk c of row r stored at chunk position c ^ (r % 8).
//   2. S = Q K^T: tcgen05.mma (A and B from shared memory, both K-major),
//      accumulated in TMEM columns [0, 128); every thread reads its row back.
//   3. P = bf16(S) is written over TMEM columns [0, 64) (two bf16 per column)
//      and O = P V is computed with A from TMEM and V as an MN-major B operand.
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

using namespace sm100;

template <int D>
__global__ void __launch_bounds__(128, 1)
tc_selftest_kernel(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *s_out, float *o_out,
                   int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int TILE = 128 * D * 2;
    uint8_t *sQ = smem, *sK = smem + TILE, *sV = smem + 2 * TILE;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 3 * TILE);
    uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(smem + 3 * TILE + 16);
    const int tid = threadIdx.x, warp = tid / 32;

    // 1. swizzled tiles
    for (int idx = tid; idx < 128 * (D / 8); idx += 128) {
        const int r = idx / (D / 8), c = idx % (D / 8);  // 16-byte chunk c of row r
        const int blk = c / 8, cc = c % 8;
        const uint32_t off = blk * (128 * 128) + r * 128 + ((cc ^ (r % 8)) * 16);
        const uint4 *src_q = reinterpret_cast<const uint4 *>(q + r * D + c * 8);
        const uint4 *src_k = reinterpret_cast<const uint4 *>(k + r * D + c * 8);
        const uint4 *src_v = reinterpret_cast<const uint4 *>(v + r * D + c * 8);
        *reinterpret_cast<uint4 *>(sQ + off) = *src_q;
        *reinterpret_cast<uint4 *>(sK + off) = *src_k;
        *reinterpret_cast<uint4 *>(sV + off) = *src_v;
    }
    fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_base_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_base_slot;
    const uint32_t tS = tbase, tO = tbase + 256;

    // 2. S = Q K^T
    if (tid == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, false);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            const uint64_t da = smem_desc_sw128(smem_u32(sQ) + koff, 16, 1024);
            const uint64_t db = smem_desc_sw128(smem_u32(sK) + koff, 16, 1024);
            mma_ss_lohi(tS, static_cast<uint32_t>(da), static_cast<uint32_t>(da >> 32), static_cast<uint32_t>(db),
                        static_cast<uint32_t>(db >> 32), idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(bar));
    }
    __syncwarp();
    bool ok = mbar_wait(smem_u32(bar), 0, 2000000000ull);
    tc_fence_after();
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int row = tid;
    float srow[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tS + lane_off + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) srow[c * 32 + i] = __uint_as_float(r[i]);
    }
    for (int i = 0; i < 128; ++i) s_out[row * 128 + i] = srow[i];

    // 3. P = bf16(S) into TMEM columns [0, 64), then O = P V
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(srow[c * 32 + 2 * i], srow[c * 32 + 2 * i + 1]);
        tmem_st16(tS + lane_off + c * 16, p);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint64_t dv = smem_desc_sw128(smem_u32(sV) + kk * 16 * 128, 128 * 128, 1024);
            mma_ts_lohi(tO, tS + kk * 8, static_cast<uint32_t>(dv), static_cast<uint32_t>(dv >> 32), idO,
                        kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(bar));
    }
    __syncwarp();
    ok = mbar_wait(smem_u32(bar), 1, 2000000000ull) && ok;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + lane_off + c * 32, r);
        tmem_wait_ld();
        for (int i = 0; i < 32; ++i) o_out[row * D + c * 32 + i] = __uint_as_float(r[i]);
    }
    if (!ok) atomicExch(status, 6);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

extern "C" int tc_selftest(const void *q, const void *k, const void *v, float *s_out, float *o_out, int *status,
                           int d)
{
    const int smem = 3 * 128 * d * 2 + 1024 + 64;
    cudaError_t e;
    if (d == 64) {
        e = cudaFuncSetAttribute(tc_selftest_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            tc_selftest_kernel<64><<<1, 128, smem>>>(static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                                                     static_cast<const uint16_t *>(v), s_out, o_out, status);
    } else if (d == 128) {
        e = cudaFuncSetAttribute(tc_selftest_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            tc_selftest_kernel<128><<<1, 128, smem>>>(static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                                                      static_cast<const uint16_t *>(v), s_out, o_out, status);
    } else {
        return -1;
    }
    if (e != cudaSuccess) return static_cast<int>(e);
    e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

// A bounded wait that must run out: an mbarrier expecting one arrival that
// never comes.  The waiting thread gives up after `limit_ns` and records 1 in
// status[0]; a wait for the phase before the current one (parity 1 on a fresh
// barrier) must succeed at once and records 1 in status[1].
__global__ void wait_timeout_kernel(int *status, unsigned long long limit_ns, unsigned long long *elapsed_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        status[1] = mbar_wait(smem_u32(&bar), 1, limit_ns) ? 1 : 0;
        const uint64_t t0 = globaltimer_ns();
        const bool ok = mbar_wait(smem_u32(&bar), 0, limit_ns);
        *elapsed_ns = globaltimer_ns() - t0;
        status[0] = ok ? 0 : 1;
    }
}

extern "C" int wait_timeout_selftest(int *status, unsigned long long limit_ns, unsigned long long *elapsed_ns)
{
    wait_timeout_kernel<<<1, 32>>>(status, limit_ns, elapsed_ns);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

// tcgen05.ld with a max reduction: 128 threads store rows of 128 fp32 values
// (in[128][128]) into tensor memory columns [0, 128), load them back in four
// 32-column pieces with tmem_ld32_max, and write the values (out_vals) and
// each piece's reported maximum (out_max[128][4]).
__global__ void __launch_bounds__(128, 1) ld_max_kernel(const float *in, float *out_vals, float *out_max)
{
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid / 32;
    if (warp == 0) {
        tmem_alloc(smem_u32(&slot), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t = slot + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(in[tid * 128 + c * 32 + i]);
        tmem_st32(t + c * 32, r);
    }
    tmem_wait_st();
    for (int c = 0; c < 4; ++c) {
        float v[32], m;
        tmem_ld32_max(t + c * 32, v, m);
        tmem_wait_ld();
        for (int i = 0; i < 32; ++i) out_vals[tid * 128 + c * 32 + i] = v[i];
        out_max[tid * 4 + c] = m;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(slot, 128);
}

extern "C" int ld_max_selftest(const float *in, float *out_vals, float *out_max)
{
    ld_max_kernel<<<1, 128>>>(in, out_vals, out_max);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}
