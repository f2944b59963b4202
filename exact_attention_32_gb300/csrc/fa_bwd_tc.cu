// Exact attention backward for GB300 (sm_103a): TMA + tcgen05 + TMEM.
//
// Given Q, K, V, the forward outputs O and LSE, and dO, computes the gradients
// of sum(O * dO) ("6.1 FlashAttention V1 in detail", section 6.1:
// dV = P^T dO, dP = dO V^T, D = rowsum(dO * O) = rowsum(dP * P),
// dS = P * (dP - D); "FlashAttention: IO-Aware Tiling, ...", section "Backward
// Pass Recomputation": dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d), the
// 1/sqrt(d) being the forward's scale).  P is recomputed from the saved LSE,
// P_ij = exp(scale * q_i . k_j - LSE_i) (section 6.2), never stored.
//
// Three launches:
//   pre   (memory-bound)  D_i = rowsum(dO_i * O_i); LSE_i * log2(e) into a
//                         padded vector (+inf on padding rows, so their P is 0);
//                         the fp32 dQ accumulator zeroed.
//   main  (tcgen05)       one CTA per 128-key block of one (b, h), looping over
//                         the 128-row query blocks (causal: from the diagonal);
//                         dK, dV accumulate in tensor memory, dQ block partials
//                         are added into the fp32 accumulator.
//   post  (memory-bound)  dQ = bf16(scale * accumulator), from the blocked
//                         accumulator layout below back to [B, H, N, d].
//
// Main kernel, per query block (S^T etc. are key-major: TMEM lane = key):
//   S^T  = K Q^T          SS MMA -> TMEM A
//   dP^T = V dO^T         SS MMA -> TMEM B
//   P^T  = exp2(S^T scale log2e - LSE log2e)      softmax warps, bf16 back into A
//   dV  += P^T dO         TS MMA (A = P^T from TMEM, B = dO MN-major) -> TMEM C
//   dS^T = P^T (dP^T - D)                         softmax warps, bf16 into B and
//                                                 into shared memory (for dQ)
//   dK  += dS^T Q         TS MMA -> TMEM D
//   dQ   = dS K           SS MMA (A = dS MN-major, B = K MN-major) -> TMEM A,
//                         read into registers (TMEM A is released at once) and
//                         staged in the Q/dO stage that block no longer needs;
//                         the load warp adds the staged block to the
//                         accumulator with one bulk reduce-add, waits until
//                         it has been read out and refills the stage
// The dQ accumulator is blocked: one 128 x d fp32 block per (b, h, query
// block), holding the block's 8 warp slices (warpgroup, 32-row group) one after
// the other, each 32 rows x d/2 columns, row-major, with the 16-byte chunk c of
// row l stored at chunk position c ^ (l mod d/8).  A warp's slice is then one
// contiguous range of global memory, and its staging writes in shared memory
// are free of bank conflicts.
// Roles (320 threads): warps 0-3 and 4-7 are two warpgroups that take query
// columns 0-63 and 64-127 of each block (and d-columns halves of dQ, dK, dV);
// warp 8 loads K, V once and Q, dO, LSE, D per block (two stages); warp 9
// issues the MMAs and owns the tensor memory.
//
// Every mbarrier wait is bounded; a wait that gives up sets FA_ERR_TIMEOUT in
// this file's status word and the CTA winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "sm100_ptx.cuh"

using namespace sm100;

namespace {

constexpr int kBlock = 128;  // keys per CTA block and queries per query block
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint64_t kCleanupLimitNs = 20000000ull;

__device__ int g_bwd_status;

__device__ __forceinline__ void report(int code) { atomicExch(&g_bwd_status, code); }

template <int D>
struct BCfg {
    static constexpr int kTile = kBlock * D * 2;  // one 128-row bf16 tile
    static constexpr int kAtoms = D / 64;
    static constexpr int kK = 0;
    static constexpr int kV = kTile;
    static constexpr int kStage0 = 2 * kTile;       // stage s: Q at kStage0 + s*kStageBytes, dO after it
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kDS = kStage0 + 2 * kStageBytes;  // dS, 128 keys x 128 queries bf16, MN-major
    static constexpr int kVec = kDS + kBlock * kBlock * 2;  // per stage: LSE*log2e (512 B), D (512 B)
    static constexpr int kBar = kVec + 2 * 1024;
    static constexpr int kNumBars = 13;
    static constexpr int kSmemBytes = kBar + kNumBars * 8 + 16;
};

enum { KV_FULL = 0, Q_FULL = 1, DQ_STAGED = 3, S_FULL = 5, DP_FULL = 6, P_READY = 7, DS_READY = 8, DQ_FULL = 9,
       DQ_CONSUMED = 10, DONE = 11, MMA_DONE = 12 };

__device__ __forceinline__ uint32_t lo32(uint64_t x) { return static_cast<uint32_t>(x); }
__device__ __forceinline__ uint32_t hi32(uint64_t x) { return static_cast<uint32_t>(x >> 32); }

// TMEM column of the packed (bf16 pairs) 16-query K-step kk: warpgroup w packs
// its 64 queries into columns [64 w, 64 w + 32).
__device__ __forceinline__ uint32_t packed_col(int kk) { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const float *__restrict__ lse2, const float *__restrict__ dvec, float *__restrict__ dq_acc,
                 __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int N, int BH, int n_blocks,
                 int n_pad, int heads_per_group, float scale, float scale_log2)
{
    using C = BCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((sb & 1023u) != 0) {  // the swizzled tiles need a 1024-byte-aligned base
        if (tid == 0) report(FA_ERR_LAUNCH);
        return;
    }
    const uint32_t bar0 = sb + C::kBar;
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kBar + C::kNumBars * 8);

    // CTA = key block kb of slice bh.  The (b, h) slices go in groups of
    // heads_per_group, so that the CTAs resident at one time share a few
    // slices' Q, dO and dQ accumulator blocks in L2; inside a group, key-block
    // major, so causal CTAs with many query blocks (small kb) start first.
    const int per_group = heads_per_group * n_blocks;
    const int grp = blockIdx.x / per_group, rem = blockIdx.x - grp * per_group;
    const int gsize = min(heads_per_group, BH - grp * heads_per_group);
    const int kb = rem / gsize, bh = grp * heads_per_group + rem % gsize;
    const int k0 = kb * kBlock;
    const int qb0 = CAUSAL ? kb : 0;
    const int nq = n_blocks - qb0;
    const bool run = *reinterpret_cast<volatile int *>(&g_bwd_status) == 0;

    if (tid == 0) {
        mbar_init(BAR(KV_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(Q_FULL + s), 1);
            mbar_init(BAR(DQ_STAGED + s), 8);  // the softmax warps, once their dQ slices are staged
        }
        mbar_init(BAR(S_FULL), 1);
        mbar_init(BAR(DP_FULL), 1);
        mbar_init(BAR(P_READY), 8);
        mbar_init(BAR(DS_READY), 8);
        mbar_init(BAR(DQ_FULL), 1);
        mbar_init(BAR(DQ_CONSUMED), 8);
        mbar_init(BAR(DONE), 1);
        mbar_init(BAR(MMA_DONE), 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tA = tmem, tB = tmem + 128, tC = tmem + 256, tD = tmem + 384;

    if (!run) {
        // nothing to do
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(BAR(KV_FULL), 2 * C::kTile);
            for (int a = 0; a < C::kAtoms; ++a) {
                tma_load_3d(sb + C::kK + a * 16384, &tm_k, BAR(KV_FULL), a * 64, k0, bh);
                tma_load_3d(sb + C::kV + a * 16384, &tm_v, BAR(KV_FULL), a * 64, k0, bh);
            }
            // add the dQ block that iteration j staged in stage j & 1 to the accumulator
            auto flush = [&](int j) -> bool {
                if (!mbar_wait(BAR(DQ_STAGED + (j & 1)), (j >> 1) & 1, kWaitLimitNs)) return false;
                bulk_reduce_add_f32(dq_acc + (static_cast<int64_t>(bh) * n_blocks + qb0 + j) * (kBlock * D),
                                    sb + C::kStage0 + (j & 1) * C::kStageBytes, kBlock * D * 4);
                bulk_commit();
                return true;
            };
            bool ok = true;
            int issued = 0;
            for (int i = 0; i < nq; ++i) {
                const int st = i & 1;
                if (i >= 2) {  // the stage is free once the block staged in it two iterations ago is read out
                    if (!(ok = flush(i - 2))) break;
                    bulk_wait_read0();
                }
                const int q0 = (qb0 + i) * kBlock;
                const uint32_t sq = sb + C::kStage0 + st * C::kStageBytes, sdo = sq + C::kTile;
                mbar_arrive_expect_tx(BAR(Q_FULL + st), 2 * C::kTile + 1024);
                for (int a = 0; a < C::kAtoms; ++a) {
                    tma_load_3d(sq + a * 16384, &tm_q, BAR(Q_FULL + st), a * 64, q0, bh);
                    tma_load_3d(sdo + a * 16384, &tm_do, BAR(Q_FULL + st), a * 64, q0, bh);
                }
                const int64_t vo = static_cast<int64_t>(bh) * n_pad + q0;
                bulk_load(sb + C::kVec + st * 1024, lse2 + vo, 512, BAR(Q_FULL + st));
                bulk_load(sb + C::kVec + st * 1024 + 512, dvec + vo, 512, BAR(Q_FULL + st));
                ++issued;
            }
            for (int j = nq >= 2 ? nq - 2 : 0; j < nq && ok; ++j) ok = flush(j);
            bulk_wait0();  // the accumulator additions complete before the CTA ends
            if (!ok) report(FA_ERR_TIMEOUT);
            const uint64_t lim = ok ? kWaitLimitNs : kCleanupLimitNs;
            mbar_wait(BAR(KV_FULL), 0, lim);
            for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i) mbar_wait(BAR(Q_FULL + (i & 1)), (i >> 1) & 1, lim);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBlock, kBlock, false);    // S^T, dP^T: K-major operands
            constexpr uint32_t idAcc = idesc_bf16_f32(kBlock, D, true);       // dV, dK: A in TMEM, B MN-major
            constexpr uint32_t idQ = idesc_bf16_f32(kBlock, D, true, true);   // dQ: A and B MN-major
            constexpr uint32_t kStage16 = C::kStageBytes >> 4, kTile16 = C::kTile >> 4;
            const uint64_t d_k_kmaj = smem_desc_sw128(sb + C::kK, 16, 1024);
            const uint64_t d_v_kmaj = smem_desc_sw128(sb + C::kV, 16, 1024);
            const uint64_t d_k_mn = smem_desc_sw128(sb + C::kK, 16384, 1024);
            const uint64_t d_ds_mn = smem_desc_sw128(sb + C::kDS, 16384, 1024);
            const uint64_t d_q_kmaj = smem_desc_sw128(sb + C::kStage0, 16, 1024);
            const uint64_t d_q_mn = smem_desc_sw128(sb + C::kStage0, 16384, 1024);
            bool ok = mbar_wait(BAR(KV_FULL), 0, kWaitLimitNs);
            for (int i = 0; i < nq && ok; ++i) {
                const int st = i & 1;
                if (!(ok = mbar_wait(BAR(Q_FULL + st), (i >> 1) & 1, kWaitLimitNs))) break;
                if (i > 0 && !(ok = mbar_wait(BAR(DQ_CONSUMED), (i - 1) & 1, kWaitLimitNs))) break;
                tc_fence_after();
                const uint32_t q_lo = lo32(d_q_kmaj) + st * kStage16, do_lo = q_lo + kTile16;
                const uint32_t qmn_lo = lo32(d_q_mn) + st * kStage16, domn_lo = qmn_lo + kTile16;
                // S^T = K Q^T and dP^T = V dO^T
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                    mma_ss_lohi(tA, lo32(d_k_kmaj) + koff, hi32(d_k_kmaj), q_lo + koff, hi32(d_q_kmaj), idS,
                                kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR(S_FULL));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                    mma_ss_lohi(tB, lo32(d_v_kmaj) + koff, hi32(d_v_kmaj), do_lo + koff, hi32(d_q_kmaj), idS,
                                kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR(DP_FULL));
                // dV += P^T dO
                if (!(ok = mbar_wait(BAR(P_READY), i & 1, kWaitLimitNs))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBlock / 16; ++kk)
                    mma_ts_lohi(tC, tA + packed_col(kk), domn_lo + kk * 128, hi32(d_q_mn), idAcc,
                                (i > 0 || kk > 0) ? 1u : 0u);
                // dK += dS^T Q, then dQ = dS K
                if (!(ok = mbar_wait(BAR(DS_READY), i & 1, kWaitLimitNs))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBlock / 16; ++kk)
                    mma_ts_lohi(tD, tB + packed_col(kk), qmn_lo + kk * 128, hi32(d_q_mn), idAcc,
                                (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < kBlock / 16; ++kk)
                    mma_ss_lohi(tA, lo32(d_ds_mn) + kk * 128, hi32(d_ds_mn), lo32(d_k_mn) + kk * 128, hi32(d_k_mn),
                                idQ, kk > 0 ? 1u : 0u);
                mma_commit(BAR(DQ_FULL));
            }
            if (ok) mma_commit(BAR(DONE));
            if (!ok) report(FA_ERR_TIMEOUT);
            mma_commit(BAR(MMA_DONE));
            mbar_wait(BAR(MMA_DONE), 0, ok ? kWaitLimitNs : kCleanupLimitNs);
        }
    } else {
        // ------------------------------------------------ softmax-side warpgroups
        const int wg = warp >> 2;  // query columns [64 wg, 64 wg + 64); d columns [wg D/2, (wg + 1) D/2)
        const int r = (warp & 3) * 32 + lane;  // TMEM lane
        const uint32_t loff = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int key = k0 + r;
        bool ok = true;
        for (int i = 0; i < nq && ok; ++i) {
            const int st = i & 1;
            const int q0 = (qb0 + i) * kBlock;
            if (!mbar_wait_warp(BAR(Q_FULL + st), (i >> 1) & 1, kWaitLimitNs) ||
                !mbar_wait_warp(BAR(S_FULL), i & 1, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *lse2_s = reinterpret_cast<const float *>(smem + C::kVec + st * 1024) + wg * 64;
            const float *d_s = lse2_s + kBlock;
            // P^T = exp2(S^T * scale * log2 e - LSE * log2 e); 0 for keys past N and, causal, keys after the query
            float p[64];
            {
                uint32_t a0[32], a1[32];
                tmem_ld32(tA + loff + wg * 64, a0);
                tmem_ld32(tA + loff + wg * 64 + 32, a1);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 l0 = *reinterpret_cast<const float2 *>(lse2_s + j);
                    const float2 l1 = *reinterpret_cast<const float2 *>(lse2_s + 32 + j);
                    const float2 x0 = fma2(make_float2(__uint_as_float(a0[j]), __uint_as_float(a0[j + 1])),
                                           make_float2(scale_log2, scale_log2), make_float2(-l0.x, -l0.y));
                    const float2 x1 = fma2(make_float2(__uint_as_float(a1[j]), __uint_as_float(a1[j + 1])),
                                           make_float2(scale_log2, scale_log2), make_float2(-l1.x, -l1.y));
                    p[j] = ex2(x0.x);
                    p[j + 1] = ex2(x0.y);
                    p[32 + j] = ex2(x1.x);
                    p[32 + j + 1] = ex2(x1.y);
                }
            }
            if (key >= N) {
#pragma unroll
                for (int j = 0; j < 64; ++j) p[j] = 0.f;
            } else if (CAUSAL && i == 0) {
                const int qb = q0 + wg * 64;  // the diagonal block: query qb + j admits key iff key <= qb + j
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (key > qb + j) p[j] = 0.f;
            }
            {
                uint32_t pk[16];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(p[h * 32 + 2 * j], p[h * 32 + 2 * j + 1]);
                    tmem_st16(tA + loff + wg * 64 + h * 16, pk);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(P_READY));

            // dS^T = P^T (dP^T - D)
            if (!mbar_wait_warp(BAR(DP_FULL), i & 1, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dsk[32];
            {
                uint32_t b0[32], b1[32];
                tmem_ld32(tB + loff + wg * 64, b0);
                tmem_ld32(tB + loff + wg * 64 + 32, b1);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 dd0 = *reinterpret_cast<const float2 *>(d_s + j);
                    const float2 dd1 = *reinterpret_cast<const float2 *>(d_s + 32 + j);
                    dsk[j / 2] = pack_bf16x2(p[j] * (__uint_as_float(b0[j]) - dd0.x),
                                             p[j + 1] * (__uint_as_float(b0[j + 1]) - dd0.y));
                    dsk[16 + j / 2] = pack_bf16x2(p[32 + j] * (__uint_as_float(b1[j]) - dd1.x),
                                                  p[32 + j + 1] * (__uint_as_float(b1[j + 1]) - dd1.y));
                }
            }
            {
                uint32_t h0[16], h1[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    h0[j] = dsk[j];
                    h1[j] = dsk[16 + j];
                }
                tmem_st16(tB + loff + wg * 64, h0);
                tmem_st16(tB + loff + wg * 64 + 16, h1);
            }
            // dS^T row (this key) into the MN-major dS tile: column block wg, 16-byte
            // chunk c (queries 8c .. 8c+7) at chunk position c ^ (key row mod 8)
            uint8_t *row_base = smem + C::kDS + wg * 16384 + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(row_base + ((c ^ (r & 7)) * 16)) =
                    make_uint4(dsk[4 * c], dsk[4 * c + 1], dsk[4 * c + 2], dsk[4 * c + 3]);
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(DS_READY));

            // dQ block partial (TMEM lane = query row): into registers, TMEM A released,
            // then staged in this block's Q/dO stage (every MMA that read it has
            // completed by DQ_FULL) for the load warp's bulk reduce
            if (!mbar_wait_warp(BAR(DQ_FULL), i & 1, kWaitLimitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t x0[32], x1[32];
            tmem_ld32(tA + loff + wg * (D / 2), x0);
            if constexpr (D == 128) tmem_ld32(tA + loff + wg * (D / 2) + 32, x1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(DQ_CONSUMED));
            constexpr int kChunks = D / 8;               // 16-byte chunks in a row of the warp slice
            constexpr int kSliceBytes = 32 * (D / 2) * 4;
            const int slot = wg * 4 + (warp & 3);
            const uint32_t stage_off = C::kStage0 + st * C::kStageBytes + slot * kSliceBytes;
            uint8_t *srow = smem + stage_off + lane * (D * 2);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const uint32_t *x = c < 8 ? x0 : x1;
                const int cl = c & 7;
                *reinterpret_cast<uint4 *>(srow + ((c ^ (lane & (kChunks - 1))) * 16)) =
                    make_uint4(x[4 * cl], x[4 * cl + 1], x[4 * cl + 2], x[4 * cl + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(DQ_STAGED + st));
        }
        if (ok) ok = mbar_wait_warp(BAR(DONE), 0, kWaitLimitNs);
        if (!ok) report(FA_ERR_TIMEOUT);
        tc_fence_after();
        // epilogue: dV (TMEM C) and scale * dK (TMEM D), this warpgroup's half of the d
        // columns; every lane takes part in the TMEM reads, only rows < N are stored
        if (ok) {
            const int64_t off = (static_cast<int64_t>(bh) * N + key) * D + wg * (D / 2);
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t tsrc = (which == 0 ? tC : tD) + loff + wg * (D / 2);
                const float mul = which == 0 ? 1.f : scale;
                __nv_bfloat16 *out = (which == 0 ? dv : dk) + off;
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t x[32];
                    tmem_ld32(tsrc + cc * 32, x);
                    tmem_wait_ld();
                    if (key >= N) continue;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v4;
                        v4.x = pack_bf16x2(__uint_as_float(x[8 * q4 + 0]) * mul, __uint_as_float(x[8 * q4 + 1]) * mul);
                        v4.y = pack_bf16x2(__uint_as_float(x[8 * q4 + 2]) * mul, __uint_as_float(x[8 * q4 + 3]) * mul);
                        v4.z = pack_bf16x2(__uint_as_float(x[8 * q4 + 4]) * mul, __uint_as_float(x[8 * q4 + 5]) * mul);
                        v4.w = pack_bf16x2(__uint_as_float(x[8 * q4 + 6]) * mul, __uint_as_float(x[8 * q4 + 7]) * mul);
                        *reinterpret_cast<uint4 *>(out + cc * 32 + 8 * q4) = v4;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// D_i = rowsum(dO_i * O_i) and LSE_i * log2(e) for padded rows (+inf and 0 on
// padding rows); the dQ accumulator rows zeroed.  One warp per padded row.
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                  const float *__restrict__ lse, float *__restrict__ lse2, float *__restrict__ dvec,
                  float *__restrict__ dq_acc, int N, int n_pad, int64_t BH)
{
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t rr = w0; rr < BH * n_pad; rr += nw) {
        const int64_t bh = rr / n_pad;
        const int i = static_cast<int>(rr - bh * n_pad);
        if (i < N) {
            const int64_t row = bh * N + i;
            const __nv_bfloat16 *a = o + row * D + lane * PER, *b = dout + row * D + lane * PER;
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc = fmaf(__bfloat162float(a[e]), __bfloat162float(b[e]), acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) {
                dvec[rr] = acc;
                lse2[rr] = lse[row] * 1.4426950408889634f;
            }
        } else if (lane == 0) {
            dvec[rr] = 0.f;
            lse2[rr] = INFINITY;
        }
        // the accumulator holds B*H*n_pad*D floats: padded row rr clears floats [rr*D, rr*D + D)
        float *z = dq_acc + rr * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) z[e] = 0.f;
    }
}

// dQ = bf16(scale * accumulator), four elements per thread; reads the blocked
// accumulator layout described at the top of this file.
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_post_kernel(const float4 *__restrict__ acc, uint2 *__restrict__ dq, int64_t n4, int N, int n_blocks,
                   float scale)
{
    constexpr int kChunks = D / 8;  // 4-float chunks per half row
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n4;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = t / (D / 4);
        const int c4 = static_cast<int>(t - row * (D / 4));
        const int64_t bh = row / N;
        const int i = static_cast<int>(row - bh * N);
        const int qb = i / kBlock, rr = i % kBlock;
        const int slot = (c4 / kChunks) * 4 + rr / 32, l = rr % 32, c = c4 % kChunks;
        const int64_t src = (bh * n_blocks + qb) * (kBlock * D / 4) + slot * (32 * kChunks) + l * kChunks +
                            (c ^ (l & (kChunks - 1)));
        const float4 x = acc[src];
        uint2 y;
        y.x = pack_bf16x2(x.x * scale, x.y * scale);
        y.y = pack_bf16x2(x.z * scale, x.w * scale);
        dq[t] = y;
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

bool make_map(CUtensorMap *m, const void *base, int64_t BH, int64_t N, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool CAUSAL>
cudaError_t launch_main(const FaBwdProblem &p, float *lse2, float *dvec, float *dq_acc, int n_pad, cudaStream_t s)
{
    using C = BCfg<D>;
    CUtensorMap mq, mk, mv, mdo;
    const int64_t BH = p.B * p.H;
    if (!make_map(&mq, p.q, BH, p.N, D) || !make_map(&mk, p.k, BH, p.N, D) || !make_map(&mv, p.v, BH, p.N, D) ||
        !make_map(&mdo, p.dout, BH, p.N, D))
        return cudaErrorInvalidValue;
    auto kern = fa_bwd_tc_kernel<D, CAUSAL>;
    cudaError_t e = set_max_dynamic_smem<fa_bwd_tc_kernel<D, CAUSAL>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t n_blocks = (p.N + kBlock - 1) / kBlock;
    const int64_t grid = n_blocks * BH;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    // about 256 CTAs per group of slices (at least one slice)
    const int64_t hpg = n_blocks >= 256 ? 1 : (256 / n_blocks < BH ? 256 / n_blocks : BH);
    kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, s>>>(
        mq, mk, mv, mdo, lse2, dvec, dq_acc, static_cast<__nv_bfloat16 *>(p.dk), static_cast<__nv_bfloat16 *>(p.dv),
        static_cast<int>(p.N), static_cast<int>(BH), static_cast<int>(n_blocks), n_pad, static_cast<int>(hpg), p.scale,
        scale_log2);
    return cudaGetLastError();
}

}  // namespace

int64_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d)
{
    const int64_t n_pad = (N + kBlock - 1) / kBlock * kBlock;
    return B * H * n_pad * d * 4 + 2 * B * H * n_pad * 4;
}

cudaError_t fa_launch_bwd(const FaBwdProblem &p, void *workspace, cudaStream_t s)
{
    const int64_t BH = p.B * p.H, n_pad = (p.N + kBlock - 1) / kBlock * kBlock;
    float *dq_acc = static_cast<float *>(workspace);
    float *lse2 = dq_acc + BH * n_pad * p.d;
    float *dvec = lse2 + BH * n_pad;
    // pre
    {
        const int64_t rows = BH * n_pad;
        const int64_t want = (rows + 7) / 8, cap = static_cast<int64_t>(p.sm_count) * 16;
        const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
        if (p.d == 64)
            fa_bwd_pre_kernel<64><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(p.o),
                                                        static_cast<const __nv_bfloat16 *>(p.dout), p.lse, lse2, dvec,
                                                        dq_acc, static_cast<int>(p.N), static_cast<int>(n_pad), BH);
        else
            fa_bwd_pre_kernel<128><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(p.o),
                                                         static_cast<const __nv_bfloat16 *>(p.dout), p.lse, lse2, dvec,
                                                         dq_acc, static_cast<int>(p.N), static_cast<int>(n_pad), BH);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // main
    cudaError_t e;
    if (p.d == 64)
        e = p.causal ? launch_main<64, true>(p, lse2, dvec, dq_acc, static_cast<int>(n_pad), s)
                     : launch_main<64, false>(p, lse2, dvec, dq_acc, static_cast<int>(n_pad), s);
    else
        e = p.causal ? launch_main<128, true>(p, lse2, dvec, dq_acc, static_cast<int>(n_pad), s)
                     : launch_main<128, false>(p, lse2, dvec, dq_acc, static_cast<int>(n_pad), s);
    if (e != cudaSuccess) return e;
    // post
    {
        const int64_t n4 = BH * p.N * p.d / 4;
        const int64_t want = (n4 + 255) / 256, cap = static_cast<int64_t>(p.sm_count) * 16;
        const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
        const int nb = static_cast<int>(n_pad / kBlock);
        if (p.d == 64)
            fa_bwd_post_kernel<64><<<grid, 256, 0, s>>>(reinterpret_cast<const float4 *>(dq_acc),
                                                         static_cast<uint2 *>(p.dq), n4, static_cast<int>(p.N), nb,
                                                         p.scale);
        else
            fa_bwd_post_kernel<128><<<grid, 256, 0, s>>>(reinterpret_cast<const float4 *>(dq_acc),
                                                          static_cast<uint2 *>(p.dq), n4, static_cast<int>(p.N), nb,
                                                          p.scale);
        return cudaGetLastError();
    }
}

int fa_bwd_take_status(cudaStream_t stream)
{
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_bwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    return h;
}
