// Forward with P apart from S (fa_fwd_dp_kernel) for GB300 (sm_103a): the bf16
// forward at d = 64 for short units, and the E4M3 forward.  The operation, the
// work order and the online softmax are those of fa_fwd_tc.cu; what differs is
// described below.  Every mbarrier wait is bounded; a wait that gives up sets
// FA_ERR_TIMEOUT in this file's device status word (read and cleared by
// fa_get_device_status) and the CTA winds down.
#include <math.h>

#include "fa_fwd_common.cuh"

using namespace sm100;

namespace {

__device__ int g_dp_status;  // sticky FA_ERR_TIMEOUT, read and cleared by fa_get_device_status

__device__ __forceinline__ void report_timeout() { atomicExch(&g_dp_status, FA_ERR_TIMEOUT); }

// ------------------------------------------------ forward with P apart from S
//
// In the forward above each query tile's chain softmax(j) -> P V(j) -> S(j+1)
// -> softmax(j+1) makes the softmax wait for every S (S_t(j+1) overwrites the
// P_t(j) that P V(j) reads).  Where memory allows, this kernel keeps P apart:
//   bf16, d = 64:   tensor memory per query tile t holds S_t [128 t, +128),
//                   O_t [256 + 64 t, +64) and P_t [384 + 64 t, +64), and
//                   P V is a TS MMA (A = P from tensor memory);
//   E4M3, d = 128:  S_t [128 t, +128), O_t [256 + 128 t, +128) fill tensor
//                   memory, so P_t (16 KB of E4M3) goes to shared memory in
//                   the 128-byte swizzle and P V is an SS MMA.
// Rows of 128 bytes (64 bf16 or 128 E4M3) make the Q, K, V and P tiles of both
// variants 16 KB with the same K steps of 32 bytes.  S_t(j+1) is computed as
// soon as the softmax has read S_t(j) into its registers (it arrives on
// s_free[t]), while it is still working on tile j; the softmax then runs from
// tile to tile without waiting.  Before storing P_t(j) (and before rescaling
// O_t) the softmax waits for P V_t(j-1), whose commit goes to o_done[t].  The
// divisor of O is summed as in the forward above (the rounded terms in heavy
// tiles; there is no ones column here).  Q is
// double-buffered, so the next unit's first S can start as soon as both
// query tiles have issued the current unit's last S.  Per K/V tile the MMA
// thread issues S_0(j) and S_1(j) (each once its tile's softmax has read the
// previous S), then the P V of item j - 1 for both tiles (each once its
// softmax has stored P), and the P V of the unit's last item at its end; a
// query tile 0 that skips a unit's last tile simply has no S or P V there.
constexpr int kD64Stages = 6;
template <bool FP8>
struct D64Cfg {
    static constexpr int kD = FP8 ? 128 : 64;                         // head dimension
    static constexpr int kTileBytes = kBlockN * 128;                  // 128 rows of 128 bytes
    static constexpr int kRingOffset = 2 * kQTiles * kTileBytes;      // two Q buffers of two tiles
    static constexpr int kPOffset = kRingOffset + kD64Stages * kTileBytes;  // E4M3: P_0, P_1
    static constexpr int kStageOffset = kPOffset + (FP8 ? kQTiles * kTileBytes : 0);
    static constexpr int kBarOffset = kStageOffset + 8 * 4096;        // O staging, 4 KB per softmax warp
    // q_full[2], q_empty[2], s_full[2], s_free[2], p_full[2], o_done[2], mma_done, kv_full[S], kv_empty[S]
    static constexpr int kNumBars = 13 + 2 * kD64Stages;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
    static constexpr int kOCol = 256;                                 // O_t at kOCol + t * kD
    static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");
};

struct D64Bars {
    uint32_t base;
    __device__ uint32_t q_full(int b) const { return base + 8u * b; }
    __device__ uint32_t q_empty(int b) const { return base + 16u + 8u * b; }
    __device__ uint32_t s_full(int t) const { return base + 32u + 8u * t; }
    __device__ uint32_t s_free(int t) const { return base + 48u + 8u * t; }
    __device__ uint32_t p_full(int t) const { return base + 64u + 8u * t; }
    __device__ uint32_t o_done(int t) const { return base + 80u + 8u * t; }
    __device__ uint32_t mma_done() const { return base + 96u; }
    __device__ uint32_t full(int s) const { return base + 104u + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 104u + 8u * (kD64Stages + s); }
};

template <bool CAUSAL, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_dp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 float *__restrict__ lse, int N, int BH, int n_mblocks, int n_units, int hg, float scale,
                 float scale_log2, const float *__restrict__ qs, const float *__restrict__ ks,
                 const float *__restrict__ vs)
{
    using C = D64Cfg<FP8>;
    constexpr int D = C::kD;
    constexpr int S = kD64Stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const D64Bars bars{s_base + C::kBarOffset};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kBarOffset + C::kNumBars * 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool run = *reinterpret_cast<volatile int *>(&g_dp_status) == 0;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.q_full(b), 1);
            mbar_init(bars.q_empty(b), 1);
            mbar_init(bars.s_full(b), 1);
            mbar_init(bars.s_free(b), kBlockM / 32);  // one arrive per softmax warp
            mbar_init(bars.p_full(b), kBlockM / 32);
            mbar_init(bars.o_done(b), 1);
        }
        mbar_init(bars.mma_done(), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), 1);
        }
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

    if (!run) {
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            bool ok = true;
            int it = 0, uc = 0;
            for (int r = 0, u = unit_index(0); u < n_units && ok; u = unit_index(++r)) {
                const Unit w = unit_of<CAUSAL, false, true>(u, N, BH, n_mblocks, 1, N, hg);
                const int qb = uc & 1;  // Q buffer of this unit: free once unit uc - 2 released it
                if (!(ok = mbar_wait(bars.q_empty(qb), ((uc >> 1) & 1) ^ 1, kWaitLimitNs))) break;
                mbar_arrive_expect_tx(bars.q_full(qb), kQTiles * C::kTileBytes);
                for (int t = 0; t < kQTiles; ++t)
                    tma_load_3d(s_base + (qb * kQTiles + t) * C::kTileBytes, &tm_q, bars.q_full(qb), 0,
                                w.q_row0 + t * kBlockM, w.bh);
                ++uc;
                for (int j = 0; j < w.n_kv && ok; ++j) {
                    for (int kind = 0; kind < 2; ++kind, ++it) {
                        const int slot = it % S, use = it / S;
                        if (!(ok = mbar_wait(bars.empty(slot), (use & 1) ^ 1, kWaitLimitNs))) break;
                        mbar_arrive_expect_tx(bars.full(slot), C::kTileBytes);
                        tma_load_3d(s_base + C::kRingOffset + slot * C::kTileBytes, kind == 0 ? &tm_k : &tm_v,
                                    bars.full(slot), 0, j * kBlockN, w.bh);
                    }
                }
            }
            if (!ok) report_timeout();
            const uint64_t lim = ok ? kWaitLimitNs : kCleanupLimitNs;
            for (int k = max(0, uc - 2); k < uc; ++k) mbar_wait(bars.q_full(k & 1), (k >> 1) & 1, lim);
            for (int k = max(0, it - S); k < it; ++k) mbar_wait(bars.full(k % S), (k / S) & 1, lim);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idS = FP8 ? idesc_e4m3_f32(kBlockM, kBlockN, false) : idesc_bf16_f32(kBlockM, kBlockN, false);
            constexpr uint32_t idO = FP8 ? idesc_e4m3_f32(kBlockM, D, true) : idesc_bf16_f32(kBlockM, D, true);
            const uint64_t dq0 = smem_desc_sw128(s_base, 16, 1024);
            const uint64_t dr0 = smem_desc_sw128(s_base + C::kRingOffset, 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(s_base + C::kRingOffset, kBlockN * 128, 1024);  // V, MN-major
            const uint32_t dq_lo = static_cast<uint32_t>(dq0), d_hi = static_cast<uint32_t>(dq0 >> 32);
            const uint32_t dr_lo = static_cast<uint32_t>(dr0), dv_lo = static_cast<uint32_t>(dv0);
            constexpr uint32_t kTile16 = C::kTileBytes >> 4;
            bool ok = true;
            int it = 0, uc = 0;    // ring position of the unit's K_0, units done
            int gs0 = 0, gs1 = 0;  // S items issued per query tile (all units)
            int gp0 = 0, gp1 = 0;  // P V items issued per query tile
            // the item whose P V is still to be issued: its V position, whether it is the
            // first of its unit, and whether query tile 0 ran it
            int pend_v = -1;
            bool pend_first = false, pend0 = false;
            auto issue_pv = [&](int t, int vpos, bool first) {
                const uint32_t bv = dv_lo + (vpos % S) * kTile16;
                if constexpr (FP8) {  // A = P_t from shared memory, 32 keys (32 bytes) per K step
                    const uint32_t ap = dq_lo + ((C::kPOffset + t * C::kTileBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 32; ++kk)
                        mma_ss_f8_lohi(tmem + C::kOCol + t * D, ap + 2 * kk, d_hi, bv + kk * 256, d_hi, idO,
                                       (!first || kk > 0) ? 1u : 0u);
                } else {  // A = P_t from tensor memory, 16 keys (8 columns) per K step
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)
                        mma_ts_lohi(tmem + C::kOCol + t * D, tmem + 384 + t * 64 + kk * 8, bv + kk * 128, d_hi, idO,
                                    (!first || kk > 0) ? 1u : 0u);
                }
                mma_commit(bars.o_done(t));
            };
            // P V of the pending item, for both query tiles (tile 0 only if it ran it)
            auto flush_pending = [&]() {
                if (pend_v < 0) return true;
                if (!mbar_wait(bars.full(pend_v % S), (pend_v / S) & 1, kWaitLimitNs)) return false;
                if (pend0) {
                    if (!mbar_wait(bars.p_full(0), gp0 & 1, kWaitLimitNs)) return false;
                    tc_fence_after();
                    issue_pv(0, pend_v, pend_first);
                    ++gp0;
                }
                if (!mbar_wait(bars.p_full(1), gp1 & 1, kWaitLimitNs)) return false;
                tc_fence_after();
                issue_pv(1, pend_v, pend_first);
                ++gp1;
                mma_commit(bars.empty(pend_v % S));  // V read by every P V it feeds
                pend_v = -1;
                return true;
            };
            auto issue_s = [&](int t, int qb, int pos) {
                const uint32_t aq = dq_lo + (qb * kQTiles + t) * kTile16;
                const uint32_t bk = dr_lo + (pos % S) * kTile16;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of each 128-byte row per K step
                    if constexpr (FP8)
                        mma_ss_f8_lohi(tmem + t * 128, aq + 2 * kk, d_hi, bk + 2 * kk, d_hi, idS, kk > 0 ? 1u : 0u);
                    else
                        mma_ss_lohi(tmem + t * 128, aq + 2 * kk, d_hi, bk + 2 * kk, d_hi, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bars.s_full(t));
            };
            for (int r = 0, u = unit_index(0); u < n_units && ok; u = unit_index(++r)) {
                const Unit w = unit_of<CAUSAL, false, true>(u, N, BH, n_mblocks, 1, N, hg);
                const int n = w.n_kv, n0 = n - (CAUSAL && w.q_row0 + kBlockM < N ? 1 : 0), qb = uc & 1;
                if (!(ok = mbar_wait(bars.q_full(qb), (uc >> 1) & 1, kWaitLimitNs))) break;
                for (int j = 0; j < n && ok; ++j) {
                    const int pos = it + 2 * j;
                    if (!(ok = mbar_wait(bars.full(pos % S), (pos / S) & 1, kWaitLimitNs))) break;
                    // S of item j, once each query tile has read its previous S into registers
                    if (j < n0) {
                        if (gs0 > 0 && !(ok = mbar_wait(bars.s_free(0), (gs0 - 1) & 1, kWaitLimitNs))) break;
                        tc_fence_after();
                        issue_s(0, qb, pos);
                        ++gs0;
                    }
                    if (gs1 > 0 && !(ok = mbar_wait(bars.s_free(1), (gs1 - 1) & 1, kWaitLimitNs))) break;
                    tc_fence_after();
                    issue_s(1, qb, pos);
                    ++gs1;
                    mma_commit(bars.empty(pos % S));                // K_j read by every S it feeds
                    if (j == n - 1) mma_commit(bars.q_empty(qb));   // the unit's last reads of its Q
                    // then the P V of the previous item, while the softmax works on this one
                    if (!(ok = flush_pending())) break;
                    pend_v = pos + 1;
                    pend_first = j == 0;
                    pend0 = j < n0;
                }
                // the unit's last P V now: the epilogue must not wait for the next unit's loads
                if (ok) ok = flush_pending();
                it += 2 * n;
                ++uc;
            }
            if (!ok) report_timeout();
            mma_commit(bars.mma_done());
            mbar_wait(bars.mma_done(), 0, ok ? kWaitLimitNs : kCleanupLimitNs);
        }
    } else {
        // --------------------------------------------------------------- softmax
        const int t = warp >> 2;
        const int row = tid & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + C::kOCol + t * D;
        const uint32_t tP = tmem + lane_off + 384 + t * 64;  // bf16 only
        // E4M3: this thread's row of P_t in shared memory (128 bytes, 16-byte pieces swizzled)
        const uint32_t sP = s_base + C::kPOffset + t * C::kTileBytes + row * 128;
        bool ok = true;
        int g = 0;  // tiles processed by this warpgroup (all units): the S, P and P V item index
        for (int r = 0, u = unit_index(0); u < n_units && ok; u = unit_index(++r)) {
            const Unit w = unit_of<CAUSAL, false, true>(u, N, BH, n_mblocks, 1, N, hg);
            // exponent constant of this slice (E4M3 scales folded in)
            const float c_u = FP8 ? scale_log2 * qs[w.bh] * ks[w.bh] : scale_log2;
            const int row_g = w.q_row0 + t * kBlockM + row;
            const int n_mine = w.n_kv - (t == 0 && CAUSAL && w.q_row0 + kBlockM < N ? 1 : 0);
            float m_ref = -INFINITY, l = 0.f, lr = 0.f;
            for (int j = 0; j < n_mine; ++j, ++g) {
                if (!mbar_wait_warp(bars.s_full(t), g & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S_t, each 32-column piece's max coming with the load
                float s[kBlockN], pm[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_ld32_max(tS + c * 32, *reinterpret_cast<float(*)[32]>(&s[c * 32]), pm[c]);
                tmem_wait_ld();
                // S_t is in registers: the next S may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.s_free(t));
                float mt = fmax3(fmaxf(pm[0], pm[1]), pm[2], pm[3]);
                const int k0 = j * kBlockN;
                if (k0 + kBlockN > N || (CAUSAL && k0 + kBlockN - 1 > w.q_row0 + t * kBlockM)) {
                    // masked keys: the max again over the admitted ones
                    const int lim = CAUSAL ? min(N - 1, row_g) : N - 1;
#pragma unroll
                    for (int i = 0; i < kBlockN; ++i)
                        if (k0 + i > lim) s[i] = -INFINITY;
                    float mx[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int b0 = 16 * q;
                        float a = fmax3(s[b0], s[b0 + 1], s[b0 + 2]);
#pragma unroll
                        for (int i = 3; i < 15; i += 2) a = fmax3(a, s[b0 + i], s[b0 + i + 1]);
                        mx[q] = fmaxf(a, s[b0 + 15]);
                    }
                    mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                }
                const float m_new = fmaxf(m_ref, mt);
                const bool need = (m_new - m_ref) * c_u > kRescaleLog2;  // true while m_ref = -inf
                float alpha = 1.f;
                if (need) {
                    alpha = ex2((m_ref - m_new) * c_u);
                    m_ref = m_new;
                }
                const float mc = (m_ref == -INFINITY ? 0.f : m_ref) * c_u;
                const bool heavy = __any_sync(0xffffffffu, ex2(fmaf(mt, c_u, -mc)) > kHeavyShare * (l * alpha));
                // P_t and O_t are free once the previous tile's P V has completed
                if (j > 0) {
                    if (!mbar_wait_warp(bars.o_done(t), (g - 1) & 1, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const float2 c2 = make_float2(c_u, c_u), nmc2 = make_float2(-mc, -mc);
                float2 lf[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                float add;  // the divisor of O: the rounded terms in heavy tiles, the fp32 terms elsewhere
                if constexpr (FP8) {
                    // P rounded to E4M3, four per word, 16-byte pieces into this row of P_t
                    uint32_t pw[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 x01 = fma2(make_float2(s[4 * i], s[4 * i + 1]), c2, nmc2);
                        const float2 x23 = fma2(make_float2(s[4 * i + 2], s[4 * i + 3]), c2, nmc2);
                        const float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
                        lf[i & 3] = add2(lf[i & 3], add2(make_float2(p0, p1), make_float2(p2, p3)));
                        pw[i] = pack_e4m3x4(p0, p1, p2, p3);
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        st_shared_v4(sP + ((q4 ^ (row & 7)) << 4),
                                     make_uint4(pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]));
                    fence_proxy_async_smem();  // visible to the P V MMA
                    const float2 lfs = add2(add2(lf[0], lf[1]), add2(lf[2], lf[3]));
                    add = lfs.x + lfs.y;
                    if (heavy) {  // the rounded terms, from the packed words still in registers
                        float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int i = 0; i < 32; ++i) lq[i & 3] = add_e4m3x4(lq[i & 3], pw[i]);
                        add = (lq[0] + lq[1]) + (lq[2] + lq[3]);
                    }
                    l = l * alpha + (lfs.x + lfs.y);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 x = fma2(make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), c2, nmc2);
                            const float p0 = ex2(x.x), p1 = ex2(x.y);
                            pk[i] = pack_bf16x2(p0, p1);
                            lf[c] = add2(lf[c], make_float2(p0, p1));
                        }
                        tmem_st16(tP + c * 16, pk);
                    }
                    const float2 lfs = add2(add2(lf[0], lf[1]), add2(lf[2], lf[3]));
                    add = lfs.x + lfs.y;
                    if (heavy) {
                        tmem_wait_st();
                        float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t rr[32];
                            tmem_ld32(tP + h * 32, rr);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) lq[i & 3] = add_bf16x2(lq[i & 3], rr[i]);
                        }
                        add = (lq[0] + lq[1]) + (lq[2] + lq[3]);
                    }
                    l = l * alpha + (lfs.x + lfs.y);
                }
                lr = lr * alpha + add;
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t rr[32];
                        tmem_ld32(tO + c * 32, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 y = mul2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                                  make_float2(alpha, alpha));
                            rr[i] = __float_as_uint(y.x);
                            rr[i + 1] = __float_as_uint(y.y);
                        }
                        tmem_st32(tO + c * 32, rr);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.p_full(t));
            }
            // epilogue once the unit's last P V (item g - 1) has completed
            if (!ok || !(ok = mbar_wait_warp(bars.o_done(t), (g - 1) & 1, kWaitLimitNs))) break;
            tc_fence_after();
            const float inv_l = lr > 0.f ? (FP8 ? vs[w.bh] : 1.f) / lr : 0.f;
            const uint32_t stage = s_base + C::kStageOffset + warp * 4096;
            const int row0 = w.q_row0 + t * kBlockM + (warp & 3) * 32;
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            // O in 32-column chunks through two 2 KB buffers (as in the forward above)
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rr[32];
                tmem_ld32(tO + c * 32, rr);
                tmem_wait_ld();
                if (c >= 2) {
                    if (lane == 0) bulk_wait_read1();
                    __syncwarp();
                }
                const uint32_t buf = stage + (c & 1) * 2048 + lane * 64;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 0]) * inv_l, __uint_as_float(rr[q4 * 8 + 1]) * inv_l);
                    v.y = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 2]) * inv_l, __uint_as_float(rr[q4 * 8 + 3]) * inv_l);
                    v.z = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 4]) * inv_l, __uint_as_float(rr[q4 * 8 + 5]) * inv_l);
                    v.w = pack_bf16x2(__uint_as_float(rr[q4 * 8 + 6]) * inv_l, __uint_as_float(rr[q4 * 8 + 7]) * inv_l);
                    st_shared_v4(buf + ((q4 ^ ((lane >> 1) & 3)) << 4), v);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < N) {
                    tma_store_3d(&tm_o, stage + (c & 1) * 2048, c * 32, row0, w.bh);
                    bulk_commit();
                }
            }
            const float scale_u = FP8 ? scale * qs[w.bh] * ks[w.bh] : scale;
            if (row_g < N) lse[static_cast<int64_t>(w.bh) * N + row_g] = l > 0.f ? m_ref * scale_u + logf(l) : -INFINITY;
        }
        if (!ok) report_timeout();
        if (lane == 0) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

template <bool CAUSAL, bool FP8>
cudaError_t launch_dp(const FaProblem &p, cudaStream_t stream, const float *qs = nullptr, const float *ks = nullptr,
                      const float *vs = nullptr)
{
    using C = D64Cfg<FP8>;
    CUtensorMap mq, mk, mv, mo;
    const int64_t BH = p.B * p.H;
    const int elem = FP8 ? 1 : 2;
    if (!make_map(&mq, p.q, BH, p.N, C::kD, elem) || !make_map(&mk, p.k, BH, p.N, C::kD, elem) ||
        !make_map(&mv, p.v, BH, p.N, C::kD, elem) || !make_out_map(&mo, p.o, BH, p.N, C::kD))
        return cudaErrorInvalidValue;
    cudaError_t e = set_max_dynamic_smem<fa_fwd_dp_kernel<CAUSAL, FP8>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t n_mblocks = (p.N + kQTiles * kBlockM - 1) / (kQTiles * kBlockM);
    const int64_t n_units = n_mblocks * BH;
    if (n_units > 0x7fffffffLL || BH > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int64_t grid = n_units < p.sm_count ? n_units : p.sm_count;  // persistent: one CTA per SM
    const int64_t kv_bytes = 2 * p.N * C::kTileBytes / kBlockN;  // K and V of one slice
    int64_t hg = BH;
    if (BH * kv_bytes > (int64_t(160) << 20)) {
        hg = (int64_t(64) << 20) / kv_bytes;
        hg = hg < 1 ? 1 : (hg > BH ? BH : hg);
    }
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    fa_fwd_dp_kernel<CAUSAL, FP8><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(
        mq, mk, mv, mo, p.lse, static_cast<int>(p.N), static_cast<int>(BH), static_cast<int>(n_mblocks),
        static_cast<int>(n_units), static_cast<int>(hg), p.scale, scale_log2, qs, ks, vs);
    return cudaGetLastError();
}

}  // namespace

cudaError_t fa_launch_dp(const FaProblem &p, cudaStream_t stream)
{
    if (p.d != 64) return cudaErrorInvalidValue;
    return p.causal ? launch_dp<true, false>(p, stream) : launch_dp<false, false>(p, stream);
}

cudaError_t fa_launch_fp8(const FaProblem &p, const float *qs, const float *ks, const float *vs,
                             cudaStream_t stream)
{
    if (p.d != 128) return cudaErrorInvalidValue;
    return p.causal ? launch_dp<true, true>(p, stream, qs, ks, vs) : launch_dp<false, true>(p, stream, qs, ks, vs);
}

int fa_dp_take_status(cudaStream_t stream)
{
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_dp_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_dp_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    return h;
}
