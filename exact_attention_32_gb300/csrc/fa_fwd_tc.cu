// Fused exact attention forward for GB300 (sm_103a): TMA + tcgen05 + TMEM.
//
// What is computed (per batch b, head h, query row i):
//   S_ij = scale * q_i . k_j,  P_i = softmax(S_i) over admitted keys,
//   O_i = sum_j P_ij v_j,      LSE_i = m_i + ln(l_i)
// ("6.1 FlashAttention V1 in detail", sections 1.1 and 5.1; LSE as in
// "FlashAttention: IO-Aware Tiling, ...", section "Backward Pass Recomputation").
//
// How: a work unit is 2 query tiles of 128 rows (256 consecutive rows of one
// (b, h) slice) that share one stream of the admitted 128-key K/V tiles.  The
// grid is persistent (one CTA per SM); each CTA walks its units longest-first,
// with barrier phases carried across units so that the next unit's Q and K/V
// loads and first S MMAs overlap the current unit's last P V and epilogue.
// Per K/V tile j and query tile t the running statistics are merged as in
// "FlashAttention: optimize data movement before counting FLOPs", section 02
// (m' = max(m, max s), l' = e^(m-m') l + sum e^(s-m'), u' = e^(m-m') u + P V):
// the numerator u lives in tensor memory and is divided by l once at the end
// (the FlashAttention-2 rescaling optimisation on the llms.blog page).
//
// Roles (320 threads):
//   warps 0-3  softmax warpgroup of query tile 0 (one thread per row)
//   warps 4-7  softmax warpgroup of query tile 1
//   warp  8    TMA producer: per unit the Q tiles (once the previous unit's last
//              S MMAs are done), then K_j, V_j into a ring of slots
//   warp  9    tcgen05 issuer (and TMEM owner):
//                S_t  = Q_t K_j^T          (A, B from shared memory)
//                O_t += P_t V_j            (A = P from tensor memory)
// Tensor memory (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256,256+d), O_1 [384,384+d); P_t (bf16, two per column) overwrites the
// first 64 columns of S_t once S_t has been read.
//
// Exponentials are base 2 with scale*log2(e) folded into one FMA; the
// reference max m is kept in unscaled dot-product units (scale > 0).  The
// numerator is rescaled only when the row max grows by more than 2^8 (any
// common shift of a row's logits leaves softmax unchanged - the identity of
// "6.1 ...", section 3.3 - so a stale reference is exact as long as the
// exponentials stay in range; LSE = m_ref + ln(l) holds for any reference).
// Keys >= N and, when causal, keys j > i are set to -inf before the max
// ("6.1 ...", section 8.3: the K/V out-of-range mask).  The row max of a tile
// with no masked key comes with the tensor-memory load of S (tcgen05.ld with
// a max reduction, sm_103a); a masked tile takes it again after masking.
//
// The epilogue (O / l to bf16) goes through shared memory: each softmax warp
// writes 32-column chunks of its 32 rows there and one thread stores each
// chunk with a TMA store, so global memory sees whole 64-byte row pieces
// rather than one 16-byte piece of 32 different rows per instruction; the
// tensor map clips the rows past N.  LSE is stored directly (a warp's 32 rows
// are contiguous).  The fp32 partials of a key split store directly from
// registers.
//
// fa_fwd_tc_kernel serves bf16 at d = 64 and 128 with its key-split and
// block-sparse variants; fa_fwd_dp.cu holds the kernel that keeps P apart from
// S (bf16 at d = 64 for short units, and the E4M3 forward).
//
// Every mbarrier wait is bounded; a wait that gives up sets FA_ERR_TIMEOUT in
// a device status word and the CTA winds down (waiting, bounded, for its own
// copies and MMAs in flight, then freeing its tensor memory).
#include <math.h>

#include <algorithm>

#include "fa_fwd_common.cuh"

using namespace sm100;

namespace {

__device__ int g_tc_status;  // sticky FA_ERR_TIMEOUT, read and cleared by fa_get_device_status

template <int D>
struct Cfg {
    static constexpr int kElem = 2;                         // bytes per element (bf16)
    static constexpr int kRowBytes = D * kElem;
    static constexpr int kTileBytes = kBlockN * kRowBytes;  // one Q, K or V tile
    static constexpr int kAtoms = kRowBytes / 128;          // 128-byte-wide column blocks per tile
    static constexpr int kStages = kTileBytes == 32768 ? 4 : 8;  // K/V ring slots
    static constexpr int kSSteps = kRowBytes / 32;          // S MMA K steps (32 bytes of each row)
    static constexpr int kPVKeys = 16;                      // keys per P V MMA
    static constexpr int kPVSteps = kBlockN / kPVKeys;
    // d = 64: the P V MMA runs at N = 80.  B's extra 16 columns come from a
    // constant block (a column of ones, then zeros), so column 64 of O accumulates
    // the row sum of exactly the bf16 P that the MMA multiplies, rescaled with O.
    static constexpr bool kOnesCol = (D == 64);
    static constexpr int kPVN = kOnesCol ? 80 : D;             // N of the P V MMA
    static constexpr int kOnesOffset = (kQTiles + kStages) * kTileBytes;
    static constexpr int kBarOffset = kOnesOffset + (kOnesCol ? kBlockN * 128 : 0);
    // barriers: q_full, q_empty, s_full[2], p_full[2], o_full[2], mma_done, kv_full[S], kv_empty[S]
    static constexpr int kNumBars = 9 + 2 * kStages;
    // block-sparse tile records: one per K/V ring slot, one per query tile
    static constexpr int kMetaOffset = kBarOffset + kNumBars * 8 + 16;
    // epilogue staging of O (bf16 output): two 32 x 32 chunks (2 KB each) per softmax warp
    static constexpr int kStageOffset = (kMetaOffset + (kStages + 2) * 4 + 1023) / 1024 * 1024;
    static constexpr int kStageBytes = 8 * 4096;
    static constexpr int kSmemBytes = 1024 + kStageOffset + kStageBytes;
    static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");
};

// Shared-memory addresses of the mbarriers, laid out from `base`: q_full,
// q_empty, s_full[2], p_full[2], o_full[2], mma_done, kv_full[S], kv_empty[S].
template <int STAGES>
struct Bars {
    uint32_t base;
    __device__ uint32_t q_full() const { return base; }
    __device__ uint32_t q_empty() const { return base + 8u; }
    __device__ uint32_t s_full(int t) const { return base + 16u + 8u * t; }
    __device__ uint32_t p_full(int t) const { return base + 32u + 8u * t; }
    __device__ uint32_t o_full(int t) const { return base + 48u + 8u * t; }
    __device__ uint32_t mma_done() const { return base + 64u; }
    __device__ uint32_t full(int s) const { return base + 72u + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 72u + 8u * (STAGES + s); }
};

__device__ __forceinline__ void report_timeout() { atomicExch(&g_tc_status, FA_ERR_TIMEOUT); }

// Block-sparse mode: K/V tile kj is processed for a unit when the block mask
// admits it for either of the unit's two 128-row query blocks (a query block
// past the last row admits nothing).  mask_word gives the tiles j0 + c .. j0 +
// c + 31 of mask rows qa and qb as a bit mask (bit i: tile j0 + c + i admitted
// by either row, tiles at or past j0 + n excluded); its 64 byte loads are
// independent, so a word costs one memory round trip.
__device__ __forceinline__ uint32_t mask_word(const uint8_t *__restrict__ bm, int nb, int qa, int qb, int j0, int c,
                                              int n)
{
    // every load is unconditional (addresses past the range are clamped to its
    // last tile and their bits dropped below), so all 64 are in flight at once
    const int last = n - 1 - c;  // >= 0: the caller asks only for words inside the range
    const uint8_t *ra = bm + static_cast<int64_t>(qa) * nb + j0 + c;
    const uint8_t *rb = bm + static_cast<int64_t>(qb) * nb + j0 + c;
    uint32_t va[32], vb[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int k = i < last ? i : last;
        va[i] = __ldg(ra + k);
        vb[i] = __ldg(rb + k);
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) m |= ((va[i] | vb[i]) != 0u ? 1u : 0u) << i;
    return last >= 31 ? m : (m & ((2u << last) - 1u));
}

// mask_word's bits for rows qa (.x) and qb (.y) separately, the 64 loads again
// all in flight at once.
__device__ __forceinline__ uint2 mask_row_words(const uint8_t *__restrict__ bm, int nb, int qa, int qb, int j0, int c,
                                                int n)
{
    const int last = n - 1 - c;
    const uint8_t *ra = bm + static_cast<int64_t>(qa) * nb + j0 + c;
    const uint8_t *rb = bm + static_cast<int64_t>(qb) * nb + j0 + c;
    uint32_t va[32], vb[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int k = i < last ? i : last;
        va[i] = __ldg(ra + k);
        vb[i] = __ldg(rb + k);
    }
    uint32_t ma = 0, mb = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        ma |= (va[i] != 0u ? 1u : 0u) << i;
        mb |= (vb[i] != 0u ? 1u : 0u) << i;
    }
    const uint32_t keep = last >= 31 ? ~0u : ((2u << last) - 1u);
    return make_uint2(ma & keep, mb & keep);
}

// Block-sparse tile record, published by the producer for every live K/V tile
// (per K ring slot) and forwarded by the MMA thread with every S tile: the
// tile index (bits 0-23), admitted by query tile 0 / 1 (bits 30 / 29), last
// live tile of the unit (bit 31).  A unit with no live tile sends one record,
// kMetaEmptyUnit (no tile has index 2^24 - 1).
constexpr uint32_t kMetaTile = 0xffffffu, kMetaOwn0 = 1u << 30, kMetaOwn1 = 1u << 29, kMetaLast = 1u << 31;
constexpr uint32_t kMetaEmptyUnit = kMetaTile | kMetaLast;

// Causal, all keys in one launch: a unit's last K/V tile starts at or past row
// q_row0 + 128 whenever query tile 1 has rows (q_row0 + 128 < N), so it is
// fully masked for query tile 0, which then skips it (its S, P and P V).
template <bool CAUSAL, bool SPLIT, bool SPARSE>
__device__ __forceinline__ bool tile0_skips_last(const Unit &w, int N)
{
    return CAUSAL && !SPLIT && !SPARSE && w.q_row0 + kBlockM < N;
}

// OUT_F32: O is written as fp32 (the partial results of a key split) instead
// of bf16; split s writes its rows at o + s * B*H*N*d and lse + s * B*H*N.
// SPARSE: bm is a [nb][nb] 0/1 block mask (nb = ceil(N/128)) over (query block,
// key block); K/V tiles no query block of the unit admits are skipped, and a
// tile is fully masked for a query tile whose block does not admit it.
// Keys outside [lo, hi] of the tile starting at key k0 to -inf.
__device__ __forceinline__ void mask_keys(float (&s)[kBlockN], int k0, int lo, int hi)
{
#pragma unroll
    for (int i = 0; i < kBlockN; ++i)
        if (k0 + i < lo || k0 + i > hi) s[i] = -INFINITY;
}

// Row max of a tile: eight independent chains of 3-input maxes.
__device__ __forceinline__ float row_max(const float (&s)[kBlockN])
{
    float mx[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const int b = 16 * g;
        float a = fmax3(s[b], s[b + 1], s[b + 2]);
#pragma unroll
        for (int i = 3; i < 15; i += 2) a = fmax3(a, s[b + i], s[b + i + 1]);
        mx[g] = fmaxf(a, s[b + 15]);
    }
    return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
}

template <int D, bool CAUSAL, bool OUT_F32, bool SPARSE>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 void *__restrict__ o, float *__restrict__ lse, int N, int BH, int n_mblocks, int n_units,
                 int n_splits, int kv_chunk, int hg, float scale, float scale_log2, const uint8_t *__restrict__ bm,
                 int nb, int split0)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t sQ = s_base;  // kQTiles tiles
    const uint32_t sRing = s_base + kQTiles * C::kTileBytes;
    const uint32_t sOnes = s_base + C::kOnesOffset;  // d = 64 only: B's columns 64..79 of the P V MMA
    const uint32_t bar0 = s_base + C::kBarOffset;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kBarOffset + C::kNumBars * 8);
    volatile uint32_t *kv_meta = reinterpret_cast<volatile uint32_t *>(smem + C::kMetaOffset);  // [kStages]
    volatile uint32_t *s_meta = kv_meta + C::kStages;                                            // [kQTiles]

    const Bars<C::kStages> bars{bar0};
    // K/V tiles a unit processes: all of its range, or in block-sparse mode those
    // the mask admits for either query block of the unit.  Only the producer
    // reads the mask (32 tiles per read): it publishes a record per live tile,
    // or one empty-unit record for a unit with none, which the MMA thread and
    // the softmax warps follow.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // after a timeout anywhere (sticky until read by the host) CTAs do no work
    const bool run = *reinterpret_cast<volatile int *>(&g_tc_status) == 0;

    if (tid == 0) {
        mbar_init(bars.q_full(), 1);
        mbar_init(bars.q_empty(), 1);
        for (int t = 0; t < 2; ++t) {
            // block-sparse: the commit and an arrive of the MMA thread that publishes s_meta[t]
            mbar_init(bars.s_full(t), SPARSE ? 2 : 1);
            mbar_init(bars.p_full(t), kBlockM / 32);  // one arrive per softmax warp
            mbar_init(bars.o_full(t), 1);
        }
        mbar_init(bars.mma_done(), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), 1);
        }
        fence_mbar_init();
    }
    if constexpr (C::kOnesCol) {
        // kBlockN key rows of 128 bytes in the 128-byte swizzle V uses: bf16 1.0 at
        // column 0 of every row (16-byte chunk 0 lands at chunk r mod 8), zeros elsewhere
        for (int i = threadIdx.x; i < kBlockN * 8; i += blockDim.x) {
            const int r = i >> 3, c = i & 7;
            reinterpret_cast<uint4 *>(smem + C::kOnesOffset)[i] =
                make_uint4(c == (r & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // visible to the tensor cores' reads
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
        // nothing to do: fall through to the teardown
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            bool ok = true;
            int it = 0, uc = 0;
            for (int r = 0, u = unit_index(0); u < n_units && ok; u = unit_index(++r)) {
                const Unit w = unit_of<CAUSAL, OUT_F32, !SPARSE>(u, N, BH, n_mblocks, n_splits, kv_chunk, hg, split0);
                if (!SPARSE && w.n_kv <= 0) continue;  // a key split with no admitted key: nothing to load
                // block-sparse: the live tiles in order, each published in its K slot's record
                // with its admission bits and a last-tile flag (found by looking one live
                // tile ahead); wa / wb are the admission bits of the two query blocks for the
                // 32-tile group `grp`
                const int qa = w.q_row0 / kBlockM;
                uint32_t wa = 0, wb = 0;
                int grp = -1;
                auto next_live = [&](int from) {  // the first live tile >= from, or -1
                    for (int c = from & ~31; c < w.n_kv; c += 32) {
                        if ((c >> 5) != grp) {
                            const uint2 wab = mask_row_words(bm, nb, qa, qa + 1 < nb ? qa + 1 : qa, w.j0, c, w.n_kv);
                            wa = wab.x;
                            wb = qa + 1 < nb ? wab.y : 0u;  // a second query block past the last row admits nothing
                            grp = c >> 5;
                        }
                        const uint32_t rest = (from > c) ? ((wa | wb) >> (from - c)) << (from - c) : (wa | wb);
                        if (rest != 0) return c + __ffs(rest) - 1;
                    }
                    return -1;
                };
                int j_live = SPARSE ? next_live(0) : 0;
                if (SPARSE && j_live < 0) {
                    // no admitted tile: one record through the K ring tells the MMA thread and the
                    // softmax warps (no Q, K or V is loaded)
                    const int slot = it % C::kStages, use = it / C::kStages;
                    if (!(ok = mbar_wait(bars.empty(slot), (use & 1) ^ 1, kWaitLimitNs))) break;
                    kv_meta[slot] = kMetaEmptyUnit;
                    mbar_arrive(bars.full(slot));  // released by this arrive
                    ++it;
                    continue;
                }
                // the Q buffers are free once the previous unit's last S MMAs have completed
                if (!mbar_wait(bars.q_empty(), (uc & 1) ^ 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bars.q_full(), kQTiles * C::kTileBytes);
                for (int t = 0; t < kQTiles; ++t)
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_3d(sQ + t * C::kTileBytes + a * 16384, &tm_q, bars.q_full(), a * (128 / C::kElem),
                                    w.q_row0 + t * kBlockM, w.bh);
                ++uc;
                for (int j = 0; j < w.n_kv && ok; ++j) {
                    uint32_t meta = 0;
                    if constexpr (SPARSE) {
                        if (j_live < 0) break;
                        j = j_live;
                        const uint32_t bit = 1u << (j & 31);
                        meta = static_cast<uint32_t>(j) | ((wa & bit) ? kMetaOwn0 : 0u) | ((wb & bit) ? kMetaOwn1 : 0u);
                        j_live = next_live(j + 1);
                        if (j_live < 0) meta |= kMetaLast;
                    }
                    for (int kind = 0; kind < 2; ++kind, ++it) {
                        const int slot = it % C::kStages, use = it / C::kStages;
                        if (!mbar_wait(bars.empty(slot), (use & 1) ^ 1, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        if (SPARSE && kind == 0) kv_meta[slot] = meta;  // released by the arrive below
                        mbar_arrive_expect_tx(bars.full(slot), C::kTileBytes);
                        const CUtensorMap *tm = kind == 0 ? &tm_k : &tm_v;
                        // K and V rows from the first key of split split0 on (a sequence shard's own rows)
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_load_3d(sRing + slot * C::kTileBytes + a * 16384, tm, bars.full(slot),
                                        a * (128 / C::kElem), (w.j0 + j) * kBlockN - (OUT_F32 ? split0 * kv_chunk : 0),
                                        w.bh);
                    }
                }
            }
            if (!ok) report_timeout();
            // every copy this thread issued has landed before the CTA may exit
            const uint64_t lim = ok ? kWaitLimitNs : kCleanupLimitNs;
            if (uc > 0) mbar_wait(bars.q_full(), (uc - 1) & 1, lim);
            for (int k = max(0, it - C::kStages); k < it; ++k)
                mbar_wait(bars.full(k % C::kStages), (k / C::kStages) & 1, lim);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBlockM, kBlockN, false);
            constexpr uint32_t idO = idesc_bf16_f32(kBlockM, C::kPVN, true);
            // descriptors are built once; a K step only moves the start address
            // (low 32 bits, in 16-byte units): +32 bytes inside a 128-byte-wide
            // column block, +16 KB to the next block (S), +2 KB per 16 keys (P V)
            const uint64_t dq = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(sRing, 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(sRing, C::kOnesCol ? sOnes - sRing : kBlockN * 128, 1024);
            const uint32_t dq_lo = static_cast<uint32_t>(dq), dq_hi = static_cast<uint32_t>(dq >> 32);
            const uint32_t dk_hi = static_cast<uint32_t>(dk0 >> 32), dv_hi = static_cast<uint32_t>(dv0 >> 32);
            constexpr uint32_t kTile16 = C::kTileBytes >> 4;
            bool ok = true;
            int it = 0, uc = 0;     // ring position, units done
            int jg0 = 0, jg1 = 0;   // items (S tiles, empty-unit records) sent to query tile 0 / 1 (all units)
            // block-sparse: an empty-unit record not yet acknowledged (on p_full) by the softmax
            // of query tile 0 / 1; its s_meta may not be written again before that
            bool tok0 = false, tok1 = false;
            auto ack_token = [&](int t) {
                bool &tk = t ? tok1 : tok0;
                if (!tk) return true;
                tk = false;
                return mbar_wait(bars.p_full(t), ((t ? jg1 : jg0) - 1) & 1, kWaitLimitNs);
            };
            for (int r = 0, u = unit_index(0); u < n_units && ok; u = unit_index(++r)) {
                const Unit w = unit_of<CAUSAL, OUT_F32, !SPARSE>(u, N, BH, n_mblocks, n_splits, kv_chunk, hg, split0);
                if (!SPARSE && w.n_kv <= 0) continue;  // a key split with no admitted key
                if constexpr (SPARSE) {
                    // a unit with no live tile: its one record goes to both softmax warpgroups
                    const int kslot = it % C::kStages, kuse = it / C::kStages;
                    if (!(ok = mbar_wait(bars.full(kslot), kuse & 1, kWaitLimitNs))) break;
                    if (kv_meta[kslot] == kMetaEmptyUnit) {
                        for (int t = 0; t < kQTiles && ok; ++t) {
                            if (!(ok = ack_token(t))) break;
                            s_meta[t] = kMetaEmptyUnit;
                            mma_commit(bars.s_full(t));
                            mbar_arrive(bars.s_full(t));
                            if (t) {
                                ++jg1;
                                tok1 = true;
                            } else {
                                ++jg0;
                                tok0 = true;
                            }
                        }
                        mma_commit(bars.empty(kslot));
                        ++it;
                        continue;
                    }
                }
                if (!(ok = mbar_wait(bars.q_full(), uc & 1, kWaitLimitNs))) break;
                tc_fence_after();
                uint32_t prev_v_lo = 0;
                int prev_v = -1;
                int jj = 0;  // K/V tiles of this unit processed so far
                const bool skip0 = tile0_skips_last<CAUSAL, OUT_F32, SPARSE>(w, N);
                bool skipped0 = false;  // query tile 0 skipped the unit's last tile
                // (block-sparse: the producer's records give the live tiles; j only counts)
                for (int j = 0; j < w.n_kv && ok; ++j) {
                    const int kslot = it % C::kStages, kuse = it / C::kStages;
                    ++it;
                    const int vslot = it % C::kStages, vuse = it / C::kStages;
                    ++it;
                    if (!(ok = mbar_wait(bars.full(kslot), kuse & 1, kWaitLimitNs))) break;
                    tc_fence_after();
                    const uint32_t meta = SPARSE ? kv_meta[kslot] : 0u;
                    const uint32_t dk_lo = static_cast<uint32_t>(dk0) + kslot * kTile16;
                    for (int t = 0; t < kQTiles && ok; ++t) {
                        if (jj > 0) {  // query tile t ran every tile before this one
                            if (!(ok = mbar_wait(bars.p_full(t), ((t == 0 ? jg0 : jg1) - 1) & 1, kWaitLimitNs))) break;
                            tc_fence_after();
#pragma unroll
                            for (int kk = 0; kk < C::kPVSteps; ++kk) {
                                const uint32_t boff = (kk * C::kPVKeys * 128) >> 4;
                                mma_ts_lohi(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, prev_v_lo + boff, dv_hi,
                                            idO, (jj > 1 || kk > 0) ? 1u : 0u);
                            }
                        }
                        // causal: the unit's last tile is fully masked for query tile 0 whenever tile 1
                        // has rows; tile 0's last P V has just been issued, so its epilogue need not
                        // wait for the rest of the unit
                        if (t == 0 && skip0 && j == w.n_kv - 1) {
                            mma_commit(bars.o_full(0));
                            skipped0 = true;
                            continue;
                        }
                        if constexpr (SPARSE) {  // this S tile's record, for the softmax (published by the arrive below)
                            if (jj == 0 && !(ok = ack_token(t))) break;
                            s_meta[t] = (meta & (kMetaTile | kMetaLast)) | (((meta >> (30 - t)) & 1u) << 30);
                        }
                        const uint32_t aq_lo = dq_lo + t * kTile16;
#pragma unroll
                        for (int kk = 0; kk < C::kSSteps; ++kk) {
                            const uint32_t koff = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                            mma_ss_lohi(tmem + t * 128, aq_lo + koff, dq_hi, dk_lo + koff, dk_hi, idS,
                                        kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bars.s_full(t));
                        if constexpr (SPARSE) mbar_arrive(bars.s_full(t));
                        if (t == 0)
                            ++jg0;
                        else
                            ++jg1;
                    }
                    if (!ok) break;
                    mma_commit(bars.empty(kslot));
                    if (jj > 0) mma_commit(bars.empty(prev_v));
                    if (!(ok = mbar_wait(bars.full(vslot), vuse & 1, kWaitLimitNs))) break;
                    tc_fence_after();
                    prev_v = vslot;
                    // d = 64: the block "after" V's 64 columns is the ones block, so the leading
                    // byte offset (bits 16..29) falls by what the start address (bits 0..13) gains
                    prev_v_lo = static_cast<uint32_t>(dv0) + vslot * (C::kOnesCol ? kTile16 - (kTile16 << 16) : kTile16);
                    ++jj;
                    if (SPARSE && (meta & kMetaLast) != 0u) break;
                }
                if (!ok) break;
                mma_commit(bars.q_empty());  // the last reads of this unit's Q are issued
                for (int t = 0; t < kQTiles && ok; ++t) {
                    if (t == 0 && skipped0) continue;  // committed with the unit's last tile
                    if (!(ok = mbar_wait(bars.p_full(t), ((t == 0 ? jg0 : jg1) - 1) & 1, kWaitLimitNs))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < C::kPVSteps; ++kk) {
                        const uint32_t boff = (kk * C::kPVKeys * 128) >> 4;
                        mma_ts_lohi(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, prev_v_lo + boff, dv_hi, idO,
                                    (jj > 1 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bars.o_full(t));
                }
                if (ok) mma_commit(bars.empty(prev_v));
                ++uc;
            }
            if (!ok) report_timeout();
            // no MMA of this CTA may still be running when tensor memory is freed
            mma_commit(bars.mma_done());
            mbar_wait(bars.mma_done(), 0, ok ? kWaitLimitNs : kCleanupLimitNs);
        }
    } else {
        // --------------------------------------------------------------- softmax
        const int t = warp >> 2;    // query tile of this warpgroup
        const int row = tid & 127;  // row within the tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * 128;
        bool ok = true;
        int jg = 0, uc = 0;
        for (int r = 0, u = unit_index(0); u < n_units && ok; u = unit_index(++r)) {
            const Unit w = unit_of<CAUSAL, OUT_F32, !SPARSE>(u, N, BH, n_mblocks, n_splits, kv_chunk, hg, split0);
            const int row_g = w.q_row0 + t * kBlockM + row;
            auto out_row_of = [&]() { return (static_cast<int64_t>(w.split) * BH + w.bh) * N + row_g; };
            const bool qb_ok = !SPARSE || (w.q_row0 / kBlockM + t < nb);
            // a unit with no admitted key in its split (or, block-sparse, in its mask rows: the
            // MMA thread's empty-unit record, acknowledged on p_full): O = 0, LSE = -inf (no
            // weight when merged)
            bool unit_live = w.n_kv > 0;
            if constexpr (SPARSE) {
                if (!mbar_wait_warp(bars.s_full(t), jg & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                unit_live = s_meta[t] != kMetaEmptyUnit;  // the first tile's record, or the empty-unit one
                if (!unit_live) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.p_full(t));
                    ++jg;
                }
            }
            if (!unit_live) {
                if (row_g < N) {
                    const int64_t out_row = out_row_of();
                    if (OUT_F32) {
                        float4 *orow = reinterpret_cast<float4 *>(static_cast<float *>(o) + out_row * D);
#pragma unroll
                        for (int i = 0; i < D / 4; ++i) orow[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
                        uint4 *orow = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o) + out_row * D);
#pragma unroll
                        for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    lse[out_row] = -INFINITY;
                }
                continue;
            }
            const float c_u = scale_log2;
            float m_ref = -INFINITY;  // reference max, unscaled units
            float l = 0.f;            // exp-sum relative to m_ref (fp32 terms; gives LSE)
            float lr = 0.f;           // the divisor of O (see the row sums below)
            int jj = 0;  // K/V tiles of this unit processed so far
            // block-sparse: the loop counts the unit's live tiles; each one's index and
            // admission bit come with its S tile (the MMA thread's record)
            const int n_mine = w.n_kv - (t == 0 && tile0_skips_last<CAUSAL, OUT_F32, SPARSE>(w, N) ? 1 : 0);
            for (int jc = 0; jc < n_mine; ++jc) {
                if (!mbar_wait_warp(bars.s_full(t), jg & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t meta = SPARSE ? s_meta[t] : 0u;
                const int j = SPARSE ? static_cast<int>(meta & kMetaTile) : jc;
                // S_t and its row max over the admitted keys
                float s[kBlockN], mt;
                const int k0 = (w.j0 + j) * kBlockN;
                const bool need_mask = k0 < w.kv_begin || k0 + kBlockN > w.kv_end ||
                                       (CAUSAL && k0 + kBlockN - 1 > w.q_row0 + t * kBlockM);
                if constexpr (SPARSE) {  // (registers at their limit: the plain load and max pass)
                    uint32_t r[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, r[c]);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[c][i]);
                    if (!qb_ok || (meta & kMetaOwn0) == 0u) {
#pragma unroll
                        for (int i = 0; i < kBlockN; ++i) s[i] = -INFINITY;  // block not admitted for this query tile
                    }
                    if (need_mask) mask_keys(s, k0, w.kv_begin, CAUSAL ? min(w.kv_end - 1, row_g) : w.kv_end - 1);
                    mt = row_max(s);
                } else {
                    // each 32-column piece's max comes with the load; a tile with masked keys
                    // takes the max again over the admitted ones
                    float pm[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_ld32_max(tS + c * 32, *reinterpret_cast<float(*)[32]>(&s[c * 32]), pm[c]);
                    tmem_wait_ld();
                    mt = fmax3(fmaxf(pm[0], pm[1]), pm[2], pm[3]);
                    if (need_mask) {
                        mask_keys(s, k0, w.kv_begin, CAUSAL ? min(w.kv_end - 1, row_g) : w.kv_end - 1);
                        mt = row_max(s);
                    }
                }
                const float m_new = fmaxf(m_ref, mt);
                const bool need = (m_new - m_ref) * c_u > kRescaleLog2;  // true while m_ref = -inf
                float alpha = 1.f;
                if (need) {
                    alpha = ex2((m_ref - m_new) * c_u);  // 0 on the first tile
                    m_ref = m_new;
                }
                // P = exp2(s * scale * log2 e - m_ref * scale * log2 e), bf16, over the first 64 columns
                // of S_t; the fp32 row sum in partial accumulators (the divisor of O: see below)
                const float mc = (m_ref == -INFINITY ? 0.f : m_ref) * c_u;
                // how the divisor of O is summed at d = 128 (see the row sums below): every
                // term inline in the key-split forward, else per tile as needed
                constexpr bool kInlineSum = !C::kOnesCol && OUT_F32;
                constexpr bool kHeavyTiles = !C::kOnesCol && !OUT_F32;
                bool heavy = false;
                if constexpr (kHeavyTiles)
                    heavy = __any_sync(0xffffffffu, ex2(fmaf(mt, c_u, -mc)) > kHeavyShare * (l * alpha));
                const float2 c2 = make_float2(c_u, c_u), nmc2 = make_float2(-mc, -mc);
                float2 lf[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 x = fma2(make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), c2, nmc2);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        p[i] = pack_bf16x2(p0, p1);
                        if constexpr (kInlineSum) {
                            lf[i & 3] = add2(lf[i & 3], make_float2(p0, p1));
                            lq[i & 3] = add_bf16x2(lq[i & 3], p[i]);
                        } else {
                            lf[c] = add2(lf[c], make_float2(p0, p1));  // one partial per chunk
                        }
                    }
                    tmem_st16(tS + c * 16, p);
                }
                const float2 lf01 = add2(lf[0], lf[1]), lf23 = add2(lf[2], lf[3]);
                const float2 lfs = add2(lf01, lf23);
                if constexpr (kInlineSum) {
                    lr = lr * alpha + ((lq[0] + lq[1]) + (lq[2] + lq[3]));
                } else if constexpr (kHeavyTiles) {
                    // d = 128: O is divided by lr, which must be the sum of the rounded P the
                    // MMA sees wherever few keys carry a row (a mismatch of the rounding step
                    // on a top weight shows in O: 2^-9), while over many comparable keys the
                    // fp32 sum's rounding differences average out.  So the exact rounded sum
                    // is taken only in "heavy" tiles, where for some row of the warp the
                    // tile's largest P exceeds kHeavyShare of the row's running sum (always
                    // the unit's first tile): P is read back from tensor memory and summed
                    // exactly (mixed-precision adds).  Any key whose final weight
                    // exceeds kHeavyShare lies in a heavy tile.  Light tiles add their fp32
                    // sum.  (d = 64 gets the rounded sum from the MMA, column 64 of O; the
                    // key-split forward, whose variants run out of registers with this
                    // branch, sums every rounded term inline.)
                    float add = lfs.x + lfs.y;
                    if (heavy) {  // 64 columns of two bf16 each
                        tmem_wait_st();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t r[32];
                            tmem_ld32(tS + h * 32, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) lq[i & 3] = add_bf16x2(lq[i & 3], r[i]);
                        }
                        add = (lq[0] + lq[1]) + (lq[2] + lq[3]);
                    }
                    lr = lr * alpha + add;
                }
                l = l * alpha + (lfs.x + lfs.y);
                // numerator rescale u *= alpha (u holds P V up to the previous tile, complete:
                // the commit that signalled this S was issued after that MMA); nothing to
                // scale on the unit's first tile
                if (jj > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 y = mul2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                                  make_float2(alpha, alpha));
                            r[i] = __float_as_uint(y.x);
                            r[i + 1] = __float_as_uint(y.y);
                        }
                        tmem_st32(tO + c * 32, r);
                    }
                    if constexpr (C::kOnesCol) {  // the rounded row sum in column 64
                        const float lc = __uint_as_float(tmem_ld1(tO + 64));
                        tmem_wait_ld();
                        tmem_st1(tO + 64, __float_as_uint(lc * alpha));
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.p_full(t));
                ++jg;
                ++jj;
                if (SPARSE && (meta & kMetaLast) != 0u) break;
            }
            if (!ok || !(ok = mbar_wait_warp(bars.o_full(t), uc & 1, kWaitLimitNs))) break;
            tc_fence_after();
            // epilogue: O = u / lr in bf16 (fp32 for the key-split forward) straight
            // from registers to global memory, LSE from the fp32 sum l.  u was built
            // from the rounded P; lr sums those same rounded terms wherever one key
            // can carry the row (see the row sums above; d = 64: column 64 of O), so
            // such a row returns its key's value without a P-rounding error.  The next
            // unit's first P V (which overwrites O_t) is issued only after this
            // warpgroup's next p_full arrive, so the reads here are safe.  A row with
            // no admitted key in this split has l = 0: O = 0, LSE = -inf.
            if constexpr (C::kOnesCol) {
                lr = __uint_as_float(tmem_ld1(tO + 64));
                tmem_wait_ld();
            }
            const int64_t out_row = out_row_of();
            const float inv_l = lr > 0.f ? 1.f / lr : 0.f;
            if constexpr (OUT_F32) {
                // the fp32 partials of a key split store straight from registers
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32, r);
                    tmem_wait_ld();
                    if (row_g < N) {
                        float4 *orow = reinterpret_cast<float4 *>(static_cast<float *>(o) + out_row * D + c * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            orow[q4] = make_float4(__uint_as_float(r[q4 * 4 + 0]) * inv_l, __uint_as_float(r[q4 * 4 + 1]) * inv_l,
                                                   __uint_as_float(r[q4 * 4 + 2]) * inv_l, __uint_as_float(r[q4 * 4 + 3]) * inv_l);
                    }
                }
            } else {
                // 32-column chunks through this warp's two 2 KB staging buffers: 32 rows of
                // 64 bytes in the 64-byte swizzle (16-byte piece q of row r at q ^ ((r >> 1) & 3)),
                // one TMA store per chunk; a buffer is refilled once the store issued from it
                // two chunks earlier (or in the previous unit) has been read
                // (the address is rebuilt here rather than kept live through the softmax loop)
                const uint32_t stage = ((smem_u32(smem_raw) + 1023u) & ~1023u) + C::kStageOffset + warp * 4096;
                const int row0 = w.q_row0 + t * kBlockM + (warp & 3) * 32;
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32, r);
                    tmem_wait_ld();
                    if (c >= 2) {
                        if (lane == 0) bulk_wait_read1();
                        __syncwarp();
                    }
                    const uint32_t buf = stage + (c & 1) * 2048 + lane * 64;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * inv_l, __uint_as_float(r[q4 * 8 + 1]) * inv_l);
                        v.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * inv_l, __uint_as_float(r[q4 * 8 + 3]) * inv_l);
                        v.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * inv_l, __uint_as_float(r[q4 * 8 + 5]) * inv_l);
                        v.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * inv_l, __uint_as_float(r[q4 * 8 + 7]) * inv_l);
                        st_shared_v4(buf + ((q4 ^ ((lane >> 1) & 3)) << 4), v);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < N) {
                        tma_store_3d(&tm_o, stage + (c & 1) * 2048, c * 32, row0, w.bh);
                        bulk_commit();
                    }
                }
            }
            if (row_g < N) lse[out_row] = l > 0.f ? m_ref * scale + logf(l) : -INFINITY;
            ++uc;
        }
        if (!ok) report_timeout();
        if (!OUT_F32 && lane == 0) bulk_wait0();  // every O store of this warp has completed
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

// kv_rows: rows of K and V per slice (N unless they hold one sequence shard:
// the keys of splits split0 .. split0 + n_splits - 1 only; 0 for a shard past
// the last key, whose K and V are never read).
template <int D, bool CAUSAL, bool OUT_F32, bool SPARSE = false>
cudaError_t launch(const FaProblem &p, void *o, float *lse, int n_splits, int kv_chunk, cudaStream_t stream,
                   const uint8_t *bm = nullptr, int split0 = 0, int64_t kv_rows = -1)
{
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv, mo;
    const int64_t BH = p.B * p.H;
    if (kv_rows < 0) kv_rows = p.N;
    if (!make_map(&mq, p.q, BH, p.N, D, C::kElem)) return cudaErrorInvalidValue;
    if (kv_rows == 0) {
        mk = mq;
        mv = mq;
    } else if (!make_map(&mk, p.k, BH, kv_rows, D, C::kElem) || !make_map(&mv, p.v, BH, kv_rows, D, C::kElem)) {
        return cudaErrorInvalidValue;
    }
    if (OUT_F32)
        mo = mq;  // not used: the key-split partials store O directly
    else if (!make_out_map(&mo, o, BH, p.N, D))
        return cudaErrorInvalidValue;
    auto kern = fa_fwd_tc_kernel<D, CAUSAL, OUT_F32, SPARSE>;
    cudaError_t e = set_max_dynamic_smem<fa_fwd_tc_kernel<D, CAUSAL, OUT_F32, SPARSE>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t n_mblocks = (p.N + kQTiles * kBlockM - 1) / (kQTiles * kBlockM);
    const int64_t n_units = n_mblocks * BH * n_splits;
    if (n_units > 0x7fffffffLL || BH > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int64_t grid = n_units < p.sm_count ? n_units : p.sm_count;  // persistent: one CTA per SM
    // slices per group: when the K and V of all slices exceed 160 MB (L2: 129 MB),
    // groups whose K and V take about 64 MB; else one group (grouping a working
    // set that L2 already holds, or the few tiles a block-sparse unit reads, only
    // costs balance)
    const int64_t kv_bytes = 2 * p.N * p.d * C::kElem;
    int64_t hg = BH;
    if (!SPARSE && BH * kv_bytes > (int64_t(160) << 20)) {
        hg = (int64_t(64) << 20) / kv_bytes;
        hg = hg < 1 ? 1 : (hg > BH ? BH : hg);
    }
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(
        mq, mk, mv, mo, o, lse, static_cast<int>(p.N), static_cast<int>(BH), static_cast<int>(n_mblocks),
        static_cast<int>(n_units), n_splits, kv_chunk, static_cast<int>(hg), p.scale, scale_log2, bm,
        static_cast<int>((p.N + kBlockN - 1) / kBlockN), split0);
    return cudaGetLastError();
}

template <bool OUT_F32>
cudaError_t dispatch(const FaProblem &p, void *o, float *lse, int n_splits, int kv_chunk, cudaStream_t s,
                     int split0 = 0, int64_t kv_rows = -1)
{
    if (p.d == 64)
        return p.causal ? launch<64, true, OUT_F32>(p, o, lse, n_splits, kv_chunk, s, nullptr, split0, kv_rows)
                        : launch<64, false, OUT_F32>(p, o, lse, n_splits, kv_chunk, s, nullptr, split0, kv_rows);
    return p.causal ? launch<128, true, OUT_F32>(p, o, lse, n_splits, kv_chunk, s, nullptr, split0, kv_rows)
                    : launch<128, false, OUT_F32>(p, o, lse, n_splits, kv_chunk, s, nullptr, split0, kv_rows);
}

}  // namespace

bool fa_fwd_takes_dp(int64_t N, int64_t d, int causal)
{
    if (d != 64) return false;
    // The d = 64 kernel (P apart from S, Q double-buffered) wins where units are
    // short and their start and end weigh; the forward above (ones column, P over
    // S) wins on long units.  Measured on one GB300: 378 against 332 TFLOP/s at
    // N = 512 causal, 482 / 467 at N = 1000 causal, 711 / 684 at N = 2048 causal,
    // 833 / 840 at N = 4096 causal, 907 / 955 at N = 16384 causal; non-causal
    // 683 / 618 at N = 512, equal at N = 1000, 861 / 869 at N = 2048.  The
    // switch is at a mean of 9 K/V tiles per 256-row unit.
    const int64_t nt = (N + kBlockN - 1) / kBlockN;
    const int64_t n_mblocks = (N + kQTiles * kBlockM - 1) / (kQTiles * kBlockM);
    int64_t tiles = 0;
    for (int64_t mb = 0; mb < n_mblocks; ++mb) tiles += causal ? std::min(nt, 2 * (mb + 1)) : nt;
    return tiles <= 9 * n_mblocks;
}

cudaError_t fa_launch_tc(const FaProblem &p, cudaStream_t stream)
{
    if (fa_fwd_takes_dp(p.N, p.d, p.causal)) return fa_launch_dp(p, stream);
    return dispatch<false>(p, p.o, p.lse, 1, static_cast<int>(p.N), stream);
}

cudaError_t fa_launch_tc_partials(const FaProblem &p, float *o_parts, float *lse_parts, int n_splits, int kv_chunk,
                                  cudaStream_t stream, int split0, int64_t kv_rows)
{
    return dispatch<true>(p, o_parts, lse_parts, n_splits, kv_chunk, stream, split0, kv_rows);
}

cudaError_t fa_launch_tc_sparse(const FaProblem &p, const uint8_t *block_mask, cudaStream_t stream)
{
    const int N = static_cast<int>(p.N);
    if (p.d == 64)
        return p.causal ? launch<64, true, false, true>(p, p.o, p.lse, 1, N, stream, block_mask)
                        : launch<64, false, false, true>(p, p.o, p.lse, 1, N, stream, block_mask);
    return p.causal ? launch<128, true, false, true>(p, p.o, p.lse, 1, N, stream, block_mask)
                    : launch<128, false, false, true>(p, p.o, p.lse, 1, N, stream, block_mask);
}

int fa_tc_take_status(cudaStream_t stream)
{
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_tc_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    return h;
}
