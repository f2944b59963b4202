// Shared by the forward kernels (fa_fwd_tc.cu, fa_fwd_dp.cu): tile sizes and
// warp roles, the persistent work order over (b, h) slices and 256-row units,
// and the TMA tensor maps of Q, K, V and O.  Everything here is internal
// linkage (an anonymous namespace), one copy per translation unit.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace {

constexpr int kBlockM = 128;  // query rows per query tile
constexpr int kBlockN = 128;  // keys per K/V tile
constexpr int kQTiles = 2;    // query tiles per CTA
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleLog2 = 8.0f;            // rescale when the max grows by more than 2^8
constexpr float kHeavyShare = 0.25f;            // d = 128: see "heavy" in the softmax
constexpr uint64_t kWaitLimitNs = 1000000000ull;    // 1 s per pipeline wait
constexpr uint64_t kCleanupLimitNs = 20000000ull;    // 20 ms per wait while winding down

// Work item u: 256 consecutive query rows of one (b, h) slice against one key
// split (keys [split * kv_chunk, (split + 1) * kv_chunk), a multiple of 128;
// a single split covers all keys).  Items are ordered by row block, heaviest
// causal block first, then by split.  Without key splits (and without a block
// mask) the (b, h) slices go in groups of `hg` (all of one group's items before
// the next group's), sized so that a group's K and V stay in L2 while its items
// run.  CTA c of a persistent grid of G CTAs
// takes, in round r, item r*G + c when r is even and r*G + (G-1-c) when r is
// odd: the zigzag pairs heavy items with light ones, so every CTA ends up with
// about the same number of K/V tiles without a shared counter.
struct Unit {
    int bh, q_row0, split, kv_begin, kv_end, j0, n_kv;
};

__device__ __forceinline__ int unit_index(int r)
{
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// SPLIT: the launch covers key splits split0 .. split0 + n_splits - 1 (the
// split-KV partials; split0 > 0 when one GPU computes one split of a sequence
// sharded over several); otherwise every item spans all N keys, and the split
// fields are compile-time constants, so the single-split variants carry none of
// the key-range arithmetic.  `split` is the index within the launch.
template <bool CAUSAL, bool SPLIT, bool GROUPED>
__device__ __forceinline__ Unit unit_of(int u, int N, int BH, int n_mblocks, int n_splits, int kv_chunk, int hg,
                                        int split0 = 0)
{
    Unit w;
    if constexpr (!SPLIT) {
        int mb;
        if constexpr (GROUPED) {
            // group g holds slices [g hg, min(BH, (g + 1) hg)); every group before it is full
            const int g = u / (hg * n_mblocks), r = u - g * hg * n_mblocks;
            const int nh = min(hg, BH - g * hg);
            mb = CAUSAL ? (n_mblocks - 1 - r / nh) : (r / nh);
            w.bh = g * hg + r % nh;
        } else {
            mb = CAUSAL ? (n_mblocks - 1 - u / BH) : (u / BH);
            w.bh = u % BH;
        }
        w.q_row0 = mb * (kQTiles * kBlockM);
        w.split = 0;
        w.kv_begin = 0;
        w.kv_end = N;
        w.j0 = 0;
        const int k_hi = CAUSAL ? min(N, w.q_row0 + kQTiles * kBlockM) : N;
        w.n_kv = (k_hi + kBlockN - 1) / kBlockN;
        return w;
    }
    const int rb = u / n_splits;  // row-block unit
    w.split = u - rb * n_splits;
    const int mb = CAUSAL ? (n_mblocks - 1 - rb / BH) : (rb / BH);
    w.bh = rb % BH;
    w.q_row0 = mb * (kQTiles * kBlockM);
    w.kv_begin = (split0 + w.split) * kv_chunk;
    w.kv_end = min(N, w.kv_begin + kv_chunk);
    // keys any row of this block admits end before k_hi
    const int k_hi = CAUSAL ? min(w.kv_end, w.q_row0 + kQTiles * kBlockM) : w.kv_end;
    w.j0 = w.kv_begin / kBlockN;
    w.n_kv = k_hi > w.kv_begin ? (k_hi + kBlockN - 1) / kBlockN - w.j0 : 0;
    return w;
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

// bf16 O [BH][N][d] as a 3-D tensor for the epilogue's TMA stores: box = 32
// columns (64 bytes) x 32 rows x 1 slice, 64-byte swizzle.
bool make_out_map(CUtensorMap *m, void *base, int64_t BH, int64_t N, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// [BH][N][d] (bf16, or E4M3 as bytes) viewed as a 3-D tensor (d fastest);
// box = 128 bytes of columns x 128 rows x 1 slice.
bool make_map(CUtensorMap *m, const void *base, int64_t BH, int64_t N, int d, int elem = 2)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem, static_cast<cuuint64_t>(N) * d * elem};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem), 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
