// Internal launch interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

// cudaFuncSetAttribute(Kernel, MaxDynamicSharedMemorySize, bytes), made once per
// kernel and device (bit d of `done` records device d) instead of on every launch.
template <auto Kernel>
cudaError_t set_max_dynamic_smem(int bytes)
{
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Size rules shared by the entry points (pure host logic, no CUDA call):
// FA_OK, FA_ERR_INVALID_ARG (sizes out of range) or FA_ERR_UNSUPPORTED (d).
int fa_check_sizes(int64_t B, int64_t H, int64_t N, int64_t d);
// Largest n_splits of fa_fwd_splitkv (and n_parts of fa_combine).
constexpr int64_t kFaMaxSplits = 32;
// Key-split geometry of fa_fwd_splitkv: chunks of a multiple of 128 keys, no empty chunk.
void fa_split_geometry(int64_t N, int64_t n_splits, int64_t *chunk, int64_t *parts);
// Workspace bytes of fa_fwd_splitkv for valid sizes and n_splits.
int64_t fa_splitkv_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int64_t n_splits);

// One validated forward problem: contiguous [B, H, N, d] bf16 tensors.
struct FaProblem {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int64_t B, H, N;
    int d;
    float scale;
    int causal;
    int sm_count;  // SMs on the current device
};

// tcgen05 kernel (TMA, tensor memory, warp-specialised): 256 query rows per CTA.
// At d = 64 it hands problems of short units to fa_launch_dp (fa_fwd_takes_dp).
cudaError_t fa_launch_tc(const FaProblem &p, cudaStream_t stream);
bool fa_fwd_takes_dp(int64_t N, int64_t d, int causal);
// The same kernel over n_splits key ranges of kv_chunk keys (a multiple of
// 128): split s (keys from (split0 + s) * kv_chunk) writes fp32 O to
// o_parts + s*B*H*N*d and LSE to lse_parts + s*B*H*N.  K and V hold kv_rows rows
// per slice starting at key split0 * kv_chunk (default: all N keys, split0 = 0).
cudaError_t fa_launch_tc_partials(const FaProblem &p, float *o_parts, float *lse_parts, int n_splits, int kv_chunk,
                                  cudaStream_t stream, int split0 = 0, int64_t kv_rows = -1);
// The same kernel restricted by a [ceil(N/128)]^2 0/1 block mask over (query block, key block).
cudaError_t fa_launch_tc_sparse(const FaProblem &p, const uint8_t *block_mask, cudaStream_t stream);
// The kernel with P apart from S (fa_fwd_dp.cu): bf16 at d = 64 (taken by
// fa_launch_tc for short units), and E4M3 Q, K, V at d = 128 with per-(b, h)
// fp32 scales qs, ks, vs.
cudaError_t fa_launch_dp(const FaProblem &p, cudaStream_t stream);
cudaError_t fa_launch_fp8(const FaProblem &p, const float *qs, const float *ks, const float *vs,
                          cudaStream_t stream);
// Read and clear that kernel's sticky device status (synchronises `stream`).
int fa_dp_take_status(cudaStream_t stream);
// Merge of n_parts partial (O fp32, LSE) results of `rows` rows into bf16 O and LSE.
cudaError_t fa_launch_combine(const float *o_parts, const float *lse_parts, int n_parts, int64_t rows, int d,
                              void *o, float *lse, int sm_count, cudaStream_t stream);
// Read and clear the tcgen05 kernel's sticky device status (synchronises `stream`).
int fa_tc_take_status(cudaStream_t stream);

// One validated backward problem: gradients of sum(O * dO).
struct FaBwdProblem {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int64_t B, H, N;
    int d;
    float scale;
    int causal;
    int sm_count;
};
// Workspace bytes of the backward: fp32 dQ accumulator and two padded fp32 row vectors.
int64_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d);
// Pre (D, LSE log2 e, zero accumulator) + tcgen05 main kernel + post (dQ to bf16).
cudaError_t fa_launch_bwd(const FaBwdProblem &p, void *workspace, cudaStream_t stream);
// Read and clear the backward kernel's sticky device status (synchronises `stream`).
int fa_bwd_take_status(cudaStream_t stream);

// Warp-level tensor-core (mma.sync) kernel: one CTA per 128-row query tile.
cudaError_t fa_launch_mma(const FaProblem &p, cudaStream_t stream);

// Forward on host buffers (fa_fwd_host): q, k, v, o, lse are host pointers,
// *_dev the caller's device staging buffers of the same shapes; the (b, h)
// slices go in n_groups consecutive groups whose copies in, forward and
// copies out are pipelined across two internal copy streams and `stream`.
struct FaHostProblem {
    const void *q, *k, *v;
    void *o;
    float *lse;
    void *q_dev, *k_dev, *v_dev, *o_dev;
    float *lse_dev;
    int64_t B, H, N;
    int d;
    float scale;
    int causal;
    int n_groups;
    int sm_count;
};
// Enqueue the pipeline; returns an fa_status.
int fa_run_host_pipeline(const FaHostProblem &p, cudaStream_t stream);
