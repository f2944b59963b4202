// Internal launch interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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
cudaError_t fa_launch_tc(const FaProblem &p, cudaStream_t stream);
// Read and clear the tcgen05 kernel's sticky device status (synchronises `stream`).
int fa_tc_take_status(cudaStream_t stream);

// Warp-level tensor-core (mma.sync) kernel: one CTA per 128-row query tile.
cudaError_t fa_launch_mma(const FaProblem &p, cudaStream_t stream);
