// fa_fwd_splitkv_noalloc: the split-KV forward with its scratch in a fixed,
// library-owned device array instead of a caller workspace.
//
// Why it exists: some host programs cannot allocate device memory at the
// point where they call attention.  Inference engines that plan every device
// buffer at start-up and forbid allocation afterwards, plugins whose host
// application owns the device allocator and hands over only the input and
// output tensors, and latency-critical loops where a cudaMalloc (which can
// synchronise the whole device) is not acceptable all fall in this group.
// They can pass their inputs and outputs and nothing else.
//
// How: the per-range partial results live in g_splitkv_scratch, a file-scope
// static device array of kScratchBytes bytes.  Every GPU that loads this
// library keeps that array for the life of the process.  Host code cannot
// use the array's name as a device address, so the first call on each device
// (with that device current) looks the address up with cudaGetSymbolAddress
// and caches it; make that first call before any stream capture.  No call
// allocates or frees device memory.
//
// Every call on a device shares the one array and leaves its parts in it.
// Nothing in it needs to start at zero: every call writes each part it reads.
// Calls whose kernels overlap on the GPU (for example on two streams without
// ordering between them) race on the array and give undefined results.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int64_t kScratchBytes = FA_SPLITKV_NOALLOC_MAX_BYTES;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once per device).
int scratch_address(int dev, void **addr)
{
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FA_ERR_LAUNCH;
        }
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return FA_OK;
}

bool overlap(const void *a, uint64_t na, const void *b, uint64_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                                      int64_t H, int64_t N, int64_t d, float scale, int causal, int64_t n_splits,
                                      void *stream)
{
    // the size rule is fa_fwd_splitkv's; beyond the array the call is refused
    const int64_t need = fa_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits);
    if (need < 0) return (d >= 1 && d != 64 && d != 128 && B >= 1 && H >= 1 && N >= 1) ? FA_ERR_UNSUPPORTED
                                                                                          : FA_ERR_INVALID_ARG;
    if (need > kScratchBytes) return FA_ERR_WORKSPACE_LIMIT;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
    }
    void *scratch = nullptr;
    const int st = scratch_address(dev, &scratch);
    if (st != FA_OK) return st;
    // inputs and outputs are the caller's and can never be the library's array,
    // but a pointer into it (from an earlier misuse) is refused all the same
    for (const void *p : {q, k, v, static_cast<const void *>(o), static_cast<const void *>(lse)})
        if (p != nullptr && overlap(p, 1, scratch, static_cast<uint64_t>(kScratchBytes))) return FA_ERR_INVALID_ARG;
    return fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, n_splits, scratch, kScratchBytes, stream);
}
