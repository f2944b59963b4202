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
// use the array's name as a device address: the address belongs to the CUDA
// context current at the call (the device's primary context, or one the host
// program made with the driver API), and it changes when a context is
// destroyed and made again (cudaDeviceReset).  So every call made outside a
// stream capture looks the address up with cudaGetSymbolAddress in the
// current context and records it for that context; a call made while its
// stream is being captured uses the address recorded for the current context
// (the lookup itself may not be legal during a capture), which is why a first
// call on each device and context must come before any stream capture, and
// again after a cudaDeviceReset.  No call allocates or frees device memory.
//
// Every call on a device shares the one array and leaves its parts in it.
// Nothing in it needs to start at zero: every call writes each part it reads.
// Calls whose kernels overlap on the GPU (for example on two streams without
// ordering between them) race on the array and give undefined results.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int64_t kScratchBytes = FA_SPLITKV_NOALLOC_MAX_BYTES;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

// Scratch address per CUDA context (contexts are few: one primary context per
// device, plus any the host program creates); the oldest entry is reused.
constexpr int kMaxContexts = 64;
struct ScratchEntry {
    CUcontext ctx;
    void *addr;
};
ScratchEntry g_entries[kMaxContexts];
int g_next_entry = 0;
std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Device address of the scratch array in the current context: looked up
// afresh unless `stream` is being captured, when the address recorded for
// this context by an earlier call is used.
int scratch_address(cudaStream_t stream, void **addr)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    const bool capturing = cs != cudaStreamCaptureStatusNone;
    void *p = nullptr;
    if (!capturing && (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr)) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get == nullptr || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return FA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    int found = -1;
    for (int i = 0; i < kMaxContexts; ++i)
        if (g_entries[i].ctx == ctx) found = i;
    if (capturing) {
        if (found < 0) return FA_ERR_LAUNCH;  // no call in this context before the capture
        *addr = g_entries[found].addr;
        return FA_OK;
    }
    if (found < 0) {
        found = g_next_entry;
        g_next_entry = (g_next_entry + 1) % kMaxContexts;
    }
    g_entries[found] = ScratchEntry{ctx, p};
    *addr = p;
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
    // the argument rules and their order are fa_fwd_splitkv's; a valid problem
    // whose parts do not fit the array is refused before anything else is done
    const int st_sizes = fa_check_sizes(B, H, N, d);
    if (st_sizes != FA_OK) return st_sizes;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (n_splits < 1 || n_splits > kFaMaxSplits) return FA_ERR_INVALID_ARG;
    if (fa_splitkv_bytes(B, H, N, d, n_splits) > kScratchBytes) return FA_ERR_WORKSPACE_LIMIT;
    void *scratch = nullptr;
    const int st = scratch_address(static_cast<cudaStream_t>(stream), &scratch);
    if (st != FA_OK) return st;
    // inputs and outputs are the caller's and can never be the library's array,
    // but a pointer into it (from an earlier misuse) is refused all the same
    for (const void *p : {q, k, v, static_cast<const void *>(o), static_cast<const void *>(lse)})
        if (p != nullptr && overlap(p, 1, scratch, static_cast<uint64_t>(kScratchBytes))) return FA_ERR_INVALID_ARG;
    return fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, n_splits, scratch, kScratchBytes, stream);
}
