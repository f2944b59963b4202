// C ABI of libfa.so: argument validation, device checks and kernel dispatch.
// The operation and every argument are documented in include/fa.h.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool checked = false;
    int status = FA_OK;  // FA_OK or FA_ERR_ARCH
    int sm_count = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

int current_device(int *dev, int *sm_count)
{
    if (cudaGetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
    }
    if (*dev < 0 || *dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_devices_mu);
    DeviceInfo &info = g_devices[*dev];
    if (!info.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_NO_DEVICE;
        }
        info.status = (major == 10 && minor == 3) ? FA_OK : FA_ERR_ARCH;
        info.sm_count = sms;
        info.checked = true;
    }
    *sm_count = info.sm_count;
    return info.status;
}

// A pointer the kernels may dereference: device (or managed) memory of the
// current device, aligned to `align` bytes (16 unless the kernels only make
// scalar 4-byte accesses through it).
int check_pointer(const void *p, int dev, uintptr_t align = 16)
{
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & (align - 1)) != 0) return FA_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return FA_ERR_INVALID_ARG;
    if (a.device != dev) return FA_ERR_NO_DEVICE;
    return FA_OK;
}

// A host pointer the copies may read or write: pinned or pageable host memory.
int check_host_pointer(const void *p)
{
    if (p == nullptr) return FA_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_INVALID_ARG;
    }
    return (a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered) ? FA_OK : FA_ERR_INVALID_ARG;
}

bool overlaps(const void *a, uint64_t na, const void *b, uint64_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

typedef cudaError_t (*Launcher)(const FaProblem &, cudaStream_t);

}  // namespace

int fa_check_sizes(int64_t B, int64_t H, int64_t N, int64_t d)
{
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (N > (int64_t(1) << 31) - 256 || B > (int64_t(1) << 31) || H > (int64_t(1) << 31))
        return FA_ERR_INVALID_ARG;
    if (B * H > (int64_t(1) << 40) / N || B * H * N > (int64_t(1) << 40) / d) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

void fa_split_geometry(int64_t N, int64_t n_splits, int64_t *chunk, int64_t *parts)
{
    const int64_t per = (N + n_splits - 1) / n_splits;
    *chunk = (per + 127) / 128 * 128;
    *parts = (N + *chunk - 1) / *chunk;
}

int64_t fa_splitkv_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int64_t n_splits)
{
    int64_t chunk, parts;
    fa_split_geometry(N, n_splits, &chunk, &parts);
    return parts * B * H * N * (d + 1) * 4;
}

namespace {

int validate_and_launch(Launcher launch, const void *q, const void *k, const void *v, void *o, float *lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal, void *stream)
{
    // sizes first: nothing is touched for an invalid problem
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;

    int dev = 0, sm_count = 0;
    st = current_device(&dev, &sm_count);
    if (st != FA_OK) return st;
    const void *ptrs[4] = {q, k, v, o};
    for (const void *p : ptrs)
        if ((st = check_pointer(p, dev)) != FA_OK) return st;
    if ((st = check_pointer(lse, dev, 4)) != FA_OK) return st;  // written by scalar stores only

    const uint64_t tbytes = static_cast<uint64_t>(B * H * N * d) * 2u;
    const uint64_t lbytes = static_cast<uint64_t>(B * H * N) * 4u;
    if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    for (const void *in : {q, k, v})
        if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes)) return FA_ERR_INVALID_ARG;

    FaProblem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.sm_count = sm_count;
    const cudaError_t e = launch(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return FA_ERR_LAUNCH;
    return FA_OK;
}

}  // namespace

extern "C" int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                      int64_t H, int64_t N, int64_t d, float scale, int causal, void *stream)
{
    return validate_and_launch(fa_launch_tc, q, k, v, o, lse, B, H, N, d, scale, causal, stream);
}

extern "C" int fa_fwd_kernel(int64_t B, int64_t H, int64_t N, int64_t d, int causal, int *kernel)
{
    const int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if ((causal != 0 && causal != 1) || kernel == nullptr) return FA_ERR_INVALID_ARG;
    *kernel = fa_fwd_takes_dp(N, d, causal) ? FA_FWD_KERNEL_DP : FA_FWD_KERNEL_TC;
    return FA_OK;
}

extern "C" int fa_bh_partition(int64_t n_slices, int64_t world, int64_t rank, int64_t *begin, int64_t *count)
{
    if (n_slices < 0 || world < 1 || rank < 0 || rank >= world || begin == nullptr || count == nullptr)
        return FA_ERR_INVALID_ARG;
    // the first n_slices % world ranks take one slice more than the others
    const int64_t base = n_slices / world, extra = n_slices % world;
    *begin = rank * base + (rank < extra ? rank : extra);
    *count = base + (rank < extra ? 1 : 0);
    return FA_OK;
}

extern "C" int fa_fwd_slab(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                           int64_t H, int64_t N, int64_t d, float scale, int causal, int64_t rank, int64_t world,
                           void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    int64_t begin = 0, count = 0;
    if ((st = fa_bh_partition(B * H, world, rank, &begin, &count)) != FA_OK) return st;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (count == 0) return FA_OK;  // more ranks than slices: nothing for this one
    // the slab is itself a contiguous problem of `count` slices: B = 1, H = count
    const int64_t t_off = begin * N * d * 2, l_off = begin * N;
    auto at = [&](const void *p) { return static_cast<const void *>(static_cast<const char *>(p) + t_off); };
    return validate_and_launch(fa_launch_tc, q ? at(q) : q, k ? at(k) : k, v ? at(v) : v,
                               o ? const_cast<void *>(at(o)) : o, lse ? lse + l_off : lse, 1, count, N, d, scale,
                               causal, stream);
}

extern "C" int fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, void *q_dev,
                           void *k_dev, void *v_dev, void *o_dev, float *lse_dev, int64_t B, int64_t H, int64_t N,
                           int64_t d, float scale, int causal, int64_t n_groups, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    const int64_t BH = B * H;
    // default: 8 groups (on one GB300, the 1x32x16384x128 causal step took 3.01 /
    // 2.59 / 2.51 / 2.41 / 2.47 / 3.17 ms with 2 / 4 / 6 / 8 / 12 / 16 groups)
    if (n_groups == 0) n_groups = BH < 8 ? BH : 8;
    if (n_groups < 1 || n_groups > BH || n_groups > 64) return FA_ERR_INVALID_ARG;

    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    const void *dptrs[5] = {q_dev, k_dev, v_dev, o_dev, lse_dev};
    for (const void *p : dptrs)
        if ((st = check_pointer(p, dev)) != FA_OK) return st;
    const void *hptrs[5] = {q, k, v, o, lse};
    for (const void *p : hptrs)
        if ((st = check_host_pointer(p)) != FA_OK) return st;
    // outputs may overlap nothing; the device staging buffers may not overlap one another
    const uint64_t tbytes = static_cast<uint64_t>(BH * N * d) * 2u;
    const uint64_t lbytes = static_cast<uint64_t>(BH * N) * 4u;
    if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    for (const void *in : {q, k, v})
        if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes)) return FA_ERR_INVALID_ARG;
    const void *dev_t[4] = {q_dev, k_dev, v_dev, o_dev};
    for (int i = 0; i < 4; ++i) {
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(dev_t[i], tbytes, dev_t[j], tbytes)) return FA_ERR_INVALID_ARG;
        if (overlaps(dev_t[i], tbytes, lse_dev, lbytes)) return FA_ERR_INVALID_ARG;
    }

    FaHostProblem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.q_dev = q_dev;
    p.k_dev = k_dev;
    p.v_dev = v_dev;
    p.o_dev = o_dev;
    p.lse_dev = lse_dev;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.n_groups = static_cast<int>(n_groups);
    p.sm_count = sm_count;
    return fa_run_host_pipeline(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_fwd_mma(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                          int64_t H, int64_t N, int64_t d, float scale, int causal, void *stream)
{
    return validate_and_launch(fa_launch_mma, q, k, v, o, lse, B, H, N, d, scale, causal, stream);
}

extern "C" int64_t fa_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int64_t n_splits)
{
    if (fa_check_sizes(B, H, N, d) != FA_OK || n_splits < 1 || n_splits > kFaMaxSplits) return -1;
    return fa_splitkv_bytes(B, H, N, d, n_splits);
}

extern "C" int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                              int64_t H, int64_t N, int64_t d, float scale, int causal, int64_t n_splits,
                              void *workspace, int64_t workspace_bytes, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (n_splits < 1 || n_splits > kFaMaxSplits) return FA_ERR_INVALID_ARG;
    const int64_t need = fa_splitkv_bytes(B, H, N, d, n_splits);
    if (workspace_bytes < need) return FA_ERR_INVALID_ARG;

    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    const void *ptrs[6] = {q, k, v, o, lse, workspace};
    for (const void *p : ptrs)
        if ((st = check_pointer(p, dev)) != FA_OK) return st;
    const uint64_t tbytes = static_cast<uint64_t>(B * H * N * d) * 2u;
    const uint64_t lbytes = static_cast<uint64_t>(B * H * N) * 4u;
    if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    for (const void *in : {q, k, v})
        if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes) ||
            overlaps(workspace, static_cast<uint64_t>(need), in, tbytes))
            return FA_ERR_INVALID_ARG;
    if (overlaps(workspace, static_cast<uint64_t>(need), o, tbytes) ||
        overlaps(workspace, static_cast<uint64_t>(need), lse, lbytes))
        return FA_ERR_INVALID_ARG;

    FaProblem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.sm_count = sm_count;
    int64_t chunk, parts;
    fa_split_geometry(N, n_splits, &chunk, &parts);
    const int64_t rows = B * H * N;
    float *o_parts = static_cast<float *>(workspace);
    float *lse_parts = o_parts + parts * rows * d;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fa_launch_tc_partials(p, o_parts, lse_parts, static_cast<int>(parts), static_cast<int>(chunk), s) !=
            cudaSuccess ||
        fa_launch_combine(o_parts, lse_parts, static_cast<int>(parts), rows, p.d, o, lse, sm_count, s) != cudaSuccess)
        return FA_ERR_LAUNCH;
    return FA_OK;
}

extern "C" int fa_kv_shard(int64_t N, int64_t world, int64_t rank, int64_t *begin, int64_t *count)
{
    if (N < 1 || world < 1 || world > kFaMaxSplits || rank < 0 || rank >= world || begin == nullptr ||
        count == nullptr)
        return FA_ERR_INVALID_ARG;
    // the key ranges of fa_fwd_splitkv with world splits; ranks past the last key get none
    int64_t chunk, parts;
    fa_split_geometry(N, world, &chunk, &parts);
    const int64_t b = rank * chunk;
    *begin = b < N ? b : N;
    *count = b < N ? (N - b < chunk ? N - b : chunk) : 0;
    return FA_OK;
}

extern "C" int fa_fwd_kv_shard(const void *q, const void *k_shard, const void *v_shard, float *o_part,
                               float *lse_part, int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                               int64_t rank, int64_t world, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    int64_t begin = 0, count = 0;
    if ((st = fa_kv_shard(N, world, rank, &begin, &count)) != FA_OK) return st;
    int64_t chunk, parts;
    fa_split_geometry(N, world, &chunk, &parts);
    if ((rank + 1) * chunk > (int64_t(1) << 31) - 1) return FA_ERR_INVALID_ARG;  // key indices are 32-bit

    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    if ((st = check_pointer(q, dev)) != FA_OK || (st = check_pointer(o_part, dev)) != FA_OK) return st;
    if ((st = check_pointer(lse_part, dev, 4)) != FA_OK) return st;
    if (count > 0)  // an empty shard's K and V are never read (and may be null)
        for (const void *p : {k_shard, v_shard})
            if ((st = check_pointer(p, dev)) != FA_OK) return st;
    const uint64_t qbytes = static_cast<uint64_t>(B * H * N * d) * 2u;
    const uint64_t kbytes = static_cast<uint64_t>(B * H * count * d) * 2u;
    const uint64_t obytes = static_cast<uint64_t>(B * H * N * d) * 4u;
    const uint64_t lbytes = static_cast<uint64_t>(B * H * N) * 4u;
    if (overlaps(o_part, obytes, lse_part, lbytes) || overlaps(o_part, obytes, q, qbytes) ||
        overlaps(lse_part, lbytes, q, qbytes))
        return FA_ERR_INVALID_ARG;
    if (count > 0)
        for (const void *in : {k_shard, v_shard})
            if (overlaps(o_part, obytes, in, kbytes) || overlaps(lse_part, lbytes, in, kbytes))
                return FA_ERR_INVALID_ARG;

    FaProblem p;
    p.q = q;
    p.k = count > 0 ? k_shard : q;
    p.v = count > 0 ? v_shard : q;
    p.o = o_part;
    p.lse = lse_part;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.sm_count = sm_count;
    if (fa_launch_tc_partials(p, o_part, lse_part, 1, static_cast<int>(chunk), static_cast<cudaStream_t>(stream),
                              static_cast<int>(rank), count) != cudaSuccess)
        return FA_ERR_LAUNCH;
    return FA_OK;
}

extern "C" int fa_combine(const float *o_parts, const float *lse_parts, int64_t n_parts, void *o, float *lse,
                          int64_t B, int64_t H, int64_t N, int64_t d, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if (n_parts < 1 || n_parts > kFaMaxSplits) return FA_ERR_INVALID_ARG;
    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    const void *ptrs[4] = {o_parts, lse_parts, o, lse};
    for (const void *p : ptrs)
        if ((st = check_pointer(p, dev)) != FA_OK) return st;
    const int64_t rows = B * H * N;
    const uint64_t pbytes = static_cast<uint64_t>(n_parts * rows * d) * 4u;
    const uint64_t plbytes = static_cast<uint64_t>(n_parts * rows) * 4u;
    const uint64_t tbytes = static_cast<uint64_t>(rows * d) * 2u, lbytes = static_cast<uint64_t>(rows) * 4u;
    if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    for (const void *out : {static_cast<const void *>(o), static_cast<const void *>(lse)}) {
        const uint64_t ob = out == o ? tbytes : lbytes;
        if (overlaps(out, ob, o_parts, pbytes) || overlaps(out, ob, lse_parts, plbytes)) return FA_ERR_INVALID_ARG;
    }
    if (fa_launch_combine(o_parts, lse_parts, static_cast<int>(n_parts), rows, static_cast<int>(d), o, lse, sm_count,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_LAUNCH;
    return FA_OK;
}

extern "C" int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                                  int64_t H, int64_t N, int64_t d, float scale, int causal,
                                  const uint8_t *block_mask, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    const void *ptrs[6] = {q, k, v, o, lse, block_mask};
    for (const void *p : ptrs)
        if ((st = check_pointer(p, dev)) != FA_OK) return st;
    const uint64_t tbytes = static_cast<uint64_t>(B * H * N * d) * 2u;
    const uint64_t lbytes = static_cast<uint64_t>(B * H * N) * 4u;
    const uint64_t nb = static_cast<uint64_t>((N + 127) / 128);
    if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    for (const void *in : {q, k, v, static_cast<const void *>(block_mask)}) {
        const uint64_t ib = in == block_mask ? nb * nb : tbytes;
        if (overlaps(o, tbytes, in, ib) || overlaps(lse, lbytes, in, ib)) return FA_ERR_INVALID_ARG;
    }
    FaProblem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.sm_count = sm_count;
    if (fa_launch_tc_sparse(p, block_mask, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_LAUNCH;
    return FA_OK;
}

extern "C" int fa_fwd_fp8(const void *q, const void *k, const void *v, const float *q_scale,
                          const float *k_scale, const float *v_scale, void *o, float *lse, int64_t B, int64_t H,
                          int64_t N, int64_t d, float scale, int causal, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    const void *ptrs[8] = {q, k, v, q_scale, k_scale, v_scale, o, lse};
    for (const void *p : ptrs)
        if ((st = check_pointer(p, dev)) != FA_OK) return st;
    const uint64_t in_bytes = static_cast<uint64_t>(B * H * N * d);  // one byte per E4M3 element
    const uint64_t o_bytes = in_bytes * 2u, lbytes = static_cast<uint64_t>(B * H * N) * 4u;
    const uint64_t sbytes = static_cast<uint64_t>(B * H) * 4u;
    if (overlaps(o, o_bytes, lse, lbytes)) return FA_ERR_INVALID_ARG;
    const void *ins[6] = {q, k, v, q_scale, k_scale, v_scale};
    const uint64_t isz[6] = {in_bytes, in_bytes, in_bytes, sbytes, sbytes, sbytes};
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, o_bytes, ins[i], isz[i]) || overlaps(lse, lbytes, ins[i], isz[i])) return FA_ERR_INVALID_ARG;
    FaProblem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.sm_count = sm_count;
    if (fa_launch_fp8(p, q_scale, k_scale, v_scale, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_LAUNCH;
    return FA_OK;
}

extern "C" int64_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d)
{
    if (fa_check_sizes(B, H, N, d) != FA_OK) return -1;
    return fa_bwd_workspace_size(B, H, N, d);
}

extern "C" int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                      const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t H, int64_t N, int64_t d,
                      float scale, int causal, void *workspace, int64_t workspace_bytes, void *stream)
{
    int st = fa_check_sizes(B, H, N, d);
    if (st != FA_OK) return st;
    if ((causal != 0 && causal != 1) || !(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    const int64_t need = fa_bwd_workspace_size(B, H, N, d);
    if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
    int dev = 0, sm_count = 0;
    if ((st = current_device(&dev, &sm_count)) != FA_OK) return st;
    const void *ptrs[11] = {q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr};
    for (int i = 0; i < 10; ++i)
        if ((st = check_pointer(ptrs[i], dev)) != FA_OK) return st;
    const uint64_t tbytes = static_cast<uint64_t>(B * H * N * d) * 2u;
    const uint64_t lbytes = static_cast<uint64_t>(B * H * N) * 4u;
    const void *outs[4] = {dq, dk, dv, workspace};
    const uint64_t osz[4] = {tbytes, tbytes, tbytes, static_cast<uint64_t>(need)};
    const void *ins[6] = {q, k, v, o, lse, dout};
    const uint64_t isz[6] = {tbytes, tbytes, tbytes, tbytes, lbytes, tbytes};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], osz[a], ins[b], isz[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], osz[a], outs[b], osz[b])) return FA_ERR_INVALID_ARG;
    }
    FaBwdProblem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.dout = dout;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = static_cast<int>(d);
    p.scale = scale;
    p.causal = causal;
    p.sm_count = sm_count;
    if (fa_launch_bwd(p, workspace, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_LAUNCH;
    return FA_OK;
}

extern "C" int fa_get_device_status(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    const int fwd = fa_tc_take_status(static_cast<cudaStream_t>(stream));
    const int dp = fa_dp_take_status(static_cast<cudaStream_t>(stream));
    const int bwd = fa_bwd_take_status(static_cast<cudaStream_t>(stream));
    return fwd != FA_OK ? fwd : (dp != FA_OK ? dp : bwd);
}

extern "C" const char *fa_status_string(int status)
{
    switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dimension must be 64 or 128";
    case FA_ERR_NO_DEVICE: return "FA_ERR_NO_DEVICE: no CUDA device, or pointer on another device";
    case FA_ERR_ARCH: return "FA_ERR_ARCH: device is not compute capability 10.3 (sm_103)";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: CUDA launch or execution error";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded in-kernel wait gave up";
    case FA_ERR_WORKSPACE_LIMIT:
        return "FA_ERR_WORKSPACE_LIMIT: the problem needs more scratch than the static array holds";
    default: return "unknown fa_status";
    }
}

extern "C" int fa_version(void) { return 100; }
