// fa_fwd_host: the forward on host buffers, with the copies overlapped.
//
// The B*H slices of a contiguous [B, H, N, d] problem are independent, and a
// run of consecutive slices is itself a contiguous problem.  The slices go in
// n_groups consecutive groups.  Group g's Q, K, V copies go to the device on
// an input stream, its forward runs on the caller's stream once they have
// landed, and its O, LSE copies come back on an output stream once it has
// run.  Group g+1's copies in therefore overlap group g's forward, and group
// g's copies out overlap group g+1's forward.  Every step is ordered by
// events only: nothing here synchronises the host.
//
// Ordering with the caller's stream: the copies in start after the work
// queued on `stream` before the call (the device staging buffers may still be
// in use by it), and the work queued on `stream` after the call starts after
// the last copy out.
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 64;

// Streams and events of one device, created on first use and kept for the
// life of the process.  `mu` serialises whole enqueue sequences, so that two
// host threads never interleave their event records and waits.
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kMaxGroups] = {}, comp[kMaxGroups] = {};
};
HostPipe g_pipes[kMaxDevices];

// Destroys whatever a failed create() made, so that a later call starts clean.
void destroy(HostPipe &hp)
{
    for (int g = 0; g < kMaxGroups; ++g) {
        if (hp.in[g]) cudaEventDestroy(hp.in[g]);
        if (hp.comp[g]) cudaEventDestroy(hp.comp[g]);
        hp.in[g] = hp.comp[g] = nullptr;
    }
    if (hp.start) cudaEventDestroy(hp.start);
    if (hp.done) cudaEventDestroy(hp.done);
    if (hp.s_in) cudaStreamDestroy(hp.s_in);
    if (hp.s_out) cudaStreamDestroy(hp.s_out);
    hp.start = hp.done = nullptr;
    hp.s_in = hp.s_out = nullptr;
}

bool create(HostPipe &hp)
{
    if (hp.ready) return true;
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, ef) == cudaSuccess;
    for (int g = 0; g < kMaxGroups && ok; ++g)
        ok = cudaEventCreateWithFlags(&hp.in[g], ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.comp[g], ef) == cudaSuccess;
    if (!ok) {
        destroy(hp);
        return false;
    }
    hp.ready = true;
    return true;
}

}  // namespace

int fa_run_host_pipeline(const FaHostProblem &p, cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
    }
    if (p.n_groups < 1 || p.n_groups > kMaxGroups) return FA_ERR_INVALID_ARG;
    HostPipe &hp = g_pipes[dev];
    std::lock_guard<std::mutex> lock(hp.mu);
    if (!create(hp)) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    const int64_t BH = p.B * p.H;
    const int64_t slice = p.N * p.d * 2, lslice = p.N * 4;  // bytes of one (b, h) slice of a tensor / of LSE
    auto at = [](const void *base, int64_t off) {
        return static_cast<char *>(const_cast<void *>(base)) + off;
    };
    bool ok = cudaEventRecord(hp.start, stream) == cudaSuccess &&
              cudaStreamWaitEvent(hp.s_in, hp.start, 0) == cudaSuccess;
    for (int g = 0; g < p.n_groups && ok; ++g) {
        const int64_t s0 = BH * g / p.n_groups, s1 = BH * (g + 1) / p.n_groups;
        const int64_t tb = (s1 - s0) * slice, lb = (s1 - s0) * lslice;
        // copies in
        ok = cudaMemcpyAsync(at(p.q_dev, s0 * slice), at(p.q, s0 * slice), tb, cudaMemcpyHostToDevice, hp.s_in) ==
                 cudaSuccess &&
             cudaMemcpyAsync(at(p.k_dev, s0 * slice), at(p.k, s0 * slice), tb, cudaMemcpyHostToDevice, hp.s_in) ==
                 cudaSuccess &&
             cudaMemcpyAsync(at(p.v_dev, s0 * slice), at(p.v, s0 * slice), tb, cudaMemcpyHostToDevice, hp.s_in) ==
                 cudaSuccess &&
             cudaEventRecord(hp.in[g], hp.s_in) == cudaSuccess;
        if (!ok) break;
        // forward of the group: slices [s0, s1) as one problem of s1 - s0 heads
        ok = cudaStreamWaitEvent(stream, hp.in[g], 0) == cudaSuccess;
        if (!ok) break;
        FaProblem fp;
        fp.q = at(p.q_dev, s0 * slice);
        fp.k = at(p.k_dev, s0 * slice);
        fp.v = at(p.v_dev, s0 * slice);
        fp.o = at(p.o_dev, s0 * slice);
        fp.lse = reinterpret_cast<float *>(at(p.lse_dev, s0 * lslice));
        fp.B = 1;
        fp.H = s1 - s0;
        fp.N = p.N;
        fp.d = p.d;
        fp.scale = p.scale;
        fp.causal = p.causal;
        fp.sm_count = p.sm_count;
        ok = fa_launch_tc(fp, stream) == cudaSuccess && cudaEventRecord(hp.comp[g], stream) == cudaSuccess;
        if (!ok) break;
        // copies out
        ok = cudaStreamWaitEvent(hp.s_out, hp.comp[g], 0) == cudaSuccess &&
             cudaMemcpyAsync(at(p.o, s0 * slice), at(p.o_dev, s0 * slice), tb, cudaMemcpyDeviceToHost, hp.s_out) ==
                 cudaSuccess &&
             cudaMemcpyAsync(at(p.lse, s0 * lslice), at(p.lse_dev, s0 * lslice), lb, cudaMemcpyDeviceToHost,
                             hp.s_out) == cudaSuccess;
    }
    // the caller's stream continues once every copy out has landed (even after a
    // failure part way, so that no copy of this call outlives it unordered)
    const bool tail = cudaEventRecord(hp.done, hp.s_out) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp.done, 0) == cudaSuccess;
    if (!ok || !tail) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    return FA_OK;
}
