/*
 * fa.h - C ABI of the GB300 (sm_103a) exact attention forward library (libfa.so).
 *
 * The operation is scaled dot-product attention for self-attention over
 * [B, H, N, d] tensors ("6.1 FlashAttention V1 in detail", section 1.1 and the
 * shapes of section 8.1):
 *
 *     S = scale * Q K^T          (per batch b and head h, N x N)
 *     P = softmax(S) row-wise    (causal: key j > query i is excluded)
 *     O = P V                    ([B, H, N, d])
 *     LSE_i = m_i + ln(l_i)      (row max m and exp-sum l of S; "FlashAttention:
 *                                 IO-Aware Tiling, ...", section "Backward Pass
 *                                 Recomputation", L = m + log(l))
 *
 * computed in one fused pass that streams K/V tiles through a running max,
 * exp-sum and unnormalised output ("FlashAttention: optimize data movement
 * before counting FLOPs", section 02: m' = max(m, max s),
 * l' = e^(m-m') l + sum e^(s-m'), u' = e^(m-m') u + sum e^(s-m') V,
 * Output = u'/l'), so no N x N matrix is ever written to device memory.
 *
 * Conventions shared by every entry point:
 *   - Tensors are device pointers on the current CUDA device, owned by the
 *     caller.  The library allocates no device memory per call.
 *   - Calls are asynchronous: they enqueue work on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream) and never synchronise.
 *   - On any error code the call has launched nothing and written nothing.
 *   - Thread safety: calls may come from several host threads; the only
 *     shared state is a per-device status word and cached device properties.
 */
#ifndef FA_H
#define FA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null/misaligned/overlapping pointer, bad size, bad scale */
    FA_ERR_UNSUPPORTED = 2, /* a valid problem the library does not handle (d not 64/128) */
    FA_ERR_NO_DEVICE = 3,   /* no CUDA device, or a pointer not on the current device */
    FA_ERR_ARCH = 4,        /* the current device is not compute capability 10.3 */
    FA_ERR_LAUNCH = 5,      /* the kernel launch itself failed (CUDA error) */
    FA_ERR_TIMEOUT = 6,     /* a bounded in-kernel wait gave up (see fa_get_device_status) */
    FA_ERR_WORKSPACE_LIMIT = 7 /* fa_fwd_splitkv_noalloc: the problem needs more scratch
                                  than FA_SPLITKV_NOALLOC_MAX_BYTES */
};

/* Size of the library-owned scratch array behind fa_fwd_splitkv_noalloc. */
#define FA_SPLITKV_NOALLOC_MAX_BYTES (32LL * 1024 * 1024)

/*
 * fa_fwd - fused exact attention forward.
 *
 *   q, k, v : const bf16, contiguous [B, H, N, d] (row-major, d fastest).
 *             May alias one another (they are only read).
 *   o       : bf16 out, contiguous [B, H, N, d]; O = P V rounded once to bf16
 *             (round-to-nearest-even).
 *   lse     : fp32 out, contiguous [B, H, N]; natural-log log-sum-exp of the
 *             scaled logits of each row over its admitted keys.
 *   B, H, N : batch, heads, sequence length (queries = keys = N); each >= 1,
 *             B*H*N*d < 2^40.
 *   d       : head dimension, 64 or 128 (else FA_ERR_UNSUPPORTED).
 *   scale   : softmax scale, finite and > 0 (1/sqrt(d) in the usual case).
 *   causal  : 0 = every key admitted; 1 = key j admitted to query i iff j <= i.
 *   stream  : cudaStream_t to enqueue on.
 *
 * Every pointer must be on the current device; q, k, v and o 16-byte
 * aligned, lse 4-byte aligned (it is written by scalar stores only, so the
 * LSE of any run of whole rows can be addressed); o and lse must not overlap
 * q, k, v or each other.  Work is split into tiles of 128
 * query rows; ragged N (not a multiple of the tile) is handled in the kernel.
 * Returns FA_OK or an fa_status code; an error found inside the kernel is
 * reported later by fa_get_device_status().
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
           void *stream);

/*
 * fa_fwd_kernel - which kernel a call of fa_fwd with these sizes launches.
 * Both compute the same forward; at d = 64 problems whose work units (256
 * query rows each) see at most 9 key/value tiles of 128 keys on average go to
 * the kernel that keeps P apart from S, the rest to the main kernel.  Meant
 * for profilers and benchmarks that attribute time to a kernel by name.
 *
 *   B, H, N, d, causal : as for fa_fwd
 *   kernel : host output, FA_FWD_KERNEL_TC (fa_fwd_tc_kernel) or
 *            FA_FWD_KERNEL_DP (fa_fwd_dp_kernel)
 * Pure host computation.  Returns FA_OK, or fa_fwd's status for invalid sizes
 * or causal flag, or FA_ERR_INVALID_ARG for a null `kernel` (nothing written).
 */
enum fa_fwd_kernel_id { FA_FWD_KERNEL_TC = 0, FA_FWD_KERNEL_DP = 1 };
int fa_fwd_kernel(int64_t B, int64_t H, int64_t N, int64_t d, int causal, int *kernel);

/*
 * fa_bh_partition - the (b, h) slices one GPU of a sharded problem takes.
 * The programs over (b, h) slices are independent and exchange nothing
 * ("6.1 FlashAttention V1 in detail", section 8.2, the parallel partition),
 * so a problem is spread over `world` GPUs by giving rank r a contiguous
 * slab of slices [begin, begin + count): the first n_slices % world ranks take
 * ceil(n_slices / world) slices, the others floor(n_slices / world).  Every
 * slice belongs to exactly one rank; a rank past n_slices gets count = 0.
 * Slices are numbered b * H + h, the order of the [B, H, N, d] layout, so a
 * slab is one contiguous range of Q, K, V, O and LSE.
 *
 *   n_slices : B * H (>= 0)
 *   world    : number of ranks (>= 1);  rank : 0 <= rank < world
 *   begin, count : host outputs
 * Pure host computation.  Returns FA_OK, or FA_ERR_INVALID_ARG (nothing
 * written) for out-of-range arguments or a null output pointer.
 */
int fa_bh_partition(int64_t n_slices, int64_t world, int64_t rank, int64_t *begin,
                    int64_t *count);

/*
 * fa_fwd_slab - fa_fwd over the slab of (b, h) slices that fa_bh_partition
 * gives rank `rank` of `world`: q, k, v, o, lse are the whole problem's
 * tensors, as for fa_fwd, and only the slab's rows of Q, K, V are read and
 * only its rows of O and LSE written (the slab runs as a problem of B = 1,
 * H = count).  Ranks on different GPUs that call it over the same problem
 * (each with the tensors in its own memory) together compute all of it, with
 * no communication.  A rank whose slab is empty launches nothing and returns
 * FA_OK.  Errors as fa_fwd, plus FA_ERR_INVALID_ARG for a bad rank or world;
 * pointers are checked at the slab's offset.
 */
int fa_fwd_slab(const void *q, const void *k, const void *v, void *o, float *lse,
                int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                int64_t rank, int64_t world, void *stream);

/*
 * fa_fwd_host - fa_fwd on HOST buffers: copies Q, K, V to the device, runs
 * the forward, and copies O and LSE back, overlapping the copies with the
 * compute.  The pages move tiles between HBM and on-chip memory
 * ("FlashAttention: optimize data movement before counting FLOPs", section
 * 02) and never discuss host memory; this entry point is this library's own.
 * It is the end-to-end path, for callers whose data lives in host memory.
 *
 *   q, k, v : host, const bf16 [B, H, N, d] as in fa_fwd.  Pinned memory
 *             (cudaHostAlloc, cudaHostRegister) copies at full speed;
 *             pageable memory works but is staged by the driver.
 *   o, lse  : host outputs, layouts as in fa_fwd; they must not overlap
 *             q, k, v or each other.
 *   q_dev, k_dev, v_dev, o_dev, lse_dev :
 *             device staging buffers of the same shapes, owned by the caller,
 *             16-byte aligned, on the current device, mutually disjoint.  On
 *             return from a completed call they hold the inputs and outputs.
 *   n_groups: the B*H (b, h) slices are processed in n_groups consecutive
 *             groups of near-equal size (1 <= n_groups <= min(B*H, 64); 0
 *             selects min(B*H, 8)).  Group g+1's copies in overlap group g's
 *             forward, and group g's copies out overlap group g+1's forward.
 *   stream  : the copies in start after the work already queued on `stream`;
 *             work queued on `stream` afterwards starts after the last copy
 *             out.  The call returns after enqueueing: synchronise `stream`
 *             before reading o and lse on the host.
 *
 * The other arguments, and the results (bit for bit those of fa_fwd on the
 * same device buffers), are as for fa_fwd.  The copies and the forward run on
 * the caller's stream and two library-owned non-blocking streams, ordered by
 * events.  Calls on one device serialise their enqueueing.  Returns FA_OK or
 * an fa_status code.  Errors found before anything is enqueued leave
 * everything untouched; FA_ERR_LAUNCH means a CUDA call failed part way.
 */
int fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                void *q_dev, void *k_dev, void *v_dev, void *o_dev, float *lse_dev,
                int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                int64_t n_groups, void *stream);

/*
 * fa_fwd_mma - the same operation, arguments, layouts and errors as fa_fwd,
 * computed by a warp-level tensor-core kernel (mma.sync m16n8k16, one CTA per
 * 128 query rows, cp.async double buffering) instead of the tcgen05 kernel.
 * Kept as an independent second implementation for cross-checks and as the
 * performance baseline of the pre-tcgen05 tensor-core path.
 */
int fa_fwd_mma(const void *q, const void *k, const void *v, void *o, float *lse,
               int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
               void *stream);

/*
 * Split-KV forward.  The keys are cut into `parts` contiguous ranges of
 * `chunk` keys (chunk = 128 * ceil(ceil(N / n_splits) / 128), parts =
 * ceil(N / chunk) <= n_splits); one launch computes, for every 256-row block
 * and every range, the attention of those rows over that range alone (fp32
 * O normalised over the range, and its LSE; a row with no admitted key in a
 * range gets O = 0, LSE = -inf), and a second launch merges the parts with
 * the two-block merge of "FlashAttention: IO-Aware Tiling, Online Softmax
 * Mathematics, ...", section "Online Softmax Mathematics":
 *     LSE = ln(sum_s e^LSE_s),   O = sum_s e^(LSE_s - LSE) O_s.
 * The result equals fa_fwd's up to rounding; splitting raises the number of
 * independent work items when B*H*ceil(N/256) is small.
 *
 *   q, k, v, o, lse, B, H, N, d, scale, causal : as for fa_fwd.
 *   n_splits        : 1..32.
 *   workspace       : device scratch owned by the caller, 16-byte aligned, at
 *                     least fa_fwd_splitkv_workspace_bytes(...) bytes, not
 *                     overlapping any other argument.  Holds the parts: fp32
 *                     O [parts][B][H][N][d] followed by fp32 LSE [parts][B][H][N].
 *                     Its contents on entry do not matter; on return they are
 *                     the per-range results.
 *   workspace_bytes : its size.
 * Errors as fa_fwd; a workspace that is too small is FA_ERR_INVALID_ARG.
 */
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                   int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                   int64_t n_splits, void *workspace, int64_t workspace_bytes,
                   void *stream);

/* Workspace bytes fa_fwd_splitkv needs for this problem, or -1 if the sizes
 * or n_splits are invalid.  Pure host computation. */
int64_t fa_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d,
                                       int64_t n_splits);

/*
 * fa_fwd_splitkv_noalloc - fa_fwd_splitkv for callers that cannot allocate
 * device memory.  The pages have no counterpart: this entry point exists for
 * host programs that must not allocate at call time (engines that plan all
 * device memory at start-up, plugins that are handed only input and output
 * tensors, latency-critical loops that cannot afford a cudaMalloc).
 *
 * Arguments, result and errors are those of fa_fwd_splitkv without the
 * workspace, checked in the same order: the parts go to a static device
 * array of FA_SPLITKV_NOALLOC_MAX_BYTES (32 MiB) that every GPU loading the
 * library holds until the process exits.  A valid problem whose
 * fa_fwd_splitkv_workspace_bytes(...) exceeds it is refused with
 * FA_ERR_WORKSPACE_LIMIT (nothing launched or written).  The array's device
 * address belongs to the CUDA context current at the call: a call outside a
 * stream capture looks it up in that context (and records it), a call on a
 * stream being captured uses the address recorded for the current context.
 * So make one call in each context (per device, and per context a host
 * program creates itself) before any stream capture, and again after a
 * cudaDeviceReset; a captured call with nothing recorded for its context
 * returns FA_ERR_LAUNCH.  No call allocates or frees device memory.  All
 * calls share the array: calls whose kernels can overlap on the GPU
 * (unordered streams) race and give undefined results.
 */
int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                           int causal, int64_t n_splits, void *stream);

/*
 * fa_kv_shard - the keys one GPU of a sequence-sharded problem holds: rank r
 * of `world` takes keys [begin, begin + count) of every (b, h) slice, the key
 * range of split r in fa_fwd_splitkv with n_splits = world (ranges of
 * 128 * ceil(ceil(N / world) / 128) keys; ranks past the last key get
 * count = 0).
 *
 *   N : keys (= queries) per slice, >= 1;  world : 1..32;  0 <= rank < world
 *   begin, count : host outputs
 * Pure host computation.  Returns FA_OK, or FA_ERR_INVALID_ARG (nothing
 * written) for out-of-range arguments or a null output pointer.
 */
int fa_kv_shard(int64_t N, int64_t world, int64_t rank, int64_t *begin, int64_t *count);

/*
 * fa_fwd_kv_shard - one GPU's part of a sequence-sharded forward: every query
 * row against the keys of this rank's shard only, as a partial result that
 * fa_combine merges with the other ranks' parts.  The pages split a row's keys
 * into blocks whose (max, sum, output) merge exactly ("FlashAttention:
 * IO-Aware Tiling, Online Softmax Mathematics, ...", section "Online Softmax
 * Mathematics", the two-block merge); spread over GPUs, that merge is
 * the one exchange a sequence-sharded attention needs.  Gathering the parts
 * (an all-gather of o_part and lse_part) is the caller's; the merge is
 * fa_combine on the gathered [world] parts.
 *
 *   q        : const bf16 [B][H][N][d], all query rows.
 *   k_shard, v_shard : const bf16 [B][H][count][d], keys begin .. begin +
 *              count - 1 of each slice (fa_kv_shard); may be NULL when count = 0.
 *   o_part   : fp32 out [B][H][N][d], O over the shard's keys (normalised by
 *              their sum).
 *   lse_part : fp32 out [B][H][N], LSE over the shard's keys; a row with no
 *              admitted key in the shard (causal rows before it, or an empty
 *              shard) gets O = 0, LSE = -inf.
 *   B, H, N, d, scale, causal : as for fa_fwd (causal compares absolute
 *              positions: key begin + j against query i).
 *   rank, world : as for fa_kv_shard.
 * Pointers as for fa_fwd (lse_part 4-byte aligned, the rest 16-byte); the
 * outputs must not overlap the inputs or each other.  Errors as fa_fwd, plus
 * FA_ERR_INVALID_ARG for a bad rank or world, or a rank whose key range would
 * pass 2^31.  Gathered on one GPU, the parts of all ranks merged by fa_combine
 * give fa_fwd_splitkv's result with n_splits = world (bit for bit when every
 * rank holds keys; ranks without keys add parts of weight 0).
 */
int fa_fwd_kv_shard(const void *q, const void *k_shard, const void *v_shard, float *o_part,
                    float *lse_part, int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                    int causal, int64_t rank, int64_t world, void *stream);

/*
 * fa_combine - merge n_parts partial attention results of the same rows over
 * disjoint key ranges (the exchange step a sequence-sharded attention needs),
 * with the two-block merge above.
 *
 *   o_parts   : const fp32 [n_parts][B][H][N][d], each part normalised over its keys
 *   lse_parts : const fp32 [n_parts][B][H][N], LSE_s (-inf: the part has no key)
 *   n_parts   : 1..32
 *   o         : bf16 out [B][H][N][d];  lse : fp32 out [B][H][N]
 * A row with LSE = -inf in every part gets O = 0, LSE = -inf.  Pointers are
 * device pointers on the current device, 16-byte aligned; outputs must not
 * overlap inputs.  Errors as fa_fwd.
 */
int fa_combine(const float *o_parts, const float *lse_parts, int64_t n_parts, void *o,
               float *lse, int64_t B, int64_t H, int64_t N, int64_t d, void *stream);

/*
 * fa_fwd_blocksparse - fa_fwd restricted by a block mask ("FlashAttention:
 * optimize data movement before counting FLOPs", section 07, names the
 * block-sparse variant without defining it; here): key j is admitted to
 * query i only if block_mask[(i / 128) * nb + j / 128] != 0, nb = ceil(N/128),
 * and, when causal, j <= i.  K/V tiles no query block of a work unit admits
 * are never loaded or multiplied.  A row that admits no key gets O = 0 and
 * LSE = -inf.
 *
 *   block_mask : const uint8 [nb][nb] device array (row = query block), shared
 *                by every (b, h); 16-byte aligned like the other pointers.
 * Other arguments and errors as fa_fwd.
 */
int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse,
                       int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                       const uint8_t *block_mask, void *stream);

/*
 * fa_fwd_fp8 - the forward of fa_fwd on 8-bit inputs ("FlashAttention: IO-Aware
 * Tiling, ...", section "FlashAttention-3": FP8 E4M3 with block quantisation
 * and scaling factors; the page fixes no scale policy, so here the block is
 * one (b, h) slice).  The real inputs are q_scale[b*H + h] * q8 (and the same
 * for k, v): S = scale * q_scale * k_scale * q8 k8^T, P = softmax(S), and P is
 * rounded to E4M3 for the P V product, O = v_scale * P v8.
 *
 *   q, k, v   : const E4M3 bytes, contiguous [B, H, N, d]
 *   q_scale, k_scale, v_scale : const fp32 [B*H], finite and > 0
 *   o         : bf16 out [B, H, N, d];  lse : fp32 out [B, H, N]
 *   d         : 128 only (else FA_ERR_UNSUPPORTED)
 * Other arguments and errors as fa_fwd.  Accuracy is set by E4M3's 3-bit
 * mantissa on P.  O is divided by the sum of the rounded P over every tile in
 * which one key can carry a quarter of the row, so the weights of a row that
 * few keys dominate still sum to one.  Elsewhere it is divided by the fp32
 * sum, whose rounding differences average out.  LSE uses the unrounded sum.
 */
int fa_fwd_fp8(const void *q, const void *k, const void *v, const float *q_scale,
               const float *k_scale, const float *v_scale, void *o, float *lse,
               int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
               void *stream);

/*
 * fa_bwd - gradients of sum(O * dO) with respect to Q, K and V for the
 * attention fa_fwd computes ("6.1 FlashAttention V1 in detail", section 6:
 * dV = P^T dO, dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D); and
 * "FlashAttention: IO-Aware Tiling, ...", section "Backward Pass
 * Recomputation": dQ = scale * dS K, dK = scale * dS^T Q).  P is recomputed
 * from the saved LSE, never stored.
 *
 *   q, k, v     : const bf16 [B, H, N, d], as passed to fa_fwd
 *   o, lse      : const, fa_fwd's outputs for q, k, v, scale, causal
 *   dout        : const bf16 [B, H, N, d], the gradient of the loss w.r.t. O
 *   dq, dk, dv  : bf16 out [B, H, N, d]
 *   B, H, N, d, scale, causal : as for fa_fwd
 *   workspace   : device scratch owned by the caller, 16-byte aligned, at least
 *                 fa_bwd_workspace_bytes(B, H, N, d) bytes (an fp32 dQ
 *                 accumulator and two fp32 row vectors); contents on entry do
 *                 not matter
 * Outputs and workspace must not overlap the inputs or each other.  Three
 * launches on `stream`; errors as fa_fwd.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int64_t B, int64_t H, int64_t N,
           int64_t d, float scale, int causal, void *workspace, int64_t workspace_bytes,
           void *stream);

/* Workspace bytes fa_bwd needs (B*H*N*d*4 + 2*B*H*ceil(N/128)*128*4), or -1
 * for invalid sizes.  Pure host computation. */
int64_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/*
 * fa_get_device_status - synchronise `stream`, then return and clear the
 * current device's sticky in-kernel status (FA_OK, or FA_ERR_TIMEOUT when a
 * bounded wait inside a kernel gave up and the kernel returned early, leaving
 * its outputs incomplete).  While FA_ERR_TIMEOUT is set, fa_fwd launches do
 * no work (their outputs are left unwritten) until this call clears it.
 * Returns FA_ERR_LAUNCH if the synchronisation itself reports a CUDA error.
 */
int fa_get_device_status(void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *fa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
