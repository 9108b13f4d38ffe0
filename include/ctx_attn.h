/*
 * ctx_attn.h -- C ABI of the ring-chunked exact attention library (sm_103a).
 *
 * What it computes.  Exact softmax attention over a sequence cut into P
 * chunks on the ring schedule of context parallelism, emulated on one GPU:
 * query chunk r meets KV chunk (r - i) mod P at ring iteration i, each
 * iteration yields a partial (O_i, LSE_i) and the partials are merged by LSE
 * weighting (diffusers issue #14265 "Ring attention backward uses stale
 * iteration-0 KV from ctx.saved_tensors ...", sections "Root cause" and
 * "How it surfaces per backend": the ring needs the LSE to merge partial
 * results).  The backward recomputes the probabilities of every (query
 * chunk, KV chunk) pair against that pair's own KV chunk, which is what the
 * same issue's "Expected behavior" asks for; the stale-K/V defect it reports
 * cannot occur.  The Ulysses sequence<->head exchange (DeepSpeed PR #8491
 * "[bugfix] _DimZeroAllToAll silently fails to send grads under
 * torch.compile"; DeepSpeed issue #7842 "[BUG] DistributedAttention produces
 * numerically incorrect results ...") is an on-device permutation.
 *
 * Conventions common to every entry point.
 *  - Device memory (inputs, outputs, workspace) is allocated and owned by the
 *    caller.  The library allocates nothing and frees nothing.
 *  - Work is enqueued on the caller's stream and is asynchronous; no entry
 *    point synchronises except ctx_get_device_status.  With the workspace
 *    and outputs given, a call may be captured in a CUDA graph (after one
 *    uncaptured call with the same head dimension on that device, which sets
 *    the kernels' shared-memory attributes once per device and looks up the
 *    device status word).  The library caches per-device addresses of its
 *    own device variables; they are invalid after cudaDeviceReset, so reload
 *    the library after a reset.
 *  - Short attention calls (about 1024 tokens and less) launch their kernels
 *    with programmatic stream serialization when the stream is not being
 *    captured: a kernel may be scheduled while the previous kernel in the
 *    stream finishes, but it waits for that kernel to complete before it
 *    reads or writes any memory, so the stream's order of memory effects is
 *    unchanged for the caller's own work before and after a call.
 *  - Diagnostics: CTX_ATTN_LOG=1 in the environment prints one line per
 *    attention call to stderr (chunks, tiles, CTAs, kernel variant, launch
 *    order); every entry point that launches work opens an NVTX range named
 *    after it.
 *  - Arguments are validated before anything is launched; an invalid call
 *    returns an error code and writes nothing (never a silent wrong result).
 *  - Element type: bf16 for q, k, v, out, dout, dq, dk, dv; fp32 for lse.
 *  - Head dimension D is 64, 128 or 256 (others: CTX_ERR_UNSUPPORTED).  D = 256
 *    is the Hugging Face causal model of the DeepSpeed Ulysses pull request
 *    ("24 attention heads, 4 key/value heads, head dimension 256"); its
 *    backward additionally needs B <= 32767.
 *  - Chunks: chunk_offsets == NULL means numpy-array_split chunking (the first
 *    S mod P chunks are one row longer); otherwise a host array of P+1
 *    strictly increasing offsets from 0 to S.  Empty chunks are rejected.
 *    Chunks need not be multiples of the 128-row tile: tails are masked.
 *  - GQA: Hq must be a multiple of Hkv; query head h uses kv head
 *    h / (Hq / Hkv) (issue #14265, "How it surfaces": the heads of K/V must
 *    divide the heads of Q).
 *  - Scale: scale <= 0 selects 1/sqrt(D).
 *  - causal != 0: key j is visible to query i iff j <= i (global row
 *    indices).  KV chunks after a query chunk are skipped entirely, the
 *    diagonal chunk is masked per element.  The diffusion workloads are not
 *    causal, the D = 256 language model is; the definition is the usual one.
 */
#ifndef CTX_ATTN_H
#define CTX_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ctx_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* Storage order of dense tensors: [B,S,H,D] or sequence-first [S,B,H,D]
 * (the DeepSpeed layout of issue #7842, "Testcase"). */
typedef enum { CTX_LAYOUT_BSHD = 0, CTX_LAYOUT_SBHD = 1 } ctx_layout_t;

typedef enum {
    CTX_OK = 0,
    CTX_ERR_INVALID_ARG = 1, /* a size, pointer, stride or offset is invalid */
    CTX_ERR_UNSUPPORTED = 2, /* valid but not implemented (D, alignment) */
    CTX_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned */
    CTX_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    CTX_ERR_TIMEOUT = 5      /* a device-side wait ran out of time (see ctx_get_device_status) */
} ctx_status_t;

/* A logical [B,S,H,D] tensor.  data is a device pointer to element
 * (0,0,0,0).  Strides are in elements, D stride is 1.  If stride_b,
 * stride_s and stride_h are all 0 the tensor is dense in the call's layout
 * and the library derives them.  Pointers and the B/S/H strides must be
 * 16-byte aligned (multiples of 8 elements) for the TMA engine. */
typedef struct {
    void* data;
    int64_t B, S, H, D;
    int64_t stride_b, stride_s, stride_h;
} ctx_tensor_t;

/* Flags for ctx_attn_fwd. */
#define CTX_FLAG_NONE 0
/* Write each ring iteration's partial (O_i, LSE_i) to the workspace and merge
 * them with a separate LSE-merge kernel, instead of merging online inside
 * the attention kernel.  Same result up to fp32 rounding order.  With causal
 * masking the iterations that meet chunks after the query's own have zero
 * weight (LSE = -inf) and are neither computed nor merged. */
#define CTX_FLAG_MATERIALIZE_PARTIALS 1
/* Visit the KV chunks in the order 0..P-1 (the K/V all-gather pattern of
 * diffusers PR #12443 "Fix Flux Context Parallel Bug ...": every query shard
 * sees the concatenated K/V) instead of the ring order (r - i) mod P.  Same
 * result up to fp32 rounding order. */
#define CTX_FLAG_KV_ALLGATHER 2

/* Bytes of device workspace the calls need for these sizes and flags:
 * max(forward, backward).  Returns 0 on invalid sizes. */
size_t ctx_attn_workspace_size(int B, int S, int Hq, int Hkv, int D, int P, int flags);

/* Chunk table (host only, no GPU needed): writes P+1 offsets of the
 * array_split chunking of S rows into P chunks.  CTX_ERR_INVALID_ARG if
 * P < 1 or P > S. */
int ctx_chunk_offsets(int S, int P, int* offsets_out);

/* Ring-chunked attention forward.
 *   q [B,S,Hq,D], k, v [B,S,Hkv,D] (bf16, read only);
 *   out [B,S,Hq,D] (bf16, written), lse [B,Hq,S] fp32 contiguous (written):
 *   lse = natural-log log-sum-exp of the scaled scores over all S keys.
 * P ring chunks (1 <= P <= min(S, 64)).  workspace may be NULL unless
 * CTX_FLAG_MATERIALIZE_PARTIALS is set.  Output rows are written once; out
 * must not alias q, k or v. */
int ctx_attn_fwd(const ctx_tensor_t* q, const ctx_tensor_t* k, const ctx_tensor_t* v, int P,
                 const int* chunk_offsets, ctx_layout_t layout, int causal, float scale,
                 const ctx_tensor_t* out, float* lse, void* workspace, size_t workspace_bytes,
                 int flags, ctx_stream_t stream);

/* Ring-chunked attention backward.
 *   q, k, v as in the forward; out, lse the forward's results; dout [B,S,Hq,D];
 *   dq [B,S,Hq,D], dk, dv [B,S,Hkv,D] (bf16, written; for GQA dk, dv are
 *   summed over the query heads of each kv head).
 * workspace: at least ctx_attn_workspace_size(...) bytes, 256-byte aligned;
 * it holds the fp32 dq accumulator and the per-row statistics. */
int ctx_attn_bwd(const ctx_tensor_t* q, const ctx_tensor_t* k, const ctx_tensor_t* v,
                 const ctx_tensor_t* out, const float* lse, const ctx_tensor_t* dout, int P,
                 const int* chunk_offsets, ctx_layout_t layout, int causal, float scale,
                 const ctx_tensor_t* dq, const ctx_tensor_t* dk, const ctx_tensor_t* dv,
                 void* workspace, size_t workspace_bytes, ctx_stream_t stream);

/* Backward without any device allocation by the caller.
 *
 * For callers that cannot call cudaMalloc: hosts whose device memory is
 * owned by a framework allocator or reserved up front (a raw allocation
 * would break the pool's accounting or fail under its budget), and code
 * that must not trigger the implicit device-wide synchronisation of
 * cudaFree.  Such callers still own q, k, v, out, lse, dout, dq, dk, dv; the
 * scratch that ctx_attn_bwd takes as `workspace` comes instead from a
 * file-scope device array of CTX_NOALLOC_SCRATCH_BYTES inside this library
 * (every GPU that loads the library holds it until the process exits).
 *
 * Arguments and results are those of ctx_attn_bwd.  Problems whose scratch
 * (ctx_attn_workspace_size with flags 0) exceeds CTX_NOALLOC_SCRATCH_BYTES
 * are rejected with CTX_ERR_WORKSPACE before anything is launched.  The
 * first call on a device looks up the array's device address on that device
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The call allocates nothing and frees nothing.
 * All calls share the one array and it keeps the last call's contents (the
 * parts that must start at zero are cleared on every call): calls that
 * overlap on the GPU, from different streams or threads, race on it.
 * The pages have no counterpart of this entry point. */
#define CTX_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int ctx_attn_bwd_noalloc(const ctx_tensor_t* q, const ctx_tensor_t* k, const ctx_tensor_t* v,
                         const ctx_tensor_t* out, const float* lse, const ctx_tensor_t* dout, int P,
                         const int* chunk_offsets, ctx_layout_t layout, int causal, float scale,
                         const ctx_tensor_t* dq, const ctx_tensor_t* dk, const ctx_tensor_t* dv,
                         ctx_stream_t stream);

/* How the attention calls of these sizes will be launched (host only, no
 * GPU needed; on a machine without one the SM count is taken as 148).
 *  fwd_ctas, bwd_ctas: CTAs of the forward and backward attention kernels.
 *  fwd_head_major, bwd_head_major: 1 when the grid is launched heads first
 *    (tile 0 of every head before tile 1 of any), which the library does for
 *    causal calls on grids of at most four CTAs per SM, so that the tiles
 *    with the most causal work start first; 0 when each head's tiles are
 *    launched together.
 *  bwd_group_split: for D = 256, the number of CTAs over which the query
 *    heads of one GQA group are split (1 = no split); always 1 otherwise.
 * Returns CTX_ERR_INVALID_ARG / CTX_ERR_UNSUPPORTED for sizes the attention
 * calls would refuse. */
typedef struct {
    int64_t fwd_ctas, bwd_ctas;
    int fwd_head_major, bwd_head_major;
    int bwd_group_split;
} ctx_launch_plan_t;
int ctx_attn_launch_plan(int B, int S, int Hq, int Hkv, int D, int P, const int* chunk_offsets, int causal,
                         ctx_launch_plan_t* plan);

/* Padded sequence length of the exchange: W * ceil(S / W), W = ring * ulysses. */
int64_t ctx_exchange_padded_len(int64_t S, int ring, int ulysses);

/* Ulysses sequence<->head exchange of 16-bit elements, bit-exact.
 * W = ring * ulysses emulated ranks; rank rho = r * ulysses + u holds rows
 * [rho * Ssh, (rho + 1) * Ssh) of the sequence padded with zero rows to
 * Sp = W * Ssh, Ssh = ceil(S / W) (padding to a multiple of the world size:
 * diffusers PR #12443 "Fix Flux Context Parallel Bug ...").  After the
 * exchange rank (r, u) holds its ring group's ulysses shards in slot order
 * and the head group [u*H/U, (u+1)*H/U) -- slot u' of a rank's output is the
 * slot that rank owns in rank (r, u')'s input (DeepSpeed PR #8491, "Testing").
 *
 * x: the whole-sequence tensor [B,S,H,D] (strided like ctx_tensor_t).
 * y: dense device buffer holding every rank's result, in the order
 *    [U][B][Sp][H/U][D] for CTX_LAYOUT_BSHD, [U][Sp][B][H/U][D] for
 *    CTX_LAYOUT_SBHD; rank (r, u) owns rows [r*U*Ssh, (r+1)*U*Ssh) of head
 *    group u.  Pad rows are written as zero.
 * dir 0: x -> y (sequence shards to head groups); dir 1: y -> x (the
 * inverse, which is also the exchange's backward).  H % ulysses == 0. */
int ctx_seq_head_exchange(const ctx_tensor_t* x, void* y, int ring, int ulysses, int dir,
                          ctx_layout_t layout, ctx_stream_t stream);

/* Synchronises the stream, then returns and clears the device status word
 * that kernels set when a bounded wait ran out (CTX_ERR_TIMEOUT) or CTX_OK;
 * CTX_ERR_CUDA if the synchronisation itself failed. */
int ctx_get_device_status(ctx_stream_t stream);

/* Failure-detection self test: launches one CTA whose single thread waits on
 * an mbarrier that nothing ever arrives on, with a limit of timeout_us
 * microseconds; the wait gives up, records CTX_ERR_TIMEOUT in the device
 * status word and returns.  Nothing faults or hangs. */
int ctx_selftest_wait_timeout(unsigned timeout_us, ctx_stream_t stream);

/* Self test of two exponentials: for n inputs x (device fp32), writes 2^x
 * computed by the SFU instruction the attention kernels use (y_sfu) and by a
 * cubic on the FMA pipe (y_poly: an alternative that was measured and not
 * adopted; no kernel calls it, it clamps x at -125 where the SFU returns 0),
 * so that a test can hold both against a reference exp2.  Device buffers,
 * n <= 2^31. */
int ctx_selftest_exp2(const float* x, float* y_poly, float* y_sfu, int64_t n, ctx_stream_t stream);

/* Kernel timing for measurement.  While enabled, every launch of the
 * attention forward kernel (kernel 0) and backward kernel (kernel 1) is
 * bracketed by a pair of CUDA events recorded on the launch stream (at most
 * 4096 launches per kernel are kept).  ctx_profile_enable(1) clears the
 * records, ctx_profile_enable(0) stops recording.  ctx_profile_read waits for
 * the recorded events and returns the summed device time of the kernel's
 * launches in milliseconds and their number.  Host-side bookkeeping only;
 * the events are created on first use. */
int ctx_profile_enable(int enable);
int ctx_profile_read(int kernel, double* total_ms, int* launches);

/* Test-only switches (failure detection; the pages have no counterpart).
 * ctx_debug_set(flags, wait_limit_ms) applies to the attention calls made
 * after it, process-wide, until it is called again; ctx_debug_set(0, 0)
 * restores normal operation.
 *  CTX_DEBUG_SKIP_ARRIVAL: the TMA producers of every attention kernel
 *    (forward and backward, every head dimension) issue no loads, and so no
 *    mbarrier arrivals, from their second load step on.  A consumer's bounded wait
 *    then runs out; the kernel records CTX_ERR_TIMEOUT in the device status
 *    word, waits (bounded) for its own copies and products in flight, frees
 *    its tensor memory and returns, with its outputs incomplete.  Nothing
 *    faults or hangs, and the next normal call computes correctly.
 *  wait_limit_ms: the limit of every device-side wait (1 .. 60000 ms); 0 keeps
 *    CTX_ATTN_WAIT_LIMIT_MS from the environment, else 2000 ms.
 * CTX_ERR_INVALID_ARG for unknown flag bits or a limit above 60 s. */
#define CTX_DEBUG_SKIP_ARRIVAL 1u
int ctx_debug_set(unsigned flags, unsigned wait_limit_ms);

/* Architecture the attention kernels' machine code was built for, as
 * cudaFuncAttributes::binaryVersion (103 for sm_103a), on the current
 * device.  CTX_ERR_CUDA if the kernels cannot run on it. */
int ctx_kernel_binary_version(int* version);

/* Human-readable text of a status code. */
const char* ctx_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* CTX_ATTN_H */
