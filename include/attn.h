/*
 * attn.h -- C ABI of libattn.so: exact attention forward with online softmax
 * on NVIDIA GB300 (sm_103a).
 *
 * The operation (all three source pages compute it; they differ only in how
 * they tile it):
 *
 *   O[b,h,i,:] = sum_j softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] ) * V[b,h,j,:]
 *
 * over the keys j visible to query i, computed tile by tile: each query row
 * keeps a running maximum m, a normaliser l and an unnormalised accumulator a,
 * and both l and a are multiplied by exp(m_old - m_new) whenever a new key
 * tile raises the maximum, so that the full score matrix is never formed.
 *   - definition and dense reference: aiml.sh "verify-tiled-attention",
 *     function standard_attention (scale 1/sqrt(d), causal limit i+1);
 *     deepnotes "flash-attention-implemented-verified-and-measured",
 *     naive_attention on [B, H, S, d] tensors;
 *   - the tiled recurrence: aiml.sh "verify-tiled-attention",
 *     tiled_flash_attention; deepnotes ..., tiled_attention_online_softmax;
 *     huhohoo "tiled-online-softmax", section "Online normalization".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout   q [B, H, Sq, d], k and v [B, H, Skv, d], o [B, H, Sq, d],
 *          lse [B, H, Sq]; all contiguous row-major, strides implied.
 *          q, k, v and o must be 16-byte aligned; lse 4-byte aligned.
 * causal   0 or 1.  Key j is visible to query i iff j <= i + (Skv - Sq)
 *          (bottom-right alignment; identical to the pages' j <= i when
 *          Sq == Skv).  A query row with no visible key gets o = 0 and
 *          lse = -inf.
 * scale    multiplies q . k.  scale <= 0 selects the pages' 1/sqrt(d); NaN or
 *          infinity is rejected.
 * lse      optional (NULL: not written).  Natural-log log-sum-exp of the
 *          scaled scores of each row, fp32.  Not on the pages; provided so a
 *          caller can merge partial results or compute a backward pass.
 * stream   a cudaStream_t (NULL = legacy default stream).  All work is
 *          enqueued on it asynchronously; no entry point synchronises except
 *          attn_check_status.  Device pointers must be valid on the current
 *          CUDA device.
 * Ownership  the caller owns every buffer.  The library keeps no per-call
 *          allocation; q, k and v are only read; o and lse must not overlap
 *          q, k or v (rejected) or each other.
 * Empty    B, H or Sq equal to 0 is a no-op returning ATTN_OK; Skv == 0 writes
 *          o = 0 and lse = -inf.
 * Errors   every entry point returns an attn_status; nothing aborts, exits or
 *          traps.  Invalid arguments are detected on the host before any
 *          launch.  attn_strerror() gives a message.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 1

/* The library is built with hidden visibility; only the functions declared
 * with ATTN_API (this header's) are exported.  The test-only entry points
 * (attn_test.h) are exported by libattn_test.so alone. */
#if defined(__GNUC__) || defined(__clang__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,        /* null/misaligned/overlapping pointer, bad size or dtype */
    ATTN_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    ATTN_ERR_LAUNCH = 3,             /* a CUDA launch or copy failed */
    ATTN_ERR_TIMEOUT = 4,            /* a kernel's bounded wait expired (see attn_check_status) */
    ATTN_ERR_CUDA = 5,               /* another CUDA runtime/driver error */
    ATTN_ERR_SCRATCH_LIMIT = 6,      /* attn_fwd_splitkv_noalloc: problem exceeds its fixed scratch */
    ATTN_ERR_BOUNDS = 7              /* bounds-checking build only: an index check failed and the
                                        access was skipped (see attn_check_status) */
} attn_status;

typedef enum attn_dtype {
    ATTN_F32 = 0,          /* fp32 q/k/v/o; CUDA-core kernel, fp32 arithmetic */
    ATTN_BF16 = 1,         /* bf16 q/k/v/o; tensor-core kernel, fp32 accumulation */
    ATTN_F16 = 2,          /* fp16 q/k/v/o; tensor-core kernel, fp32 accumulation */
    ATTN_BF16_OUT_F32 = 3, /* bf16 q/k/v, fp32 o (no output rounding) */
    ATTN_F16_OUT_F32 = 4   /* fp16 q/k/v, fp32 o */
} attn_dtype;

/*
 * attn_fwd -- exact attention forward (the operation above).
 *
 * Supported head widths: ATTN_F32: d in {16, 32, 64, 128};
 * ATTN_BF16/F16 and their _OUT_F32 variants: d in {64, 128}.
 * ATTN_F32 runs the CUDA-core kernel with 32-row query blocks and 64-key
 * blocks (the key block of deepnotes "Correctness first"); the 16-bit types
 * run the tensor-core kernel with 128 x 128 tiles.
 * Requires a compute capability 10.3 device (GB300) for every dtype.
 *
 * CUDA graphs: the first call that uses a kernel variant on a device sets
 * up its per-device state (the kernel's shared-memory attribute, for the fp32
 * kernel its occupancy, the address of the status word); the variant follows
 * from dtype, d and the problem shape.  After that a call of the same shape
 * only enqueues one kernel on `stream` (two for attn_fwd_splitkv) and may be
 * captured into a CUDA graph; a replay reads whatever the captured pointers
 * hold at replay time.  Make one ordinary call of the shape before capturing.
 *
 * Work distribution (16-bit types): each launch of the tensor-core kernel
 * takes its work units from one of 256 device counters of the library,
 * chosen in turn, and returns that counter to zero when it ends.  At most
 * 256 such launches may therefore be in flight on one device at once, and a
 * CUDA graph containing the call must not be replayed concurrently with
 * itself (its replays share the counter captured with it).
 */
ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int Sq, int Skv, int d, int causal, float scale,
             int dtype, void *stream);

/*
 * attn_validate -- the host-side argument check of attn_fwd, without any CUDA
 * call or launch.  Returns ATTN_OK or ATTN_ERR_INVALID_ARG.  Pointers are only
 * compared and tested for alignment, never dereferenced.
 */
ATTN_API int attn_validate(const void *q, const void *k, const void *v, const void *o,
                  const float *lse, int B, int H, int Sq, int Skv, int d,
                  int causal, float scale, int dtype);

/*
 * attn_fwd_staged -- attn_fwd on HOST buffers: copies q, k, v from host memory
 * to the caller's device buffers dq, dk, dv, runs attn_fwd into do_ / dlse,
 * and copies o (and lse when both lse_host and dlse are non-NULL) back to
 * host memory (one cudaMemcpyAsync per tensor, or per tensor and chunk).
 * Host buffers should be pinned for the copies to be asynchronous.  The call
 * returns after enqueueing; synchronise the stream before reading o_host.
 * Problems with at least 4 MiB of input are cut into up to 4 chunks of
 * (batch, head) slices, with shares 2 : 3 : 3.5 : 1.5 (small first and last
 * chunks, so the kernels start early and little is left after the last
 * copy in), that run on two streams the library creates once per device:
 * the copies of one chunk overlap the kernel of the other.  Those streams
 * start after the work queued on `stream` and `stream` waits for them, so the
 * call behaves as if everything ran on `stream`; concurrent staged calls on
 * one device share the two streams.  attn_shutdown releases them; call it
 * before a cudaDeviceReset that the process survives.
 * Sizes and dtype as attn_fwd; host pointers must not be NULL when their
 * tensor is non-empty.
 */
ATTN_API int attn_fwd_staged(const void *q_host, const void *k_host, const void *v_host,
                    void *o_host, float *lse_host, void *dq, void *dk, void *dv,
                    void *do_, float *dlse, int B, int H, int Sq, int Skv,
                    int d, int causal, float scale, int dtype, void *stream);

/*
 * Split-KV forward for a few query rows per head (decode)
 * --------------------------------------------------------
 * The keys of every (batch, head) are cut into n_splits contiguous ranges of
 * equal length (a multiple of 32 keys); each range is processed by its own
 * CTAs on CUDA cores (fp32 arithmetic for every input type), which write a
 * partial result -- the softmax-weighted average of the range's values and
 * the log-sum-exp of its scaled scores -- into `workspace`; attn_merge's
 * kernel then combines the partial results of every row.  The result is the
 * same operation as attn_fwd: only the order of the sums differs (the pages'
 * point that the tiling, here the split, changes nothing but rounding:
 * aiml.sh "verify-tiled-attention", tile-size sweep; huhohoo
 * "tiled-online-softmax", block size seven).
 */

/*
 * attn_splitkv_workspace_size -- bytes of the workspace attn_fwd_splitkv
 * needs: 4 * n_splits * B * H * Sq * (d + 1) (partial outputs
 * [n_splits][B*H][Sq][d] followed by partial lse [n_splits][B*H][Sq], fp32).
 * Host only.  d in {16, 32, 64, 128}; 1 <= n_splits <= 256.
 */
ATTN_API int attn_splitkv_workspace_size(int B, int H, int Sq, int d, int n_splits, size_t *bytes);

/*
 * attn_splitkv_plan -- the split count the library would pick on the current
 * device and, if workspace_bytes is not NULL, the workspace size for it.
 * The count minimises an estimate of the time: waves of CTAs over the
 * device's resident CTA slots times the 32-key tiles each warp walks plus a
 * fixed cost per CTA (about two tiles), with at least two tiles per warp in
 * each split.  Needs a compute capability 10.3 device.
 */
ATTN_API int attn_splitkv_plan(int B, int H, int Sq, int Skv, int d, int dtype, int *n_splits,
                      size_t *workspace_bytes);

/*
 * attn_fwd_splitkv -- attn_fwd computed by key splits.
 *
 * Arguments and layouts as attn_fwd, except:
 *   d          in {16, 32, 64, 128} for every dtype;
 *   Sq         <= 524280;
 *   n_splits   1 .. 256 (see attn_splitkv_plan); empty trailing splits are
 *              skipped;
 *   workspace  device memory of at least attn_splitkv_workspace_size bytes,
 *              16-byte aligned, owned by the caller and not overlapping any
 *              other argument; its contents are scratch (overwritten).
 *              May be NULL when Skv == 0.
 * Enqueues two kernels on `stream` (partial results, merge).  Returns
 * ATTN_ERR_INVALID_ARG for a missing, small, misaligned or overlapping
 * workspace; otherwise as attn_fwd.
 */
ATTN_API int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int Sq, int Skv, int d, int causal, float scale,
                     int dtype, int n_splits, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv for callers that must not
 * allocate memory.  No passage of the source pages corresponds to it: it is
 * an interface for code that cannot call cudaMalloc, for example code
 * running inside a custom allocator or a memory-pool callback, a runtime
 * that forbids allocation on its serving path, or a caller whose memory
 * budget is fixed in advance.
 *
 * Instead of a caller-provided workspace it uses a scratch array of
 * ATTN_NOALLOC_SCRATCH_BYTES (8 MiB) that is part of the library's device
 * image: every GPU on which the library is used holds it until the process
 * exits.  The call calls no allocating routine (no cudaMalloc, no library
 * allocator).
 *   - Size limit: the problem must fit, i.e.
 *     4 * n_splits * B * H * Sq * (d + 1) <= ATTN_NOALLOC_SCRATCH_BYTES
 *     (see attn_splitkv_workspace_size) whenever Skv > 0; otherwise
 *     ATTN_ERR_SCRATCH_LIMIT is returned before anything is launched.
 *   - Set-up on a device: the first call of ANY entry point on a device
 *     (with that device current) looks up the array's device address, which
 *     makes CUDA load the module holding it and reserve the 8 MiB there.  The
 *     first launch of each kernel variant may also make the driver load that
 *     kernel's code.  Both happen once per device; so, before entering code
 *     that must not allocate, make one call of this entry point on the
 *     device with the same dtype and head width (and before capturing a
 *     stream).  Later calls change nothing in the device's free memory.
 *   - Sharing: every call uses the same array, which keeps the contents of
 *     the last call.  Nothing in it needs to start at zero (each partial
 *     result is written before it is read), but calls that overlap on the GPU
 *     (different streams, or different host threads without ordering) race
 *     on it: order them, e.g. on one stream.
 * Other arguments, results and errors as attn_fwd_splitkv.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
ATTN_API int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int Sq, int Skv, int d, int causal, float scale,
                             int dtype, int n_splits, void *stream);

/*
 * attn_merge -- combines partial attention results of the same query rows
 * over disjoint key sets (key splits, or key shards held by different
 * devices) into the result over the union of the keys.  Each partial result
 * is the state (m, l, a) of the online softmax in the form o_part = a / l,
 * lse_part = m + ln l; the merge is the update of huhohoo
 * "tiled-online-softmax" ("Online normalization") applied to whole states:
 *   M = max_p lse_p,  w_p = exp(lse_p - M),
 *   o = sum_p w_p o_p / sum_p w_p,  lse = M + ln(sum_p w_p).
 * A part with lse = -inf (no visible key) contributes nothing; a row whose
 * parts are all -inf gets o = 0 and lse = -inf.
 *
 *   n_parts    1 .. 4096;  rows 0 .. 2^31 - 1;  d >= 1
 *   o_parts    [n_parts][rows][d] fp32, device memory
 *   lse_parts  [n_parts][rows]    fp32, natural log
 *   o          [rows][d] of out_dtype: ATTN_F32, ATTN_BF16 or ATTN_F16
 *   lse        [rows] fp32, or NULL
 * fp32 arithmetic; asynchronous on `stream`.  Outputs must not overlap the
 * inputs or each other (ATTN_ERR_INVALID_ARG).
 */
ATTN_API int attn_merge(const float *o_parts, const float *lse_parts, int n_parts, int64_t rows, int d,
               void *o, float *lse, int out_dtype, void *stream);

/*
 * attn_check_status -- synchronises `stream`, then reads and clears the
 * library's device status word on the current device.  Returns
 * ATTN_ERR_BOUNDS if, in the bounds-checking build (libattn_checked.so,
 * compiled with ATTN_BOUNDS_CHECK), a kernel since the last check computed
 * a global-memory index or TMA coordinate outside its buffer (the access was
 * skipped, so the output is incomplete); ATTN_ERR_TIMEOUT if any tensor-core
 * kernel since the last check gave up a bounded wait (its output is then
 * incomplete); ATTN_ERR_CUDA if the stream reports an error; ATTN_OK
 * otherwise.  The normal build never sets ATTN_ERR_BOUNDS.
 */
ATTN_API int attn_check_status(void *stream);

/*
 * attn_shutdown -- releases what the library created on the current device
 * and forgets what it cached about it.  It destroys the two streams and three
 * events of attn_fwd_staged, after waiting for those streams to finish.  It
 * clears the cached capability check, SM count and kernel shared-memory
 * limits, and the device addresses of the status word, of the no-alloc
 * scratch and of the tensor-core kernel's schedule counters.  Work the caller queued on its own streams is not waited for.
 * The next call on the device sets everything up again.  Call it before
 * cudaDeviceReset if the process goes on using the library, since a reset
 * invalidates those handles.  It must not run concurrently with other calls
 * on the same device.  Returns ATTN_OK, or ATTN_ERR_CUDA if destroying a
 * handle failed; the state is forgotten either way.  Not on the source
 * pages: resource management of this library.
 */
ATTN_API int attn_shutdown(void);

/* Human-readable text for an attn_status value (static storage). */
ATTN_API const char *attn_strerror(int status);

/* ATTN_ABI_VERSION of the loaded library. */
ATTN_API int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
