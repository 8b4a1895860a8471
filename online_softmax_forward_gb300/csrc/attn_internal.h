// attn_internal.h -- declarations shared by the translation units of libattn.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Bit set in the device status word when a bounded wait expired.
constexpr int kStatusTimeout = 1;
// Bit set by the bounds-checking build when an index check failed.
constexpr int kStatusBounds = 2;

// The bounds-checking build (compiled with ATTN_BOUNDS_CHECK; the library
// libattn_checked.so) tests every global-memory index and every TMA
// coordinate a kernel computes against the extent of its buffer before the
// access.  A failed test ORs kStatusBounds into the status word and the
// access is skipped (a TMA load that fails its test also stops the CTA the
// way an expired wait does); nothing traps.  attn_check_status then reports
// ATTN_ERR_BOUNDS.  In the normal build the tests compile to nothing.
#ifdef ATTN_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

#ifdef __CUDACC__
// true if `ok`; otherwise records the failure in *status and returns false,
// so that the caller skips the access.  Always true in the normal build.
__device__ __forceinline__ bool in_bounds(bool ok, int *status) {
    if constexpr (kBoundsCheck) {
        if (!ok) {
            atomicOr(status, kStatusBounds);
            return false;
        }
    }
    return true;
}
#endif

// Host-side view of one problem.
struct Problem {
    int B, H, Sq, Skv, d, causal;
    float scale;  // resolved (> 0)
    int dtype;
    int64_t bh() const { return (int64_t)B * H; }
};

size_t elem_bytes_in(int dtype);
size_t elem_bytes_out(int dtype);

// fp32 CUDA-core path (attn_f32.cu).
int launch_f32(const float *q, const float *k, const float *v, float *o,
               float *lse, const Problem &p, int block_q, int block_kv,
               cudaStream_t stream);
bool f32_tiles_fit(int d, int block_q, int block_kv);
// Register-tiled fp32 kernel with fixed 32 x 64 tiles (the attn_fwd path).
int launch_f32_tiled(const float *q, const float *k, const float *v, float *o,
                     float *lse, const Problem &p, cudaStream_t stream);

// 16-bit tensor-core path (attn_tc.cu).
int launch_tc(const void *q, const void *k, const void *v, void *o, float *lse,
              const Problem &p, cudaStream_t stream);
void forget_sched_counters(int dev);  // attn_shutdown: look the address up again next time

// Split-KV path for few query rows (attn_splitkv.cu).
constexpr int kSplitRowBlock = 8;  // query rows per split-KV CTA when Sq > 1
constexpr int kMaxSplits = 256;    // upper bound of n_splits
constexpr int kMaxSplitRows = 65535 * kSplitRowBlock;  // grid limit on Sq
int splitkv_row_block(int Sq);
void splitkv_chunking(int Skv, int n_splits, int *chunk, int *n_eff);
int splitkv_choose(const Problem &p, int sms);
// part_o [n_splits][B*H][Sq][d] and part_lse [n_splits][B*H][Sq] fp32.
int launch_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                   const Problem &p, int n_splits, float *part_o, float *part_lse,
                   cudaStream_t stream);
// Merges [n_parts][rows][d] / [n_parts][rows] into o [rows][d] (out_dtype
// ATTN_F32, ATTN_BF16 or ATTN_F16) and lse [rows] (may be null).
int launch_merge(const float *po, const float *pl, int n_parts, int64_t rows, int d, void *o,
                 float *lse, int out_dtype, cudaStream_t stream);

// Fixed device scratch of attn_fwd_splitkv_noalloc (attn_splitkv.cu): its
// size, and its device address on the current device (looked up once per
// device).
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
int noalloc_scratch_ptr(void **ptr);
void forget_noalloc_scratch(int dev);  // attn_shutdown: look the address up again next time

// Writes o = 0 and lse = -inf (Skv == 0).
int launch_empty_keys(void *o, float *lse, const Problem &p, cudaStream_t stream);

// Sets the dynamic shared-memory limit of a kernel on the current device the
// first time it is asked for that (kernel, device) pair; later calls only
// look it up.  Returns false if the CUDA call fails.
bool set_smem_limit_once(const void *func, int bytes);
// Number of SMs of the current device, cached per device (0 on error).
int device_sm_count();

// Host-staged calls (attn_fwd_staged) of at least kStagedMinBytes of input
// run in chunks of (batch, head) slices on two library streams of the
// device, so that copies overlap the kernels.  Chunk i takes a share of the
// slices in proportion to kStagedWeights[i] (fewer chunks when there are
// fewer slices).  A small first chunk starts the kernels early; a small last
// chunk shortens what is left after the last host-to-device copy (its kernel
// and its copy back); the shares grow in between so that each copy lands
// before the kernel before it ends.
constexpr double kStagedWeights[] = {2.0, 3.0, 3.5, 1.5};
constexpr int kStagedChunks = (int)(sizeof(kStagedWeights) / sizeof(kStagedWeights[0]));
constexpr size_t kStagedMinBytes = (size_t)4 << 20;
struct StagedStreams {
    cudaStream_t st[2];
    cudaEvent_t start, done[2];
};
StagedStreams *staged_streams();  // created once per device; nullptr on failure

// Device status word helpers (attn_api.cu).
int *status_word_device_ptr();

// Watchdog settings for the tensor-core kernel.
int test_hook();
uint64_t watchdog_ns();

}  // namespace attn
