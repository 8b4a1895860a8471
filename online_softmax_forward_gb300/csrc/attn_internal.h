// attn_internal.h -- declarations shared by the translation units of libattn.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Bit set in the device status word when a bounded wait expired.
constexpr int kStatusTimeout = 1;

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

// 16-bit tensor-core path (attn_tc.cu).
int launch_tc(const void *q, const void *k, const void *v, void *o, float *lse,
              const Problem &p, cudaStream_t stream);

// Writes o = 0 and lse = -inf (Skv == 0).
int launch_empty_keys(void *o, float *lse, const Problem &p, cudaStream_t stream);

// Device status word helpers (attn_api.cu).
int *status_word_device_ptr();

// Watchdog settings for the tensor-core kernel.
int test_hook();
uint64_t watchdog_ns();

}  // namespace attn
