/*
 * attn_test.h -- entry points of libattn_test.so only: the test library is
 * the product library (every function of attn.h, the same kernels) plus the
 * two functions below, which the test suite needs and a production caller
 * does not.  libattn.so does not export them.
 *
 * Conventions, status codes and dtypes are those of attn.h.
 */
#ifndef ATTN_GB300_ATTN_TEST_H
#define ATTN_GB300_ATTN_TEST_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_fwd_f32_blocked -- the fp32 CUDA-core path with caller-chosen tile
 * sizes, so that block-size invariance (including sizes that do not divide
 * the sequence, e.g. 7, or 13 x 19) can be tested as the pages do
 * (aiml.sh "verify-tiled-attention" test_lab.py tile sweep; huhohoo
 * "tiled-online-softmax" exercise with block size seven).
 * block_q in [1, 128], block_kv in [1, 256]; the key tile must fit in shared
 * memory (ATTN_ERR_INVALID_ARG otherwise).  Other arguments as attn_fwd with
 * dtype ATTN_F32.
 */
ATTN_API int attn_fwd_f32_blocked(const float *q, const float *k, const float *v,
                                  float *o, float *lse, int B, int H, int Sq, int Skv,
                                  int d, int causal, float scale, int block_q,
                                  int block_kv, void *stream);

/*
 * Test hook for the watchdog of the tensor-core kernel.  hook = 0 (default)
 * disables it; hook = 1 makes the next launches of this library's
 * tensor-core kernel skip one internal completion signal, so that a bounded
 * wait expires, the kernel stops cleanly and attn_check_status reports
 * ATTN_ERR_TIMEOUT.  timeout_ns sets the bounded-wait limit (0 keeps the
 * current value; default 1e9 ns).  Process-wide within this library; not
 * thread-safe against concurrent attn_fwd calls.  Not on the source pages:
 * it exercises the failure detection of the kernel without a GPU fault.
 */
ATTN_API int attn_test_set_hook(int hook, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_TEST_H */
