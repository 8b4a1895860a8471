// attn_api.cu -- the extern "C" entry points of libattn.so: argument
// validation, device check, dispatch to the fp32 or tensor-core kernel,
// host-staged variant and the device status word.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <string.h>

#include "attn.h"
#include "attn_internal.h"
#ifdef ATTN_TEST_EXPORTS
#include "attn_test.h"  // the test library's build of this file
#endif

namespace attn {

// One status word per device (a module-scope __device__ variable: no
// allocation).  Kernels receive its address as a parameter and atomically OR
// error bits into it; attn_check_status reads and clears it.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices];  // device address of g_status_word per device
int g_hook = 0;
uint64_t g_watchdog_ns = 1000000000ull;

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// [lo, hi) byte ranges overlap?
bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    uintptr_t a0 = (uintptr_t)a, a1 = a0 + an, b0 = (uintptr_t)b, b1 = b0 + bn;
    return a0 < b1 && b0 < a1;
}

bool dtype_known(int dtype) { return dtype >= ATTN_F32 && dtype <= ATTN_F16_OUT_F32; }

bool d_supported(int dtype, int d) {
    if (dtype == ATTN_F32) return d == 16 || d == 32 || d == 64 || d == 128;
    return d == 64 || d == 128;
}

int resolve_scale(float scale, int d, float *out) {
    if (isnan(scale) || isinf(scale)) return ATTN_ERR_INVALID_ARG;
    *out = scale > 0.f ? scale : (float)(1.0 / sqrt((double)d));
    return ATTN_OK;
}

int cuda_to_status(cudaError_t e) {
    if (e == cudaSuccess) return ATTN_OK;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return ATTN_ERR_UNSUPPORTED_DEVICE;
    return ATTN_ERR_CUDA;
}

// The current device must be compute capability 10.3 (GB300).  The answer
// is cached per device (1 = supported, 2 = not), so that small calls do not
// pay for the attribute queries each time.
int g_device_ok[kMaxDevices];

int check_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ATTN_ERR_UNSUPPORTED_DEVICE;
    if (dev >= 0 && dev < kMaxDevices) {
        const int known = __atomic_load_n(&g_device_ok[dev], __ATOMIC_ACQUIRE);
        if (known) return known == 1 ? ATTN_OK : ATTN_ERR_UNSUPPORTED_DEVICE;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_UNSUPPORTED_DEVICE;
    const bool ok = (major == 10 && minor == 3);
    if (ok) {
        // Looking the no-alloc scratch up loads its module (and reserves the
        // array) on this device now, in the first call of any entry point,
        // rather than inside a later attn_fwd_splitkv_noalloc.  A failure
        // here is not this call's concern: that entry point reports it.
        void *scratch = nullptr;
        (void)noalloc_scratch_ptr(&scratch);
    }
    if (dev >= 0 && dev < kMaxDevices) __atomic_store_n(&g_device_ok[dev], ok ? 1 : 2, __ATOMIC_RELEASE);
    return ok ? ATTN_OK : ATTN_ERR_UNSUPPORTED_DEVICE;
}

// (kernel, device) pairs whose shared-memory limit has been set.
struct SmemDone {
    const void *func;
    int dev;
    int bytes;
};
std::mutex g_smem_mu;
SmemDone g_smem_done[256];
int g_smem_n = 0;
int g_sms[kMaxDevices];

}  // namespace

size_t elem_bytes_in(int dtype) { return dtype == ATTN_F32 ? 4 : 2; }
size_t elem_bytes_out(int dtype) {
    return (dtype == ATTN_F32 || dtype == ATTN_BF16_OUT_F32 || dtype == ATTN_F16_OUT_F32) ? 4 : 2;
}

bool set_smem_limit_once(const void *func, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(g_smem_mu);
    for (int i = 0; i < g_smem_n; ++i)
        if (g_smem_done[i].func == func && g_smem_done[i].dev == dev && g_smem_done[i].bytes >= bytes)
            return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    if (g_smem_n < 256) g_smem_done[g_smem_n++] = SmemDone{func, dev, bytes};
    return true;
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        const int n = __atomic_load_n(&g_sms[dev], __ATOMIC_ACQUIRE);
        if (n > 0) return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) __atomic_store_n(&g_sms[dev], n, __ATOMIC_RELEASE);
    return n;
}

int *status_word_device_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = (int *)p;
    }
    return g_status_ptr[dev];
}

namespace {
StagedStreams g_staged[kMaxDevices];  // the staged path's streams and events per device
bool g_staged_made[kMaxDevices];

// Destroys whatever part of a StagedStreams exists (null handles are skipped).
cudaError_t destroy_staged(StagedStreams &r) {
    cudaError_t first = cudaSuccess;
    auto keep = [&](cudaError_t e) { if (first == cudaSuccess) first = e; };
    for (int j = 0; j < 2; ++j) {
        if (r.st[j]) {
            keep(cudaStreamSynchronize(r.st[j]));
            keep(cudaStreamDestroy(r.st[j]));
        }
        if (r.done[j]) keep(cudaEventDestroy(r.done[j]));
    }
    if (r.start) keep(cudaEventDestroy(r.start));
    r = StagedStreams{};
    return first;
}
}  // namespace

StagedStreams *staged_streams() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_staged_made[dev]) {
        StagedStreams r{};
        bool ok = true;
        for (int j = 0; j < 2 && ok; ++j)
            ok = cudaStreamCreateWithFlags(&r.st[j], cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&r.done[j], cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&r.start, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            destroy_staged(r);  // nothing half-made is kept
            return nullptr;
        }
        g_staged[dev] = r;
        g_staged_made[dev] = true;
    }
    return &g_staged[dev];
}

int test_hook() { return g_hook; }
uint64_t watchdog_ns() { return g_watchdog_ns; }

// Validation shared by attn_validate / attn_fwd / attn_fwd_staged /
// attn_fwd_splitkv.  any_width: every head width of the fp32 path is allowed
// for every dtype (the split-KV path).
static int validate(const void *q, const void *k, const void *v, const void *o,
                    const float *lse, int B, int H, int Sq, int Skv, int d,
                    int causal, float scale, int dtype, Problem *out, bool any_width = false) {
    if (!dtype_known(dtype)) return ATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Sq < 0 || Skv < 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!d_supported(any_width ? ATTN_F32 : dtype, d)) return ATTN_ERR_INVALID_ARG;
    float sc = 0.f;
    if (resolve_scale(scale, d, &sc) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
    const int64_t bh = (int64_t)B * H;
    if (bh > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    const size_t ein = elem_bytes_in(dtype), eout = elem_bytes_out(dtype);
    const size_t nq = (size_t)bh * Sq * d, nkv = (size_t)bh * Skv * d;
    if (nq > 0) {
        if (!q || !o) return ATTN_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(o, 16)) return ATTN_ERR_INVALID_ARG;
        if (lse && !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
    }
    if (nkv > 0 && nq > 0) {
        if (!k || !v) return ATTN_ERR_INVALID_ARG;
        if (!aligned(k, 16) || !aligned(v, 16)) return ATTN_ERR_INVALID_ARG;
    }
    if (nq > 0) {
        const size_t ob = nq * eout, lb = lse ? (size_t)bh * Sq * 4 : 0;
        const void *ins[3] = {q, k, v};
        const size_t inb[3] = {nq * ein, nkv * ein, nkv * ein};
        for (int i = 0; i < 3; ++i) {
            if (overlap(o, ob, ins[i], inb[i])) return ATTN_ERR_INVALID_ARG;
            if (overlap(lse, lb, ins[i], inb[i])) return ATTN_ERR_INVALID_ARG;
        }
        if (overlap(o, ob, lse, lb)) return ATTN_ERR_INVALID_ARG;
    }
    if (out) {
        out->B = B; out->H = H; out->Sq = Sq; out->Skv = Skv; out->d = d;
        out->causal = causal; out->scale = sc; out->dtype = dtype;
    }
    return ATTN_OK;
}

// Bytes of the split-KV workspace: partial outputs [n][B*H][Sq][d] and
// partial lse [n][B*H][Sq], fp32.  Returns false on overflow.
static bool splitkv_bytes(int64_t bh, int Sq, int d, int n_splits, size_t *bytes) {
    const double est = (double)n_splits * (double)bh * (double)Sq * (double)(d + 1) * 4.0;
    if (est > 9.0e18) return false;
    *bytes = (size_t)n_splits * (size_t)bh * (size_t)Sq * (size_t)(d + 1) * 4u;
    return true;
}

static int fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                    const Problem &p, cudaStream_t stream) {
    if (p.bh() == 0 || p.Sq == 0) return ATTN_OK;
    int st = check_device();
    if (st != ATTN_OK) return st;
    if (p.Skv == 0) return launch_empty_keys(o, lse, p, stream);
    if (p.dtype == ATTN_F32)
        return launch_f32_tiled((const float *)q, (const float *)k, (const float *)v, (float *)o,
                                lse, p, stream);
    return launch_tc(q, k, v, o, lse, p, stream);
}

}  // namespace attn

using namespace attn;

extern "C" {

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

int attn_shutdown(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_OK;  // nothing is ever kept for it
    cudaError_t e = cudaSuccess;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_staged_made[dev]) {
            e = destroy_staged(g_staged[dev]);
            g_staged_made[dev] = false;
        }
        g_status_ptr[dev] = nullptr;
    }
    __atomic_store_n(&g_device_ok[dev], 0, __ATOMIC_RELEASE);
    __atomic_store_n(&g_sms[dev], 0, __ATOMIC_RELEASE);
    {
        std::lock_guard<std::mutex> lk(g_smem_mu);
        int n = 0;
        for (int i = 0; i < g_smem_n; ++i)
            if (g_smem_done[i].dev != dev) g_smem_done[n++] = g_smem_done[i];
        g_smem_n = n;
    }
    forget_noalloc_scratch(dev);
    forget_sched_counters(dev);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

const char *attn_strerror(int status) {
    switch (status) {
    case ATTN_OK: return "success";
    case ATTN_ERR_INVALID_ARG: return "invalid argument (null, misaligned or overlapping pointer, bad size, head width or dtype)";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "unsupported device: a compute capability 10.3 (GB300) GPU is required";
    case ATTN_ERR_LAUNCH: return "kernel launch or copy failed";
    case ATTN_ERR_TIMEOUT: return "a kernel gave up a bounded wait; its output is incomplete";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_SCRATCH_LIMIT: return "the problem needs more scratch than the fixed device array of attn_fwd_splitkv_noalloc holds";
    case ATTN_ERR_BOUNDS: return "bounds-checking build: a kernel computed an index outside its buffer (the access was skipped)";
    default: return "unknown status";
    }
}

int attn_validate(const void *q, const void *k, const void *v, const void *o,
                  const float *lse, int B, int H, int Sq, int Skv, int d,
                  int causal, float scale, int dtype) {
    return validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, nullptr);
}

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int Sq, int Skv, int d, int causal, float scale,
             int dtype, void *stream) {
    Problem p;
    int st = validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, &p);
    if (st != ATTN_OK) return st;
    return fwd_impl(q, k, v, o, lse, p, (cudaStream_t)stream);
}

#ifdef ATTN_TEST_EXPORTS
int attn_fwd_f32_blocked(const float *q, const float *k, const float *v,
                         float *o, float *lse, int B, int H, int Sq, int Skv,
                         int d, int causal, float scale, int block_q,
                         int block_kv, void *stream) {
    Problem p;
    int st = validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, ATTN_F32, &p);
    if (st != ATTN_OK) return st;
    if (block_q < 1 || block_q > 128 || block_kv < 1 || block_kv > 256 ||
        !f32_tiles_fit(d, block_q, block_kv))
        return ATTN_ERR_INVALID_ARG;
    if (p.bh() == 0 || p.Sq == 0) return ATTN_OK;
    st = check_device();
    if (st != ATTN_OK) return st;
    if (p.Skv == 0) return launch_empty_keys(o, lse, p, (cudaStream_t)stream);
    return launch_f32(q, k, v, o, lse, p, block_q, block_kv, (cudaStream_t)stream);
}
#endif  // ATTN_TEST_EXPORTS

int attn_fwd_staged(const void *q_host, const void *k_host, const void *v_host,
                    void *o_host, float *lse_host, void *dq, void *dk, void *dv,
                    void *do_, float *dlse, int B, int H, int Sq, int Skv,
                    int d, int causal, float scale, int dtype, void *stream) {
    Problem p;
    int st = validate(dq, dk, dv, do_, dlse, B, H, Sq, Skv, d, causal, scale, dtype, &p);
    if (st != ATTN_OK) return st;
    const size_t nq = (size_t)p.bh() * Sq * d, nkv = (size_t)p.bh() * Skv * d;
    if (nq == 0) return ATTN_OK;
    if (!q_host || !o_host || (nkv > 0 && (!k_host || !v_host))) return ATTN_ERR_INVALID_ARG;
    st = check_device();
    if (st != ATTN_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t ein = elem_bytes_in(dtype), eout = elem_bytes_out(dtype);
    const int64_t BH = p.bh();
    const size_t in_bytes = (nq + 2 * nkv) * ein;
    const int nchunks = (BH >= 2 && in_bytes >= kStagedMinBytes)
                            ? (int)(BH < kStagedChunks ? BH : kStagedChunks) : 1;
    // chunk i holds the (batch, head) slices [bound[i], bound[i + 1]): shares
    // in proportion to the weights, rounded, at least one slice each
    int64_t bound[kStagedChunks + 1];
    {
        double total = 0.0, cum = 0.0;
        for (int i = 0; i < nchunks; ++i) total += kStagedWeights[i];
        bound[0] = 0;
        for (int i = 1; i < nchunks; ++i) {
            cum += kStagedWeights[i - 1];
            int64_t b = (int64_t)((double)BH * cum / total + 0.5);
            if (b < bound[i - 1] + 1) b = bound[i - 1] + 1;
            if (b > BH - (nchunks - i)) b = BH - (nchunks - i);
            bound[i] = b;
        }
        bound[nchunks] = BH;
    }
    StagedStreams *res = nullptr;
    if (nchunks > 1) {
        res = staged_streams();
        if (!res) return ATTN_ERR_CUDA;
        // the chunks start after the work the caller has queued on `stream`
        if (cudaEventRecord(res->start, s) != cudaSuccess ||
            cudaStreamWaitEvent(res->st[0], res->start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(res->st[1], res->start, 0) != cudaSuccess)
            return ATTN_ERR_LAUNCH;
    }
    int err = ATTN_OK;
    for (int i = 0; i < nchunks && err == ATTN_OK; ++i) {
        // (batch, head) slices [b0, b1) on alternating streams: the copies of
        // one chunk overlap the kernel and the copies of the other
        const int64_t b0 = bound[i], b1 = bound[i + 1];
        cudaStream_t cs = nchunks > 1 ? res->st[i & 1] : s;
        const size_t oq = (size_t)b0 * Sq * d, okv = (size_t)b0 * Skv * d;
        const size_t cq = (size_t)(b1 - b0) * Sq * d, ckv = (size_t)(b1 - b0) * Skv * d;
        char *dqc = (char *)dq + oq * ein, *dkc = (char *)dk + okv * ein, *dvc = (char *)dv + okv * ein;
        char *doc = (char *)do_ + oq * eout;
        float *dlc = dlse ? dlse + (size_t)b0 * Sq : nullptr;
        if (cudaMemcpyAsync(dqc, (const char *)q_host + oq * ein, cq * ein, cudaMemcpyHostToDevice,
                            cs) != cudaSuccess) {
            err = ATTN_ERR_LAUNCH;
            break;
        }
        if (ckv > 0 &&
            (cudaMemcpyAsync(dkc, (const char *)k_host + okv * ein, ckv * ein,
                             cudaMemcpyHostToDevice, cs) != cudaSuccess ||
             cudaMemcpyAsync(dvc, (const char *)v_host + okv * ein, ckv * ein,
                             cudaMemcpyHostToDevice, cs) != cudaSuccess)) {
            err = ATTN_ERR_LAUNCH;
            break;
        }
        Problem sub = p;
        sub.B = 1;
        sub.H = (int)(b1 - b0);
        err = fwd_impl(dqc, dkc, dvc, doc, dlc, sub, cs);
        if (err != ATTN_OK) break;
        if (cudaMemcpyAsync((char *)o_host + oq * eout, doc, cq * eout, cudaMemcpyDeviceToHost,
                            cs) != cudaSuccess ||
            (lse_host && dlse &&
             cudaMemcpyAsync(lse_host + (size_t)b0 * Sq, dlc, (size_t)(b1 - b0) * Sq * 4,
                             cudaMemcpyDeviceToHost, cs) != cudaSuccess))
            err = ATTN_ERR_LAUNCH;
    }
    if (nchunks > 1) {
        // the caller's stream continues once both chunk streams are done --
        // also after a failure, so that work already queued on the library's
        // streams is ordered before whatever the caller does next
        for (int j = 0; j < 2; ++j)
            if (cudaEventRecord(res->done[j], res->st[j]) != cudaSuccess ||
                cudaStreamWaitEvent(s, res->done[j], 0) != cudaSuccess) {
                if (err == ATTN_OK) err = ATTN_ERR_LAUNCH;
            }
    }
    return err;
}

int attn_splitkv_workspace_size(int B, int H, int Sq, int d, int n_splits, size_t *bytes) {
    if (!bytes || B < 0 || H < 0 || Sq < 0 || !d_supported(ATTN_F32, d)) return ATTN_ERR_INVALID_ARG;
    if (n_splits < 1 || n_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
    return splitkv_bytes((int64_t)B * H, Sq, d, n_splits, bytes) ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

int attn_splitkv_plan(int B, int H, int Sq, int Skv, int d, int dtype, int *n_splits,
                      size_t *workspace_bytes) {
    Problem p;
    int st = validate(nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0, 0, 0, d, 0, 0.f, dtype,
                      &p, true);
    if (st != ATTN_OK || !n_splits || B < 0 || H < 0 || Sq < 0 || Skv < 0)
        return ATTN_ERR_INVALID_ARG;
    st = check_device();
    if (st != ATTN_OK) return st;
    const int sms = device_sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    p.B = B; p.H = H; p.Sq = Sq; p.Skv = Skv;
    *n_splits = splitkv_choose(p, sms);
    if (workspace_bytes)
        return attn_splitkv_workspace_size(B, H, Sq, d, *n_splits, workspace_bytes);
    return ATTN_OK;
}

int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int Sq, int Skv, int d, int causal, float scale,
                     int dtype, int n_splits, void *workspace, size_t workspace_bytes,
                     void *stream) {
    Problem p;
    int st = validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, &p, true);
    if (st != ATTN_OK) return st;
    if (n_splits < 1 || n_splits > kMaxSplits || Sq > kMaxSplitRows) return ATTN_ERR_INVALID_ARG;
    if (p.bh() == 0 || Sq == 0) return ATTN_OK;
    size_t need = 0;
    if (!splitkv_bytes(p.bh(), Sq, d, n_splits, &need)) return ATTN_ERR_INVALID_ARG;
    if (Skv > 0) {
        if (!workspace || !aligned(workspace, 16) || workspace_bytes < need)
            return ATTN_ERR_INVALID_ARG;
        const size_t nq = (size_t)p.bh() * Sq * d, nkv = (size_t)p.bh() * Skv * d;
        const size_t ein = elem_bytes_in(dtype), eout = elem_bytes_out(dtype);
        if (overlap(workspace, need, q, nq * ein) || overlap(workspace, need, k, nkv * ein) ||
            overlap(workspace, need, v, nkv * ein) || overlap(workspace, need, o, nq * eout) ||
            overlap(workspace, need, lse, lse ? (size_t)p.bh() * Sq * 4 : 0))
            return ATTN_ERR_INVALID_ARG;
    }
    st = check_device();
    if (st != ATTN_OK) return st;
    if (Skv == 0) return launch_empty_keys(o, lse, p, (cudaStream_t)stream);
    float *part_o = (float *)workspace;
    float *part_lse = part_o + (size_t)n_splits * p.bh() * Sq * d;
    return launch_splitkv(q, k, v, o, lse, p, n_splits, part_o, part_lse, (cudaStream_t)stream);
}

int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int Sq, int Skv, int d, int causal, float scale,
                             int dtype, int n_splits, void *stream) {
    Problem p;
    int st = validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, &p, true);
    if (st != ATTN_OK) return st;
    if (n_splits < 1 || n_splits > kMaxSplits || Sq > kMaxSplitRows) return ATTN_ERR_INVALID_ARG;
    if (p.bh() == 0 || Sq == 0) return ATTN_OK;
    size_t need = 0;
    if (!splitkv_bytes(p.bh(), Sq, d, n_splits, &need)) return ATTN_ERR_INVALID_ARG;
    // an empty key set needs no scratch (it only writes o = 0, lse = -inf)
    if (Skv > 0 && need > kNoAllocScratchBytes) return ATTN_ERR_SCRATCH_LIMIT;
    st = check_device();
    if (st != ATTN_OK) return st;
    if (Skv == 0) return launch_empty_keys(o, lse, p, (cudaStream_t)stream);
    void *scratch = nullptr;
    st = noalloc_scratch_ptr(&scratch);
    if (st != ATTN_OK) return st;
    // every partial result the merge reads is written first: nothing to clear
    float *part_o = (float *)scratch;
    float *part_lse = part_o + (size_t)n_splits * p.bh() * Sq * d;
    return launch_splitkv(q, k, v, o, lse, p, n_splits, part_o, part_lse, (cudaStream_t)stream);
}

int attn_merge(const float *o_parts, const float *lse_parts, int n_parts, int64_t rows, int d,
               void *o, float *lse, int out_dtype, void *stream) {
    if (n_parts < 1 || n_parts > 4096 || rows < 0 || rows > INT32_MAX || d < 1)
        return ATTN_ERR_INVALID_ARG;
    if (out_dtype != ATTN_F32 && out_dtype != ATTN_BF16 && out_dtype != ATTN_F16)
        return ATTN_ERR_INVALID_ARG;
    if (rows == 0) return ATTN_OK;
    const size_t eout = out_dtype == ATTN_F32 ? 4 : 2;
    const double est = (double)n_parts * (double)rows * (double)d * 4.0;
    if (est > 9.0e18) return ATTN_ERR_INVALID_ARG;
    const size_t po_b = (size_t)n_parts * rows * d * 4, pl_b = (size_t)n_parts * rows * 4;
    const size_t o_b = (size_t)rows * d * eout, l_b = lse ? (size_t)rows * 4 : 0;
    if (!o_parts || !lse_parts || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned(o_parts, 4) || !aligned(lse_parts, 4) || !aligned(o, eout) ||
        (lse && !aligned(lse, 4)))
        return ATTN_ERR_INVALID_ARG;
    if (overlap(o, o_b, o_parts, po_b) || overlap(o, o_b, lse_parts, pl_b) ||
        overlap(lse, l_b, o_parts, po_b) || overlap(lse, l_b, lse_parts, pl_b) ||
        overlap(o, o_b, lse, l_b))
        return ATTN_ERR_INVALID_ARG;
    const int st = check_device();
    if (st != ATTN_OK) return st;
    return launch_merge(o_parts, lse_parts, n_parts, rows, d, o, lse, out_dtype,
                        (cudaStream_t)stream);
}

int attn_check_status(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_to_status(e);
    int *dptr = status_word_device_ptr();
    if (!dptr) return ATTN_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, dptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(dptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (word & kStatusBounds) return ATTN_ERR_BOUNDS;
    if (word & kStatusTimeout) return ATTN_ERR_TIMEOUT;
    return ATTN_OK;
}

#ifdef ATTN_TEST_EXPORTS
int attn_test_set_hook(int hook, uint64_t timeout_ns) {
    if (hook < 0 || hook > 1) return ATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_hook = hook;
    if (timeout_ns) g_watchdog_ns = timeout_ns;
    return ATTN_OK;
}
#endif  // ATTN_TEST_EXPORTS

}  // extern "C"
