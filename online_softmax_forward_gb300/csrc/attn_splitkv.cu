// attn_splitkv.cu -- split-KV attention forward for a few query rows per head
// (decode), and the merge of partial results.
//
// For Sq much smaller than Skv one CTA per (batch, head) leaves most of the
// GPU idle.  The keys of every head are cut into n_splits contiguous ranges;
// each range is processed by its own CTAs, which write a partial result
// (o_part = the softmax-weighted average of the range's values, lse_part =
// the log-sum-exp of the range's scaled scores) into a caller-provided
// workspace.  A second kernel merges the partial results of each row with
// the online-softmax update of huhohoo "tiled-online-softmax" ("Online
// normalization") applied to whole states, the step aiml.sh
// "verify-tiled-attention" (tiled_flash_attention) takes whenever a new key
// block raises the running maximum:
//     M = max_s lse_s,  w_s = exp(lse_s - M),  o = sum_s w_s o_s / sum_s w_s,
//     lse = M + ln(sum_s w_s).
// The merge is also exported on its own (attn_merge), for results computed
// over key shards elsewhere.  Up to 32 parts it runs one warp per row (8 rows
// per CTA, lane s holds w_s, the lanes split the columns); beyond that, one
// CTA per row.
//
// Partial kernel: CTA (bh, split, block of RB query rows).  Each warp walks
// its own 32-key tiles of the split (tiles warp, warp + W, ...), staged in
// shared memory with 16-byte cp.async (each instruction of the warp copies
// 512 contiguous bytes) in a ring of kStages tiles per warp, and keeps
// its own running max m, normaliser l and accumulator a for every row:
// lane = key for the scores (q pre-multiplied by scale * log2 e), warp
// shuffles for the tile max and sum, lanes over the head dimension for P.V.
// The warps' states are merged through shared memory at the end.  All
// arithmetic is fp32 (16-bit inputs are widened on use).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "attn_internal.h"

namespace attn {

// Scratch of attn_fwd_splitkv_noalloc: a fixed array in device memory, so
// that the call needs no allocation.  Every device that loads the library
// holds it until the process exits.  Host code cannot use the name as an
// address; the address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kTileKeys = 32;  // keys per warp tile: one per lane
constexpr size_t kSkvSmemLimit = 227 * 1024;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte global -> shared copy; src_bytes = 0 writes zeros without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// 16 bytes of T widened to fp32.
template <typename T>
struct Unpack16;
template <>
struct Unpack16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void run(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
};
template <>
struct Unpack16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void run(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // a bf16 is the high half of an fp32
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <>
struct Unpack16<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void run(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
};

template <int D, typename T>
struct SkvCfg {
    static constexpr int kElems16 = 16 / (int)sizeof(T);  // elements per 16-byte chunk
    static constexpr int kChunks = D / kElems16;            // 16-byte chunks per row
    // Staged row stride: D elements + 16 bytes, an odd number of 16-byte
    // units, so that the 8 lanes of one shared-memory phase reading chunk c
    // of 8 different rows hit 8 different bank groups.
    static constexpr int kRow = D * (int)sizeof(T) + 16;
    static constexpr int kTile = kTileKeys * kRow;  // one K or V tile
    static constexpr int kStage = 2 * kTile;        // K and V
    // 3 stages per warp keep two tiles in flight while one is computed
    static constexpr int kStages = 3;
    static constexpr int kWarpRing = kStages * kStage;
    static constexpr int kWarps = (4 * kWarpRing <= 210 * 1024) ? 4 : 2;
    static_assert((kRow / 16) % 2 == 1, "row stride must be an odd number of 16-byte units");
};

template <int D, typename T, int RB>
constexpr size_t skv_smem_bytes() {
    using C = SkvCfg<D, T>;
    return (size_t)RB * D * 4 + (size_t)C::kWarps * ((size_t)C::kWarpRing + (size_t)RB * kTileKeys * 4);
}

template <int D, typename T, int RB>
__global__ void __launch_bounds__(SkvCfg<D, T>::kWarps * 32)
splitkv_partial_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       float *__restrict__ part_o, float *__restrict__ part_lse, int BH, int Sq,
                       int Skv, int causal, float sl2, int chunk, int *status) {
    using C = SkvCfg<D, T>;
    using U = Unpack16<T>;
    constexpr int W = C::kWarps;
    constexpr int CPL = (D + 31) / 32;  // output columns per lane
    extern __shared__ __align__(16) uint8_t sm[];
    float *Qs = reinterpret_cast<float *>(sm);  // [RB][D], scaled into log2 units

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, split = blockIdx.y;
    const int row0 = blockIdx.z * RB;
    const int nrows = min(RB, Sq - row0);
    // the merge kernel that follows may be scheduled now; it waits for this
    // grid to complete before it reads anything (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the whole block (bh, split and row0 are block-uniform); the partial
    // results it skips are then never written
    if (!in_bounds(bh < BH && row0 < Sq, status)) return;
    const int off = Skv - Sq;  // causal: key j visible to query i iff j <= i + off
    const int kb = split * chunk;
    int ke = min(Skv, kb + chunk);
    if (causal) ke = min(ke, row0 + nrows + off);  // past the last row's limit
    const int ntiles = ke > kb ? (ke - kb + kTileKeys - 1) / kTileKeys : 0;

    for (int t = threadIdx.x; t < RB * D; t += blockDim.x) {
        const int i = t / D, c = t % D;
        const size_t qi = ((size_t)bh * Sq + row0 + i) * D + c;
        Qs[t] = i < nrows && in_bounds(qi < (size_t)BH * Sq * D, status)
                    ? to_f32<T>(q[qi]) * sl2 : 0.f;
    }
    __syncthreads();

    uint8_t *ring = sm + (size_t)RB * D * 4 + (size_t)warp * (C::kWarpRing + RB * kTileKeys * 4);
    float *Ps = reinterpret_cast<float *>(ring + C::kWarpRing);  // [RB][32] probabilities
    const T *kg = k + (size_t)bh * Skv * D;
    const T *vg = v + (size_t)bh * Skv * D;

    float m[RB], l[RB], acc[RB][CPL];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) acc[i][u] = 0.f;
    }

    // K and V rows of tile `tile` into ring stage `stage`: 16-byte piece g of
    // the tile (row g / kChunks, chunk g % kChunks) is copied by lane g % 32,
    // so each instruction of the warp reads 512 contiguous bytes.  Keys past
    // the range are zero-filled (never read from global memory).
    auto issue = [&](int tile, int stage) {
        const uint32_t kbase = smem_u32(ring + stage * C::kStage);
#pragma unroll
        for (int it2 = 0; it2 < C::kChunks; ++it2) {
            const int g = it2 * 32 + lane;
            const int r = g / C::kChunks, c = g % C::kChunks;
            const int j = kb + tile * kTileKeys + r;
            const bool in = j < ke &&
                            in_bounds((size_t)j * D + (c + 1) * C::kElems16 <= (size_t)Skv * D, status);
            const size_t src = (size_t)(in ? j : kb) * D + c * C::kElems16;
            const uint32_t dst = kbase + r * C::kRow + c * 16;
            cp_async16(dst, kg + src, in ? 16 : 0);
            cp_async16(dst + C::kTile, vg + src, in ? 16 : 0);
        }
    };

    // prologue: the first kStages - 1 tiles of this warp
#pragma unroll
    for (int s = 0; s < C::kStages - 1; ++s) {
        if (warp + s * W < ntiles) issue(warp + s * W, s);
        cp_async_commit();
    }
    int it = 0;
    for (int tile = warp; tile < ntiles; tile += W, ++it) {
        const int stage = it % C::kStages;
        const int ahead = tile + (C::kStages - 1) * W;
        if (ahead < ntiles) issue(ahead, (it + C::kStages - 1) % C::kStages);
        cp_async_commit();
        cp_async_wait<C::kStages - 1>();  // this tile's copies have landed
        __syncwarp();  // ... for every lane, which also copied other lanes' rows
        const uint8_t *Kt = ring + stage * C::kStage;
        const uint8_t *Vt = Kt + C::kTile;
        const int j = kb + tile * kTileKeys + lane;

        // scores of this lane's key against every row (log2 units)
        float sc[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) sc[i] = 0.f;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
            float kf[U::N];
            U::run(*reinterpret_cast<const uint4 *>(Kt + lane * C::kRow + c * 16), kf);
#pragma unroll
            for (int e = 0; e < U::N; e += 4) {
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(Qs + i * D + c * U::N + e);
                    sc[i] = fmaf(q4.x, kf[e], sc[i]);
                    sc[i] = fmaf(q4.y, kf[e + 1], sc[i]);
                    sc[i] = fmaf(q4.z, kf[e + 2], sc[i]);
                    sc[i] = fmaf(q4.w, kf[e + 3], sc[i]);
                }
            }
        }
        // online softmax update per row; m and l are the same in every lane
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const bool vis = i < nrows && j < ke && (!causal || j <= row0 + i + off);
            const float s = vis ? sc[i] : -INFINITY;
            const float mn = fmaxf(m[i], warp_max(s));
            float p = 0.f, alpha = 1.f;
            if (mn != -INFINITY) {
                p = ex2(s - mn);         // 0 for an excluded key
                alpha = ex2(m[i] - mn);  // 0 while nothing has been accumulated
            }
            l[i] = l[i] * alpha + warp_sum(p);
            m[i] = mn;
#pragma unroll
            for (int u = 0; u < CPL; ++u) acc[i][u] *= alpha;
            Ps[i * kTileKeys + lane] = p;
        }
        __syncwarp();
        // a += P . V, lanes over the head dimension
#pragma unroll
        for (int jj = 0; jj < kTileKeys; jj += 4) {
            float vv[4][CPL];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const T *vrow = reinterpret_cast<const T *>(Vt + (jj + e) * C::kRow);
#pragma unroll
                for (int u = 0; u < CPL; ++u) {
                    const int c = lane + 32 * u;
                    vv[e][u] = c < D ? to_f32<T>(vrow[c]) : 0.f;
                }
            }
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const float4 p4 = *reinterpret_cast<const float4 *>(Ps + i * kTileKeys + jj);
#pragma unroll
                for (int u = 0; u < CPL; ++u) {
                    acc[i][u] = fmaf(p4.x, vv[0][u], acc[i][u]);
                    acc[i][u] = fmaf(p4.y, vv[1][u], acc[i][u]);
                    acc[i][u] = fmaf(p4.z, vv[2][u], acc[i][u]);
                    acc[i][u] = fmaf(p4.w, vv[3][u], acc[i][u]);
                }
            }
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the warps' states row by row (the staging area is reused)
    float *Mw = reinterpret_cast<float *>(sm + (size_t)RB * D * 4);  // [W][RB]
    float *Lw = Mw + W * RB;                                          // [W][RB]
    float *Aw = Lw + W * RB;                                          // [W][RB][D]
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            Mw[warp * RB + i] = m[i];
            Lw[warp * RB + i] = l[i];
        }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
            const int c = lane + 32 * u;
            if (c < D) Aw[(warp * RB + i) * D + c] = acc[i][u];
        }
    __syncthreads();
    const size_t prow = ((size_t)split * BH + bh) * Sq + row0;  // first row of this block
    const size_t part_rows = (size_t)gridDim.y * BH * Sq;        // rows of the workspace used
    if (!in_bounds(prow + nrows <= part_rows, status)) return;   // block-uniform
    for (int t = threadIdx.x; t < nrows * D; t += blockDim.x) {
        const int i = t / D, c = t % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, Mw[w * RB + i]);
        float o = 0.f;
        if (M != -INFINITY) {
            float L = 0.f, A = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float e = ex2(Mw[w * RB + i] - M);
                L = fmaf(Lw[w * RB + i], e, L);
                A = fmaf(Aw[(w * RB + i) * D + c], e, A);
            }
            o = A / L;
        }
        part_o[(prow + i) * D + c] = o;
    }
    for (int i = threadIdx.x; i < nrows; i += blockDim.x) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, Mw[w * RB + i]);
        float L = 0.f;
        if (M != -INFINITY)
#pragma unroll
            for (int w = 0; w < W; ++w) L = fmaf(Lw[w * RB + i], ex2(Mw[w * RB + i] - M), L);
        part_lse[prow + i] = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f;
    }
}

// Merge of n_parts partial results [n_parts][rows][d] / [n_parts][rows] into
// o [rows][d] and lse [rows].  merge_kernel, for more than 32 parts: one CTA
// of kMergeThreads per row; the weights exp(lse_p - M) are computed once
// into shared memory; each thread then sums its columns over the parts.
constexpr int kMergeThreads = 128;

__device__ __forceinline__ float block_reduce(float x, float *red, bool is_max) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    x = is_max ? warp_max(x) : warp_sum(x);
    __syncthreads();  // red may still be read by a previous reduction
    if (lane == 0) red[warp] = x;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

template <typename TO>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const float *__restrict__ po, const float *__restrict__ pl, int n_parts,
             int64_t rows, int d, TO *__restrict__ o, float *__restrict__ lse, int *status) {
    extern __shared__ float wts[];  // [n_parts]
    // launched as a programmatic dependent of the partial kernel: its results
    // are complete and visible after this wait (no-op without a predecessor)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float red[kMergeThreads / 32];
    const int64_t row = blockIdx.x;
    // every index below is p * rows + row or (p * rows + row) * d + c with
    // p < n_parts, c < d: inside the buffers once row < rows
    if (!in_bounds(row < rows, status)) return;  // block-uniform
    TO *orow = o + row * d;
    float M = -INFINITY;
    for (int p = threadIdx.x; p < n_parts; p += kMergeThreads)
        M = fmaxf(M, pl[(int64_t)p * rows + row]);
    M = block_reduce(M, red, true);
    if (M == -INFINITY) {  // no part saw a key: o = 0, lse = -inf
        for (int c = threadIdx.x; c < d; c += kMergeThreads) orow[c] = from_f32<TO>(0.f);
        if (lse && threadIdx.x == 0) lse[row] = -INFINITY;
        return;
    }
    float L = 0.f;
    for (int p = threadIdx.x; p < n_parts; p += kMergeThreads) {
        const float lp = pl[(int64_t)p * rows + row];
        const float w = lp == -INFINITY ? 0.f : expf(lp - M);  // a part with no key weighs 0
        wts[p] = w;
        L += w;
    }
    L = block_reduce(L, red, false);  // also makes wts visible to every thread
    const float inv = 1.f / L;
    for (int c = threadIdx.x; c < d; c += kMergeThreads) {
        float a = 0.f;
        const float *col = po + row * d + c;
#pragma unroll 4
        for (int p = 0; p < n_parts; ++p) {
            const float w = wts[p];
            if (w != 0.f) a = fmaf(w, col[(int64_t)p * rows * d], a);
        }
        orow[c] = from_f32<TO>(a * inv);
    }
    if (lse && threadIdx.x == 0) lse[row] = M + logf(L);
}

// One warp per row, for up to 32 parts: lane p holds the weight of part p,
// the lanes split the columns, so each part's row is one coalesced read and
// no block barrier is needed.  With many rows (the heads and queries of a
// sequence-sharded prefill: 262,144 rows) this runs at memory speed, where
// one CTA per row spends its time on CTA scheduling and block reductions.
// The sums are taken in the same order as merge_kernel's, so both give the
// same bits.
constexpr int kMergeRowWarps = 8;  // rows per CTA

template <typename TO>
__global__ void __launch_bounds__(kMergeRowWarps * 32)
merge_rows_kernel(const float *__restrict__ po, const float *__restrict__ pl, int n_parts,
                  int64_t rows, int d, TO *__restrict__ o, float *__restrict__ lse,
                  int *status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kMergeRowWarps + (threadIdx.x >> 5);
    if (row >= rows) return;  // the whole warp: one row per warp
    // lane p < n_parts reads part p: the indices stay inside the buffers when
    // the parts fit one lane each
    if (!in_bounds(n_parts <= 32 && row >= 0, status)) return;
    const float lp = lane < n_parts ? pl[(int64_t)lane * rows + row] : -INFINITY;
    const float M = warp_max(lp);
    TO *orow = o + row * d;
    if (M == -INFINITY) {  // no part saw a key: o = 0, lse = -inf
        for (int c = lane; c < d; c += 32) orow[c] = from_f32<TO>(0.f);
        if (lse && lane == 0) lse[row] = -INFINITY;
        return;
    }
    const float w = lp == -INFINITY ? 0.f : expf(lp - M);  // a part with no key weighs 0
    const float L = warp_sum(w);
    const float inv = 1.f / L;
    const float *prow = po + row * d;
    const int64_t pstride = rows * d;
    for (int c0 = 0; c0 < d; c0 += 128) {  // four columns per lane in flight
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        for (int q = 0; q < n_parts; ++q) {
            const float wq = __shfl_sync(0xffffffffu, w, q);
            if (wq == 0.f) continue;  // the same for the whole warp
            const float *col = prow + (int64_t)q * pstride;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < d) a[u] = fmaf(wq, col[c], a[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + lane + 32 * u;
            if (c < d) orow[c] = from_f32<TO>(a[u] * inv);
        }
    }
    if (lse && lane == 0) lse[row] = M + logf(L);
}

template <typename TO>
int launch_merge_t(const float *po, const float *pl, int n_parts, int64_t rows, int d, void *o,
                   float *lse, cudaStream_t stream) {
    if (rows == 0) return ATTN_OK;
    if (rows > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    const bool by_warp = n_parts <= 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(by_warp ? (unsigned)((rows + kMergeRowWarps - 1) / kMergeRowWarps)
                               : (unsigned)rows);
    cfg.blockDim = dim3(by_warp ? kMergeRowWarps * 32 : kMergeThreads);
    cfg.dynamicSmemBytes = by_warp ? 0 : (size_t)n_parts * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int *status = status_word_device_ptr();
    if (!status) return ATTN_ERR_CUDA;
    const cudaError_t e =
        by_warp ? cudaLaunchKernelEx(&cfg, merge_rows_kernel<TO>, po, pl, n_parts, rows, d,
                                     reinterpret_cast<TO *>(o), lse, status)
                : cudaLaunchKernelEx(&cfg, merge_kernel<TO>, po, pl, n_parts, rows, d,
                                     reinterpret_cast<TO *>(o), lse, status);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

template <int D, typename T, int RB>
int launch_partial(const void *q, const void *k, const void *v, float *po, float *pl,
                   const Problem &p, int n_eff, int chunk, cudaStream_t stream) {
    constexpr size_t smem = skv_smem_bytes<D, T, RB>();
    static_assert(smem <= kSkvSmemLimit, "split-KV shared memory");
    auto kern = splitkv_partial_kernel<D, T, RB>;
    if (!set_smem_limit_once(reinterpret_cast<const void *>(kern), (int)smem)) return ATTN_ERR_LAUNCH;
    const dim3 grid((unsigned)p.bh(), (unsigned)n_eff, (unsigned)((p.Sq + RB - 1) / RB));
    int *status = status_word_device_ptr();
    if (!status) return ATTN_ERR_CUDA;
    kern<<<grid, SkvCfg<D, T>::kWarps * 32, smem, stream>>>(
        reinterpret_cast<const T *>(q), reinterpret_cast<const T *>(k),
        reinterpret_cast<const T *>(v), po, pl, (int)p.bh(), p.Sq, p.Skv, p.causal,
        p.scale * 1.4426950408889634f, chunk, status);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

template <int D, typename T>
int launch_partial_rb(const void *q, const void *k, const void *v, float *po, float *pl,
                      const Problem &p, int n_eff, int chunk, cudaStream_t stream) {
    if (p.Sq <= 1) return launch_partial<D, T, 1>(q, k, v, po, pl, p, n_eff, chunk, stream);
    return launch_partial<D, T, kSplitRowBlock>(q, k, v, po, pl, p, n_eff, chunk, stream);
}

template <typename T>
int launch_partial_d(const void *q, const void *k, const void *v, float *po, float *pl,
                     const Problem &p, int n_eff, int chunk, cudaStream_t stream) {
    switch (p.d) {
    case 16: return launch_partial_rb<16, T>(q, k, v, po, pl, p, n_eff, chunk, stream);
    case 32: return launch_partial_rb<32, T>(q, k, v, po, pl, p, n_eff, chunk, stream);
    case 64: return launch_partial_rb<64, T>(q, k, v, po, pl, p, n_eff, chunk, stream);
    case 128: return launch_partial_rb<128, T>(q, k, v, po, pl, p, n_eff, chunk, stream);
    default: return ATTN_ERR_INVALID_ARG;
    }
}

int warps_for(int d, int dtype) {
    const size_t row = (size_t)d * elem_bytes_in(dtype) + 16;
    return 4 * 3 * 2 * kTileKeys * row <= 210 * 1024 ? 4 : 2;
}

// Resident CTAs per SM of the partial kernel for this problem (>= 1).
template <int D, typename T, int RB>
int occupancy_t() {
    constexpr size_t smem = skv_smem_bytes<D, T, RB>();
    auto kern = splitkv_partial_kernel<D, T, RB>;
    int n = 0;
    if (!set_smem_limit_once(reinterpret_cast<const void *>(kern), (int)smem) ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, SkvCfg<D, T>::kWarps * 32,
                                                      smem) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}
template <int D, typename T>
int occupancy_rb(int Sq) {
    return Sq <= 1 ? occupancy_t<D, T, 1>() : occupancy_t<D, T, kSplitRowBlock>();
}
template <typename T>
int occupancy_d(int d, int Sq) {
    switch (d) {
    case 16: return occupancy_rb<16, T>(Sq);
    case 32: return occupancy_rb<32, T>(Sq);
    case 64: return occupancy_rb<64, T>(Sq);
    default: return occupancy_rb<128, T>(Sq);
    }
}
int splitkv_occupancy(const Problem &p) {
    if (p.dtype == ATTN_F32) return occupancy_d<float>(p.d, p.Sq);
    if (p.dtype == ATTN_BF16 || p.dtype == ATTN_BF16_OUT_F32)
        return occupancy_d<__nv_bfloat16>(p.d, p.Sq);
    return occupancy_d<__half>(p.d, p.Sq);
}

}  // namespace

int splitkv_row_block(int Sq) { return Sq <= 1 ? 1 : kSplitRowBlock; }

namespace {
constexpr int kScratchMaxDev = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kScratchMaxDev];
}  // namespace

// Device address of g_noalloc_scratch on the current device, looked up with
// cudaGetSymbolAddress the first time a device asks and cached after that.
int noalloc_scratch_ptr(void **ptr) {
    constexpr int kMaxDev = kScratchMaxDev;
    void **addr = g_scratch_addr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
                return ATTN_ERR_UNSUPPORTED_DEVICE;
            return ATTN_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return ATTN_OK;
}

void forget_noalloc_scratch(int dev) {
    if (dev < 0 || dev >= kScratchMaxDev) return;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    g_scratch_addr[dev] = nullptr;
}

// Keys per split (a multiple of 32) and the number of non-empty splits for a
// requested split count.
void splitkv_chunking(int Skv, int n_splits, int *chunk, int *n_eff) {
    int c = (Skv + n_splits - 1) / n_splits;
    c = ((c + kTileKeys - 1) / kTileKeys) * kTileKeys;
    if (c < kTileKeys) c = kTileKeys;
    *chunk = c;
    *n_eff = Skv > 0 ? (Skv + c - 1) / c : 1;
}

// Cost of one CTA beyond its key tiles, in units of one 32-key tile step per
// warp.  Fitted to split-count sweeps of a 4 x 32-head, 32768-key decode on
// GB300, where each CTA costs about 3 us on top of its tiles (about two tile
// steps): time grows with the split count through the merge kernel and the
// partial kernel alike.
constexpr double kCtaFixedTiles = 2.0;

// The split count with the smallest estimated time: waves of CTAs over the
// GPU's resident slots times (the key tiles each warp walks + the fixed cost
// per CTA), plus a small charge per split for the merge; at least two tiles
// per warp in a split.

int splitkv_choose(const Problem &p, int sms) {
    const int64_t rows_blocks = (p.Sq + splitkv_row_block(p.Sq) - 1) / splitkv_row_block(p.Sq);
    const int64_t base = p.bh() * rows_blocks;
    const int W = warps_for(p.d, p.dtype);
    const int64_t slots = (int64_t)(sms > 0 ? sms : 1) * splitkv_occupancy(p);
    const int64_t min_keys = 2LL * W * kTileKeys;
    int64_t max_n = (p.Skv + min_keys - 1) / min_keys;
    if (max_n < 1) max_n = 1;
    if (max_n > kMaxSplits) max_n = kMaxSplits;
    int best = 1;
    double best_cost = 1e300;
    for (int n = 1; n <= max_n; ++n) {
        int chunk = 0, n_eff = 0;
        splitkv_chunking(p.Skv, n, &chunk, &n_eff);
        if (n_eff != n) continue;  // the same chunking as a smaller count
        const int64_t waves = (base * n + slots - 1) / slots;
        const int64_t tiles = ((chunk + kTileKeys - 1) / kTileKeys + W - 1) / W;
        const double cost = (double)waves * ((double)tiles + kCtaFixedTiles) + 0.02 * n;
        if (cost < best_cost) {
            best_cost = cost;
            best = n;
        }
    }
    return best;
}

int launch_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                   const Problem &p, int n_splits, float *part_o, float *part_lse,
                   cudaStream_t stream) {
    int chunk = 0, n_eff = 0;
    splitkv_chunking(p.Skv, n_splits, &chunk, &n_eff);
    int st = ATTN_ERR_INVALID_ARG;
    switch (p.dtype) {
    case ATTN_F32:
        st = launch_partial_d<float>(q, k, v, part_o, part_lse, p, n_eff, chunk, stream);
        break;
    case ATTN_BF16:
    case ATTN_BF16_OUT_F32:
        st = launch_partial_d<__nv_bfloat16>(q, k, v, part_o, part_lse, p, n_eff, chunk, stream);
        break;
    case ATTN_F16:
    case ATTN_F16_OUT_F32:
        st = launch_partial_d<__half>(q, k, v, part_o, part_lse, p, n_eff, chunk, stream);
        break;
    }
    if (st != ATTN_OK) return st;
    const int out = (p.dtype == ATTN_BF16) ? ATTN_BF16 : (p.dtype == ATTN_F16) ? ATTN_F16 : ATTN_F32;
    return launch_merge(part_o, part_lse, n_eff, p.bh() * p.Sq, p.d, o, lse, out, stream);
}

int launch_merge(const float *po, const float *pl, int n_parts, int64_t rows, int d, void *o,
                 float *lse, int out_dtype, cudaStream_t stream) {
    switch (out_dtype) {
    case ATTN_F32: return launch_merge_t<float>(po, pl, n_parts, rows, d, o, lse, stream);
    case ATTN_BF16: return launch_merge_t<__nv_bfloat16>(po, pl, n_parts, rows, d, o, lse, stream);
    case ATTN_F16: return launch_merge_t<__half>(po, pl, n_parts, rows, d, o, lse, stream);
    default: return ATTN_ERR_INVALID_ARG;
    }
}

}  // namespace attn
