// attn_f32.cu -- fp32 exact attention forward on CUDA cores.
//
// The tiled online-softmax loop of aiml.sh "verify-tiled-attention"
// (tiled_flash_attention) with the update of huhohoo "tiled-online-softmax"
// ("Online normalization"), in fp32, for small and latency-bound shapes and
// for tile-size invariance tests.  Tile sizes are runtime values.
//
// Three kernels compute the same thing:
//
// attn_f32_tiled_kernel (attn_fwd): fixed tiles of 32 query rows by 64 keys,
// 128 threads, register-blocked.  Thread (ty, tx), ty in [0, 8), tx in
// [0, 16), owns the 4 x 4 scores of rows ty + 8i and keys tx + 16j, so every
// float4 read from shared memory feeds four FMAs; the row maximum is reduced
// over the 16 lanes of a half-warp every tile, the row sum once at the end.
// It also owns O for rows ty + 8i and columns tx*W + 64c (W = 4 for d >= 64),
// kept in registers across the whole key loop together with the row state
// (m, l), so only P goes through shared memory (written and read by the same
// half-warp).  Only tiles that some row of the block cannot see whole are
// masked.  K/V tiles go through cp.async, in two stages per warpgroup or in
// one, where the next K loads while this tile's softmax and P V run and the
// next V while the next scores are taken.  On grids with fewer blocks than
// SMs, 2 or 4 warpgroups per block take the key tiles in turn and merge their
// states at the end, each warpgroup finishing a quarter (or half) of the rows.
//
// attn_f32_keysplit_kernel (attn_fwd at d = 64 on grids of fewer than four
// blocks per SM): 32 query rows per block, 8 warps; each warp walks every
// eighth 32-key tile with its own online-softmax state for all 32 rows, in
// 8 x 4 score and 8 x 8 output blocks per thread (12 float4 shared-memory
// reads per 128 FMAs, against 8 per 64 above), and the warps' states are
// combined at the end.
//
// attn_f32_kernel (attn_fwd_f32_blocked): runtime tile sizes, down to 1 x 1,
// for the tile-size invariance tests.  One CTA owns one block of block_q
// query rows and walks the key/value blocks of block_kv rows; each block is
// staged in shared memory once and used by every query row of the CTA.  One
// warp handles one query row at a time: lanes split the keys of the tile for
// the scores, warp shuffles give the tile maximum and the sum of
// exponentials, and lanes split the head dimension for the P.V product.
// Per-row state (running max m, normaliser l, accumulator a) lives in shared
// memory between key tiles.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kWarps = 8;     // warps per CTA
constexpr int kPad = 4;       // row padding of the Q and K tiles, in floats
constexpr size_t kSmemLimit = 200 * 1024;

__host__ __device__ inline size_t f32_smem_bytes(int d, int bq, int bkv) {
    return sizeof(float) * ((size_t)bq * (d + kPad) + (size_t)bkv * (d + kPad) +
                            (size_t)bkv * d + (size_t)bq * d + 2 * (size_t)bq +
                            (size_t)kWarps * bkv);
}

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

// Copy `rows` rows of D floats from global (row-major, contiguous) into a
// shared tile with row stride `ld` floats, 16 bytes per thread per step.
// `avail` is the number of rows from src to the end of its [S, D] slice
// (the extent the bounds-checking build tests each row against).
template <int D>
__device__ __forceinline__ void stage_rows(float *dst, int ld, const float *__restrict__ src,
                                           int rows, int avail, int *status) {
    constexpr int V4 = D / 4;
    const int n = rows * V4;
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const int r = t / V4, c = (t % V4) * 4;
        if (!in_bounds(r < avail, status)) continue;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(src + (size_t)r * D + c));
        *reinterpret_cast<float4 *>(dst + r * ld + c) = x;
    }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                int BH, int Sq, int Skv, int causal, float scale, int block_q, int block_kv,
                int nqb, int *status) {
    extern __shared__ __align__(16) float sm[];
    constexpr int LD = D + kPad;
    constexpr int CPL = (D + 31) / 32;  // output columns per lane
    float *Qs = sm;                                  // [block_q][LD]
    float *Ks = Qs + (size_t)block_q * LD;           // [block_kv][LD]
    float *Vs = Ks + (size_t)block_kv * LD;          // [block_kv][D]
    float *As = Vs + (size_t)block_kv * D;           // [block_q][D] accumulators
    float *Ms = As + (size_t)block_q * D;            // [block_q] running max
    float *Ls = Ms + block_q;                        // [block_q] running sum
    float *Ps = Ls + block_q;                        // [kWarps][block_kv] scores / probabilities

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.x / nqb;
    const int qb = blockIdx.x % nqb;
    const int q_start = qb * block_q;
    const int q_end = min(q_start + block_q, Sq);
    const int rows = q_end - q_start;
    const int off = Skv - Sq;  // causal: key j visible to query i iff j <= i + off
    float *Pw = Ps + warp * block_kv;
    if (!in_bounds(bh < BH, status)) return;  // the whole block: bh is block-uniform

    const float *qg = q + ((size_t)bh * Sq + q_start) * D;
    const float *kg = k + (size_t)bh * Skv * D;
    const float *vg = v + (size_t)bh * Skv * D;

    stage_rows<D>(Qs, LD, qg, rows, Sq - q_start, status);
    for (int t = threadIdx.x; t < rows * D; t += blockDim.x) As[t] = 0.f;
    for (int t = threadIdx.x; t < rows; t += blockDim.x) {
        Ms[t] = -INFINITY;
        Ls[t] = 0.f;
    }

    // Keys beyond kv_stop are invisible to every row of this block.
    const int kv_stop = causal ? min(Skv, q_end + off) : Skv;
    for (int kv_start = 0; kv_start < kv_stop; kv_start += block_kv) {
        const int kv_end = min(kv_start + block_kv, Skv);
        __syncthreads();  // previous tile fully consumed (and Q staged)
        stage_rows<D>(Ks, LD, kg + (size_t)kv_start * D, kv_end - kv_start, Skv - kv_start, status);
        stage_rows<D>(Vs, D, vg + (size_t)kv_start * D, kv_end - kv_start, Skv - kv_start, status);
        __syncthreads();

        for (int r = warp; r < rows; r += kWarps) {
            const int i = q_start + r;
            const int lim = causal ? min(kv_end, i + off + 1) : kv_end;
            const int nvis = lim - kv_start;  // visible keys of this row in this tile
            if (nvis <= 0) continue;          // the row skips a tile with no visible key

            // scores of this tile and their maximum
            const float *qr = Qs + r * LD;
            float tmax = -INFINITY;
            for (int jj = lane; jj < nvis; jj += 32) {
                const float *kr = Ks + jj * LD;
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < D; c += 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(qr + c);
                    const float4 b = *reinterpret_cast<const float4 *>(kr + c);
                    acc = fmaf(a.x, b.x, acc);
                    acc = fmaf(a.y, b.y, acc);
                    acc = fmaf(a.z, b.z, acc);
                    acc = fmaf(a.w, b.w, acc);
                }
                const float s = acc * scale;
                Pw[jj] = s;
                tmax = fmaxf(tmax, s);
            }
            tmax = warp_max(tmax);
            const float m_old = Ms[r];
            const float m_new = fmaxf(m_old, tmax);
            // rescale of the previous state; nothing to rescale before the first tile
            const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
            float psum = 0.f;
            for (int jj = lane; jj < nvis; jj += 32) {
                const float p = expf(Pw[jj] - m_new);
                Pw[jj] = p;
                psum += p;
            }
            psum = warp_sum(psum);
            __syncwarp();

            // a = a * alpha + P @ V_tile, lanes over the head dimension
            float *ar = As + r * D;
#pragma unroll
            for (int u = 0; u < CPL; ++u) {
                const int c = lane + 32 * u;
                if (c < D) {
                    float acc = ar[c] * alpha;
                    for (int jj = 0; jj < nvis; ++jj) acc = fmaf(Pw[jj], Vs[jj * D + c], acc);
                    ar[c] = acc;
                }
            }
            __syncwarp();
            if (lane == 0) {
                Ls[r] = Ls[r] * alpha + psum;
                Ms[r] = m_new;
            }
            __syncwarp();
        }
    }
    __syncthreads();

    // output = a / l; lse = m + ln l; rows that saw no key: 0 and -inf
    for (int r = warp; r < rows; r += kWarps) {
        const int i = q_start + r;
        const float l = Ls[r];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *orow = o + ((size_t)bh * Sq + i) * D;
        const bool row_in = in_bounds(((size_t)bh * Sq + i + 1) * D <= (size_t)BH * Sq * D, status);
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
            const int c = lane + 32 * u;
            if (c < D && row_in) orow[c] = As[r * D + c] * inv;
        }
        if (lse && lane == 0 && row_in) lse[(size_t)bh * Sq + i] = l > 0.f ? Ms[r] + logf(l) : -INFINITY;
    }
}

// ---------------------------------------------------------------- tiled kernel
constexpr int kTQ = 32;         // query rows per CTA
constexpr int kTK = 64;         // keys per tile
constexpr int kWG = 128;        // threads of one warpgroup
constexpr int kLdP = kTK + 16;  // P row stride: rows 2 apart land 32 banks apart

// KS warpgroups share the query block and take the key tiles in turn
// (tile j goes to warpgroup j mod KS); each has its own P and NS stages of
// K and V.  With two stages the next tile loads whole during this one; with
// one, the next K loads once this tile's scores are taken and the next V once
// its P V is done.
template <int D, int KS, int NS>
struct TiledCfg {
    static constexpr int kLd = D + 4;                // Q and K row stride, floats
    static constexpr int kW = D >= 64 ? 4 : D / 16;  // contiguous O columns per group
    static constexpr int kNC = D / (16 * kW);        // column groups per thread
    static constexpr int kNS = NS;
    static constexpr int kStageK = kNS * kTK * kLd;  // floats of one warpgroup's K stages
    static constexpr int kStageV = kNS * kTK * D;
    static constexpr int kOffK = kTQ * kLd;
    static constexpr int kOffV = kOffK + KS * kStageK;
    static constexpr int kOffP = kOffV + KS * kStageV;
    static constexpr size_t kSmemBytes = sizeof(float) * (size_t)(kOffP + KS * kTQ * kLdP);
    // per-thread state a second warpgroup hands over: m, l and O, 4 rows each
    static constexpr int kStateFloats = 8 + 4 * kNC * kW;
    static_assert(KS == 1 || kStateFloats * kWG <= kStageK, "state must fit the K stages");
    static_assert(NS == 1 || NS == 2, "one or two stages");
};

__device__ __forceinline__ uint32_t smem_addr(const void *ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
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
__device__ __forceinline__ void cp_async_wait1() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait0() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// barrier of the 128 threads of warpgroup g (ids 1.., 0 is __syncthreads)
__device__ __forceinline__ void wg_sync(int g) {
    asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "n"(kWG) : "memory");
}

// rows [row0, row0 + n) of a [S, D] slice into a shared tile of row stride
// ld by `nthr` threads (this one is `tid`); rows at or past `valid` are
// zero-filled.
template <int D>
__device__ __forceinline__ void stage_async(float *dst, int ld, const float *__restrict__ src,
                                            int row0, int n, int valid, int tid, int nthr,
                                            int *status) {
    constexpr int V4 = D / 4;
    for (int f = tid; f < n * V4; f += nthr) {
        const int r = f / V4, c = (f - r * V4) * 4;
        const bool in = row0 + r < valid &&
                        in_bounds((size_t)(row0 + r) * D + c + 4 <= (size_t)valid * D, status);
        const float *s = in ? src + (size_t)(row0 + r) * D + c : src;
        cp_async16(smem_addr(dst + r * ld + c), s, in ? 16 : 0);
    }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int D, int KS, int NS>
__global__ void __launch_bounds__(KS * kWG, 1)
attn_f32_tiled_kernel(const float *__restrict__ q, const float *__restrict__ k,
                      const float *__restrict__ v, float *__restrict__ o,
                      float *__restrict__ lse, int BH, int Sq, int Skv, int causal,
                      float scale_log2, int nqb, int *status) {
    using C = TiledCfg<D, KS, NS>;
    constexpr int LD = C::kLd, W = C::kW, NC = C::kNC;
    extern __shared__ __align__(16) float sm[];
    const int g = threadIdx.x / kWG;    // warpgroup
    const int tid = threadIdx.x % kWG;  // thread inside the warpgroup
    float *Qs = sm;
    float *Ks = sm + C::kOffK + g * C::kStageK;  // [kNS][kTK][LD]
    float *Vs = sm + C::kOffV + g * C::kStageV;  // [kNS][kTK][D]
    float *Ps = sm + C::kOffP + g * kTQ * kLdP;  // [kTQ][kLdP]

    const int tx = tid & 15, ty = tid >> 4;
    const int64_t bh = blockIdx.x / nqb;
    const int q0 = (blockIdx.x % nqb) * kTQ;
    const int q_end = min(q0 + kTQ, Sq);
    const int off = Skv - Sq;  // causal: key j visible to query i iff j <= i + off
    if (!in_bounds(bh < BH, status)) return;  // the whole block: bh is block-uniform
    const float *qg = q + (size_t)bh * Sq * D;
    const float *kg = k + (size_t)bh * Skv * D;
    const float *vg = v + (size_t)bh * Skv * D;

    // keys visible to each of this thread's rows: [0, lim[i])
    int lim[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        lim[i] = causal ? min(Skv, q0 + ty + 8 * i + off + 1) : Skv;
    const int kv_stop = causal ? min(Skv, q_end + off) : Skv;
    const int ntiles = kv_stop > 0 ? (kv_stop + kTK - 1) / kTK : 0;
    // keys below kv_all are visible to every row of the block: tiles that end
    // there need no mask
    const int kv_all = causal ? min(Skv, q0 + off + 1) : Skv;

    // m in log2 units; l is this thread's share of the row sum (its own keys),
    // summed over the half-warp once at the end
    float m[4], l[4], acc[4][NC][W];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int w = 0; w < W; ++w) acc[i][c][w] = 0.f;
    }

    // Q and the first K of each warpgroup, then its first V as a second
    // group, so the first S starts while V is still arriving; one CTA barrier:
    // from here on Q is read-only and each warpgroup syncs alone
    if (ntiles > 0) {
        stage_async<D>(Qs, LD, qg, q0, kTQ, Sq, threadIdx.x, KS * kWG, status);
        if (g < ntiles) stage_async<D>(Ks, LD, kg, g * kTK, kTK, Skv, tid, kWG, status);
        cp_async_commit();
        if (g < ntiles) stage_async<D>(Vs, D, vg, g * kTK, kTK, Skv, tid, kWG, status);
        cp_async_commit();
        cp_async_wait1();
    }
    __syncthreads();
    for (int jt = g, n = 0; jt < ntiles; jt += KS, ++n) {
        const int st = C::kNS == 2 ? (n & 1) : 0, kv0 = jt * kTK;
        const bool more = jt + KS < ntiles;
        if constexpr (C::kNS == 2) {
            if (more) {  // the other stage was released at the end of the last tile
                stage_async<D>(Ks + (st ^ 1) * kTK * LD, LD, kg, kv0 + KS * kTK, kTK, Skv, tid, kWG, status);
                stage_async<D>(Vs + (st ^ 1) * kTK * D, D, vg, kv0 + KS * kTK, kTK, Skv, tid, kWG, status);
            }
            cp_async_commit();
            cp_async_wait1();  // everything but the copies just issued has landed
            wg_sync(g);
        }
        // one stage: K of this tile has landed and is visible (prologue or
        // the end of the last tile); V may still be arriving
        const float *Kt = Ks + st * kTK * LD;
        const float *Vt = Vs + st * kTK * D;

        // raw scores Q K^T for rows ty + 8i, keys tx + 16j
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; c += 4) {
            float4 qa[4], kb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                qa[i] = *reinterpret_cast<const float4 *>(Qs + (ty + 8 * i) * LD + c);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                kb[j] = *reinterpret_cast<const float4 *>(Kt + (tx + 16 * j) * LD + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x = s[i][j];
                    x = fmaf(qa[i].x, kb[j].x, x);
                    x = fmaf(qa[i].y, kb[j].y, x);
                    x = fmaf(qa[i].z, kb[j].z, x);
                    x = fmaf(qa[i].w, kb[j].w, x);
                    s[i][j] = x;
                }
        }
        if constexpr (C::kNS == 1) {
            cp_async_wait0();  // V of this tile, the only copy in flight
            wg_sync(g);        // K is free for the next tile and V is visible
            if (more) {
                stage_async<D>(Ks, LD, kg, kv0 + KS * kTK, kTK, Skv, tid, kWG, status);
                cp_async_commit();
            }
        }

        // online softmax per row: the maximum of the raw scores (the scale is
        // positive, so it commutes with the maximum), then one FMA scales and
        // shifts each score into log2 units before exp2; masked keys are -inf
        if (kv0 + kTK > kv_all) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (kv0 + tx + 16 * j >= lim[i]) s[i][j] = -INFINITY;
        }
        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = fmaxf(fmax3(s[i][0], s[i][1], s[i][2]), s[i][3]);
#pragma unroll
        for (int w = 8; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], w));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float m_new = fmaxf(m[i], mx[i] * scale_log2);
            float alpha = 1.f, sum = 0.f;
            if (m_new == -INFINITY) {  // no visible key yet: P = 0, nothing to rescale
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
            } else {
                alpha = m[i] == -INFINITY ? 0.f : exp2f(m[i] - m_new);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = exp2f(fmaf(s[i][j], scale_log2, -m_new));
                    sum += s[i][j];
                }
            }
            m[i] = m_new;
            l[i] = l[i] * alpha + sum;
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int w = 0; w < W; ++w) acc[i][c][w] *= alpha;
#pragma unroll
            for (int j = 0; j < 4; ++j) Ps[(ty + 8 * i) * kLdP + tx + 16 * j] = s[i][j];
        }
        __syncwarp();  // the rows of P this half-warp reads were written by it

        // O += P V for rows ty + 8i, columns tx*W + 64c
#pragma unroll 2
        for (int kk = 0; kk < kTK; kk += 4) {
            float4 pa[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                pa[i] = *reinterpret_cast<const float4 *>(Ps + (ty + 8 * i) * kLdP + kk);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float *vr = Vt + (kk + u) * D + tx * W;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    float vv[W];
                    if constexpr (W == 4) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(vr + 64 * c);
                        vv[0] = t4.x; vv[1] = t4.y; vv[2] = t4.z; vv[3] = t4.w;
                    } else if constexpr (W == 2) {
                        const float2 t2 = *reinterpret_cast<const float2 *>(vr + 64 * c);
                        vv[0] = t2.x; vv[1] = t2.y;
                    } else {
                        vv[0] = vr[64 * c];
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float pi = u == 0 ? pa[i].x : u == 1 ? pa[i].y : u == 2 ? pa[i].z : pa[i].w;
#pragma unroll
                        for (int w = 0; w < W; ++w) acc[i][c][w] = fmaf(pi, vv[w], acc[i][c][w]);
                    }
                }
            }
        }
        wg_sync(g);  // this stage and P are free for the next tile
        if constexpr (C::kNS == 1) {
            if (more) {
                stage_async<D>(Vs, D, vg, kv0 + KS * kTK, kTK, Skv, tid, kWG, status);
                cp_async_commit();
                cp_async_wait1();  // the next K; the next V may still be arriving
                wg_sync(g);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int w = 8; w > 0; w >>= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], w);

    if constexpr (KS > 1) {
        // every warpgroup leaves (m, l, O) in its own K stages, laid out
        // [field][thread]; warpgroup g then finishes rows i = g, g + KS, ...
        // of every thread position, combining the KS partial states the way
        // partial softmax states combine: rescale each to the largest max
        {
            float *xs = sm + C::kOffK + g * C::kStageK;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xs[i * kWG + tid] = m[i];
                xs[(4 + i) * kWG + tid] = l[i];
#pragma unroll
                for (int c = 0; c < NC; ++c)
#pragma unroll
                    for (int w = 0; w < W; ++w)
                        xs[(8 + (i * NC + c) * W + w) * kWG + tid] = acc[i][c][w];
            }
        }
        __syncthreads();
#pragma unroll 1
        for (int i = g; i < 4; i += KS) {
            const int row = q0 + ty + 8 * i;
            if (row >= Sq) continue;
            // the last element this thread stores (o; lse lies inside the same rows)
            if (!in_bounds(((size_t)bh * Sq + row) * D + tx * W + 64 * (NC - 1) + W <=
                               (size_t)BH * Sq * D, status))
                continue;
            float mm = -INFINITY;
#pragma unroll
            for (int h = 0; h < KS; ++h) mm = fmaxf(mm, sm[C::kOffK + h * C::kStageK + i * kWG + tid]);
            float ll = 0.f, a[NC][W];
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int w = 0; w < W; ++w) a[c][w] = 0.f;
#pragma unroll
            for (int h = 0; h < KS; ++h) {
                const float *xs = sm + C::kOffK + h * C::kStageK;
                const float mh = xs[i * kWG + tid];
                const float sc = mh == -INFINITY ? 0.f : exp2f(mh - mm);
                ll = fmaf(xs[(4 + i) * kWG + tid], sc, ll);
#pragma unroll
                for (int c = 0; c < NC; ++c)
#pragma unroll
                    for (int w = 0; w < W; ++w)
                        a[c][w] = fmaf(xs[(8 + (i * NC + c) * W + w) * kWG + tid], sc, a[c][w]);
            }
            const float inv = ll > 0.f ? 1.f / ll : 0.f;
            float *orow = o + ((size_t)bh * Sq + row) * D + tx * W;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if constexpr (W == 4) {
                    *reinterpret_cast<float4 *>(orow + 64 * c) =
                        make_float4(a[c][0] * inv, a[c][1] * inv, a[c][2] * inv, a[c][3] * inv);
                } else {
#pragma unroll
                    for (int w = 0; w < W; ++w) orow[64 * c + w] = a[c][w] * inv;
                }
            }
            if (lse && tx == 0)
                lse[(size_t)bh * Sq + row] =
                    ll > 0.f ? (mm + log2f(ll)) * 0.69314718055994530942f : -INFINITY;
        }
    } else {
    // O = acc / l and lse = m + log2(l), in natural units; rows that saw no key: 0 and -inf
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = q0 + ty + 8 * i;
        if (row >= Sq) continue;
        if (!in_bounds(((size_t)bh * Sq + row) * D + tx * W + 64 * (NC - 1) + W <=
                           (size_t)BH * Sq * D, status))
            continue;
        const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
        float *orow = o + ((size_t)bh * Sq + row) * D + tx * W;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            if constexpr (W == 4) {
                *reinterpret_cast<float4 *>(orow + 64 * c) =
                    make_float4(acc[i][c][0] * inv, acc[i][c][1] * inv, acc[i][c][2] * inv,
                                acc[i][c][3] * inv);
            } else {
#pragma unroll
                for (int w = 0; w < W; ++w) orow[64 * c + w] = acc[i][c][w] * inv;
            }
        }
        if (lse && tx == 0)
            lse[(size_t)bh * Sq + row] =
                l[i] > 0.f ? (m[i] + log2f(l[i])) * 0.69314718055994530942f : -INFINITY;
    }
    }
}

// ---------------------------------------------------------------- key-split kernel (d = 64)
// 32 query rows per CTA, 8 warps; warp w takes the 32-key tiles w, w + 8, ...
// of the block and keeps its own online-softmax state for all 32 rows, so one
// thread owns an 8 x 4 block of scores (rows rg + 4i, keys kg + 8j; rg = lane
// / 8, kg = lane % 8) and an 8 x 8 block of O (rows rg + 4i, columns
// 4 kg + 32h + e).  Per head-dimension step of four, 12 float4 reads from
// shared memory feed 128 FMAs (the 4 x 4 blocks of the tiled kernel: 8 per
// 64), and every read instruction is one shared-memory wavefront.  P goes to
// a per-warp transposed tile, so that the P V loop reads 8 rows' P with two
// float4.  The row maximum and sum are reduced over the 8 lanes of a row
// group with shuffles.  At the end the 8 warps' states are combined the way
// partial softmax states combine (rescaled to the largest max).
constexpr int kSW = 8;           // warps
constexpr int kSQ = 32;          // query rows per CTA
constexpr int kSK = 32;          // keys per warp tile
constexpr int kSLd = 64 + 4;     // Q and K row stride: consecutive rows 4 banks apart
constexpr int kSLdP = kSQ + 4;   // row stride of the transposed P tile
constexpr int kSWarpFloats = kSK * kSLd + kSK * 64 + kSK * kSLdP;  // K, V, P^T of one warp
constexpr int kSOffW = kSQ * kSLd;                                 // after Q
constexpr size_t kSSmemBytes = sizeof(float) * (size_t)(kSOffW + kSW * kSWarpFloats);
// the combination reuses the warps' areas: O [warp][row][64], then m, l [warp][row]
static_assert(kSW * kSQ * 64 + 2 * kSW * kSQ <= kSW * kSWarpFloats, "state must fit");

__global__ void __launch_bounds__(kSW * 32, 1)
attn_f32_keysplit_kernel(const float *__restrict__ q, const float *__restrict__ k,
                         const float *__restrict__ v, float *__restrict__ o,
                         float *__restrict__ lse, int BH, int Sq, int Skv, int causal,
                         float scale_log2, int nqb, int *status) {
    constexpr int D = 64;
    extern __shared__ __align__(16) float sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 3, kg = lane & 7;
    float *Qs = sm;
    float *Kw = sm + kSOffW + warp * kSWarpFloats;  // [kSK][kSLd]
    float *Vw = Kw + kSK * kSLd;                    // [kSK][64]
    float *Pw = Vw + kSK * 64;                      // [kSK][kSLdP]: P^T, rows in the order rg*8 + i

    const int64_t bh = blockIdx.x / nqb;
    const int q0 = (blockIdx.x % nqb) * kSQ;
    const int q_end = min(q0 + kSQ, Sq);
    const int off = Skv - Sq;  // causal: key j visible to query i iff j <= i + off
    if (!in_bounds(bh < BH, status)) return;  // block-uniform
    const float *qg = q + (size_t)bh * Sq * D;
    const float *kgp = k + (size_t)bh * Skv * D;
    const float *vg = v + (size_t)bh * Skv * D;

    int lim[8];  // keys visible to row rg + 4i: [0, lim[i])
#pragma unroll
    for (int i = 0; i < 8; ++i) lim[i] = causal ? min(Skv, q0 + rg + 4 * i + off + 1) : Skv;
    const int kv_stop = causal ? min(Skv, q_end + off) : Skv;
    const int ntiles = kv_stop > 0 ? (kv_stop + kSK - 1) / kSK : 0;
    const int kv_all = causal ? min(Skv, q0 + off + 1) : Skv;  // visible to every row

    float m[8], l[8], acc[8][2][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][h][e] = 0.f;
    }

    // Q by the whole block; this warp's first K and V as two more groups
    stage_async<D>(Qs, kSLd, qg, q0, kSQ, Sq, threadIdx.x, kSW * 32, status);
    cp_async_commit();
    if (warp < ntiles) stage_async<D>(Kw, kSLd, kgp, warp * kSK, kSK, Skv, lane, 32, status);
    cp_async_commit();
    if (warp < ntiles) stage_async<D>(Vw, D, vg, warp * kSK, kSK, Skv, lane, 32, status);
    cp_async_commit();
    cp_async_wait1();  // Q and K have landed; V may still be arriving
    __syncthreads();

    for (int tile = warp; tile < ntiles; tile += kSW) {
        const int kv0 = tile * kSK;
        const bool more = tile + kSW < ntiles;
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 2
        for (int c = 0; c < D; c += 4) {
            float4 qa[8], kb[4];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                qa[i] = *reinterpret_cast<const float4 *>(Qs + (rg + 4 * i) * kSLd + c);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                kb[j] = *reinterpret_cast<const float4 *>(Kw + (kg + 8 * j) * kSLd + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x = s[i][j];
                    x = fmaf(qa[i].x, kb[j].x, x);
                    x = fmaf(qa[i].y, kb[j].y, x);
                    x = fmaf(qa[i].z, kb[j].z, x);
                    x = fmaf(qa[i].w, kb[j].w, x);
                    s[i][j] = x;
                }
        }
        __syncwarp();  // every lane is done with K: the next K may load
        if (more) stage_async<D>(Kw, kSLd, kgp, kv0 + kSW * kSK, kSK, Skv, lane, 32, status);
        cp_async_commit();

        // online softmax per row, as in the tiled kernel: max of the raw scores
        // over the row group's 8 lanes, one FMA into log2 units, exp2
        if (kv0 + kSK > kv_all) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (kv0 + kg + 8 * j >= lim[i]) s[i][j] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmax3(s[i][0], s[i][1], s[i][2]), s[i][3]);
#pragma unroll
        for (int w = 4; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], w));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float m_new = fmaxf(m[i], mx[i] * scale_log2);
            float alpha = 1.f, sum = 0.f;
            if (m_new == -INFINITY) {  // no visible key yet: P = 0, nothing to rescale
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
            } else {
                alpha = m[i] == -INFINITY ? 0.f : exp2f(m[i] - m_new);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = exp2f(fmaf(s[i][j], scale_log2, -m_new));
                    sum += s[i][j];
                }
            }
            m[i] = m_new;
            l[i] = l[i] * alpha + sum;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][h][e] *= alpha;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float *pr = Pw + (kg + 8 * j) * kSLdP + rg * 8;
            *reinterpret_cast<float4 *>(pr) = make_float4(s[0][j], s[1][j], s[2][j], s[3][j]);
            *reinterpret_cast<float4 *>(pr + 4) = make_float4(s[4][j], s[5][j], s[6][j], s[7][j]);
        }
        cp_async_wait1();  // this tile's V (the next K may still be arriving)
        __syncwarp();      // P and V written by the other lanes are visible

        // O += P V for rows rg + 4i, columns 4 kg + 32h + e
#pragma unroll 4
        for (int kk = 0; kk < kSK; ++kk) {
            const float4 p0 = *reinterpret_cast<const float4 *>(Pw + kk * kSLdP + rg * 8);
            const float4 p1 = *reinterpret_cast<const float4 *>(Pw + kk * kSLdP + rg * 8 + 4);
            const float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 vv = *reinterpret_cast<const float4 *>(Vw + kk * D + 4 * kg + 32 * h);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[i][h][0] = fmaf(pr[i], vv.x, acc[i][h][0]);
                    acc[i][h][1] = fmaf(pr[i], vv.y, acc[i][h][1]);
                    acc[i][h][2] = fmaf(pr[i], vv.z, acc[i][h][2]);
                    acc[i][h][3] = fmaf(pr[i], vv.w, acc[i][h][3]);
                }
            }
        }
        __syncwarp();  // every lane is done with V and P: the next V may load
        if (more) stage_async<D>(Vw, D, vg, kv0 + kSW * kSK, kSK, Skv, lane, 32, status);
        cp_async_commit();
        cp_async_wait1();  // the next K (the next V may still be arriving)
        __syncwarp();
    }
    cp_async_wait0();
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int w = 4; w > 0; w >>= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], w);

    // combine the 8 warps' states: each leaves (m, l, O) in the shared area
    __syncthreads();  // every warp is done with its K, V and P
    float *Os = sm + kSOffW;          // [warp][row][64]
    float *Ms = Os + kSW * kSQ * 64;  // [warp][row]
    float *Ls = Ms + kSW * kSQ;       // [warp][row]
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = rg + 4 * i;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<float4 *>(Os + (warp * kSQ + r) * 64 + 4 * kg + 32 * h) =
                make_float4(acc[i][h][0], acc[i][h][1], acc[i][h][2], acc[i][h][3]);
        if (kg == 0) {
            Ms[warp * kSQ + r] = m[i];
            Ls[warp * kSQ + r] = l[i];
        }
    }
    __syncthreads();
    // thread t finishes row t / 8, columns 8 (t % 8) .. + 7
    const int r = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * 8;
    const int row = q0 + r;
    if (row >= Sq) return;
    if (!in_bounds(((size_t)bh * Sq + row) * D + c0 + 8 <= (size_t)BH * Sq * D, status)) return;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSW; ++w) mm = fmaxf(mm, Ms[w * kSQ + r]);
    float ll = 0.f;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kSW; ++w) {
        const float mw = Ms[w * kSQ + r];
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - mm);
        ll = fmaf(Ls[w * kSQ + r], sc, ll);
        const float4 x0 = *reinterpret_cast<const float4 *>(Os + (w * kSQ + r) * 64 + c0);
        const float4 x1 = *reinterpret_cast<const float4 *>(Os + (w * kSQ + r) * 64 + c0 + 4);
        a[0] = fmaf(x0.x, sc, a[0]); a[1] = fmaf(x0.y, sc, a[1]);
        a[2] = fmaf(x0.z, sc, a[2]); a[3] = fmaf(x0.w, sc, a[3]);
        a[4] = fmaf(x1.x, sc, a[4]); a[5] = fmaf(x1.y, sc, a[5]);
        a[6] = fmaf(x1.z, sc, a[6]); a[7] = fmaf(x1.w, sc, a[7]);
    }
    const float inv = ll > 0.f ? 1.f / ll : 0.f;
    float *orow = o + ((size_t)bh * Sq + row) * D + c0;
    *reinterpret_cast<float4 *>(orow) = make_float4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
    *reinterpret_cast<float4 *>(orow + 4) = make_float4(a[4] * inv, a[5] * inv, a[6] * inv, a[7] * inv);
    if (lse && c0 == 0)
        lse[(size_t)bh * Sq + row] = ll > 0.f ? (mm + log2f(ll)) * 0.69314718055994530942f : -INFINITY;
}

int launch_keysplit(const float *q, const float *k, const float *v, float *o, float *lse,
                    const Problem &p, cudaStream_t stream) {
    const int nqb = (p.Sq + kSQ - 1) / kSQ;
    const int64_t grid = p.bh() * nqb;
    if (grid > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    if (!set_smem_limit_once(reinterpret_cast<const void *>(attn_f32_keysplit_kernel),
                             (int)kSSmemBytes))
        return ATTN_ERR_LAUNCH;
    int *status = status_word_device_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn_f32_keysplit_kernel<<<(unsigned)grid, kSW * 32, kSSmemBytes, stream>>>(
        q, k, v, o, lse, (int)p.bh(), p.Sq, p.Skv, p.causal, p.scale * 1.4426950408889634f, nqb,
        status);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

template <int D, int KS, int NS>
int launch_tiled_ks(const float *q, const float *k, const float *v, float *o, float *lse,
                    const Problem &p, int64_t grid, int nqb, cudaStream_t stream) {
    constexpr size_t smem = TiledCfg<D, KS, NS>::kSmemBytes;
    if (!set_smem_limit_once(reinterpret_cast<const void *>(attn_f32_tiled_kernel<D, KS, NS>),
                             (int)smem))
        return ATTN_ERR_LAUNCH;
    int *status = status_word_device_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn_f32_tiled_kernel<D, KS, NS><<<(unsigned)grid, KS * kWG, smem, stream>>>(
        q, k, v, o, lse, (int)p.bh(), p.Sq, p.Skv, p.causal, p.scale * 1.4426950408889634f, nqb,
        status);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// Blocks of one warpgroup with two stages that one SM holds at once (shared
// memory bounds it: one at d = 128, two at d = 64), 0 while unknown.  A
// property of the kernel and the architecture, so it is asked once.
template <int D>
int two_stage_blocks_per_sm() {
    static std::atomic<int> cached{0};
    int n = cached.load(std::memory_order_acquire);
    if (n > 0) return n;
    constexpr size_t smem = TiledCfg<D, 1, 2>::kSmemBytes;
    if (!set_smem_limit_once(reinterpret_cast<const void *>(attn_f32_tiled_kernel<D, 1, 2>),
                             (int)smem))
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_f32_tiled_kernel<D, 1, 2>, kWG,
                                                      smem) != cudaSuccess) {
        (void)cudaGetLastError();  // a failed query is not a launch error
        return 0;
    }
    cached.store(n, std::memory_order_release);
    return n;
}

// Fewer query blocks than SMs and more than one key tile: several warpgroups
// per block split its key tiles, so that each SM runs more warps -- four with
// one K/V stage each at d = 32 and 64, two with two stages at d = 16 (where a
// warpgroup's state would not fit one stage for the merge).  With one key
// tile there is nothing to split and the merge would only cost (10.9 -> 8.9 us
// at B=2, H=4, S=64, d=64).  Otherwise one warpgroup per block:
// with two stages while the whole grid is resident at once, and with one
// stage beyond that, which halves the block's K/V memory so that twice as
// many blocks share an SM and hide one another's copies (+20 % at
// B=2, H=40, S=1024, d=64 and at B=2, H=16, S=2048, d=128).
template <int D>
int launch_tiled_d(const float *q, const float *k, const float *v, float *o, float *lse,
                   const Problem &p, cudaStream_t stream) {
    const int nqb = (p.Sq + kTQ - 1) / kTQ;
    const int64_t grid = p.bh() * nqb;
    if (grid > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    const int key_tiles = (p.Skv + kTK - 1) / kTK;  // of the block that sees the most keys
    // d = 64 below four blocks per SM: the key-split kernel (B=2, H=4, S=512:
    // 24.4 -> 22.5 us; B=1, H=8, S=2048 causal: +20 %); on larger grids the
    // one-warpgroup blocks below are 3-4 % faster (B=2, H=40, S=1024)
    if constexpr (D == 64) {
        if (sms > 0 && grid < 4 * (int64_t)sms) return launch_keysplit(q, k, v, o, lse, p, stream);
    }
    if constexpr (D <= 64) {
        if (sms > 0 && grid < sms && key_tiles > 1) {
            if constexpr (D >= 32) return launch_tiled_ks<D, 4, 1>(q, k, v, o, lse, p, grid, nqb, stream);
            return launch_tiled_ks<D, 2, 2>(q, k, v, o, lse, p, grid, nqb, stream);
        }
    }
    const int per_sm = two_stage_blocks_per_sm<D>();
    if (sms > 0 && per_sm > 0 && grid <= (int64_t)sms * per_sm)
        return launch_tiled_ks<D, 1, 2>(q, k, v, o, lse, p, grid, nqb, stream);
    return launch_tiled_ks<D, 1, 1>(q, k, v, o, lse, p, grid, nqb, stream);
}

__global__ void fill_empty_kernel(uint8_t *o, size_t o_bytes, float *lse, size_t n_lse) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < o_bytes; t += stride)
        o[t] = 0;
    if (lse)
        for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n_lse; t += stride)
            lse[t] = -INFINITY;
}

template <int D>
int launch_d(const float *q, const float *k, const float *v, float *o, float *lse,
             const Problem &p, int bq, int bkv, cudaStream_t stream) {
    const size_t smem = f32_smem_bytes(D, bq, bkv);
    if (!set_smem_limit_once(reinterpret_cast<const void *>(attn_f32_kernel<D>), (int)kSmemLimit))
        return ATTN_ERR_LAUNCH;
    const int nqb = (p.Sq + bq - 1) / bq;
    const int64_t grid = p.bh() * nqb;
    if (grid > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    int *status = status_word_device_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn_f32_kernel<D><<<(unsigned)grid, kWarps * 32, smem, stream>>>(
        q, k, v, o, lse, (int)p.bh(), p.Sq, p.Skv, p.causal, p.scale, bq, bkv, nqb, status);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

bool f32_tiles_fit(int d, int block_q, int block_kv) {
    return f32_smem_bytes(d, block_q, block_kv) <= kSmemLimit;
}

int launch_f32(const float *q, const float *k, const float *v, float *o, float *lse,
               const Problem &p, int block_q, int block_kv, cudaStream_t stream) {
    if (!f32_tiles_fit(p.d, block_q, block_kv)) return ATTN_ERR_INVALID_ARG;
    switch (p.d) {
    case 16: return launch_d<16>(q, k, v, o, lse, p, block_q, block_kv, stream);
    case 32: return launch_d<32>(q, k, v, o, lse, p, block_q, block_kv, stream);
    case 64: return launch_d<64>(q, k, v, o, lse, p, block_q, block_kv, stream);
    case 128: return launch_d<128>(q, k, v, o, lse, p, block_q, block_kv, stream);
    default: return ATTN_ERR_INVALID_ARG;
    }
}

int launch_f32_tiled(const float *q, const float *k, const float *v, float *o, float *lse,
                     const Problem &p, cudaStream_t stream) {
    switch (p.d) {
    case 16: return launch_tiled_d<16>(q, k, v, o, lse, p, stream);
    case 32: return launch_tiled_d<32>(q, k, v, o, lse, p, stream);
    case 64: return launch_tiled_d<64>(q, k, v, o, lse, p, stream);
    case 128: return launch_tiled_d<128>(q, k, v, o, lse, p, stream);
    default: return ATTN_ERR_INVALID_ARG;
    }
}

int launch_empty_keys(void *o, float *lse, const Problem &p, cudaStream_t stream) {
    const size_t o_bytes = (size_t)p.bh() * p.Sq * p.d * elem_bytes_out(p.dtype);
    const size_t n_lse = (size_t)p.bh() * p.Sq;
    fill_empty_kernel<<<256, 256, 0, stream>>>((uint8_t *)o, o_bytes, lse, n_lse);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace attn
