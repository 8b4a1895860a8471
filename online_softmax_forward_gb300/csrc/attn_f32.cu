// attn_f32.cu -- fp32 exact attention forward on CUDA cores.
//
// The tiled online-softmax loop of aiml.sh "verify-tiled-attention"
// (tiled_flash_attention) with the update of huhohoo "tiled-online-softmax"
// ("Online normalization"), in fp32, for small and latency-bound shapes and
// for tile-size invariance tests.  Tile sizes are runtime values.
//
// One CTA owns one block of block_q query rows of one (batch, head) slice and
// walks the key/value blocks of block_kv rows; each block is staged in shared
// memory once and used by every query row of the CTA.  One warp handles one
// query row at a time: lanes split the keys of the tile for the scores
// (q . k, q broadcast from shared memory), warp shuffles give the tile
// maximum and the sum of exponentials, and lanes split the head dimension for
// the P.V product.  Per-row state (running max m, normaliser l, accumulator a)
// lives in shared memory between key tiles.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

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
template <int D>
__device__ __forceinline__ void stage_rows(float *dst, int ld, const float *__restrict__ src,
                                           int rows) {
    constexpr int V4 = D / 4;
    const int n = rows * V4;
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const int r = t / V4, c = (t % V4) * 4;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(src + (size_t)r * D + c));
        *reinterpret_cast<float4 *>(dst + r * ld + c) = x;
    }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                int Sq, int Skv, int causal, float scale, int block_q, int block_kv, int nqb) {
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

    const float *qg = q + ((size_t)bh * Sq + q_start) * D;
    const float *kg = k + (size_t)bh * Skv * D;
    const float *vg = v + (size_t)bh * Skv * D;

    stage_rows<D>(Qs, LD, qg, rows);
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
        stage_rows<D>(Ks, LD, kg + (size_t)kv_start * D, kv_end - kv_start);
        stage_rows<D>(Vs, D, vg + (size_t)kv_start * D, kv_end - kv_start);
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
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
            const int c = lane + 32 * u;
            if (c < D) orow[c] = As[r * D + c] * inv;
        }
        if (lse && lane == 0) lse[(size_t)bh * Sq + i] = l > 0.f ? Ms[r] + logf(l) : -INFINITY;
    }
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
    attn_f32_kernel<D><<<(unsigned)grid, kWarps * 32, smem, stream>>>(
        q, k, v, o, lse, p.Sq, p.Skv, p.causal, p.scale, bq, bkv, nqb);
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

int launch_empty_keys(void *o, float *lse, const Problem &p, cudaStream_t stream) {
    const size_t o_bytes = (size_t)p.bh() * p.Sq * p.d * elem_bytes_out(p.dtype);
    const size_t n_lse = (size_t)p.bh() * p.Sq;
    fill_empty_kernel<<<256, 256, 0, stream>>>((uint8_t *)o, o_bytes, lse, n_lse);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace attn
