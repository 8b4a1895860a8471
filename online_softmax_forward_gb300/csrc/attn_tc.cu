// attn_tc.cu -- bf16/fp16 exact attention forward on the sm_103a tensor cores.
//
// The computation is the tiled online softmax of aiml.sh
// "verify-tiled-attention" (tiled_flash_attention: query blocks, key/value
// blocks, causal early stop, per-row running max / sum / accumulator) with the
// update of huhohoo "tiled-online-softmax" ("Online normalization"):
//     m_new = max(m, max S);  r = exp(m - m_new);  P = exp(S - m_new)
//     a = a * r + P V;  l = l * r + sum P;  out = a / l
// Tiles are 128 query rows x 128 keys.  How the work maps onto GB300:
//
//  * Persistent grid, one CTA per SM.  A work unit is two consecutive 128-row
//    query tiles (Q0, Q1) of one (batch, head) slice; they share every K/V
//    tile.  Units are handed out longest-first (causal) in a snake order.
//  * Warp 8 (producer) streams Q0/Q1 and then K_j, V_j tiles with TMA (128-byte
//    swizzle) into a ring of shared-memory stages guarded by mbarriers.
//  * Warp 9 (MMA issuer, one thread) runs tcgen05.mma kind::f16:
//        S_t = Q_t K_j^T  (both operands in shared memory, fp32 in TMEM)
//        O_t += P_t V_j   (P_t read from TMEM, V_j from shared memory)
//    in the order S0(j) S1(j) | PV0(j) S0(j+1) | PV1(j) S1(j+1) | ..., so the
//    tensor core works on one query tile while the other one's softmax runs.
//    P_t is written over S_t; S_t(j+1) is issued after PV_t(j) by the same
//    thread and relies on tcgen05.mma operations of a CTA executing in issue
//    order.
//  * Warps 0-3 / 4-7 (softmax warpgroups, one per query tile; one thread per
//    query row) read S from TMEM, apply the causal / tail mask, take the row
//    max, exponentiate with ex2 (scores pre-multiplied by scale*log2 e), sum,
//    write P back to TMEM as 16-bit pairs, and rescale O in TMEM when needed.
//    The running max is updated lazily: O and l are rescaled only when the
//    max grows by more than 2^8 (the P values then stay <= 256); O, l and m
//    always refer to the same stale max, so the result is the same softmax.
//    After the last tile they write O / l and lse = m + ln l.
//  * Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0, O1 after.
//  * Every mbarrier wait is bounded (globaltimer).  On expiry the CTA sets an
//    abort flag, records ATTN timeout in the status word, lets every role
//    leave its loop, waits for its own TMA loads and MMAs in flight, frees
//    tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per query tile (MMA M)
constexpr int BN = 128;  // keys per key/value tile
constexpr int kStages = 4;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units)

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head width");
    static constexpr int kChunks = D / 64;            // 128-byte swizzle atoms along d
    static constexpr int kChunkBytes = BN * 128;      // one atom column of a tile: 16 KB
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // Q, K or V tile
    static constexpr int kOffQ = 0;                   // Q0, Q1
    static constexpr int kOffKV = 2 * kTileBytes;     // ring stages
    static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
    static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
    // tensor-memory columns of S_t and O_t
    __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
    __device__ static constexpr uint32_t col_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
};

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

struct TcParams {
    void *o;
    float *lse;
    int *status;
    int BH, Sq, Skv, causal;
    int nqb;      // units per (batch, head): ceil(Sq / 256)
    int n_units;  // BH * nqb
    float scale_log2;  // scale * log2(e)
    int out_f32;       // 1: o is fp32; 0: o has the input type
    int hook;
    unsigned long long timeout_ns;
};

struct Unit {
    int bh, q0;
    int nkv[2];
};

__device__ __forceinline__ Unit decode_unit(int u, const TcParams &p) {
    Unit r;
    const int level = u / p.BH;
    r.bh = u % p.BH;
    const int qb = p.causal ? (p.nqb - 1 - level) : level;  // causal: longest first
    r.q0 = qb * 2 * BM;
    const int off = p.Skv - p.Sq;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qs = r.q0 + t * BM;
        int n = 0;
        if (qs < p.Sq) {
            const int q_end = min(qs + BM, p.Sq);
            const int kv_end = p.causal ? min(p.Skv, q_end + off) : p.Skv;
            n = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
        }
        r.nkv[t] = n;
    }
    return r;
}

// Snake-ordered static schedule: round r hands unit r*G + c (even r) or
// r*G + G-1-c (odd r) to CTA c.  Returns -1 when done.
__device__ __forceinline__ int unit_of(int round, const TcParams &p) {
    const int G = gridDim.x, c = blockIdx.x;
    const long base = (long)round * G;
    if (base >= p.n_units) return -2;
    const long u = base + ((round & 1) ? (G - 1 - c) : c);
    return u < p.n_units ? (int)u : -1;
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   K-major operands: rows of 64 16-bit elements (128 B), 8-row groups
//   1024 B apart (SBO); the K offset inside the atom is added to the start
//   address.  MN-major operands (V for P.V): 64 contiguous N elements per
//   128-byte row, 8 K-rows per 1024-B atom (SBO), atoms along N 16 KB apart
//   (LBO).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
    d |= (uint64_t)2 << 61;  // swizzle: 128 B
    return d;
}

// Instruction descriptor, kind::f16, fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool b_mn_major) {
    return (1u << 4)                          // D format: f32
           | ((bf16 ? 1u : 0u) << 7)          // A format
           | ((bf16 ? 1u : 0u) << 10)         // B format
           | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Bounded wait shared by all roles.  Returns false if the CTA is aborting
// (another role gave up) or this wait expired (then it starts the abort).
struct Watch {
    volatile int *abort_flag;
    int *status;
    unsigned long long limit;

    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (true) {
#pragma unroll 1
            for (int i = 0; i < 16; ++i)
                if (ptx::mbar_try_wait(bar, parity)) return true;
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > limit) {
                *abort_flag = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
    // Waits for hardware completion (TMA / MMA in flight) during teardown,
    // regardless of the abort flag; bounded by the same limit.
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (ptx::globaltimer_ns() - t0 > limit) {
                atomicOr(status, kStatusTimeout);
                return;
            }
        }
    }
};

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (kBF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

// Keeps the compiler from reading tcgen05.ld destination registers before
// tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::kOffBar);
    const uint32_t sQ = ptx::smem_addr(smem + C::kOffQ);
    const uint32_t sKV = ptx::smem_addr(smem + C::kOffKV);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Watch watch{&bars->abort_flag, p.status, p.timeout_ns};

    auto bar = [&](uint64_t &b) { return ptx::smem_addr(&b); };

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(bars->q_full), 1);
        ptx::mbar_init(bar(bars->q_empty), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(bars->kv_full[s]), 1);
            ptx::mbar_init(bar(bars->kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(bars->s_full[t]), 1);
            ptx::mbar_init(bar(bars->p_full[t]), 128);
            ptx::mbar_init(bar(bars->o_full[t]), 1);
            ptx::mbar_init(bar(bars->o_empty[t]), 128);
        }
        ptx::mbar_init(bar(bars->mma_done), 1);
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t pos = 0, qn = 0;
            bool loaded_q = false;
            uint32_t last_q_par = 0;
            bool ok = true;
            for (int round = 0; ok; ++round) {
                const int u = unit_of(round, p);
                if (u == -2) break;
                if (u < 0) continue;
                const Unit w = decode_unit(u, p);
                const int nmax = max(w.nkv[0], w.nkv[1]);
                if (nmax == 0) continue;
                if (!watch.wait(bar(bars->q_empty), (qn & 1) ^ 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(bar(bars->q_full), 2 * C::kTileBytes);
                for (int t = 0; t < 2; ++t)
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tm_q,
                                         bar(bars->q_full), c * 64, w.q0 + t * BM, w.bh);
                last_q_par = qn & 1;
                loaded_q = true;
                ++qn;
                for (int j = 0; j < nmax && ok; ++j) {
                    for (int which = 0; which < 2; ++which) {  // K_j then V_j
                        const int s = pos % kStages;
                        if (!watch.wait(bar(bars->kv_empty[s]), ((pos / kStages) & 1) ^ 1)) {
                            ok = false;
                            break;
                        }
                        ptx::mbar_arrive_expect_tx(bar(bars->kv_full[s]), C::kTileBytes);
                        const CUtensorMap *tm = which ? &tm_v : &tm_k;
                        for (int c = 0; c < C::kChunks; ++c)
                            ptx::tma_load_3d(sKV + s * C::kTileBytes + c * C::kChunkBytes, tm,
                                             bar(bars->kv_full[s]), c * 64, j * BN, w.bh);
                        ++pos;
                    }
                }
            }
            // teardown: wait until every load this thread issued has landed
            for (uint32_t s = 0; s < (uint32_t)kStages && s < pos; ++s) {
                const uint32_t last = s + ((pos - 1 - s) / kStages) * kStages;  // last use of s
                watch.drain(bar(bars->kv_full[s]), (last / kStages) & 1);
            }
            if (loaded_q) watch.drain(bar(bars->q_full), last_q_par);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_f16(kBF16, BM, BN, false);
            constexpr uint32_t kIdescO = idesc_f16(kBF16, BM, D, true);
            uint32_t pos = 0, qn = 0;
            uint32_t pn[2] = {0, 0}, on[2] = {0, 0};
            bool ok = true;
            bool first_unit = true;

            auto issue_s = [&](int t, int stage) {
                const uint32_t d_tmem = tmem + C::col_s(t);
                const uint32_t a0 = sQ + t * C::kTileBytes, b0 = sKV + stage * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    ptx::mma_ss(d_tmem, sdesc(a0 + koff, 16, 1024), sdesc(b0 + koff, 16, 1024),
                                kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int stage, bool acc) {
                const uint32_t d_tmem = tmem + C::col_o(t);
                const uint32_t b0 = sKV + stage * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t a_tmem = tmem + C::col_s(t) + kk * 8;  // 16 keys = 8 columns
                    ptx::mma_ts(d_tmem, a_tmem, sdesc(b0 + kk * 16 * 128, C::kChunkBytes, 1024),
                                kIdescO, (acc || kk > 0) ? 1u : 0u);
                }
            };

            for (int round = 0; ok; ++round) {
                const int u = unit_of(round, p);
                if (u == -2) break;
                if (u < 0) continue;
                const Unit w = decode_unit(u, p);
                const int nmax = max(w.nkv[0], w.nkv[1]);
                if (nmax == 0) continue;
                if (!watch.wait(bar(bars->q_full), qn & 1)) { ok = false; break; }
                ++qn;
                ptx::tc_fence_after();
                // K_0: S0(0), S1(0)
                uint32_t posK = pos++;
                int stK = posK % kStages;
                if (!watch.wait(bar(bars->kv_full[stK]), (posK / kStages) & 1)) { ok = false; break; }
                ptx::tc_fence_after();
                for (int t = 0; t < 2; ++t) {
                    if (w.nkv[t] > 0) {
                        issue_s(t, stK);
                        const bool skip = p.hook == 1 && first_unit && t == 0 && blockIdx.x == 0;
                        if (!skip) ptx::mma_commit(bar(bars->s_full[t]));
                    }
                }
                ptx::mma_commit(bar(bars->kv_empty[stK]));
                first_unit = false;
                for (int j = 0; j < nmax && ok; ++j) {
                    const uint32_t posV = pos++;
                    const int stV = posV % kStages;
                    if (!watch.wait(bar(bars->kv_full[stV]), (posV / kStages) & 1)) { ok = false; break; }
                    const bool has_next = j + 1 < nmax;
                    if (has_next) {
                        posK = pos++;
                        stK = posK % kStages;
                        if (!watch.wait(bar(bars->kv_full[stK]), (posK / kStages) & 1)) { ok = false; break; }
                    }
                    ptx::tc_fence_after();
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= w.nkv[t]) continue;
                        if (!watch.wait(bar(bars->p_full[t]), pn[t] & 1)) { ok = false; break; }
                        ++pn[t];
                        if (j == 0) {
                            if (!watch.wait(bar(bars->o_empty[t]), (on[t] & 1) ^ 1)) { ok = false; break; }
                            ++on[t];
                        }
                        ptx::tc_fence_after();
                        issue_pv(t, stV, j > 0);
                        if (j == w.nkv[t] - 1) ptx::mma_commit(bar(bars->o_full[t]));
                        if (j + 1 < w.nkv[t]) {
                            issue_s(t, stK);
                            ptx::mma_commit(bar(bars->s_full[t]));
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(bar(bars->kv_empty[stV]));
                    if (has_next) ptx::mma_commit(bar(bars->kv_empty[stK]));
                }
                if (!ok) break;
                ptx::mma_commit(bar(bars->q_empty));
            }
            // teardown: every MMA issued by this thread has completed
            ptx::mma_commit(bar(bars->mma_done));
            watch.drain(bar(bars->mma_done), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;        // query tile of this warpgroup
        const int wq = warp & 3;        // TMEM lane quarter of this warp
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::col_s(t);
        const uint32_t tO = tmem + lane_base + C::col_o(t);
        const float sl2 = p.scale_log2;
        const int off = p.Skv - p.Sq;
        uint32_t sn = 0, ofn = 0;
        bool ok = true;

        for (int round = 0; ok; ++round) {
            const int u = unit_of(round, p);
            if (u == -2) break;
            if (u < 0) continue;
            const Unit w = decode_unit(u, p);
            const int nk = w.nkv[t];
            const int row = w.q0 + t * BM + wq * 32 + lane;  // query index of this thread
            const int limit = p.causal ? min(p.Skv, row + off + 1) : p.Skv;  // keys < limit visible
            float m = -INFINITY;  // running max, log2-scaled units
            float l = 0.f;        // running normaliser relative to m

            for (int j = 0; j < nk; ++j) {
                const bool got = watch.wait(bar(bars->s_full[t]), sn & 1);
                ++sn;
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t r[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, r[c]);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence(r[c]);

                float s[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[c][i]);
                const int kv0 = j * BN;
                if (kv0 + BN > limit) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (kv0 + i >= limit) s[i] = -INFINITY;
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int i = 4; i < 128; i += 4) {
                    mx0 = fmaxf(mx0, s[i]);
                    mx1 = fmaxf(mx1, s[i + 1]);
                    mx2 = fmaxf(mx2, s[i + 2]);
                    mx3 = fmaxf(mx3, s[i + 3]);
                }
                const float tile_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const float m_new = fmaxf(m, tile_max);
                bool rescale = false;
                float alpha = 1.f;
                if (m == -INFINITY) {
                    m = m_new;  // first visible keys: nothing accumulated yet
                } else if (m_new - m > kRescaleLog2) {
                    rescale = true;
                    alpha = ptx::ex2_approx(m - m_new);
                    m = m_new;
                    l *= alpha;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O_t holds P V of tiles < j (complete: S_t(j) was issued after them)
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + c * 32, o);
                        ptx::tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        ptx::tmem_st32(tO + c * 32, o);
                    }
                    ptx::tmem_wait_st();
                }
                const float mb = (m == -INFINITY) ? 0.f : m;
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[2][32];
#pragma unroll
                for (int i = 0; i < 128; i += 2) {
                    const float p0 = ptx::ex2_approx(fmaf(s[i], sl2, -mb));
                    const float p1 = ptx::ex2_approx(fmaf(s[i + 1], sl2, -mb));
                    sum0 += p0;
                    sum1 += p1;
                    pk[i >> 6][(i >> 1) & 31] = pack2<kBF16>(p0, p1);
                }
                l += sum0 + sum1;
                __syncwarp();  // tcgen05.st needs the whole warp converged
                ptx::tmem_st32(tS, pk[0]);
                ptx::tmem_st32(tS + 32, pk[1]);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(bars->p_full[t]));
            }
            if (!ok) break;

            // epilogue: O / l and lse for the rows of this thread
            if (nk > 0) {
                const bool got = watch.wait(bar(bars->o_full[t]), ofn & 1);
                ++ofn;
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                ptx::tc_fence_after();
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool live = row < p.Sq;
            const size_t orow = ((size_t)w.bh * p.Sq + row) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                __syncwarp();  // tcgen05.ld needs the whole warp converged
                if (nk > 0) {
                    ptx::tmem_ld32(tO + c * 32, o);
                    ptx::tmem_wait_ld();
                    reg_fence(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (!live) {
                    // rows past Sq: nothing to store
                } else if (p.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + orow + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv,
                                             __uint_as_float(o[4 * i + 1]) * inv,
                                             __uint_as_float(o[4 * i + 2]) * inv,
                                             __uint_as_float(o[4 * i + 3]) * inv);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.o) + orow + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 v;
                        v.x = pack2<kBF16>(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
                        v.y = pack2<kBF16>(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
                        v.z = pack2<kBF16>(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
                        v.w = pack2<kBF16>(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
                        dst[i] = v;
                    }
                }
            }
            if (live && p.lse)
                p.lse[(size_t)w.bh * p.Sq + row] =
                    l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            if (nk > 0) {
                __syncwarp();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(bars->o_empty[t]));
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [BH, S, d] 16-bit tensor as a 3-D TMA map, box 64 (d) x 128 (rows) x 1,
// 128-byte swizzle; rows past S read as zeros.
bool make_map(CUtensorMap *m, const void *base, bool bf16, int d, int S, int64_t BH) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int D, bool kBF16>
int launch_typed(const void *q, const void *k, const void *v, void *o, float *lse,
                 const Problem &pr, cudaStream_t stream) {
    using C = Cfg<D>;
    CUtensorMap tq, tk, tv;
    const int64_t BH = pr.bh();
    if (!make_map(&tq, q, kBF16, D, pr.Sq, BH) || !make_map(&tk, k, kBF16, D, pr.Skv, BH) ||
        !make_map(&tv, v, kBF16, D, pr.Skv, BH))
        return ATTN_ERR_CUDA;
    int *status = status_word_device_ptr();
    if (!status) return ATTN_ERR_CUDA;
    TcParams p;
    p.o = o;
    p.lse = lse;
    p.status = status;
    p.BH = (int)BH;
    p.Sq = pr.Sq;
    p.Skv = pr.Skv;
    p.causal = pr.causal;
    p.nqb = (pr.Sq + 2 * BM - 1) / (2 * BM);
    const int64_t n_units = BH * p.nqb;
    if (n_units > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    p.n_units = (int)n_units;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.out_f32 = (pr.dtype == ATTN_BF16_OUT_F32 || pr.dtype == ATTN_F16_OUT_F32) ? 1 : 0;
    p.hook = test_hook();
    p.timeout_ns = watchdog_ns();
    const int sms = num_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const int grid = (int)(n_units < sms ? n_units : sms);
    auto kern = attn_tc_kernel<D, kBF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return ATTN_ERR_LAUNCH;
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return ATTN_ERR_UNSUPPORTED_DEVICE;
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_tc(const void *q, const void *k, const void *v, void *o, float *lse,
              const Problem &p, cudaStream_t stream) {
    const bool bf16 = (p.dtype == ATTN_BF16 || p.dtype == ATTN_BF16_OUT_F32);
    if (p.d == 128)
        return bf16 ? launch_typed<128, true>(q, k, v, o, lse, p, stream)
                    : launch_typed<128, false>(q, k, v, o, lse, p, stream);
    if (p.d == 64)
        return bf16 ? launch_typed<64, true>(q, k, v, o, lse, p, stream)
                    : launch_typed<64, false>(q, k, v, o, lse, p, stream);
    return ATTN_ERR_INVALID_ARG;
}

}  // namespace attn
