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
//  * Persistent grid, one CTA per SM, 12 warps.  A work unit is two
//    consecutive 128-row query tiles (Q0, Q1) of one (batch, head) slice; they
//    share every K/V tile.  Units are handed out dynamically: the producer
//    of a CTA claims the next unit index from a device counter when it has
//    issued the loads of the current one, decodes it, and passes the decoded
//    unit to the CTA's other roles through a small ring in shared memory.
//    The order of the indices (decode_unit) takes the (batch, head) slices
//    in groups of about one round of units, longest first inside a group, so
//    the CTAs running at any time share the K and V of a few heads through
//    L2: each K/V tile is read from HBM about once.
//  * Warp 8 (producer) streams Q0/Q1 and the K/V tiles with TMA (128-byte
//    swizzle) into a ring of shared-memory stages guarded by mbarriers, in
//    the order the tensor core consumes them: K_0, then K_{j+1}, V_j for each
//    j.  Each query tile has its own Q buffer and barriers, so the next unit's
//    Q_t is fetched as soon as the last S_t of the current unit is computed;
//    it is prefetched into L2 when the unit is published.
//  * Warps 9 and 10 issue the tcgen05.mma (kind::f16, fp32 accumulate) of
//    query tile 0 and 1 respectively, as whole warps with one elected lane:
//        S_t = Q_t K_j^T  (shared-memory operands, fp32 result in TMEM)
//        O_t += P_t V_j   (V_j in shared memory, O_t in TMEM; P_t in shared
//                          memory at d = 128, in TMEM at d = 64)
//    S_t(j+1) is issued as soon as the softmax has copied S_t(j) out of tensor
//    memory, so the tensor core computes the next scores while the softmax
//    exponentiates the current ones; PV_t(j) follows once P_t(j) is written.
//    A K/V stage is released when both issuers are done with it.
//  * Warps 0-3 / 4-7 (softmax warpgroups, one per query tile; one thread per
//    query row, 224 registers each via setmaxnreg) read S from TMEM with the
//    load-and-reduce form of sm_103a (tcgen05.ld.red with .max: two 64-column
//    loads that also return their maximum, so a tile's row max costs no
//    instructions; only a diagonal or tail tile masks keys and takes its max
//    in software), exponentiate with ex2 (scores pre-multiplied by
//    scale*log2 e, paired fp32 arithmetic), sum, and write P as 16-bit
//    values: at d = 128 into a shared-memory tile in the MMA's
//    128-byte-swizzled layout, at d = 64 into tensor memory with two
//    32-column stores (no swizzle, no proxy fence; 7-9 % faster).  The
//    running max is updated lazily: O and l are rescaled (O in TMEM, after
//    the previous P.V has completed) only when the max grows by more than
//    2^8, so P stays <= 256; O, l and m always refer to the same stale max,
//    so the result is the same softmax.  Each row keeps two normalisers: l,
//    the sum of the exact P, gives the lse; lr adds to it, tile by tile, the
//    rounding error of the tile's largest P in its 16-bit form -- the term a
//    stale max makes large (up to 256 * 2^-9) -- so that O / lr divides by
//    (almost exactly) the sum of the weights P.V multiplied.  After the last
//    tile they write O / lr and lse = m + ln l.
//  * Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0, O1 after;
//    at d = 64 also P0 [384,448) and P1 [448,512), 16-bit pairs per column.
//  * Every mbarrier wait is bounded (globaltimer).  On expiry the CTA sets an
//    abort flag, records ATTN timeout in the status word, lets every role
//    leave its loop, waits for its own TMA loads and MMAs in flight, frees
//    tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per query tile (MMA M)
constexpr int BN = 128;  // keys per key/value tile
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp0 = 9;  // issuer of query tile 0; kMmaWarp0 + 1 issues tile 1
constexpr int kThreads = 12 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units)
// Work units are claimed from a device counter by the producer and passed to
// the other roles through a ring of kSchedRing shared-memory slots; every warp
// that reads a slot (issuers, softmax) releases it.
constexpr int kSchedRing = 4;
constexpr int kSchedReaders = 10;
// Device counters of the dynamic schedule: kSchedSlots pairs (next unit,
// CTAs done); each launch takes the next pair, and its last CTA resets it.
constexpr int kSchedSlots = 256;
// Register split: the block is launched with kLaunchRegs per thread; the two
// softmax warpgroups grow to kSoftmaxRegs and the third warpgroup (producer,
// issuers) shrinks to kOtherRegs.  The totals must match exactly.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 224;
constexpr int kOtherRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs == kThreads * kLaunchRegs, "register split");

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head width");
    static constexpr int kChunks = D / 64;            // 128-byte swizzle atoms along d
    static constexpr int kChunkBytes = BN * 128;      // one atom column of a 128-row tile: 16 KB
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // Q, K or V tile
    static constexpr int kPBytes = 2 * kChunkBytes;   // P tile: 128 rows x 128 keys, 16-bit
    // at d = 64 tensor memory has room for P next to S and O: P_t in columns
    // 384 + 64 t, and the P.V MMAs read it from there
    static constexpr bool kTmemP = D == 64;
    static constexpr int kStages = D == 128 ? 3 : 6;  // K/V ring depth (fills 227 KB)
    static constexpr int kOffQ = 0;                   // Q0, Q1
    static constexpr int kOffP = 2 * kTileBytes;      // P0, P1 (shared memory at d = 128)
    static constexpr int kOffKV = kOffP + (kTmemP ? 0 : 2 * kPBytes);  // ring stages
    static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
    static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // + barriers + alignment slack
    // tensor-memory columns of S_t and O_t
    __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
    __device__ static constexpr uint32_t col_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
    __device__ static constexpr uint32_t col_p(int t) { return 384u + (t ? 64u : 0u); }
};
constexpr int kMaxStages = 6;

struct Unit {
    int bh, q0;
    int nkv[2];
};

struct Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
    uint64_t s_full[2];   // S_t computed (MMA commit)
    uint64_t s_free[2];   // S_t copied to registers by the softmax (128 arrivals)
    uint64_t p_full[2];   // P_t written to shared memory (128 arrivals)
    uint64_t p_free[2];   // P_t . V done: P buffer free, O_t up to date (MMA commit)
    uint64_t o_empty[2];  // epilogue has read O_t (128 arrivals)
    uint64_t mma_done[2];
    uint64_t sched_full[kSchedRing], sched_empty[kSchedRing];
    Unit sched_unit[kSchedRing];  // the decoded unit; bh = -2: no more units
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct TcParams {
    void *o;
    float *lse;
    int *status;
    unsigned int *sched;  // this launch's counter pair: next unit, CTAs done
    int BH, Sq, Skv, causal;
    int nqb;      // units per (batch, head): ceil(Sq / 256)
    int hg;       // (batch, head) slices per schedule group (K/V of a group fit in L2)
    int n_units;  // BH * nqb
    float scale_log2;  // scale * log2(e)
    int out_f32;       // 1: o is fp32; 0: o has the input type
    int stage_o;       // 1: O leaves through shared memory (d = 128, Skv <= 8192)
    int hook;
    unsigned long long timeout_ns;
};

// Unit u of the schedule.  The (batch, head) slices are taken in groups of
// hg (about one unit per CTA in a group); inside a group the units go level
// by level, longest first for causal, and round-robin over the group's heads,
// so the CTAs running at any time share the K/V of a few heads through L2.
__device__ __forceinline__ Unit decode_unit(int u, const TcParams &p) {
    Unit r;
    const int per_group = p.hg * p.nqb;
    const int g = u / per_group;
    const int rem = u - g * per_group;
    const int heads = min(p.hg, p.BH - g * p.hg);  // the last group may be smaller
    const int level = rem / heads;
    r.bh = g * p.hg + (rem - level * heads);
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

// Shared-memory matrix descriptor, 128-byte swizzle.
//   K-major operands: rows of 64 16-bit elements (128 B), 8-row groups
//   1024 B apart (SBO); the K offset inside the atom is added to the start
//   address.  MN-major operands (V for P.V): 64 contiguous N elements per
//   128-byte row, 8 K-rows per 1024-B atom (SBO), atoms along N 16 KB apart
//   (LBO).  The start address occupies the low 14 bits (address / 16), so
//   an offset inside the same shared-memory window is added to the
//   descriptor directly.
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
// tcgen05.wait::ld (and from recycling tcgen05.st source registers before
// tcgen05.wait::st when placed after it).
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// A 64-key half tile of S held as two 32-column tcgen05.ld results.
struct Half {
    uint32_t a[32], b[32];
};

__device__ __forceinline__ void fence_half(Half &h) {
    reg_fence(h.a);
    reg_fence(h.b);
}

// Keys >= limit of a 64-key half tile starting at key kv0 get a score of
// -inf (excluded), so that they contribute exp(-inf) = 0.
__device__ __forceinline__ void mask_half(Half &h, int kv0, int limit) {
    if (kv0 + 64 > limit) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (kv0 + i >= limit) h.a[i] = __float_as_uint(-INFINITY);
            if (kv0 + 32 + i >= limit) h.b[i] = __float_as_uint(-INFINITY);
        }
    }
}

// Maximum raw score of a 64-key half tile.
__device__ __forceinline__ float max_half(const Half &h) {
    float x0 = __uint_as_float(h.a[0]), x1 = __uint_as_float(h.a[1]);
    float x2 = __uint_as_float(h.b[0]), x3 = __uint_as_float(h.b[1]);
#pragma unroll
    for (int i = 2; i + 3 < 30; i += 4) {  // elements 2..29 of a and b
        x0 = ptx::max3(x0, __uint_as_float(h.a[i]), __uint_as_float(h.a[i + 1]));
        x1 = ptx::max3(x1, __uint_as_float(h.a[i + 2]), __uint_as_float(h.a[i + 3]));
        x2 = ptx::max3(x2, __uint_as_float(h.b[i]), __uint_as_float(h.b[i + 1]));
        x3 = ptx::max3(x3, __uint_as_float(h.b[i + 2]), __uint_as_float(h.b[i + 3]));
    }
    // elements 30 and 31 of a and b
    return fmaxf(ptx::max3(x0, __uint_as_float(h.a[30]), __uint_as_float(h.a[31])),
                 ptx::max3(fmaxf(x1, x3), x2, fmaxf(__uint_as_float(h.b[30]), __uint_as_float(h.b[31]))));
}

// P = 2^(s * sl2 - mb) for 32 keys: packed 16-bit pairs into pk, fp32
// partial sums of the exact values into acc.
template <bool kBF16>
__device__ __forceinline__ void exp32(const uint32_t (&r)[32], float sl2, float mb,
                                      uint32_t *pk, float2 (&acc)[4]) {
    const float2 sc = make_float2(sl2, sl2), nb = make_float2(-mb, -mb);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc, nb);
        const float p0 = ptx::ex2_approx(x.x), p1 = ptx::ex2_approx(x.y);
        acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
        pk[i] = pack2<kBF16>(p0, p1);
    }
}

// Rounding error of the largest probability of a tile, 2^(smax * sl2 - mb),
// when it is stored as a 16-bit P: its 16-bit value minus its exact value.
// The value is computed by the same instructions as in exp32, so it is the
// same number P.V multiplies.
template <bool kBF16>
__device__ __forceinline__ float max_p_rounding(float smax, float sl2, float mb) {
    const float p = ptx::ex2_approx(fmaf(smax, sl2, -mb));
    return ptx::add_f32_half<kBF16, false>(0.f, pack2<kBF16>(p, p)) - p;
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    using C = Cfg<D>;
    constexpr int kStages = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::kOffBar);
    const uint32_t sQ = ptx::smem_addr(smem + C::kOffQ);
    const uint32_t sP = ptx::smem_addr(smem + C::kOffP);
    const uint32_t sKV = ptx::smem_addr(smem + C::kOffKV);

    // The warp index is broadcast from lane 0 so that the compiler knows it is
    // warp-uniform: role branches and every value derived from it (MMA
    // descriptors, tensor-memory addresses) can then live in uniform registers.
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const Watch watch{&bars->abort_flag, p.status, p.timeout_ns};

    auto bar = [&](uint64_t &b) { return ptx::smem_addr(&b); };

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(bars->q_full[t]), 1);
            ptx::mbar_init(bar(bars->q_empty[t]), 1);
            ptx::mbar_init(bar(bars->s_full[t]), 1);
            ptx::mbar_init(bar(bars->s_free[t]), 128);
            ptx::mbar_init(bar(bars->p_full[t]), 128);
            ptx::mbar_init(bar(bars->p_free[t]), 1);
            ptx::mbar_init(bar(bars->o_empty[t]), 128);
            ptx::mbar_init(bar(bars->mma_done[t]), 1);
        }
        for (int s = 0; s < kSchedRing; ++s) {
            ptx::mbar_init(bar(bars->sched_full[s]), 1);
            ptx::mbar_init(bar(bars->sched_empty[s]), kSchedReaders);
        }
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(bars->kv_full[s]), 1);
            ptx::mbar_init(bar(bars->kv_empty[s]), 2);  // one arrival per issuer
        }
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == kMmaWarp0) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, bars->tmem_base, 0);

    // Ring position of the K/V tiles of a unit with n key tiles whose first
    // tile sits at position `base`: the order is K_0, then K_{j+1}, V_j for
    // j = 0 .. n-2, then V_{n-1} -- the order in which the MMAs consume them.
    auto pos_k = [](uint32_t base, int j) { return base + (j == 0 ? 0u : (uint32_t)(2 * j - 1)); };
    auto pos_v = [](uint32_t base, int j, int n) {
        return base + (j + 1 < n ? (uint32_t)(2 * j + 2) : (uint32_t)(2 * j + 1));
    };

    // The next work unit for a consumer warp (issuer, softmax): the
    // producer's k-th claim, read from ring slot k mod kSchedRing and released
    // by one arrival per warp.  False if the CTA is aborting.
    auto next_unit = [&](uint32_t &k, Unit &w) {
        const uint32_t s = k % kSchedRing;
        if (!__all_sync(0xffffffffu, watch.wait(bar(bars->sched_full[s]), (k / kSchedRing) & 1)))
            return false;
        const volatile Unit *su = &bars->sched_unit[s];
        w.bh = su->bh;
        w.q0 = su->q0;
        w.nkv[0] = su->nkv[0];
        w.nkv[1] = su->nkv[1];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(bars->sched_empty[s]));
        ++k;
        return true;
    };

    // Each role changes its register budget at the top of its own branch, so
    // the compiler sees which limit holds for which code.
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        ptx::setmaxnreg_dec<kOtherRegs>();
        if (lane == 0) {
            uint32_t pos = 0;
            uint32_t qn[2] = {0, 0}, q_last_par[2] = {0, 0};
            bool q_loaded[2] = {false, false};
            bool ok = true;
            // a TMA coordinate that fails the bounds-checking build's test stops
            // the CTA the way an expired wait does
            auto stop = [&]() {
                *watch.abort_flag = 1;
                return false;
            };
            auto load_kv = [&](const CUtensorMap *tm, int j, int bh) {
                const int s = pos % kStages;
                if (!watch.wait(bar(bars->kv_empty[s]), ((pos / kStages) & 1) ^ 1)) return false;
                if (!in_bounds(j >= 0 && j * BN < p.Skv && bh >= 0 && bh < p.BH, p.status))
                    return stop();
                ptx::mbar_arrive_expect_tx(bar(bars->kv_full[s]), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    ptx::tma_load_3d(sKV + s * C::kTileBytes + c * C::kChunkBytes, tm,
                                     bar(bars->kv_full[s]), c * 64, j * BN, bh);
                ++pos;
                return true;
            };
            // Dynamic schedule: the next unit is claimed from the launch's counter
            // once this unit's last load is issued (the claim's latency hides
            // behind the ring), and published to the other roles.
            unsigned claim = atomicAdd(p.sched, 1u);
            for (uint32_t k = 0; ok; ++k) {
                const uint32_t slot = k % kSchedRing;
                if (!watch.wait(bar(bars->sched_empty[slot]), ((k / kSchedRing) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                // the unit is decoded once here and published whole, so that
                // the other roles start it without integer divisions
                Unit w{-2, 0, {0, 0}};
                if (claim < (unsigned)p.n_units) w = decode_unit((int)claim, p);
                volatile Unit *su = &bars->sched_unit[slot];
                su->bh = w.bh;
                su->q0 = w.q0;
                su->nkv[0] = w.nkv[0];
                su->nkv[1] = w.nkv[1];
                ptx::mbar_arrive(bar(bars->sched_full[slot]));
                if (w.bh < 0) break;
                // The Q tiles of the new unit into L2 now.  Their loads below
                // wait until the current unit's last S of that tile is computed,
                // and Q is read only once, so they would otherwise start from
                // HBM about one key tile before the softmax needs them.
                for (int t = 0; t < 2; ++t)
                    if (w.nkv[t] > 0 &&
                        in_bounds(w.q0 + t * BM < p.Sq && w.bh >= 0 && w.bh < p.BH, p.status))
                        for (int c = 0; c < C::kChunks; ++c)
                            ptx::tma_prefetch_3d(&tm_q, c * 64, w.q0 + t * BM, w.bh);
                const int nmax = max(w.nkv[0], w.nkv[1]);
                if (nmax == 0) {
                    claim = atomicAdd(p.sched, 1u);
                    continue;
                }
                for (int t = 0; t < 2 && ok; ++t) {
                    if (w.nkv[t] == 0) continue;
                    if (!watch.wait(bar(bars->q_empty[t]), (qn[t] & 1) ^ 1)) { ok = false; break; }
                    if (!in_bounds(w.q0 + t * BM < p.Sq && w.bh >= 0 && w.bh < p.BH, p.status)) {
                        ok = stop();
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(bar(bars->q_full[t]), C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tm_q,
                                         bar(bars->q_full[t]), c * 64, w.q0 + t * BM, w.bh);
                    q_last_par[t] = qn[t] & 1;
                    q_loaded[t] = true;
                    ++qn[t];
                }
                ok = ok && load_kv(&tm_k, 0, w.bh);
                for (int j = 0; j < nmax && ok; ++j)
                    ok = (j + 1 >= nmax || load_kv(&tm_k, j + 1, w.bh)) && load_kv(&tm_v, j, w.bh);
                if (ok) claim = atomicAdd(p.sched, 1u);
            }
            // teardown: wait until every load this thread issued has landed
            for (uint32_t s = 0; s < (uint32_t)kStages && s < pos; ++s) {
                const uint32_t last = s + ((pos - 1 - s) / kStages) * kStages;  // last use of s
                watch.drain(bar(bars->kv_full[s]), (last / kStages) & 1);
            }
            for (int t = 0; t < 2; ++t)
                if (q_loaded[t]) watch.drain(bar(bars->q_full[t]), q_last_par[t]);
        }
        __syncwarp();
    } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
        // ------------------------------------------------------------ MMA issuer of tile t
        // The whole warp runs this loop; one elected lane issues each MMA and commit.
        ptx::setmaxnreg_dec<kOtherRegs>();
        // a wait's outcome is made warp-uniform so that the warp stays converged
        auto wait_all = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, watch.wait(b, parity));
        };
        const int t = warp - kMmaWarp0;
        constexpr uint32_t kIdescS = idesc_f16(kBF16, BM, BN, false);
        constexpr uint32_t kIdescO = idesc_f16(kBF16, BM, D, true);
        const uint64_t dq = sdesc(sQ + t * C::kTileBytes, 16, 1024);
        const uint64_t dp = sdesc(sP + t * C::kPBytes, 16, 1024);
        const uint64_t dk = sdesc(sKV, 16, 1024);
        const uint64_t dv = sdesc(sKV, C::kChunkBytes, 1024);
        const uint32_t tS = tmem + C::col_s(t), tO = tmem + C::col_o(t);
        uint32_t pos = 0, qn = 0, sn = 0, pn = 0, on = 0;
        bool ok = true;
        bool first = true;
        auto stage_of = [&](uint32_t at, int &st) {
            st = at % kStages;
            return (at / kStages) & 1;
        };
        // S_t(jj) = Q_t K_jj^T, K_jj at ring position `at`
        auto issue_s = [&](uint32_t at, int jj, int my) {
            int st;
            const uint32_t par = stage_of(at, st);
            if (!wait_all(bar(bars->kv_full[st]), par)) return false;
            if (jj >= my) {  // this tile needs no more keys: release the stage in order
                ptx::mbar_arrive_warp(bar(bars->kv_empty[st]));
                return true;
            }
            // the softmax must have copied the previous S_t out of tensor memory
            if (sn > 0 && !wait_all(bar(bars->s_free[t]), (sn - 1) & 1)) return false;
            ptx::tc_fence_after();
            const uint64_t dkj = dk + (uint64_t)((st * C::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t koff = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                ptx::mma_ss_warp(tS, dq + koff, dkj + koff, kIdescS, kk > 0 ? 1u : 0u);
            }
            const bool skip = p.hook == 1 && first && t == 0 && blockIdx.x == 0;
            if (!skip) ptx::mma_commit_warp(bar(bars->s_full[t]));
            first = false;
            ++sn;
            ptx::mma_commit_warp(bar(bars->kv_empty[st]));
            if (jj == my - 1) ptx::mma_commit_warp(bar(bars->q_empty[t]));
            return true;
        };
        // O_t += P_t(jj) V_jj once the softmax has written P_t(jj)
        auto issue_pv = [&](uint32_t at, int jj, int my) {
            int st;
            const uint32_t par = stage_of(at, st);
            if (!wait_all(bar(bars->kv_full[st]), par)) return false;
            if (jj >= my) {
                ptx::mbar_arrive_warp(bar(bars->kv_empty[st]));
                return true;
            }
            if (!wait_all(bar(bars->p_full[t]), pn & 1)) return false;
            ++pn;
            if (jj == 0) {  // the epilogue of the previous unit has read O_t
                if (!wait_all(bar(bars->o_empty[t]), (on & 1) ^ 1)) return false;
                ++on;
            }
            ptx::tc_fence_after();
            const uint64_t dvj = dv + (uint64_t)((st * C::kTileBytes) >> 4);
            if constexpr (C::kTmemP) {
                // A = P_t from tensor memory: 16 keys (8 columns of bf16 pairs) per MMA
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    ptx::mma_ts_warp(tO, tmem + C::col_p(t) + kk * 8,
                                     dvj + (uint64_t)((kk * 16 * 128) >> 4), kIdescO,
                                     (jj > 0 || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t koff = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_ss_warp(tO, dp + koff, dvj + (uint64_t)((kk * 16 * 128) >> 4),
                                     kIdescO, (jj > 0 || kk > 0) ? 1u : 0u);
                }
            }
            ptx::mma_commit_warp(bar(bars->p_free[t]));
            ptx::mma_commit_warp(bar(bars->kv_empty[st]));
            return true;
        };
        for (uint32_t k = 0; ok;) {
            Unit w;
            if (!next_unit(k, w)) { ok = false; break; }
            if (w.bh < 0) break;
            const int nmax = max(w.nkv[0], w.nkv[1]);
            const int my = w.nkv[t];
            if (nmax == 0) continue;
            if (my > 0) {
                if (!wait_all(bar(bars->q_full[t]), qn & 1)) { ok = false; break; }
                ++qn;
            }
            // every stage is waited for and released in ring order, also by a
            // tile that needs fewer key tiles than the other
            ok = issue_s(pos_k(pos, 0), 0, my);
            for (int j = 0; j < nmax && ok; ++j)
                ok = (j + 1 >= nmax || issue_s(pos_k(pos, j + 1), j + 1, my)) &&
                     issue_pv(pos_v(pos, j, nmax), j, my);
            pos += 2 * nmax;
        }
        // teardown: every MMA issued by this warp has completed
        ptx::mma_commit_warp(bar(bars->mma_done[t]));
        watch.drain(bar(bars->mma_done[t]), 0);
        __syncwarp();
    } else if (warp < kProducerWarp) {
        // ------------------------------------------------------------ softmax
        ptx::setmaxnreg_inc<kSoftmaxRegs>();
        const int t = warp >> 2;        // query tile of this warpgroup
        const int wq = warp & 3;        // TMEM lane quarter of this warp
        const int r = wq * 32 + lane;   // row of this thread inside the tile
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::col_s(t);
        const uint32_t tO = tmem + lane_base + C::col_o(t);
        const uint32_t pRow = sP + t * C::kPBytes + r * 128;  // this row in both P atom columns
        const uint32_t tP = tmem + lane_base + C::col_p(t);  // this warp's lanes of P_t (d = 64)
        const uint32_t swz = (uint32_t)(r & 7);               // 128-byte swizzle phase of the row
        const float sl2 = p.scale_log2;
        const int off = p.Skv - p.Sq;
        uint32_t sn = 0, pfn = 0;
        bool ok = true;

        for (uint32_t k = 0; ok;) {
            Unit w;
            if (!next_unit(k, w)) { ok = false; break; }
            if (w.bh < 0) break;
            const int nk = w.nkv[t];
            const int row = w.q0 + t * BM + r;  // query index of this thread
            const int limit = p.causal ? min(p.Skv, row + off + 1) : p.Skv;  // keys < limit visible
            float m = -INFINITY;  // running max, log2-scaled units
            // running normalisers relative to m: l sums the exact P (for the
            // lse); lr is l with each tile's largest P taken at its 16-bit
            // value, the one P.V multiplies (for the output)
            float l = 0.f;
            float lr = 0.f;

            for (int j = 0; j < nk; ++j) {
                const bool got = watch.wait(bar(bars->s_full[t]), sn & 1);
                ++sn;
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                ptx::tc_fence_after();
                const int kv0 = j * BN;
                Half ra, rb;
                // Both halves in flight at once.  The load-and-reduce form also
                // returns each half's maximum, which is the row maximum of the
                // tile unless some of its keys are masked.
                float mxa, mxb;
                ptx::tmem_ld64_max(tS, ra.a, ra.b, mxa);
                ptx::tmem_ld64_max(tS + 64, rb.a, rb.b, mxb);
                ptx::tmem_wait_ld();
                fence_half(ra);
                fence_half(rb);
                asm volatile("" : "+f"(mxa), "+f"(mxb));  // read only after the wait
                // S_t is in registers: the next S_t may be written
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(bars->s_free[t]));
                float smax;  // raw maximum of the tile's visible keys
                if (kv0 + BN > limit) {
                    // diagonal or tail tile: masked keys must not set the maximum
                    mask_half(ra, kv0, limit);
                    mask_half(rb, kv0 + 64, limit);
                    smax = fmaxf(max_half(ra), max_half(rb));
                } else {
                    smax = fmaxf(mxa, mxb);
                }
                const float m_new = fmaxf(m, smax * sl2);
                bool rescale = false;
                float alpha = 1.f;
                if (m == -INFINITY) {
                    m = m_new;  // first visible keys: nothing accumulated yet
                } else if (m_new - m > kRescaleLog2) {
                    rescale = true;
                    alpha = ptx::ex2_approx(m - m_new);
                    m = m_new;
                    l *= alpha;
                    lr *= alpha;
                }
                // P_t(j-1) . V must be complete before O_t is rescaled or the P
                // buffer is overwritten
                bool pv_done = (j == 0);
                if (__any_sync(0xffffffffu, rescale)) {
                    if (!pv_done) {
                        const bool g2 = watch.wait(bar(bars->p_free[t]), pfn & 1);
                        ++pfn;
                        pv_done = true;
                        if (!__all_sync(0xffffffffu, g2)) { ok = false; break; }
                        ptx::tc_fence_after();
                    }
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + c * 32, o);
                        ptx::tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
                            o[i] = __float_as_uint(v.x);
                            o[i + 1] = __float_as_uint(v.y);
                        }
                        ptx::tmem_st32(tO + c * 32, o);
                        ptx::tmem_wait_st();
                    }
                }
                const float mb = (m == -INFINITY) ? 0.f : m;
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                uint32_t pa[32], pb[32];
                exp32<kBF16>(ra.a, sl2, mb, pa, acc);
                exp32<kBF16>(ra.b, sl2, mb, pa + 16, acc);
                if (!pv_done) {
                    const bool g2 = watch.wait(bar(bars->p_free[t]), pfn & 1);
                    ++pfn;
                    if (!__all_sync(0xffffffffu, g2)) { ok = false; break; }
                }
                if constexpr (C::kTmemP) {
                    // P row into tensor memory: column c holds keys 2c, 2c + 1
                    ptx::tmem_st32(tP, pa);
                    exp32<kBF16>(rb.a, sl2, mb, pb, acc);
                    exp32<kBF16>(rb.b, sl2, mb, pb + 16, acc);
                    ptx::tmem_st32(tP + 32, pb);
                    ptx::tmem_wait_st();
                } else {
                    // P row into the K-major, 128-byte-swizzled tile: 16-byte chunk c
                    // of a 128-byte row is stored at chunk c ^ (row mod 8)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        ptx::st_shared_v4(pRow + ((((uint32_t)c) ^ swz) << 4), pa[4 * c],
                                          pa[4 * c + 1], pa[4 * c + 2], pa[4 * c + 3]);
                    exp32<kBF16>(rb.a, sl2, mb, pb, acc);
                    exp32<kBF16>(rb.b, sl2, mb, pb + 16, acc);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        ptx::st_shared_v4(pRow + C::kChunkBytes + ((((uint32_t)c) ^ swz) << 4),
                                          pb[4 * c], pb[4 * c + 1], pb[4 * c + 2], pb[4 * c + 3]);
                    ptx::fence_proxy_async_smem();
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(bars->p_full[t]));
                const float2 s01 = __fadd2_rn(acc[0], acc[1]), s23 = __fadd2_rn(acc[2], acc[3]);
                const float tile_sum = (s01.x + s01.y) + (s23.x + s23.y);
                l += tile_sum;
                lr += tile_sum + max_p_rounding<kBF16>(smax, sl2, mb);
            }
            if (!ok) break;

            // epilogue: O / l and lse for the rows of this thread
            if (nk > 0) {  // the last P_t . V of the unit has completed
                const bool got = watch.wait(bar(bars->p_free[t]), pfn & 1);
                ++pfn;
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                ptx::tc_fence_after();
            }
            const float inv = lr > 0.f ? 1.f / lr : 0.f;
            const bool live = row < p.Sq;
            const size_t orow = ((size_t)w.bh * p.Sq + row) * D;
            const size_t o_elems = (size_t)p.BH * p.Sq * D;  // extent of o (and lse / D)
            if (D == 128 && p.stage_o && nk > 0) {
                // Staged stores: each warp writes O / lr of its 32 rows into its
                // rows of the P tile (free: the last P.V has completed) -- 16
                // chunks of 16 bytes per row, columns 0-63 of a 16-bit row (or
                // the first 32 of a 64-column fp32 half) in the rows of the first
                // 64-key atom, the rest in the second, chunk c at c ^ (row mod 8)
                // -- and stores them back two rows (16-bit) or two half rows
                // (fp32) per warp instruction: whole 128-byte lines instead of 32
                // rows of 16 bytes each.  fp32 output takes two passes.
                const uint32_t sw = sP + t * C::kPBytes + (uint32_t)(wq * 32) * 128;
                const int rbase = w.q0 + t * BM + wq * 32;
                const int passes = p.out_f32 ? 2 : 1;
#pragma unroll 1
                for (int h = 0; h < passes; ++h) {
#pragma unroll 1
                    for (int c = 0; c < (p.out_f32 ? 2 : 4); ++c) {
                        uint32_t o[32];
                        __syncwarp();  // tcgen05.ld needs the whole warp converged
                        ptx::tmem_ld32(tO + h * 64 + c * 32, o);
                        ptx::tmem_wait_ld();
                        reg_fence(o);
                        if (p.out_f32) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int ch = 8 * c + i;
                                ptx::st_shared_v4(
                                    sw + (uint32_t)(ch >> 3) * C::kChunkBytes + (uint32_t)lane * 128 +
                                        ((uint32_t)((ch & 7) ^ (lane & 7)) << 4),
                                    __float_as_uint(__uint_as_float(o[4 * i]) * inv),
                                    __float_as_uint(__uint_as_float(o[4 * i + 1]) * inv),
                                    __float_as_uint(__uint_as_float(o[4 * i + 2]) * inv),
                                    __float_as_uint(__uint_as_float(o[4 * i + 3]) * inv));
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int ch = 4 * c + i;
                                ptx::st_shared_v4(
                                    sw + (uint32_t)(ch >> 3) * C::kChunkBytes + (uint32_t)lane * 128 +
                                        ((uint32_t)((ch & 7) ^ (lane & 7)) << 4),
                                    pack2<kBF16>(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                                    pack2<kBF16>(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                                    pack2<kBF16>(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                                    pack2<kBF16>(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
                            }
                        }
                    }
                    if (h == passes - 1) {  // O_t is read: the next unit's P.V may overwrite it
                        __syncwarp();
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(bar(bars->o_empty[t]));
                    }
                    __syncwarp();  // the staged rows of the other lanes are visible
                    // lanes 0-15: row 2i, lanes 16-31: row 2i + 1; 16 bytes each
#pragma unroll 4
                    for (int i = 0; i < 16; ++i) {
                        const int rr = 2 * i + (lane >> 4);  // row inside the warp's 32
                        const int ch = lane & 15;
                        uint4 v;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                     : "r"(sw + (uint32_t)(ch >> 3) * C::kChunkBytes + (uint32_t)rr * 128 +
                                           ((uint32_t)((ch & 7) ^ (rr & 7)) << 4)));
                        const int grow = rbase + rr;
                        if (grow >= p.Sq) continue;
                        if (p.out_f32) {
                            const size_t go = ((size_t)w.bh * p.Sq + grow) * D + (size_t)h * 64 + (size_t)ch * 4;
                            if (in_bounds(go + 4 <= o_elems, p.status))
                                *reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.o) + go) = v;
                        } else {
                            const size_t go = ((size_t)w.bh * p.Sq + grow) * D + (size_t)ch * 8;
                            if (in_bounds(go + 8 <= o_elems, p.status))
                                *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.o) + go) = v;
                        }
                    }
                    __syncwarp();  // every lane is done with the staged rows
                }
            } else {
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
                } else if (!in_bounds(orow + (size_t)(c + 1) * 32 <= o_elems, p.status)) {
                    // bounds-checking build: the store is skipped
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
            }
            if (live && p.lse && in_bounds(orow < o_elems, p.status))
                p.lse[(size_t)w.bh * p.Sq + row] =
                    l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            if (nk > 0 && !(D == 128 && p.stage_o)) {  // the staged path released O_t above
                __syncwarp();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(bars->o_empty[t]));
            }
        }
    } else {
        // warp 11: no role; it only gives up its registers
        ptx::setmaxnreg_dec<kOtherRegs>();
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp0) ptx::tmem_dealloc(tmem, kTmemCols);
    // every CTA has made its last claim: the last one to finish resets the
    // counter pair for a later launch
    if (threadIdx.x == 0 && atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 1, 0u);
    }
}

// Counter pairs of the dynamic schedule (zero at module load; each launch
// leaves its pair at zero again).
__device__ unsigned int g_sched[kSchedSlots * 2];

// ------------------------------------------------------------------ host side
std::mutex g_sched_mu;
unsigned int *g_sched_addr[64];
std::atomic<unsigned> g_sched_seq{0};

// The counter pair of the next launch on the current device; nullptr on error.
unsigned int *next_sched_pair() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    unsigned int *base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_sched_mu);
        if (!g_sched_addr[dev]) {
            void *a = nullptr;
            if (cudaGetSymbolAddress(&a, g_sched) != cudaSuccess) return nullptr;
            g_sched_addr[dev] = static_cast<unsigned int *>(a);
        }
        base = g_sched_addr[dev];
    }
    return base + 2 * (g_sched_seq.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
}
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
    unsigned int *sched = next_sched_pair();
    if (!status || !sched) return ATTN_ERR_CUDA;
    TcParams p;
    p.o = o;
    p.lse = lse;
    p.status = status;
    p.sched = sched;
    p.BH = (int)BH;
    p.Sq = pr.Sq;
    p.Skv = pr.Skv;
    p.causal = pr.causal;
    p.nqb = (pr.Sq + 2 * BM - 1) / (2 * BM);
    const int sms = device_sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    {
        // heads per schedule group: about one round of units (one per CTA), so
        // that the CTAs running at any time work on the K and V of a few heads,
        // which stay in L2 between the units that read them
        // (the smallest divisor of B*H that covers a round: equal groups, so
        // that no short group is left for the end, where it would run alone).
        // Without such a divisor all heads form one group -- unless their K and
        // V exceed what L2 holds, where round-sized groups with a smaller last
        // one cost less than reading K and V from HBM once per round of units.
        int64_t h0 = ((int64_t)sms + p.nqb - 1) / p.nqb;
        if (h0 < 1) h0 = 1;
        int64_t hg = h0;
        while (hg < BH && BH % hg != 0) ++hg;
        const int64_t kv_bytes = BH * 2LL * pr.Skv * D * 2;
        if (hg >= BH && kv_bytes > (96LL << 20)) hg = h0;
        if (hg > BH) hg = BH;
        p.hg = (int)hg;
    }
    const int64_t n_units = BH * p.nqb;
    if (n_units > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    p.n_units = (int)n_units;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.out_f32 = (pr.dtype == ATTN_BF16_OUT_F32 || pr.dtype == ATTN_F16_OUT_F32) ? 1 : 0;
    // Staged O stores (see the epilogue) pay with up to 8192 keys: +0.4-1.6 % at 8k
    // causal, +2.6 % at 4k, +8.6 % at 8k queries x 2k keys with fp32 output; with
    // 16k and 32k keys they measured 1-4 % slower, so those keep the direct stores.
    p.stage_o = (pr.d == 128 && pr.Skv <= 8192) ? 1 : 0;
    p.hook = test_hook();
    p.timeout_ns = watchdog_ns();
    const int grid = (int)(n_units < sms ? n_units : sms);
    auto kern = attn_tc_kernel<D, kBF16>;
    // The register split inside the kernel (setmaxnreg) needs exactly the pool
    // it was sized for; a build with another entry register count would block
    // in setmaxnreg.inc, so it is refused here instead of launched.
    static std::atomic<int> regs_ok{-1};  // a property of the binary: the same on every device
    int ok = regs_ok.load(std::memory_order_relaxed);
    if (ok < 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return ATTN_ERR_UNSUPPORTED_DEVICE;
        ok = (fa.numRegs == kLaunchRegs && fa.maxThreadsPerBlock >= kThreads) ? 1 : 0;
        regs_ok.store(ok, std::memory_order_relaxed);
    }
    if (!ok) return ATTN_ERR_LAUNCH;
    if (!set_smem_limit_once(reinterpret_cast<const void *>(kern), C::kSmemBytes))
        return ATTN_ERR_LAUNCH;
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return ATTN_ERR_UNSUPPORTED_DEVICE;
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

void forget_sched_counters(int dev) {
    if (dev < 0 || dev >= 64) return;
    std::lock_guard<std::mutex> lk(g_sched_mu);
    g_sched_addr[dev] = nullptr;
}

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
