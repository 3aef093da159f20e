// route_tc.cu -- Step 1, Route, for bf16 routers (1 <= E <= 256): the
// router GEMM on the tensor cores with the score, top-k and gates fused into
// the epilogue (Ultralytics glossary "Expert Parallelism", "How Tokens Move
// Between GPUs", step 1; DeepSeek-V3 selection-only bias from "Load Balancing
// and Capacity").
//
// logits[T, E] = x[T, d] . Wr[E, d]^T with bf16 operands and fp32
// accumulation in tensor memory.  Every product of two bf16 values is exact
// in fp32; on inputs whose partial sums stay representable (the dyadic test
// grid: multiples of 2^-12 below 2^10) the accumulation is exact too, so the
// logits -- and every routing decision -- equal the FFMA kernels' bit for bit.
//
// Persistent kernel, one CTA per SM (192 or 320 threads, ~200 KB of shared
// memory so that exactly one CTA holds the SM's 512 TMEM columns):
//   warp 0     TMA: a 128-token x 64 tile of x and the E x 64 tile of Wr
//              (rows past E zero-filled) per stage;
//   warp 1     TMEM allocation; one lane issues tcgen05.mma (M=128, N=Np,
//              Np = E rounded up to a multiple of 16, at least 16) into one of
//              two accumulators;
//   warps 2-5  epilogue (and warps 6-9 when CTAs have several tiles: the two
//              groups take alternate tiles, one TMEM buffer each, so two
//              tiles' epilogues overlap): each thread owns one token (one TMEM lane), reads
//              its E logits 32 at a time and keeps a sorted top-k in registers
//              (ties to the lower expert index), then computes the gates and
//              writes topk_idx / topk_gate.
// Sigmoid routers: the exact score fp32(1/(1+exp(-L))) needs double
// precision, which is slow on this part.  The epilogue ranks all experts by
// an approximation a of the key (score + selection bias) with a known bound
// |a - key| <= eps, finds the k-th largest approximation A_k, and evaluates
// the exact score only for experts with a >= A_k - 2*delta, delta > eps.  The
// k experts with the largest a have keys >= A_k - eps, so the k-th exact key
// is >= A_k - eps; any expert of the exact top-k therefore has key >= A_k -
// eps and a >= A_k - 2*eps > A_k - 2*delta.  The exact top-k over these
// candidates is the exact top-k over all experts, ties included.  The main
// pass uses a fast fp32 sigmoid (delta = 2^-14, over 100x its bound, plus
// 2^-21 |A_k| for the rounding of large keys) and keeps the k + 4 best
// experts with their logits, so the candidates are almost always in that list;
// the rank pass of rank-limited routing uses 1/2 + tanh(L/2)/2 with the
// hardware tanh (documented relative error 2^-11, so eps < 2.5e-4) and
// delta = 2^-8.
//
// Epilogue layout: per 32-logit chunk, one compact unrolled pass stashes the
// logits in shared memory (one padded row per thread) and builds a 32-bit
// mask of the values that beat the current k-th key; only those are inserted
// (sorted insertion, ties to the lower index), so the insertion code exists
// once and runs rarely.
#include <float.h>

#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int RM = 128, RK = 64;
// Per epilogue thread: 32 stashed logits (+1 pad), and with rank limiting two
// rows of 32 rank scores; odd pitches keep the per-thread rows conflict-free.
constexpr int STASH_PITCH = 33;
constexpr int STASH_PITCH_RANKS = 97;
constexpr int R_THREADS_MAX = 64 + 2 * 128;  // producer, MMA, up to two epilogue warp groups
constexpr int R_MAX_STAGES = 12;  // deep rings for few experts (18 KB stages): more of x in flight
constexpr uint32_t R_TMEM_COLS = 512;
constexpr int R_SMEM_TILES = 221184;  // bytes of stage ring (at most)
constexpr int R_SMEM_FIXED = 1024 /*align*/ + 256 /*barriers*/ + 2 * 256 * 4 /*biases*/;
constexpr int R_SMEM_MAX = 232448;  // 227 KB per block
constexpr float kApproxDelta = 1.0f / 256.0f;
static_assert((2 * R_MAX_STAGES + 5) * 8 <= 240, "barriers overlap the flags");

struct RtParams {
    int64_t T;
    int d, E, Np, k, score, renorm;
    int R, max_ranks;   // rank-limited routing when max_ranks > 0
    int stash_pitch;    // floats of shared memory per epilogue thread
    int epi_groups;     // epilogue warp groups (1 or 2); group g owns TMEM buffer g when 2
    const float* logit_bias;
    const float* sel_bias;
    int32_t* idx;
    float* gate;
    uint32_t* status;
    int num_kb, m_tiles, stages, stage_bytes;
    int kbs;        // K blocks per ring stage (their x boxes are issued back to back)
    int num_st;     // ring stages per tile: num_kb / kbs
    int tile_rows;  // tokens per tile (multiple of 8, <= 128); the MMA always runs M = 128
    int tx_bytes;   // bytes one stage's TMA loads deliver
    // Expert split: each tile's experts are cut into `split` slices of Eh
    // experts (one work unit each, units = m_tiles * split).  With split > 1
    // every unit writes its exact partial top-k to `part` (and, for softmax
    // gates without renormalisation, its partial softmax sum to `zpart`), and
    // route_merge_kernel forms the final top-k and gates.
    int split, Eh, units;
    // 1 (split only, one unit per CTA): the split units of a tile form a
    // thread-block cluster; each leaves its partial list in its stash rows and
    // the slice-0 CTA merges them through distributed shared memory (no merge
    // kernel, no partial lists in global memory)
    int cmerge;
    // 1: epilogue group 0 first runs its code once on the unused TMEM buffer,
    // storing nothing, while the K loop streams x (see the epilogue)
    int warm;
    RoutePartial* part;
    float2* zpart;
};

__device__ __forceinline__ float sigmoid_exact(float L) {
    return (float)(1.0 / (1.0 + exp(-(double)L)));
}
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sigmoid_approx(float L) {
    return fmaf(0.5f, tanh_approx(0.5f * L), 0.5f);
}
// A fast fp32 sigmoid for ranking.  With e = exp(-L), the documented bounds of
// the intrinsics (__expf: 2 + floor(|1.173 L|) ulp; the fp32 add: 1/2 ulp;
// __fdividef: 2 ulp for divisors up to 2^126, and 0 beyond, where the true
// value is below 2^-126) give |f - s| <= s (1 - s) (2 + 1.2 |L|) 2^-23 + 3 s 2^-23,
// at most ~4e-7 over all L (s (1 - s) decays like e^-|L|).  kFastDelta = 2^-14
// is over 100 times that.
__device__ __forceinline__ float sigmoid_fast(float L) { return __fdividef(1.f, 1.f + __expf(-L)); }
constexpr float kFastDelta = 1.0f / 16384.0f;

// Sorted top-k (k <= 8) in registers: key, a payload value and the index.
// The list always has 8 entries, in descending key order: 8 - k sentinels
// (key +inf, never displaced) followed by the k best so far, so the k-th best
// is always entry 7.  A fixed position keeps the list in registers (reading
// entry k - 1 for a runtime k would make it an indexed array in local memory).
template <int N>
struct TopKN {
    float key[N], val[N];
    int idx[N];
    // n (<= N) real entries, behind N - n sentinels
    __device__ __forceinline__ void init(int n) {
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const bool sentinel = j < N - n;
            key[j] = sentinel ? INFINITY : -INFINITY;
            val[j] = 0.f;
            idx[j] = sentinel ? -1 : 0x7fffffff;
        }
    }
    __device__ __forceinline__ float last_key() const { return key[N - 1]; }
    // Sorted insertion.  The new entry's place is the number of entries that
    // rank before it (the list is sorted, so they form a prefix); every slot's
    // new content then depends only on the old list and that place, so the
    // eight compares and the shifts are independent instructions rather than
    // one chain of compare-and-swap steps.
    __device__ __forceinline__ void insert(float kv, float v, int e) {
        if (!key_better(kv, e, key[N - 1], idx[N - 1])) return;
        int pos = 0;
#pragma unroll
        for (int j = 0; j < N - 1; ++j) pos += key_better(key[j], idx[j], kv, e) ? 1 : 0;
#pragma unroll
        for (int j = N - 1; j > 0; --j) {
            const bool shift = j > pos, here = j == pos;
            key[j] = shift ? key[j - 1] : (here ? kv : key[j]);
            val[j] = shift ? val[j - 1] : (here ? v : val[j]);
            idx[j] = shift ? idx[j - 1] : (here ? e : idx[j]);
        }
        if (pos == 0) {
            key[0] = kv;
            val[0] = v;
            idx[0] = e;
        }
    }
};
// The router's top-k: 8 - k sentinels, then the k best, the k-th always entry 7.
struct TopK : TopKN<8> {
    __device__ __forceinline__ float kth_key() const { return key[7]; }
};

// The best m of R scores s[0..R) by rounds of selection (ties to the lower
// rank): returns the bit set of chosen ranks and, in *mth, the m-th score.
__device__ __forceinline__ uint32_t pick_ranks(const float* sc, int R, int m, float* mth) {
    uint32_t chosen = 0;
    float last = -INFINITY;
    for (int j = 0; j < m; ++j) {
        int best = -1;
        for (int r = 0; r < R; ++r)
            if (!((chosen >> r) & 1u) && (best < 0 || sc[r] > sc[best])) best = r;
        chosen |= 1u << best;
        last = sc[best];
    }
    *mth = last;
    return chosen;
}

// First K block of a tile.  Every tile reads the same router weights; if all
// CTAs walked K in the same order they would all hit the few L2 slices that
// hold the current weight block at once.  Rotating the start per tile spreads
// them over the whole matrix.  (The summation order then differs between
// tiles; on inputs whose sums are exact in fp32 this changes nothing.)
__device__ __forceinline__ int k_start(int tile, int num_kb) { return (int)(((unsigned)tile * 37u) % (unsigned)num_kb); }

// SPLIT: the launch cuts each tile's experts into p.split slices (never with
// rank-limited routing); a separate instantiation keeps the unsplit kernel's
// register budget as it is.
template <bool SPLIT>
__global__ void __launch_bounds__(R_THREADS_MAX, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const RtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* extra = smem + p.stages * p.stage_bytes;
    // full[R_MAX_STAGES] empty[R_MAX_STAGES] accf[2] acce[2] drain: 232 bytes
    uint64_t* bars = reinterpret_cast<uint64_t*>(extra);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(extra + 240);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(extra + 244);
    float* lb_s = reinterpret_cast<float*>(extra + 256);
    float* sb_s = lb_s + 256;
    float* stash_all = sb_s + 256;  // [128][p.stash_pitch]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + R_MAX_STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * R_MAX_STAGES);
    const uint32_t acce0 = smem_u32(bars + 2 * R_MAX_STAGES + 2);
    const uint32_t drain = smem_u32(bars + 2 * R_MAX_STAGES + 4);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), R_TMEM_COLS);
    // programmatic dependent launch: everything above touched no global data
    pdl_wait();
    if (warp >= 2) {
        for (int e = threadIdx.x - 64; e < 256; e += (int)blockDim.x - 64) {
            lb_s[e] = (p.logit_bias && e < p.E) ? p.logit_bias[e] : 0.f;
            sb_s[e] = (p.sel_bias && e < p.E) ? p.sel_bias[e] : 0.f;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int unit = blockIdx.x; unit < p.units && !*abort_flag; unit += gridDim.x) {
                const int tile = SPLIT ? unit / p.split : unit;
                const int e0 = SPLIT ? (unit - tile * p.split) * p.Eh : 0;  // first expert of the slice
                const int ks0 = k_start(unit, p.num_st);
                for (int i = 0; i < p.num_st; ++i) {
                    int ks = ks0 + i;
                    if (ks >= p.num_st) ks -= p.num_st;
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status,
                                   MOE_DEV_GEMM_TIMEOUT))
                        break;
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, p.tx_bytes);
                    const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
                    const uint32_t sw = sa + p.kbs * (RM * RK * 2);
                    for (int j = 0; j < p.kbs; ++j)
                        tma_load_2d(sa + j * (RM * RK * 2), &tmX, (ks * p.kbs + j) * RK,
                                    tile * p.tile_rows, fb);
                    for (int j = 0; j < p.kbs; ++j)
                        tma_load_2d(sw + j * (p.Np * RK * 2), &tmW, (ks * p.kbs + j) * RK, e0, fb);
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(RM, p.Np);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < p.units && ok; unit += gridDim.x) {
                if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1, abort_flag, p.status,
                               MOE_DEV_GEMM_TIMEOUT)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
                for (int i = 0; i < p.num_st; ++i) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status,
                                   MOE_DEV_GEMM_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
                    const uint32_t sw = sa + p.kbs * (RM * RK * 2);
                    for (int j = 0; j < p.kbs; ++j) {
#pragma unroll
                        for (int kk = 0; kk < RK / 16; ++kk)
                            mma_bf16(d_tmem, sw128_desc(sa + j * (RM * RK * 2) + kk * 32),
                                     sw128_desc(sw + j * (p.Np * RK * 2) + kk * 32), idesc,
                                     (i | j | kk) != 0 ? 1u : 0u);
                    }
                    commit(empty0 + 8 * stage);
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                commit(accf0 + 8 * acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            if (!ok) {
                // drain this thread's MMAs before TMEM is released (bounded)
                commit(drain);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
                }
            }
        }
    } else {
        // ---------------- epilogue: one token per thread ----------------
        // With two warp groups, group g takes this CTA's tiles i with i % 2 == g
        // (they land in TMEM buffer g), so two tiles' epilogues run at once.
        const int q = warp & 3;
        const int egroup = (warp - 2) >> 2;
        const bool sigmoid = p.score == MOE_SCORE_SIGMOID;
        const bool has_lb = p.logit_bias != nullptr;
        const bool has_sb = p.sel_bias != nullptr;
        float* stash = stash_all + (threadIdx.x - 64) * p.stash_pitch;
        float* rank_a = stash + 33;  // rank scores (rank-limited routing only)
        float* rank_x = stash + 65;
        const bool limited = !SPLIT && p.max_ranks > 0;
        const int per = p.E / p.R;
        const float inv_per = 1.0f / (float)per;  // (e + 1/2) * inv_per truncates to e / per exactly
        // Warm-up: with one tile per CTA and few experts the epilogue is a
        // short stretch of code that runs once, after the K loop, mostly
        // waiting for its instructions to arrive.  Group 0 then first runs the
        // same code on TMEM buffer 1 (allocated, never written by this CTA's
        // MMAs) while the K loop streams x, with every store, status bit and
        // barrier arrival suppressed (`dry`), so that the real pass finds its
        // instructions cached.
        const bool warm_up = p.warm && egroup == 0;
        int local = warm_up ? -2 : -1;
        for (int unit = (int)blockIdx.x - (warm_up ? (int)gridDim.x : 0); unit < p.units;
             unit += gridDim.x) {
            ++local;
            const bool dry = local < 0;
            if (!dry && local % p.epi_groups != egroup) continue;
            const int acc = dry ? 1 : local & 1;  // the MMA alternates buffers per tile
            const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;  // n-th use of that buffer
            if (!dry) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait(accf0 + 8 * acc, acc_phase,
                                                                  abort_flag, p.status,
                                                                  MOE_DEV_GEMM_TIMEOUT));
                if (!ok) break;
            }
            fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
            // rows past tile_rows hold whatever the stage held before: computed, never stored
            const bool row_ok = !dry && q * 32 + lane < p.tile_rows;
            const int tile = SPLIT ? unit / p.split : unit;
            const int h = SPLIT ? unit - tile * p.split : 0;
            const int e0 = SPLIT ? h * p.Eh : 0;  // this unit's experts: [e0, e_end)
            const int e_end = SPLIT ? e0 + p.Eh : p.E;  // slices are whole 32-expert chunks
            const int nchunks = SPLIT ? p.Eh / 32 : (p.E + 31) / 32;
            const int64_t t = (int64_t)tile * p.tile_rows + q * 32 + lane;
            TopK top;
            top.init(p.k);
            float v[32];
            bool nonfinite = false;  // a NaN or infinite logit among this token's
            // Rank-limited routing: rank score = best key among the rank's
            // experts; keep the max_ranks best ranks (ties to the lower rank).
            uint32_t allowed = 0xffffffffu;
            if (limited) {
                for (int r = 0; r < p.R; ++r) rank_a[r] = -INFINITY;
                for (int c = 0; c < nchunks; ++c) {
                    tmem_ld32(tb + (uint32_t)(c * 32), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = e0 + c * 32 + i;
                        if ((SPLIT || e < e_end)) {
                            const float L = has_lb ? __fadd_rn(v[i], lb_s[e]) : v[i];
                            const float key =
                                sigmoid ? __fadd_rn(sigmoid_approx(L), sb_s[e]) : L;
                            const int r = (int)(((float)e + 0.5f) * inv_per);
                            if (key > rank_a[r]) rank_a[r] = key;
                        }
                    }
                }
                float mth;
                if (!sigmoid) {
                    allowed = pick_ranks(rank_a, p.R, p.max_ranks, &mth);
                } else {
                    // Approximate rank scores are within delta of the exact
                    // ones: a rank of the exact best set has approximate score
                    // >= (m-th approximate) - 2 delta, and its best expert has
                    // approximate key >= its approximate score - 2 delta.
                    pick_ranks(rank_a, p.R, p.max_ranks, &mth);
                    const float rthr = mth - 2.f * kApproxDelta;
                    for (int r = 0; r < p.R; ++r) rank_x[r] = -INFINITY;
                    for (int c = 0; c < nchunks; ++c) {
                        tmem_ld32(tb + (uint32_t)(c * 32), v);
                        uint32_t mask = 0;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int e = e0 + c * 32 + i;
                            const float L = has_lb ? __fadd_rn(v[i], lb_s[e & 255]) : v[i];
                            stash[i] = L;
                            if ((SPLIT || e < e_end)) {
                                const float a = __fadd_rn(sigmoid_approx(L), sb_s[e]);
                                const float ra = rank_a[(int)(((float)e + 0.5f) * inv_per)];
                                if (ra >= rthr && a >= ra - 2.f * kApproxDelta) mask |= 1u << i;
                            }
                        }
                        while (mask) {
                            const int i = __ffs(mask) - 1;
                            mask &= mask - 1;
                            const int e = e0 + c * 32 + i;
                            const float key = __fadd_rn(sigmoid_exact(stash[i]), sb_s[e]);
                            const int r = (int)(((float)e + 0.5f) * inv_per);
                            if (key > rank_x[r]) rank_x[r] = key;
                        }
                    }
                    allowed = pick_ranks(rank_x, p.R, p.max_ranks, &mth);
                }
            }
            auto rank_ok = [&](int e) -> bool {
                return !limited || ((allowed >> (int)(((float)e + 0.5f) * inv_per)) & 1u);
            };
            if (!sigmoid) {
                for (int c = 0; c < nchunks; ++c) {
                    tmem_ld32(tb + (uint32_t)(c * 32), v);
                    const float thr = top.kth_key();
                    uint32_t mask = 0;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = e0 + c * 32 + i;
                        const float L = has_lb ? __fadd_rn(v[i], lb_s[e & 255]) : v[i];
                        v[i] = L;
                        nonfinite |= (SPLIT || e < e_end) && !(fabsf(L) <= FLT_MAX);
                        if ((SPLIT || e < e_end) && L > thr && rank_ok(e)) mask |= 1u << i;
                    }
                    // stored after the loop: a store between the bias loads would
                    // order them (the compiler cannot tell the areas apart)
#pragma unroll
                    for (int i = 0; i < 32; ++i) stash[i] = v[i];
                    while (mask) {
                        const int i = __ffs(mask) - 1;
                        mask &= mask - 1;
                        const float L = stash[i];
                        top.insert(L, L, e0 + c * 32 + i);
                    }
                }
            } else {
                // One pass ranks the experts by the fast score (plus the selection
                // bias) and keeps the k + 4 best with their logits.  The exact
                // score is then needed only for kept experts within 2 delta of the
                // k-th fast key: every expert of the exact top-k is that close (see
                // the proof at the top of this file, with the fast score's bound
                // and the fp32 rounding of large keys, 2^-21 |key|, in delta).  If
                // even the (k+4)-th kept key is that close, the list may have
                // dropped a candidate, and a second pass visits every expert (with
                // k + 2 kept, that pass ran in a few warps of every large batch and
                // set the kernel's end).
                TopKN<12> approx;
                approx.init(p.k + 4);
                for (int c = 0; c < nchunks; ++c) {
                    tmem_ld32(tb + (uint32_t)(c * 32), v);
                    const float thr = approx.last_key();
                    uint32_t mask = 0;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = e0 + c * 32 + i;
                        const float L = has_lb ? __fadd_rn(v[i], lb_s[e & 255]) : v[i];
                        stash[i] = L;
                        nonfinite |= (SPLIT || e < e_end) && !(fabsf(L) <= FLT_MAX);
                        const float a = __fadd_rn(sigmoid_fast(L), sb_s[e & 255]);
                        if ((SPLIT || e < e_end) && a > thr && rank_ok(e)) mask |= 1u << i;
                    }
                    while (mask) {
                        const int i = __ffs(mask) - 1;
                        mask &= mask - 1;
                        const int e = e0 + c * 32 + i;
                        const float L = stash[i];
                        approx.insert(__fadd_rn(sigmoid_fast(L), sb_s[e]), L, e);
                    }
                }
                const float ak = approx.key[7];  // the k-th fast key
                const float band = ak - 2.f * (kFastDelta + fabsf(ak) * (1.0f / 2097152.0f));
                const bool every = approx.key[11] >= band;
                if (!every) {
#pragma unroll
                    for (int j = 0; j < 12; ++j) {
                        if (approx.idx[j] >= 0 && approx.key[j] >= band) {
                            const int e = approx.idx[j];
                            const float s = sigmoid_exact(approx.val[j]);
                            top.insert(has_sb ? __fadd_rn(s, sb_s[e]) : s, s, e);
                        }
                    }
                }
                if (__any_sync(0xffffffffu, every)) {
                    for (int c = 0; c < nchunks; ++c) {
                        tmem_ld32(tb + (uint32_t)(c * 32), v);
                        uint32_t mask = 0;
                        if (every) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int e = e0 + c * 32 + i;
                                const float L = has_lb ? __fadd_rn(v[i], lb_s[e & 255]) : v[i];
                                stash[i] = L;
                                const float a = __fadd_rn(sigmoid_fast(L), sb_s[e & 255]);
                                if ((SPLIT || e < e_end) && a >= band && rank_ok(e)) mask |= 1u << i;
                            }
                        }
                        while (mask) {
                            const int i = __ffs(mask) - 1;
                            mask &= mask - 1;
                            const int e = e0 + c * 32 + i;
                            const float s = sigmoid_exact(stash[i]);
                            top.insert(has_sb ? __fadd_rn(s, sb_s[e]) : s, s, e);
                        }
                    }
                }
            }
            // gates; the k chosen experts are entries 8-k .. 7, best first
            const int j0 = 8 - p.k;
            float g[8];
            float m = -INFINITY;  // softmax: the best logit (of this unit's experts)
            float z = 0.f;        // softmax: the gate denominator
            if (!sigmoid) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j == j0) m = top.val[j];
            }
            if (!sigmoid && !p.renorm) {
                // full softmax: the sum over every expert (of this unit)
                for (int c = 0; c < nchunks; ++c) {
                    tmem_ld32(tb + (uint32_t)(c * 32), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = e0 + c * 32 + i;
                        if ((SPLIT || e < e_end)) {
                            const float L = has_lb ? __fadd_rn(v[i], lb_s[e]) : v[i];
                            z += expf(L - m);
                        }
                    }
                }
            }
            if (SPLIT && p.cmerge) {
                // this slice's exact top-k (and partial softmax sum), left in the
                // thread's stash row for the cluster merge at the end
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j >= j0) {
                        stash[3 * (j - j0)] = top.key[j];
                        stash[3 * (j - j0) + 1] = top.val[j];
                        stash[3 * (j - j0) + 2] = __int_as_float(top.idx[j]);
                    }
                stash[24] = m;
                stash[25] = z;
            } else if (SPLIT) {
                // this slice's exact top-k (and partial softmax sum) for the merge
                if (row_ok && t < p.T) {
                    RoutePartial* pp = p.part + ((int64_t)t * p.split + h) * p.k;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j >= j0) {
                            pp[j - j0].key = top.key[j];
                            pp[j - j0].val = top.val[j];
                            pp[j - j0].idx = top.idx[j];
                        }
                    if (!sigmoid && !p.renorm) p.zpart[t * p.split + h] = make_float2(m, z);
                }
            } else if (!sigmoid) {
                if (p.renorm) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j >= j0) z += expf(top.val[j] - m);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) g[j] = expf(top.val[j] - m) / z;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j >= j0) z += top.val[j];
#pragma unroll
                for (int j = 0; j < 8; ++j) g[j] = p.renorm ? top.val[j] / z : top.val[j];
            }
            if (nonfinite && row_ok && t < p.T) atomicOr(p.status, MOE_DEV_NONFINITE);
            fence_before();
            __syncwarp();
            if (lane == 0 && !dry) mbar_arrive(acce0 + 8 * acc);
            if (!SPLIT && row_ok && t < p.T) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j >= j0) {
                        p.idx[t * p.k + (j - j0)] = top.idx[j];
                        p.gate[t * p.k + (j - j0)] = g[j];
                    }
            }
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, R_TMEM_COLS);
    }
    if (SPLIT && p.cmerge) {
        // Cluster merge: every slice's lists are in its CTA's stash rows (the same
        // offsets in every CTA of the cluster, one row per token of the tile).
        cluster_sync();
        if (warp >= 2 && warp < 6 && (int)blockIdx.x < p.units && (int)blockIdx.x % p.split == 0) {
            const int row = (warp & 3) * 32 + lane;
            const int64_t t = (int64_t)((int)blockIdx.x / p.split) * p.tile_rows + row;
            const float* own = stash_all + (threadIdx.x - 64) * p.stash_pitch;
            TopK top;
            top.init(p.k);
            for (int h = 0; h < p.split; ++h) {
                for (int jj = 0; jj < p.k; ++jj) {
                    float kv, vv, iv;
                    if (h == 0) {
                        kv = own[3 * jj];
                        vv = own[3 * jj + 1];
                        iv = own[3 * jj + 2];
                    } else {
                        kv = ld_cluster_f32(cluster_addr(own + 3 * jj, (uint32_t)h));
                        vv = ld_cluster_f32(cluster_addr(own + 3 * jj + 1, (uint32_t)h));
                        iv = ld_cluster_f32(cluster_addr(own + 3 * jj + 2, (uint32_t)h));
                    }
                    top.insert(kv, vv, __float_as_int(iv));
                }
            }
            const int j0 = 8 - p.k;
            float g[8];
            if (p.score != MOE_SCORE_SIGMOID) {
                float m = -INFINITY;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j == j0) m = top.val[j];
                float z = 0.f;
                if (p.renorm) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j >= j0) z += expf(top.val[j] - m);
                } else {
                    for (int h = 0; h < p.split; ++h) {
                        const float mh = h == 0 ? own[24] : ld_cluster_f32(cluster_addr(own + 24, (uint32_t)h));
                        const float zh = h == 0 ? own[25] : ld_cluster_f32(cluster_addr(own + 25, (uint32_t)h));
                        z += zh * expf(mh - m);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) g[j] = expf(top.val[j] - m) / z;
            } else {
                float z = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j >= j0) z += top.val[j];
#pragma unroll
                for (int j = 0; j < 8; ++j) g[j] = p.renorm ? top.val[j] / z : top.val[j];
            }
            if (row < p.tile_rows && t < p.T) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j >= j0) {
                        p.idx[t * p.k + (j - j0)] = top.idx[j];
                        p.gate[t * p.k + (j - j0)] = g[j];
                    }
            }
        }
        cluster_sync();  // no CTA leaves while the merge reads its shared memory
    }
}

// The final top-k of a router whose experts were split across work units:
// one thread per token inserts every slice's exact partial top-k into one
// list (the same key order and tie rule, so the result is the top-k over all
// experts), then computes the gates as the unsplit epilogue does.  Softmax
// gates without renormalisation rescale the slices' partial sums to the
// common maximum.
__global__ void __launch_bounds__(256) route_merge_kernel(const RtParams p) {
    pdl_wait();  // the router's partial lists
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= p.T) return;
    TopK top;
    top.init(p.k);
    for (int h = 0; h < p.split; ++h) {
        const RoutePartial* pp = p.part + (t * p.split + h) * p.k;
        for (int jj = 0; jj < p.k; ++jj) top.insert(pp[jj].key, pp[jj].val, pp[jj].idx);
    }
    const int j0 = 8 - p.k;
    float g[8];
    if (p.score != MOE_SCORE_SIGMOID) {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j == j0) m = top.val[j];
        float z = 0.f;
        if (p.renorm) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j >= j0) z += expf(top.val[j] - m);
        } else {
            for (int h = 0; h < p.split; ++h) {
                const float2 mz = p.zpart[t * p.split + h];
                z += mz.y * expf(mz.x - m);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = expf(top.val[j] - m) / z;
    } else {
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j >= j0) z += top.val[j];
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = p.renorm ? top.val[j] / z : top.val[j];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j >= j0) {
            p.idx[t * p.k + (j - j0)] = top.idx[j];
            p.gate[t * p.k + (j - j0)] = g[j];
        }
}

}  // namespace

// Expert slices per router tile.  A unit's time is about proportional to its
// experts (tensor work and the epilogue's passes over the logits) plus a fixed
// part (streaming x, the exact scores of the candidates), counted here as 32
// experts; split when fewer waves of smaller units finish sooner.  Slices are
// multiples of 32 experts.  Only unlimited routing with a partial-list buffer.
int route_split(int64_t T, int E, int sms, bool allowed) {
    if (!allowed || T <= 0 || T > kRouteSplitMaxT) return 1;
    const int64_t m = (T + RM - 1) / RM;
    int best = 1;
    int64_t best_cost = (m + sms - 1) / sms * (32 + E);
    for (int S = 2; S <= kRouteSplitMax; S *= 2) {
        if (E % (32 * S) != 0) continue;
        const int64_t cost = (m * S + sms - 1) / sms * (32 + E / S);
        if (cost < best_cost) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

int64_t route_partial_bytes(int64_t T, int E) {
    if (T <= 0 || T > kRouteSplitMaxT || E < 64 || E % 64 != 0) return 0;
    return T * kRouteSplitMax * (8 * (int64_t)sizeof(RoutePartial) + (int64_t)sizeof(float2));
}

// Tokens per router tile.  With few experts (Np <= 64) the K loop is bound by
// reading x, so what matters is the most rows any CTA streams: the tile height
// (a multiple of 8, the swizzle atom's row count) that minimises
// ceil(tiles / SMs) * height, the larger height on a tie.  With more experts
// the M = 128 MMA (whatever the height) sets the tile's time: 128.
int route_tile_rows(int64_t T, int Np, int sms) {
    if (Np > 64 || T <= 0) return RM;
    int best = RM;
    int64_t best_cost = ((T + RM - 1) / RM + sms - 1) / sms * RM;
    for (int tr = RM - 8; tr >= 8; tr -= 8) {
        const int64_t cost = ((T + tr - 1) / tr + sms - 1) / sms * tr;
        if (cost < best_cost) {
            best_cost = cost;
            best = tr;
        }
    }
    return best;
}

int route_tc_supported(const RouteArgs& a) {
    if (a.dtype != MOE_DTYPE_BF16) return 1;
    if (a.E < 1 || a.E > 256) return 2;
    if (a.d % 8 != 0) return 3;
    if ((reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.w)) & 15) return 4;
    return 0;
}

cudaError_t launch_route_tc(const RouteArgs& a, cudaStream_t s) {
    if (route_tc_supported(a) != 0) return cudaErrorInvalidValue;
    if (a.T == 0) return cudaSuccess;
    RtParams p;
    p.T = a.T;
    p.d = a.d;
    p.E = a.E;
    p.Np = a.E <= 16 ? 16 : (a.E + 15) / 16 * 16;  // MMA N: a multiple of 16, at least 16
    p.k = a.k;
    p.score = a.score;
    p.renorm = a.renorm;
    p.logit_bias = a.logit_bias;
    p.sel_bias = a.sel_bias;
    p.idx = a.idx;
    p.gate = a.gate;
    p.status = a.status;
    p.num_kb = (a.d + RK - 1) / RK;
    p.R = a.R > 0 ? a.R : 1;
    p.max_ranks = (a.max_ranks > 0 && a.max_ranks < p.R && p.R <= 32) ? a.max_ranks : 0;
    p.part = a.part;
    p.zpart = a.part ? reinterpret_cast<float2*>(a.part + a.T * kRouteSplitMax * 8) : nullptr;
    p.stash_pitch = p.max_ranks > 0 ? STASH_PITCH_RANKS : STASH_PITCH;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    p.split = route_split(a.T, a.E, sms, p.max_ranks == 0 && a.part != nullptr);
    p.Eh = p.E / p.split;
    if (p.split > 1) p.Np = p.Eh;  // a multiple of 32
    p.tile_rows = p.split > 1 ? RM : route_tile_rows(a.T, p.Np, sms);
    p.m_tiles = (int)((a.T + p.tile_rows - 1) / p.tile_rows);
    p.units = p.m_tiles * p.split;
    const int grid = p.units < sms ? p.units : sms;
    p.cmerge = (p.split > 1 && p.units <= grid) ? 1 : 0;
    // K blocks per ring stage (their x boxes issued back to back, so each row is
    // read in runs of kbs * 128 bytes).  Measured (moe_route alone, CUDA events,
    // L2 flushed): 8 experts 41.0 / 38.9 / 41.0 us for 1 / 2 / 4 blocks; 64-expert
    // slices of a small batch 108.5 / 102.4 / 98.3 us; 64 experts unsliced (many
    // tiles per CTA, where the deeper ring matters more) 38.9 / 45.1 / 45.1 us.
    p.kbs = 1;
    if (p.split > 1 && p.Np <= 64 && p.num_kb % 4 == 0) p.kbs = 4;
    else if (p.Np <= 16 && p.num_kb % 2 == 0) p.kbs = 2;
    p.num_st = p.num_kb / p.kbs;
    // stage stride: full 128-row A tiles
    p.stage_bytes = p.kbs * (RM * RK * 2 + p.Np * RK * 2);
    p.tx_bytes = p.kbs * (p.tile_rows * RK * 2 + p.Np * RK * 2);
    auto stages_for = [&](int groups) {
        const int extra = R_SMEM_FIXED + 128 * groups * p.stash_pitch * 4;
        const int ring = (R_SMEM_MAX - extra) < R_SMEM_TILES ? (R_SMEM_MAX - extra) : R_SMEM_TILES;
        const int st = ring / p.stage_bytes;
        return st < R_MAX_STAGES ? st : R_MAX_STAGES;
    };
    // A second epilogue group overlaps the epilogues of a CTA's tiles.  It pays
    // off once CTAs average two tiles; with fewer, only if its stash leaves the
    // TMA ring at least 4 stages deep (small E: stages are small).
    // the warm-up pass: one 32-expert chunk and at most one tile per CTA
    // (A/B, moe_route alone, CUDA events: Mixtral shape ~35 -> ~33 us)
    p.warm = (p.Np <= 32 && p.split == 1 && p.units <= grid) ? 1 : 0;
    p.epi_groups = (p.max_ranks == 0 && (p.units >= 2 * grid ||
                                         (p.units > grid && stages_for(2) >= 4)))
                       ? 2 : 1;
    const int extra = R_SMEM_FIXED + 128 * p.epi_groups * p.stash_pitch * 4;
    p.stages = stages_for(p.epi_groups);
    CUtensorMap tmX, tmW;
    if (!make_tmap_bf16(&tmX, a.x, (uint64_t)a.d, (uint64_t)a.T, 1, (uint32_t)p.tile_rows, 2) ||
        !make_tmap_bf16(&tmW, a.w, (uint64_t)a.d, (uint64_t)a.E, 1, (uint32_t)p.Np, 2))
        return cudaErrorInvalidValue;
    const int smem = p.stages * p.stage_bytes + extra;
    // the shared-memory limit is a per-device function attribute: raise it once per
    // device to the largest size used so far
    constexpr int kDevs = 64;
    static int attr_bytes[kDevs][2] = {};
    const int form = p.split > 1 ? 1 : 0;
    auto kern = p.split > 1 ? route_tc_kernel<true> : route_tc_kernel<false>;
    if (dev < 0 || dev >= kDevs || attr_bytes[dev][form] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kDevs) attr_bytes[dev][form] = smem;
    }
    if (p.cmerge) {
        // only if the cluster fits beside nothing else (it needs p.split SMs of one GPC)
        static int fits[kDevs][5] = {};  // 0 unknown, 1 yes, 2 no
        int& f = fits[dev >= 0 && dev < kDevs ? dev : 0][p.split];
        if (f == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(grid);
            cfg.blockDim = dim3(64 + 128 * p.epi_groups);
            cfg.dynamicSmemBytes = (size_t)smem;
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)p.split;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            f = (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) ? 1 : 2;
            cudaGetLastError();  // a refused query leaves no error behind
        }
        if (f != 1) p.cmerge = 0;
    }
    if (p.cmerge)
        return launch_pdl_cluster(kern, dim3(grid), 64 + 128 * p.epi_groups, (size_t)smem, s,
                                  dim3((unsigned)p.split, 1, 1), tmX, tmW, p);
    cudaError_t e =
        launch_pdl(kern, dim3(grid), 64 + 128 * p.epi_groups, (size_t)smem, s, tmX, tmW, p);
    if (e != cudaSuccess || p.split == 1) return e;
    return launch_pdl(route_merge_kernel, dim3((unsigned)((a.T + 255) / 256)), 256, 0, s, p);
}

}  // namespace moe
