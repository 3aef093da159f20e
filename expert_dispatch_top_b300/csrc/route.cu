// route.cu -- Step 1, Route: router logits (fp32 FFMA), score, top-k, gates.
// fp32 routers run here; bf16 routers run on the tensor cores (route_tc.cu).
//
// Ultralytics glossary "Expert Parallelism", section "How Tokens Move Between
// GPUs", step 1: every token gets a score for every expert and keeps the k
// best.  Selection-only bias: DeepSeek-V3 bias-based balancing (same page,
// "Load Balancing and Capacity").
//
// Logits are fp32 FFMA sums.  On inputs whose products and partial sums are
// all representable (the dyadic test grid), every summation order gives the
// same fp32 value, so the selection is reproducible bit for bit.  The sigmoid
// score is fp32(1/(1+exp(-L))) evaluated in double, i.e. the correctly
// rounded fp32 sigmoid except in vanishingly rare double-rounding cases.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr float kNegInf = -INFINITY;
constexpr int kNoExpert = 0x7fffffff;

__device__ __forceinline__ float sigmoid_score(float L) {
    return (float)(1.0 / (1.0 + exp(-(double)L)));
}

// Segmented argmax over groups of W lanes (W a power of two <= 32).
template <int W>
__device__ __forceinline__ void seg_argmax(float& v, int& i) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (key_better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

template <int W>
__device__ __forceinline__ float seg_sum(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Top-k and gates for one token whose E logits are spread over a group of W
// lanes, lane e' of the group holding the values of experts e' + W*i
// (i < NV).  L: logits (logit bias included); valid[i]: e < E.
// Rank-limited routing (0 < max_ranks < R): a rank's score is the best key of
// its E/R experts, the max_ranks best ranks are kept (ties to the lower rank)
// and the top-k is taken among their experts.  The best remaining rank is the
// rank of the best key among experts of ranks not yet kept: ranks are
// contiguous blocks of experts, so the lower expert index that wins a tie of
// keys also names the lower rank.
template <int W, int NV>
__device__ __forceinline__ void select_and_gate(const float (&L)[NV], int e_base, int E, int k,
                                                int score, int renorm, const float* sel_bias,
                                                int R, int max_ranks, int32_t* out_idx,
                                                float* out_gate, uint32_t* status) {
    float key[NV], s[NV];
    int slot[NV];
    bool ok[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = e_base + W * i;
        slot[i] = -1;
        if (e < E) {
            if (score == MOE_SCORE_SIGMOID) {
                s[i] = sigmoid_score(L[i]);
                key[i] = sel_bias ? __fadd_rn(s[i], sel_bias[e]) : s[i];
            } else {
                s[i] = 0.f;
                key[i] = L[i];
            }
        } else {
            s[i] = 0.f;
            key[i] = kNegInf;
        }
        ok[i] = e < E;
        if (status && e < E && !(fabsf(L[i]) <= FLT_MAX)) atomicOr(status, MOE_DEV_NONFINITE);
    }
    if (max_ranks > 0 && max_ranks < R) {
        const int per = E / R;
        uint32_t kept = 0;  // bit r: rank r kept
        for (int m = 0; m < max_ranks; ++m) {
            float bv = kNegInf;
            int bi = kNoExpert;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = e_base + W * i;
                if (e < E && !((kept >> (e / per)) & 1u) && key_better(key[i], e, bv, bi)) {
                    bv = key[i];
                    bi = e;
                }
            }
            seg_argmax<W>(bv, bi);
            if (bi != kNoExpert) kept |= 1u << (bi / per);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = e_base + W * i;
            ok[i] = e < E && ((kept >> (e / per)) & 1u);
        }
    }
    float top_logit = 0.f;
    for (int j = 0; j < k; ++j) {
        // local best among not-yet-chosen values of this lane
        float bv = kNegInf;
        int bi = kNoExpert;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = e_base + W * i;
            if (ok[i] && slot[i] < 0 && key_better(key[i], e, bv, bi)) {
                bv = key[i];
                bi = e;
            }
        }
        seg_argmax<W>(bv, bi);
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (e_base + W * i == bi) {
                slot[i] = j;
                out_idx[j] = bi;
                if (j == 0) top_logit = L[i];
            }
        if (j == 0) {
            // broadcast the winner's logit: the owner is the only lane with it set
            float tl = (bi == kNoExpert) ? 0.f : top_logit;
            top_logit = seg_sum<W>(tl);
        }
    }
    // Gates.
    if (score == MOE_SCORE_SOFTMAX) {
        const float m = top_logit;  // the largest logit overall (first choice)
        float ex[NV];
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = e_base + W * i;
            ex[i] = (e < E) ? expf(L[i] - m) : 0.f;
            if (e < E && (!renorm || slot[i] >= 0)) part += ex[i];
        }
        const float z = seg_sum<W>(part);
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (slot[i] >= 0) out_gate[slot[i]] = ex[i] / z;
    } else {
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (slot[i] >= 0) part += s[i];
        const float z = renorm ? seg_sum<W>(part) : 1.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (slot[i] >= 0) out_gate[slot[i]] = renorm ? s[i] / z : s[i];
    }
}

// ---------------------------------------------------------------------------
// E <= 32: each warp scores TPW tokens at once (so every weight vector loaded
// serves TPW tokens); lanes split d into 16-byte vectors.  A transposing
// butterfly then leaves lane l with the full sum of value l = (token l / EMAX,
// expert l % EMAX), and the top-k runs on segments of EMAX lanes.
// ---------------------------------------------------------------------------
template <typename T, int EMAX>
__global__ void __launch_bounds__(256) route_small_kernel(RouteArgs a) {
    pdl_wait();  // programmatic dependent launch: the previous kernel's writes
    constexpr int TPW = 32 / EMAX;
    constexpr int V = Elem<T>::kPerVec;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * 8 + warp) * TPW;
    if (t0 >= a.T) return;
    const int nvec = a.d / V;
    const T* x = static_cast<const T*>(a.x);
    const T* w = static_cast<const T*>(a.w);

    float acc[TPW * EMAX];
#pragma unroll
    for (int i = 0; i < TPW * EMAX; ++i) acc[i] = 0.f;

    for (int c = lane; c < nvec; c += 32) {
        float xv[TPW][V];
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt) {
            if (t0 + tt < a.T) {
                Elem<T>::unpack(ld_nc_v4(x + (t0 + tt) * a.d + (int64_t)c * V), xv[tt]);
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) xv[tt][v] = 0.f;
            }
        }
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            if (e < a.E) {
                float wv[V];
                Elem<T>::unpack(ld_v4(w + (int64_t)e * a.d + (int64_t)c * V), wv);
#pragma unroll
                for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
                    for (int v = 0; v < V; ++v) acc[tt * EMAX + e] = fmaf(xv[tt][v], wv[v], acc[tt * EMAX + e]);
            }
        }
    }
    // Transposing butterfly: 31 shuffles for 32 sums.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int v = 0; v < o; ++v) {
            const float send = hi ? acc[v] : acc[v + o];
            const float keep = hi ? acc[v + o] : acc[v];
            acc[v] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    const int tt = lane / EMAX;
    const int e = lane % EMAX;
    const int64_t t = t0 + tt;
    float L[1];
    L[0] = acc[0];
    if (e < a.E && a.logit_bias) L[0] = __fadd_rn(L[0], a.logit_bias[e]);
    const bool live = t < a.T;
    // Every lane takes part in the shuffles; only live tokens write.
    int32_t idx_buf[8];
    float gate_buf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        idx_buf[j] = -1;
        gate_buf[j] = 0.f;
    }
    select_and_gate<EMAX, 1>(L, e, a.E, a.k, a.score, a.renorm, a.sel_bias, a.R, a.max_ranks,
                             idx_buf, gate_buf, live ? a.status : nullptr);
    if (live) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < a.k && idx_buf[j] == e) {
                a.idx[t * a.k + j] = e;
                a.gate[t * a.k + j] = gate_buf[j];
            }
    }
}

// ---------------------------------------------------------------------------
// E > 32: a 64-token x EP-expert fp32 FFMA tile per block (EP = E rounded up
// to 64, 128 or 256), K staged through shared memory in chunks of 32, then
// one warp per token for the top-k with E/32 values per lane.
// ---------------------------------------------------------------------------
constexpr int kTT = 64;   // tokens per block
constexpr int kKC = 32;   // K chunk

template <int EP>
constexpr int big_smem_bytes() {
    return (kTT * (EP + 1) * 4) > ((kKC * kTT + kKC * EP) * 4) ? (kTT * (EP + 1) * 4)
                                                               : ((kKC * kTT + kKC * EP) * 4);
}

template <typename T, int EP>
__global__ void __launch_bounds__(256) route_big_kernel(RouteArgs a) {
    extern __shared__ __align__(16) float sm[];
    pdl_wait();  // programmatic dependent launch: the previous kernel's writes
    float* xs = sm;                // [kKC][kTT]
    float* ws = sm + kKC * kTT;    // [kKC][EP]
    float* Ls = sm;                // [kTT][EP+1] after the GEMM
    constexpr int V = Elem<T>::kPerVec;
    constexpr int NJ = EP / 64;    // expert groups of 4 per thread
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t tbase = (int64_t)blockIdx.x * kTT;
    const T* x = static_cast<const T*>(a.x);
    const T* w = static_cast<const T*>(a.w);

    float acc[4][NJ * 4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NJ * 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < a.d; k0 += kKC) {
        // x tile: kTT x kKC elements, 16-byte vectors
        constexpr int XV = kTT * kKC / V;
        for (int v = tid; v < XV; v += 256) {
            const int tok = v / (kKC / V), kc = (v % (kKC / V)) * V;
            float f[V];
            const int64_t t = tbase + tok;
            if (t < a.T && k0 + kc < a.d) {
                Elem<T>::unpack(ld_nc_v4(x + t * a.d + k0 + kc), f);
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q) f[q] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < V; ++q) xs[(kc + q) * kTT + tok] = f[q];
        }
        constexpr int WV = EP * kKC / V;
        for (int v = tid; v < WV; v += 256) {
            const int e = v / (kKC / V), kc = (v % (kKC / V)) * V;
            float f[V];
            if (e < a.E && k0 + kc < a.d) {
                Elem<T>::unpack(ld_v4(w + (int64_t)e * a.d + k0 + kc), f);
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q) f[q] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < V; ++q) ws[(kc + q) * EP + e] = f[q];
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kKC; ++kk) {
            const float4 xa = *reinterpret_cast<const float4*>(&xs[kk * kTT + ty * 4]);
            const float xr[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float4 wb = *reinterpret_cast<const float4*>(&ws[kk * EP + 64 * j + tx * 4]);
                const float wr[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[i][j * 4 + c] = fmaf(xr[i], wr[c], acc[i][j * 4 + c]);
            }
        }
        __syncthreads();
    }
    // logits to shared memory
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) Ls[(ty * 4 + i) * (EP + 1) + 64 * j + tx * 4 + c] = acc[i][j * 4 + c];
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    constexpr int NV = EP / 32;
    for (int tok = warp; tok < kTT; tok += 8) {
        const int64_t t = tbase + tok;
        if (t >= a.T) break;
        float L[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            float v = Ls[tok * (EP + 1) + e];
            if (e < a.E && a.logit_bias) v = __fadd_rn(v, a.logit_bias[e]);
            L[i] = v;
        }
        int32_t idx_buf[8];
        float gate_buf[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            idx_buf[j] = -1;
            gate_buf[j] = 0.f;
        }
        select_and_gate<32, NV>(L, lane, a.E, a.k, a.score, a.renorm, a.sel_bias, a.R, a.max_ranks,
                                idx_buf, gate_buf, a.status);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < a.k && idx_buf[j] >= 0) {
                a.idx[t * a.k + j] = idx_buf[j];
                a.gate[t * a.k + j] = gate_buf[j];
            }
    }
}

template <typename T>
cudaError_t launch_typed(const RouteArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    if (a.E <= 8) {
        const int64_t blocks = (a.T + 8 * 4 - 1) / (8 * 4);
        return launch_pdl(route_small_kernel<T, 8>, dim3((unsigned)blocks), 256, 0, s, a);
    } else if (a.E <= 16) {
        const int64_t blocks = (a.T + 8 * 2 - 1) / (8 * 2);
        return launch_pdl(route_small_kernel<T, 16>, dim3((unsigned)blocks), 256, 0, s, a);
    } else if (a.E <= 32) {
        const int64_t blocks = (a.T + 8 - 1) / 8;
        return launch_pdl(route_small_kernel<T, 32>, dim3((unsigned)blocks), 256, 0, s, a);
    } else {
        const unsigned blocks = (unsigned)((a.T + kTT - 1) / kTT);
        if (a.E <= 64) {
            constexpr int B = big_smem_bytes<64>();
            return launch_pdl(route_big_kernel<T, 64>, dim3(blocks), 256, (size_t)B, s, a);
        } else if (a.E <= 128) {
            constexpr int B = big_smem_bytes<128>();
            return launch_pdl(route_big_kernel<T, 128>, dim3(blocks), 256, (size_t)B, s, a);
        } else {
            constexpr int B = big_smem_bytes<256>();
            // the shared-memory limit is a per-device function attribute
            constexpr int kDevs = 64;
            static bool attr[kDevs] = {};
            int dev = 0;
            cudaGetDevice(&dev);
            if (dev < 0 || dev >= kDevs || !attr[dev]) {
                cudaError_t e = cudaFuncSetAttribute(route_big_kernel<T, 256>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, B);
                if (e != cudaSuccess) return e;
                if (dev >= 0 && dev < kDevs) attr[dev] = true;
            }
            return launch_pdl(route_big_kernel<T, 256>, dim3(blocks), 256, (size_t)B, s, a);
        }
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
    if (route_tc_supported(a) == 0) return launch_route_tc(a, s);
    if (a.dtype == MOE_DTYPE_F32) return launch_typed<float>(a, s);
    return launch_typed<__nv_bfloat16>(a, s);
}

}  // namespace moe
