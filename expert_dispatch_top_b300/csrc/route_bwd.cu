// route_bwd.cu -- backward of Step 1, Route: the router is trained through
// its gates (topicspectrum "Training teaches both experts and router").
//
// The choice of experts is piecewise constant in the logits, so no gradient
// flows through the selection (nor into the selection-only bias); it flows
// through the gates.  For a token with chosen experts e_j, gates g_j and
// incoming gradients dg_j = dL/dg_j:
//   softmax, renormalised:  dL[e_j] = g_j (dg_j - sum_i g_i dg_i), 0 elsewhere;
//   softmax, full:          dL[e]   = p_e (dg_e - sum_j p_(e_j) dg_j) for every e
//                           (p the softmax over all experts, dg_e = 0 off the choice);
//   sigmoid, renormalised:  dL[e_j] = (dg_j - sum_i g_i dg_i) / (sum_i s_i) * s_j (1 - s_j);
//   sigmoid:                dL[e_j] = dg_j s_j (1 - s_j).
// Then dx[t] = sum_e dL[t,e] W[e], dW[e] = sum_t dL[t,e] x[t] and
// d_logit_bias[e] = sum_t dL[t,e].
//
// route_bwd_token_kernel: one warp per token recomputes the logits it needs
// (the chosen experts', or all of them for full-softmax gates) as fp32 dot
// products, forms the gates and dL in fp32 (fast divisions: a few ulp, well
// inside the gradient's tolerance), writes the token's dense dL row,
// and, when asked, dx[t] from the nonzero dL entries (fp32 accumulation, one
// rounding).  route_bwd_weight_kernel (below) forms dW and d_logit_bias from
// the dL rows and x with sums in a fixed order (deterministic), rounding dW
// once.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

template <typename T>
__device__ __forceinline__ float dot_row(const T* a, const T* b, int nvec, int lane) {
    constexpr int V = Elem<T>::kPerVec;
    float acc = 0.f;
    for (int c = lane; c < nvec; c += 32) {
        float fa[V], fb[V];
        Elem<T>::unpack(ld_nc_v4(a + (int64_t)c * V), fa);
        Elem<T>::unpack(ld_nc_v4(b + (int64_t)c * V), fb);
#pragma unroll
        for (int q = 0; q < V; ++q) acc = fmaf(fa[q], fb[q], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(256) route_bwd_token_kernel(RouteBwdArgs a) {
    constexpr int V = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    const T* x = static_cast<const T*>(a.x) + t * a.d;
    const T* w = static_cast<const T*>(a.w);
    const int nvec = a.d / V;
    const bool full = a.score == MOE_SCORE_SOFTMAX && !a.renorm;
    float* dL = a.d_logits + t * a.E;
    // lane j < k holds slot j: expert, incoming gradient, logit
    int e_l = 0;
    float dg_l = 0.f, L_l = 0.f;
    if (lane < a.k) {
        e_l = a.idx[t * a.k + lane];
        dg_l = a.d_gate[t * a.k + lane];
        if ((unsigned)e_l >= (unsigned)a.E) {  // not a forward choice: expert 0, no gradient
            e_l = 0;
            dg_l = 0.f;
        }
    }
    for (int j = 0; j < a.k; ++j) {
        const int e = __shfl_sync(0xffffffffu, e_l, j);
        float L = dot_row<T>(x, w + (int64_t)e * a.d, nvec, lane);
        if (a.logit_bias) L = __fadd_rn(L, a.logit_bias[e]);
        if (lane == j) L_l = L;
    }
    const bool mine = lane < a.k;
    // sum over the chosen slots i of g_i (dg_l - dg_i).  With gates that sum to 1
    // this equals dg_l - sum_i g_i dg_i, without that difference's cancellation
    // when one gate is close to 1 (the other slots' terms are then tiny and the
    // fp32 difference would lose most of their digits).
    auto centred = [&](float g) {
        float acc = 0.f;
        for (int i = 0; i < a.k; ++i) {
            const float gi = __shfl_sync(0xffffffffu, g, i);
            const float dgi = __shfl_sync(0xffffffffu, dg_l, i);
            acc = fmaf(gi, dg_l - dgi, acc);
        }
        return acc;
    };
    if (!full) {
        float v = 0.f;  // dL of this lane's slot
        if (a.score == MOE_SCORE_SOFTMAX) {
            float m = -INFINITY;
            for (int j = 0; j < a.k; ++j) m = fmaxf(m, __shfl_sync(0xffffffffu, L_l, j));
            const float ex = mine ? expf(L_l - m) : 0.f;
            float z = ex;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            const float g = __fdividef(ex, z);
            v = g * centred(g);
        } else {
            const float s = mine ? __fdividef(1.f, 1.f + expf(-L_l)) : 0.f;
            float ds = dg_l;
            if (a.renorm) {
                float sum = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const float g = __fdividef(s, sum);
                ds = __fdividef(centred(g), sum);
            }
            v = ds * s * (1.f - s);
        }
        for (int e = lane; e < a.E; e += 32) dL[e] = 0.f;
        __syncwarp();
        if (mine) dL[e_l] = v;
    } else {
        // full softmax: every logit, p over all experts
        float m = -INFINITY;
        for (int e = 0; e < a.E; ++e) {
            float L = dot_row<T>(x, w + (int64_t)e * a.d, nvec, lane);
            if (a.logit_bias) L = __fadd_rn(L, a.logit_bias[e]);
            if (lane == 0) dL[e] = L;  // stash the logits in the output row
            m = fmaxf(m, L);
        }
        __syncwarp();
        float z = 0.f;
        for (int e = lane; e < a.E; e += 32) z += expf(dL[e] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        const float pj = mine ? __fdividef(expf(L_l - m), z) : 0.f;
        float dot = pj * dg_l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        // A chosen slot j: dL = p_j (dg_j - dot) = p_j (dg_j (1 - p_j) - sum_(i!=j) p_i dg_i),
        // with 1 - p_j summed over the other experts rather than subtracted from 1
        // (stable when p_j is close to 1).
        float zx = 0.f;  // slot lane < k: the exp sum over every expert but its own
        for (int j = 0; j < a.k; ++j) {
            const int ej = __shfl_sync(0xffffffffu, e_l, j);
            float part = 0.f;
            for (int e = lane; e < a.E; e += 32)
                if (e != ej) part += expf(dL[e] - m);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == j) zx = part;
        }
        float other = 0.f;
        for (int i = 0; i < a.k; ++i) {
            const float pi = __shfl_sync(0xffffffffu, pj, i);
            const float dgi = __shfl_sync(0xffffffffu, dg_l, i);
            if (i != lane) other = fmaf(pi, dgi, other);
        }
        const float dl_slot = pj * (dg_l * __fdividef(zx, z) - other);
        __syncwarp();
        // every lane runs the same number of rounds (the shuffles need all 32)
        for (int e0 = 0; e0 < a.E; e0 += 32) {
            const int e = e0 + lane;
            int js = -1;
            for (int j = 0; j < a.k; ++j)
                if (__shfl_sync(0xffffffffu, e_l, j) == e) js = j;
            const float vs = __shfl_sync(0xffffffffu, dl_slot, js < 0 ? 0 : js);
            if (e < a.E) dL[e] = js >= 0 ? vs : -__fdividef(expf(dL[e] - m), z) * dot;
        }
    }
    if (!a.dx) return;
    __syncwarp();
    // dx[t] = sum_e dL[t,e] W[e] over the nonzero entries (the chosen experts, or all)
    T* dx = static_cast<T*>(a.dx) + t * a.d;
    const int ne = full ? a.E : a.k;
    int ej[8];  // the chosen experts, known to every lane
#pragma unroll
    for (int j = 0; j < 8; ++j) ej[j] = __shfl_sync(0xffffffffu, e_l, j);
    for (int c = lane; c < nvec; c += 32) {
        float acc[V];
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = 0.f;
        for (int i = 0; i < ne; ++i) {
            int e = i;
            if (!full) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j == i) e = ej[j];
            }
            const float v = dL[e];
            if (v == 0.f) continue;
            float fw[V];
            Elem<T>::unpack(ld_nc_v4(w + (int64_t)e * a.d + (int64_t)c * V), fw);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = fmaf(v, fw[q], acc[q]);
        }
        st_v4(dx + (int64_t)c * V, Elem<T>::pack(acc));
    }
}

// dW[e, cols] = sum over t of dL[t,e] x[t, cols], and d_logit_bias[e] = sum
// over t of dL[t,e].  A CTA owns 8 experts and 32 column vectors (256 bf16 or
// 128 fp32 columns) for a contiguous range of tokens; its 8 warps take
// interleaved groups of 32 tokens.  Per group, lane l reads token l's 8 dL
// entries (32 contiguous bytes), then the warp walks the group's tokens with
// any nonzero entry four at a time: each lane loads its column vector of the
// four x rows, and for every expert whose dL is nonzero (a warp-uniform test)
// adds dL * x into its accumulators -- x is read once per token for all 8
// experts.  The token range is split over the S CTAs of a thread-block
// cluster when there are too few (expert block, column block) pairs to fill
// the GPU; the partial sums are then added through distributed shared memory.
// Every sum is taken in a fixed order (warps in index order, cluster ranks in
// rank order, lanes by a fixed shuffle tree), so the result is deterministic.
constexpr int kWExperts = 8;
constexpr int kWWarps = 8;
constexpr int kWMaxSplit = 8;
constexpr int kWBatch = 4;  // x rows in flight per lane

template <typename T>
__global__ void __launch_bounds__(kWWarps * 32) route_bwd_weight_kernel(RouteBwdArgs a, int S) {
    constexpr int V = Elem<T>::kPerVec;
    constexpr int COLS = 32 * V;
    __shared__ float part[kWExperts][COLS];  // this CTA's sums (warps added in order)
    __shared__ float bpart[kWExperts];       // this CTA's d_logit_bias sums
    pdl_wait();  // the token kernel's dL rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * kWExperts;
    const int ne = a.E - e0 < kWExperts ? a.E - e0 : kWExperts;
    const int nvec = a.d / V;
    const int c = blockIdx.y * 32 + lane;  // this lane's column vector
    const bool has_col = c < nvec;
    const T* x = static_cast<const T*>(a.x);
    // this CTA's tokens: split z of S
    const int z = S > 1 ? (int)cluster_rank() : 0;
    const int64_t groups = (a.T + 31) / 32;
    const int64_t g_lo = groups * z / S, g_hi = groups * (z + 1) / S;
    const bool vec_dl = (a.E % 4) == 0 && (reinterpret_cast<uintptr_t>(a.d_logits) & 15) == 0;
    float acc[kWExperts][V];
#pragma unroll
    for (int j = 0; j < kWExperts; ++j)
#pragma unroll
        for (int q = 0; q < V; ++q) acc[j][q] = 0.f;
    float bsum[kWExperts];
#pragma unroll
    for (int j = 0; j < kWExperts; ++j) bsum[j] = 0.f;
    for (int64_t g = g_lo + warp; g < g_hi; g += kWWarps) {
        const int64_t t = g * 32 + lane;
        float dv[kWExperts];
#pragma unroll
        for (int j = 0; j < kWExperts; ++j) dv[j] = 0.f;
        if (t < a.T) {
            const float* row = a.d_logits + t * a.E + e0;
            if (vec_dl && ne == kWExperts) {
                const float4 u0 = *reinterpret_cast<const float4*>(row);
                const float4 u1 = *reinterpret_cast<const float4*>(row + 4);
                dv[0] = u0.x; dv[1] = u0.y; dv[2] = u0.z; dv[3] = u0.w;
                dv[4] = u1.x; dv[5] = u1.y; dv[6] = u1.z; dv[7] = u1.w;
            } else {
#pragma unroll
                for (int j = 0; j < kWExperts; ++j)
                    if (j < ne) dv[j] = row[j];
            }
        }
        bool nz = false;
#pragma unroll
        for (int j = 0; j < kWExperts; ++j) {
            bsum[j] += dv[j];
            nz |= dv[j] != 0.f;
        }
        uint32_t mask = __ballot_sync(0xffffffffu, nz);
        while (mask) {
            // up to kWBatch tokens of the group: their x vectors in flight together
            int src[kWBatch];
            uint4 raw[kWBatch];
#pragma unroll
            for (int u = 0; u < kWBatch; ++u) {
                src[u] = mask ? __ffs(mask) - 1 : -1;
                if (mask) mask &= mask - 1;
                if (src[u] >= 0 && has_col)
                    raw[u] = ld_nc_v4(x + (g * 32 + src[u]) * a.d + (int64_t)c * V);
            }
#pragma unroll
            for (int u = 0; u < kWBatch; ++u) {
                if (src[u] < 0) break;  // warp-uniform
                float f[V];
                if (has_col) Elem<T>::unpack(raw[u], f);
#pragma unroll
                for (int j = 0; j < kWExperts; ++j) {
                    const float v = __shfl_sync(0xffffffffu, dv[j], src[u]);
                    if (v != 0.f && has_col) {
#pragma unroll
                        for (int q = 0; q < V; ++q) acc[j][q] = fmaf(v, f[q], acc[j][q]);
                    }
                }
            }
        }
    }
    // d_logit_bias: lanes by a fixed butterfly, then warps in order below
#pragma unroll
    for (int j = 0; j < kWExperts; ++j)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bsum[j] += __shfl_xor_sync(0xffffffffu, bsum[j], o);
    // warps add their sums into part[] one after another (fixed order)
    for (int w = 0; w < kWWarps; ++w) {
        if (warp == w) {
#pragma unroll
            for (int j = 0; j < kWExperts; ++j) {
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    float* dst = &part[j][lane * V + q];
                    *dst = (w == 0 ? 0.f : *dst) + acc[j][q];
                }
                if (lane == 0) bpart[j] = (w == 0 ? 0.f : bpart[j]) + bsum[j];
            }
        }
        __syncthreads();
    }
    if (S > 1) cluster_sync();  // every rank's part[] is complete
    // CTA rank z finalises its share of the 8 x COLS outputs, adding the ranks in order
    const int n_out = kWExperts * COLS;
    for (int i = z * (n_out / S) + (int)threadIdx.x; i < (z + 1) * (n_out / S); i += kWWarps * 32) {
        const int j = i / COLS, col = i - j * COLS;
        float sum = part[j][col];
        if (S > 1) {
            sum = 0.f;
            for (int r = 0; r < S; ++r) sum += ld_cluster_f32(cluster_addr(&part[j][col], (uint32_t)r));
        }
        const int cc = blockIdx.y * COLS + col;  // element column
        if (a.d_w && j < ne && cc < a.d) {
            T* out = static_cast<T*>(a.d_w) + (int64_t)(e0 + j) * a.d + cc;
            *out = Elem<T>::from_f(sum);
        }
    }
    if (a.d_logit_bias && blockIdx.y == 0 && z == 0 && threadIdx.x < kWExperts &&
        (int)threadIdx.x < ne) {
        float b = 0.f;
        for (int r = 0; r < S; ++r)
            b += S > 1 ? ld_cluster_f32(cluster_addr(&bpart[threadIdx.x], (uint32_t)r))
                       : bpart[threadIdx.x];
        a.d_logit_bias[e0 + threadIdx.x] = b;
    }
    if (S > 1) cluster_sync();  // no CTA leaves while another reads its shared memory
}

template <typename T>
cudaError_t launch_typed(const RouteBwdArgs& a, cudaStream_t s) {
    const unsigned blocks = (unsigned)((a.T + 7) / 8);  // 8 warps (tokens) per block
    route_bwd_token_kernel<T><<<blocks, 256, 0, s>>>(a);
    cudaError_t e = noted_launch();
    if (e != cudaSuccess || (!a.d_w && !a.d_logit_bias)) return e;
    constexpr int V = Elem<T>::kPerVec;
    const int nvec = a.d / V;
    const unsigned eb = (unsigned)((a.E + kWExperts - 1) / kWExperts);
    const unsigned cb = (unsigned)((nvec + 31) / 32);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // token splits (a power of two <= 8) until there are about two CTAs per SM
    // (two fit an SM), with at least 64 token groups per split.  Measured with 8
    // warps per CTA (Mixtral shape 0.133 ms, DeepSeek shape 0.441 ms) against
    // 16 warps and one CTA per SM (0.186 / 0.515 ms).
    int S = 1;
    while (S < kWMaxSplit && (int64_t)eb * cb * S < 2 * (int64_t)sms &&
           (a.T + 31) / 32 >= 64 * 2 * S)
        S *= 2;
    return launch_pdl_cluster(route_bwd_weight_kernel<T>, dim3(eb, cb, (unsigned)S), kWWarps * 32, 0,
                              s, dim3(1, 1, (unsigned)S), a, S);
}

}  // namespace

cudaError_t launch_route_backward(const RouteBwdArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    if (a.dtype == MOE_DTYPE_F32) return launch_typed<float>(a, s);
    return launch_typed<__nv_bfloat16>(a, s);
}

}  // namespace moe
