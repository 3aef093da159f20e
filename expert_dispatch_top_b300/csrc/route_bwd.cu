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
// rounding).  route_bwd_weight_kernel: one CTA per (expert, 32 column
// vectors), eight warps over interleaved tokens, accumulates dL[t,e] x[t] over
// the nonzero dL entries and adds the warps' sums in a fixed order
// (deterministic), rounding dW once; the chunk-0 CTA also sums d_logit_bias.
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
            float dot = g * dg_l;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            v = g * (dg_l - dot);
        } else {
            const float s = mine ? __fdividef(1.f, 1.f + expf(-L_l)) : 0.f;
            float ds = dg_l;
            if (a.renorm) {
                float sum = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const float g = __fdividef(s, sum);
                float dot = g * dg_l;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                ds = __fdividef(dg_l - dot, sum);
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
        __syncwarp();
        // every lane runs the same number of rounds (the shuffles need all 32)
        for (int e0 = 0; e0 < a.E; e0 += 32) {
            const int e = e0 + lane;
            float dge = 0.f;
            for (int j = 0; j < a.k; ++j) {
                const int ej = __shfl_sync(0xffffffffu, e_l, j);
                const float dgj = __shfl_sync(0xffffffffu, dg_l, j);
                if (ej == e) dge = dgj;
            }
            if (e < a.E) dL[e] = __fdividef(expf(dL[e] - m), z) * (dge - dot);
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

// dW[e, cols] = sum over t of dL[t,e] x[t, cols].  One CTA per (expert, 32
// column vectors); its 8 warps take every 8th token (warp w: t = w, w+8, ...),
// each lane one 16-byte column vector, and the 8 partial sums are added in warp
// order through shared memory: a fixed order, so the result is deterministic.
constexpr int kWGroups = 8;
template <typename T>
__global__ void __launch_bounds__(256) route_bwd_weight_kernel(RouteBwdArgs a) {
    constexpr int V = Elem<T>::kPerVec;
    __shared__ float red[kWGroups][32][V + 1];
    __shared__ float bias_red[kWGroups];
    pdl_wait();  // the token kernel's dL rows
    const int e = blockIdx.x;
    const int gi = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.y * 32 + lane;  // column vector
    const int nvec = a.d / V;
    const bool has_col = c < nvec;
    const T* x = static_cast<const T*>(a.x);
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
    float bias_acc = 0.f;
    for (int64_t t = gi; t < a.T; t += kWGroups) {
        const float v = a.d_logits[t * a.E + e];
        bias_acc += v;
        if (v == 0.f || !has_col) continue;
        float f[V];
        Elem<T>::unpack(ld_nc_v4(x + t * a.d + (int64_t)c * V), f);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = fmaf(v, f[q], acc[q]);
    }
#pragma unroll
    for (int q = 0; q < V; ++q) red[gi][lane][q] = acc[q];
    if (lane == 0) bias_red[gi] = bias_acc;
    __syncthreads();
    if (gi != 0) return;
    float sum[V];
#pragma unroll
    for (int q = 0; q < V; ++q) {
        sum[q] = 0.f;
        for (int g = 0; g < kWGroups; ++g) sum[q] += red[g][lane][q];
    }
    if (a.d_w && has_col)
        st_v4(static_cast<T*>(a.d_w) + (int64_t)e * a.d + (int64_t)c * V, Elem<T>::pack(sum));
    if (a.d_logit_bias && blockIdx.y == 0 && lane == 0) {
        float b = 0.f;
        for (int g = 0; g < kWGroups; ++g) b += bias_red[g];
        a.d_logit_bias[e] = b;
    }
}

template <typename T>
cudaError_t launch_typed(const RouteBwdArgs& a, cudaStream_t s) {
    const unsigned blocks = (unsigned)((a.T + 7) / 8);  // 8 warps (tokens) per block
    route_bwd_token_kernel<T><<<blocks, 256, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || (!a.d_w && !a.d_logit_bias)) return e;
    constexpr int V = Elem<T>::kPerVec;
    const int nvec = a.d / V;
    const dim3 grid((unsigned)a.E, (unsigned)((nvec + 31) / 32));
    return launch_pdl(route_bwd_weight_kernel<T>, grid, 256, 0, s, a);
}

}  // namespace

cudaError_t launch_route_backward(const RouteBwdArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    if (a.dtype == MOE_DTYPE_F32) return launch_typed<float>(a, s);
    return launch_typed<__nv_bfloat16>(a, s);
}

}  // namespace moe
