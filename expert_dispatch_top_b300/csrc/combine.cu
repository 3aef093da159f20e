// combine.cu -- Step 4, Combine: gate-weighted un-permute back to token order.
//
// Ultralytics glossary "Expert Parallelism", "How Tokens Move Between GPUs",
// step 4 (outputs return to their token and are summed with the router
// gates as weights); ai360xpert "The All-to-All Bottleneck" (Gather).  A
// dropped assignment (slot_row < 0) contributes nothing; the optional
// residual carries a fully dropped token through unchanged (ai360xpert "Load
// Balancing and Dropped Tokens"; Ultralytics "Load Balancing and Capacity").
//
// One warp per token, grid-stride; each lane moves 16-byte vectors.  The k
// expert rows of a token, for U column vectors at a time, are independent
// loads issued back to back (8 in flight per lane); with one vector per step
// (k > 4) and a shared-expert or residual row to add, those rows' vectors
// join the same batch (PRE) instead of costing a second round trip.  fp32
// accumulation in slot order, one rounding to the output type.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

#ifdef MOE_CHECKED
// Bounds violations found by calls that have no workspace (checked build).
__device__ uint32_t g_checked_status;
#endif

// Checked build: a kept row outside [0, rows_cap) is reported and dropped.
__device__ __forceinline__ int checked_row(int r, int64_t rows_cap) {
#ifdef MOE_CHECKED
    if (r < -1 || (r >= 0 && r >= rows_cap)) {
        atomicOr(&g_checked_status, MOE_DEV_BOUNDS);
        return -1;
    }
#endif
    return r;
}

// Checked build: the offsets the expert FFN kernels read, made non-decreasing
// within [0, rows_cap] (one warp).
__global__ void sanitize_offsets_kernel(const int32_t* in, int32_t* out, int G, int64_t rows_cap,
                                        uint32_t* status) {
    if (threadIdx.x != 0) return;
    bool bad = false;
    int64_t prev = 0;
    for (int g = 0; g <= G; ++g) {
        int64_t v = in[g];
        if (v < prev || v > rows_cap) {
            bad = true;
            v = v < prev ? prev : rows_cap;
        }
        out[g] = (int32_t)v;
        prev = v;
    }
    if (bad) atomicOr(status, MOE_DEV_BOUNDS);
}

// KMAX: compile-time bound on k; U: 16-byte column vectors per lane in flight.
// U * KMAX = 8 keeps eight independent row loads in flight per lane (k = 1 has
// its own variant, so that top-1 layers also keep eight).
template <typename T, int KMAX, int U, bool PRE>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
    constexpr int V = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nvec = a.d / V;
    const int64_t row_bytes = (int64_t)a.d * sizeof(T);
    const char* yp = static_cast<const char*>(a.yp);
    const char* sh = static_cast<const char*>(a.shared);
    const char* rs = static_cast<const char*>(a.resid);
    char* y = static_cast<char*>(a.y);
    pdl_wait();  // the expert FFN's (or dispatch's) rows
    for (int64_t t = warp0; t < a.T; t += nwarps) {
        int r_l = -1;
        float g_l = 0.f;
        if (lane < a.k) {
            r_l = a.slot_row[t * a.k + lane];
            g_l = a.gate ? a.gate[t * a.k + lane] : 1.f;  // no gates: the plain sum of rows
        }
        if (kChecked && lane < a.k) r_l = checked_row(r_l, a.rows_cap);
        int r[KMAX];
        float g[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            r[j] = __shfl_sync(0xffffffffu, r_l, j);
            g[j] = __shfl_sync(0xffffffffu, g_l, j);
            if (j >= a.k) r[j] = -1;
        }
        for (int c0 = lane; c0 < nvec; c0 += 32 * U) {
            uint4 v[U][KMAX];
            uint4 vs = make_uint4(0u, 0u, 0u, 0u), vr = vs;  // PRE: shared / residual vectors
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (c < nvec && r[j] >= 0)
                        v[u][j] = ld_nc_v4(yp + (int64_t)r[j] * row_bytes + (int64_t)c * 16);
                if (PRE && c < nvec && sh) vs = ld_nc_v4(sh + t * row_bytes + (int64_t)c * 16);
                if (PRE && c < nvec && rs) vr = ld_nc_v4(rs + t * row_bytes + (int64_t)c * 16);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                if (c >= nvec) break;
                float acc[V];
#pragma unroll
                for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (r[j] >= 0) {
                        float f[V];
                        Elem<T>::unpack(v[u][j], f);
#pragma unroll
                        for (int q = 0; q < V; ++q) acc[q] = fmaf(g[j], f[q], acc[q]);
                    }
                if (sh) {
                    float f[V];
                    Elem<T>::unpack(PRE ? vs : ld_nc_v4(sh + t * row_bytes + (int64_t)c * 16), f);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[q] += f[q];
                }
                if (rs) {
                    float f[V];
                    Elem<T>::unpack(PRE ? vr : ld_nc_v4(rs + t * row_bytes + (int64_t)c * 16), f);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[q] += f[q];
                }
                st_cs_v4(y + t * row_bytes + (int64_t)c * 16, Elem<T>::pack(acc));
            }
        }
    }
}

template <typename T>
cudaError_t launch_combine_typed(const CombineArgs& a, unsigned blocks, cudaStream_t s) {
    const dim3 g(blocks);
    if (a.k == 1) return launch_pdl(combine_kernel<T, 1, 8, false>, g, 256, 0, s, a);
    if (a.k <= 2) return launch_pdl(combine_kernel<T, 2, 4, false>, g, 256, 0, s, a);
    if (a.k <= 4) return launch_pdl(combine_kernel<T, 4, 2, false>, g, 256, 0, s, a);
    if (a.shared || a.resid) return launch_pdl(combine_kernel<T, 8, 1, true>, g, 256, 0, s, a);
    return launch_pdl(combine_kernel<T, 8, 1, false>, g, 256, 0, s, a);
}

// Backward of combine, one warp per token: for every kept slot j,
// d_yp[slot_row[t,j]] = g[t,j] * dy[t] (one rounding) and
// d_gate[t,j] = <dy[t], yp[slot_row[t,j]]> (fp32, lane partials then a
// butterfly); dropped slots get d_gate = 0.
template <typename T, int KMAX>
__global__ void __launch_bounds__(256) combine_bwd_kernel(CombineBwdArgs a) {
    constexpr int V = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nvec = a.d / V;
    const int64_t row_bytes = (int64_t)a.d * sizeof(T);
    const char* dy = static_cast<const char*>(a.dy);
    const char* yp = static_cast<const char*>(a.yp);
    char* dyp = static_cast<char*>(a.d_yp);
    for (int64_t t = warp0; t < a.T; t += nwarps) {
        int r_l = -1;
        float g_l = 0.f;
        if (lane < a.k) {
            r_l = a.slot_row[t * a.k + lane];
            g_l = a.gate[t * a.k + lane];
        }
        if (kChecked && lane < a.k) r_l = checked_row(r_l, a.rows_cap);
        int r[KMAX];
        float g[KMAX], dot[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            r[j] = __shfl_sync(0xffffffffu, r_l, j);
            g[j] = __shfl_sync(0xffffffffu, g_l, j);
            if (j >= a.k) r[j] = -1;
            dot[j] = 0.f;
        }
        for (int c = lane; c < nvec; c += 32) {
            float f[V];
            Elem<T>::unpack(ld_nc_v4(dy + t * row_bytes + (int64_t)c * 16), f);
            uint4 v[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (r[j] >= 0) v[j] = ld_nc_v4(yp + (int64_t)r[j] * row_bytes + (int64_t)c * 16);
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (r[j] >= 0) {
                    float y[V], o[V];
                    Elem<T>::unpack(v[j], y);
#pragma unroll
                    for (int q = 0; q < V; ++q) {
                        dot[j] = fmaf(f[q], y[q], dot[j]);
                        o[q] = g[j] * f[q];
                    }
                    st_v4(dyp + (int64_t)r[j] * row_bytes + (int64_t)c * 16, Elem<T>::pack(o));
                }
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < a.k) a.d_gate[t * a.k + j] = r[j] >= 0 ? dot[j] : 0.f;
        }
    }
}

template <typename T>
void launch_combine_bwd_typed(const CombineBwdArgs& a, unsigned blocks, cudaStream_t s) {
    if (a.k <= 2)
        combine_bwd_kernel<T, 2><<<blocks, 256, 0, s>>>(a);
    else if (a.k <= 4)
        combine_bwd_kernel<T, 4><<<blocks, 256, 0, s>>>(a);
    else
        combine_bwd_kernel<T, 8><<<blocks, 256, 0, s>>>(a);
}

}  // namespace

cudaError_t launch_combine_backward(const CombineBwdArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (a.T + 7) / 8;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    if (a.dtype == MOE_DTYPE_F32)
        launch_combine_bwd_typed<float>(a, (unsigned)blocks, s);
    else
        launch_combine_bwd_typed<__nv_bfloat16>(a, (unsigned)blocks, s);
    return noted_launch();
}

cudaError_t launch_sanitize_offsets(const int32_t* in, int32_t* out, int G, int64_t rows_cap,
                                    uint32_t* status, cudaStream_t s) {
    sanitize_offsets_kernel<<<1, 32, 0, s>>>(in, out, G, rows_cap, status);
    return noted_launch();
}

cudaError_t take_checked_status(uint32_t* out, cudaStream_t s) {
#ifdef MOE_CHECKED
    uint32_t v = 0;
    void* addr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&addr, g_checked_status);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&v, addr, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(addr, 0, 4, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) *out |= v;
    return e;
#else
    (void)out;
    (void)s;
    return cudaSuccess;
#endif
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (a.T + 7) / 8;  // 8 warps (tokens) per block
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    if (a.dtype == MOE_DTYPE_F32) return launch_combine_typed<float>(a, (unsigned)blocks, s);
    return launch_combine_typed<__nv_bfloat16>(a, (unsigned)blocks, s);
}

}  // namespace moe
