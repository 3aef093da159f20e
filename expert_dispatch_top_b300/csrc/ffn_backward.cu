// ffn_backward.cu -- backward through the expert FFNs (training, the pages'
// main setting: topicspectrum "Training teaches both experts and router").
//
// For each expert's rows (forward: pre = x W_up^T, h = act(pre), y = h W_down^T):
//   1. pre  = xp . W_up^T                  recomputed (grouped GEMM, no epilogue)
//   2. dh   = d_yp . W_down                (grouped GEMM on W_down^T)
//   3. d_pre, h from pre and dh            (elementwise activation backward)
//   4. d_xp = d_pre . W_up                 (grouped GEMM on W_up^T)
//   5. dW_down[e] = sum over rows d_yp^T h, dW_up[e] = sum over rows d_pre^T xp
// The GEMMs of steps 1, 2 and 4 run on the forward's grouped GEMMs.  bf16: on
// the tensor cores, steps 2 and 4 reading the weights as stored through the
// GEMM's MN-major B mode; fp32: with the weights transposed once per call by a
// batched tiled transpose, on the tensor cores as three tf32 products per
// product when d and d_ff are multiples of 16 (the operands split into tf32
// high and low parts in the scratch: xp, d_yp and both weights before step 1,
// d_pre after step 3), else on FFMA.  Step 5 sums over each expert's ragged
// rows: bf16 runs it on the tensor cores in the grouped GEMM's K-grouped mode
// over transposed, 64-row-padded copies of the activations (that mode also
// writes the zero gradients of experts without rows); fp32 runs a tiled FFMA
// kernel that reads the rows directly.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// out[b][c][r] = in[b][r][c] for a batch of R x C matrices (32 x 32 tiles).
template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T* in, T* out, int R, int C) {
    __shared__ T tile[32][33];
    const int b = blockIdx.z;
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const T* src = in + (int64_t)b * R * C;
    T* dst = out + (int64_t)b * R * C;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        if (r < R && c < C) tile[i][tx] = src[(int64_t)r * C + c];
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (r < R && c < C) dst[(int64_t)c * R + r] = tile[tx][i];
    }
}

__device__ __forceinline__ float sigm(float v) { return 1.f / (1.f + expf(-v)); }

// Activation backward over the kept rows (offsets[E] of them), one thread per
// hidden column.  SwiGLU: pre = [g | u]; GELU: pre = a.  Writes d_pre (same
// shape as pre) and, when h is not null, the recomputed activation h.
template <typename T>
__global__ void __launch_bounds__(256) act_backward_kernel(const T* pre, const T* dh, T* d_pre, T* h,
                                                           const int32_t* offsets, int E, int f,
                                                           int gated, int64_t rows_cap) {
    const int64_t rows = offsets[E] < rows_cap ? offsets[E] : rows_cap;
    const int up = gated ? 2 * f : f;
    const int64_t n = rows * f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / f;
        const int c = (int)(i - r * f);
        const float gd = Elem<T>::to_f(dh[r * f + c]);
        if (gated) {
            const float g = Elem<T>::to_f(pre[r * up + c]);
            const float u = Elem<T>::to_f(pre[r * up + f + c]);
            const float s = sigm(g);
            d_pre[r * up + c] = Elem<T>::from_f(gd * u * s * (1.f + g * (1.f - s)));
            d_pre[r * up + f + c] = Elem<T>::from_f(gd * g * s);
            if (h) h[r * f + c] = Elem<T>::from_f(g * s * u);
        } else {
            const float a = Elem<T>::to_f(pre[r * up + c]);
            const float cdf = 0.5f * (1.f + erff(a * 0.70710678118654752440f));
            const float pdf = 0.39894228040143267794f * expf(-0.5f * a * a);
            d_pre[r * up + c] = Elem<T>::from_f(gd * (cdf + a * pdf));
            if (h) h[r * f + c] = Elem<T>::from_f(a * cdf);
        }
    }
}

// Padded row layout of the weight-gradient GEMMs: expert e's rows start at
// padded row poff[e] = sum over e' < e of ceil(rows_e' / 64) * 64, and the rows
// from its last row up to the next multiple of 64 are zero, so that each
// expert's rows are a whole number of 64-row K blocks.  poff[E] = padded total.
// Computed by the whole block (256 threads, E <= 256).
__device__ __forceinline__ void pad_offsets(const int32_t* offsets, int E, int* poff,
                                            int* wsum /* 8 ints */) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v = tid < E ? (offsets[tid + 1] - offsets[tid] + 63) / 64 * 64 : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wsum[w];
    if (tid < E) poff[tid] = base + incl - v;
    if (tid == 255) poff[E] = base + incl;
    __syncthreads();
}

// Expert owning padded row p: the last e with poff[e] <= p.
__device__ __forceinline__ int pad_owner(const int* poff, int E, int p) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (poff[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// bf16 activation backward that also lays out the weight-gradient operands:
// one padded row per block iteration, 8 columns per thread and vector.  Real
// rows write d_pre (expert-major rows, for the input gradient) and the padded
// copies d_pre_pad and h_pad; padding rows write zeros.
template <bool GATED>
__global__ void __launch_bounds__(256) act_backward_pad_kernel(
    const __nv_bfloat16* pre, const __nv_bfloat16* dh, __nv_bfloat16* d_pre,
    __nv_bfloat16* d_pre_pad, __nv_bfloat16* h_pad, const int32_t* offsets, int E, int f) {
    __shared__ int poff[257];
    __shared__ int wsum[8];
    pad_offsets(offsets, E, poff, wsum);
    const int up = GATED ? 2 * f : f;
    const int nv = f / 8;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int p = blockIdx.x; p < poff[E]; p += gridDim.x) {
        const int e = pad_owner(poff, E, p);
        const int j = p - poff[e];
        const bool real = j < offsets[e + 1] - offsets[e];
        const int64_t r = (int64_t)offsets[e] + j;
        for (int v = threadIdx.x; v < nv; v += blockDim.x) {
            const int c = v * 8;
            if (!real) {
                *reinterpret_cast<uint4*>(h_pad + (int64_t)p * f + c) = zero;
                *reinterpret_cast<uint4*>(d_pre_pad + (int64_t)p * up + c) = zero;
                if (GATED) *reinterpret_cast<uint4*>(d_pre_pad + (int64_t)p * up + f + c) = zero;
                continue;
            }
            float gd[8], a[8], hv[8], da[8];
            Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(dh + r * f + c), gd);
            Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(pre + r * up + c), a);
            if (GATED) {
                float u[8], du[8];
                Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(pre + r * up + f + c), u);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float sg = sigm(a[i]);
                    da[i] = gd[i] * u[i] * sg * (1.f + a[i] * (1.f - sg));
                    du[i] = gd[i] * a[i] * sg;
                    hv[i] = a[i] * sg * u[i];
                }
                const uint4 qu = Elem<__nv_bfloat16>::pack(du);
                *reinterpret_cast<uint4*>(d_pre + r * up + f + c) = qu;
                *reinterpret_cast<uint4*>(d_pre_pad + (int64_t)p * up + f + c) = qu;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float cdf = 0.5f * (1.f + erff(a[i] * 0.70710678118654752440f));
                    const float pdf = 0.39894228040143267794f * expf(-0.5f * a[i] * a[i]);
                    da[i] = gd[i] * (cdf + a[i] * pdf);
                    hv[i] = a[i] * cdf;
                }
            }
            const uint4 qa = Elem<__nv_bfloat16>::pack(da);
            *reinterpret_cast<uint4*>(d_pre + r * up + c) = qa;
            *reinterpret_cast<uint4*>(d_pre_pad + (int64_t)p * up + c) = qa;
            *reinterpret_cast<uint4*>(h_pad + (int64_t)p * f + c) = Elem<__nv_bfloat16>::pack(hv);
        }
    }
}

// Padded copies of two expert-major [rows, C] bf16 buffers (xp and d_yp).
__global__ void __launch_bounds__(256) pad_rows_kernel(const __nv_bfloat16* in0, __nv_bfloat16* out0,
                                                       const __nv_bfloat16* in1, __nv_bfloat16* out1,
                                                       const int32_t* offsets, int E, int C) {
    __shared__ int poff[257];
    __shared__ int wsum[8];
    pad_offsets(offsets, E, poff, wsum);
    const int nv = C / 8;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int p = blockIdx.x; p < poff[E]; p += gridDim.x) {
        const int e = pad_owner(poff, E, p);
        const int j = p - poff[e];
        const bool real = j < offsets[e + 1] - offsets[e];
        const int64_t r = (int64_t)offsets[e] + j;
        for (int v = threadIdx.x; v < nv; v += blockDim.x) {
            const int64_t o = (int64_t)p * C + v * 8;
            if (real) {
                const int64_t i = r * C + v * 8;
                *reinterpret_cast<uint4*>(out0 + o) = ld_nc_v4(in0 + i);
                *reinterpret_cast<uint4*>(out1 + o) = ld_nc_v4(in1 + i);
            } else {
                *reinterpret_cast<uint4*>(out0 + o) = zero;
                *reinterpret_cast<uint4*>(out1 + o) = zero;
            }
        }
    }
}

// fp32 weight gradient: dW[g][m][n] = sum over rows r of group g of A[r][m] * B[r][n]
// (64 x 64 tiles, 4 x 4 per thread, 16 rows per step).
__global__ void __launch_bounds__(256) wgrad_simt_kernel(const float* A, const float* B, float* dW,
                                                         const int32_t* offsets, int M, int N) {
    __shared__ __align__(16) float As[16][64];
    __shared__ __align__(16) float Bs[16][64];
    const int g = blockIdx.z;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int lo = offsets[g], hi = offsets[g + 1];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[4][4] = {};
    for (int r0 = lo; r0 < hi; r0 += 16) {
        for (int i = tid; i < 16 * 64; i += 256) {
            const int rr = i / 64, cc = i % 64;
            const int r = r0 + rr;
            As[rr][cc] = (r < hi && m0 + cc < M) ? A[(int64_t)r * M + m0 + cc] : 0.f;
            Bs[rr][cc] = (r < hi && n0 + cc < N) ? B[(int64_t)r * N + n0 + cc] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float ar[4] = {a.x, a.y, a.z, a.w}, br[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* out = dW + (int64_t)g * M * N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n < N) out[(int64_t)m * N + n] = acc[i][j];
        }
    }
}

template <typename T>
cudaError_t transpose_batched(const void* in, void* out, int B, int R, int C, cudaStream_t s) {
    dim3 grid((C + 31) / 32, (R + 31) / 32, B);
    transpose_kernel<T><<<grid, 256, 0, s>>>(static_cast<const T*>(in), static_cast<T*>(out), R, C);
    return noted_launch();
}

}  // namespace

size_t ffn_backward_scratch_bytes(int64_t rows_cap, int E, int d, int f, int gated, int eb,
                                  int weight_grads) {
    const int up = gated ? 2 * f : f;
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t P = (size_t)((rows_cap + 64 * (int64_t)E + 63) / 64 * 64);  // padded rows bound
    size_t n = 0;
    n += al((size_t)rows_cap * up * eb);   // pre
    n += al((size_t)rows_cap * f * eb);    // dh
    n += al((size_t)rows_cap * up * eb);   // d_pre
    if (eb == 4) {
        n += al((size_t)E * up * d * eb);  // W_up^T
        n += al((size_t)E * d * f * eb);   // W_down^T
        if (weight_grads) n += al((size_t)rows_cap * f * eb);  // h
        if (d % 16 == 0 && f % 16 == 0) {
            // tf32 high and low parts: xp, W_up, d_yp, W_down^T, d_pre, W_up^T
            const size_t part[6] = {(size_t)rows_cap * d, (size_t)E * up * d, (size_t)rows_cap * d,
                                    (size_t)E * f * d, (size_t)rows_cap * up, (size_t)E * d * up};
            for (int i = 0; i < 6; ++i) n += 2 * al(part[i] * 4);
        }
    } else if (weight_grads) {
        n += al(P * f * 2);     // h, padded rows
        n += al(P * up * 2);    // d_pre, padded rows
        n += al(P * d * 2);     // xp, padded rows
        n += al(P * d * 2);     // d_yp, padded rows
    }
    return n;
}

cudaError_t launch_ffn_backward(const FfnBwdArgs& a, cudaStream_t s) {
    const int gated = a.epi == EPI_SWIGLU;
    const int up = gated ? 2 * a.f : a.f;
    const int eb = a.dtype == MOE_DTYPE_F32 ? 4 : 2;
    const bool tc = eb == 2;
    const bool wg = a.d_w_up || a.d_w_down;
    const bool x3 = !tc && a.d % 16 == 0 && a.f % 16 == 0;  // fp32 on the tensor cores
    if (tc && a.E > 256) return cudaErrorInvalidValue;
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t P = (size_t)((a.rows_cap + 64 * (int64_t)a.E + 63) / 64 * 64);
    char* sp = static_cast<char*>(a.scratch);
    auto take = [&](size_t bytes) {
        void* q = sp;
        sp += al(bytes);
        return q;
    };
    void* pre = take((size_t)a.rows_cap * up * eb);
    void* dh = take((size_t)a.rows_cap * a.f * eb);
    void* d_pre = take((size_t)a.rows_cap * up * eb);
    void *w_upT = nullptr, *w_downT = nullptr, *h = nullptr;
    void *h_pad = nullptr, *d_pre_pad = nullptr, *xp_pad = nullptr, *dyp_pad = nullptr;
    if (!tc) {
        w_upT = take((size_t)a.E * up * a.d * eb);
        w_downT = take((size_t)a.E * a.d * a.f * eb);
        if (wg) h = take((size_t)a.rows_cap * a.f * eb);
    } else if (wg) {
        h_pad = take(P * a.f * 2);
        d_pre_pad = take(P * up * 2);
        xp_pad = take(P * a.d * 2);
        dyp_pad = take(P * a.d * 2);
    }
    // fp32 on the tensor cores: high / low tf32 parts of each GEMM operand
    enum { XP, WU, DYP, WDT, DPRE, WUT };
    void *hi[6] = {}, *lo[6] = {};
    if (x3) {
        const size_t part[6] = {(size_t)a.rows_cap * a.d, (size_t)a.E * up * a.d,
                                (size_t)a.rows_cap * a.d, (size_t)a.E * a.f * a.d,
                                (size_t)a.rows_cap * up, (size_t)a.E * a.d * up};
        for (int i = 0; i < 6; ++i) {
            hi[i] = take(part[i] * 4);
            lo[i] = take(part[i] * 4);
        }
    }
    cudaError_t e;
    if (!tc) {
        // transposed weights: W_up [E, up, d] -> [E, d, up]; W_down [E, d, f] -> [E, f, d]
        if ((e = transpose_batched<float>(a.w_up, w_upT, a.E, up, a.d, s)) != cudaSuccess) return e;
        if ((e = transpose_batched<float>(a.w_down, w_downT, a.E, a.d, a.f, s)) != cudaSuccess)
            return e;
    }
    // the split of n fp32 values at src into operand op's high / low parts
    auto job = [&](int op, const void* src, int64_t n) {
        Tf32SplitJob j;
        j.src = static_cast<const float*>(src);
        j.hi = static_cast<float*>(hi[op]);
        j.lo = static_cast<float*>(lo[op]);
        j.n = n;
        return j;
    };
    if (x3) {
        const Tf32SplitJob inputs[3] = {job(XP, a.xp, a.rows_cap * a.d),
                                        job(WU, a.w_up, (int64_t)a.E * up * a.d),
                                        job(DYP, a.d_yp, a.rows_cap * a.d)};
        if ((e = launch_tf32_split(inputs, 3, s)) != cudaSuccess) return e;
        const Tf32SplitJob transposed[2] = {job(WDT, w_downT, (int64_t)a.E * a.f * a.d),
                                            job(WUT, w_upT, (int64_t)a.E * a.d * up)};
        if ((e = launch_tf32_split(transposed, 2, s)) != cudaSuccess) return e;
    }
    // out = A . B^T with B [E, N, K] (b_mn = 0), or out = A . B with B [E, K, N] (b_mn = 1)
    auto gemm = [&](const void* A, const void* B, void* out, int N, int K, int b_mn) {
        GemmArgs g;
        g.A = A;
        g.B = B;
        g.out = out;
        g.offsets = a.offsets;
        g.rows_cap = a.rows_cap;
        g.m_rows = 0;
        g.G = a.E;
        g.N = N;
        g.K = K;
        g.epi = EPI_NONE;
        g.dtype = a.dtype;
        g.status = a.status;
        g.b_mn = b_mn;
        return tc ? launch_gemm_tc(g, s) : launch_gemm_simt(g, s);
    };
    // the same on the tensor cores from split fp32 operands (K-major B)
    auto gemm3 = [&](int ia, int ib, void* out, int N, int K) {
        GemmArgs g;
        g.A = hi[ia];
        g.A_lo = lo[ia];
        g.B = hi[ib];
        g.B_lo = lo[ib];
        g.out = out;
        g.offsets = a.offsets;
        g.rows_cap = a.rows_cap;
        g.m_rows = 0;
        g.G = a.E;
        g.N = N;
        g.K = K;
        g.epi = EPI_NONE;
        g.dtype = a.dtype;
        g.status = a.status;
        return launch_gemm_x3(g, s);
    };
    e = x3 ? gemm3(XP, WU, pre, up, a.d) : gemm(a.xp, a.w_up, pre, up, a.d, 0);  // 1
    if (e != cudaSuccess) return e;
    e = x3 ? gemm3(DYP, WDT, dh, a.f, a.d)
           : gemm(a.d_yp, tc ? a.w_down : w_downT, dh, a.f, a.d, tc);  // 2
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // 3: activation backward (bf16 with weight gradients: also the padded operands)
    if (tc && wg) {
        if (gated)
            act_backward_pad_kernel<true><<<sms * 8, 256, 0, s>>>(
                static_cast<const __nv_bfloat16*>(pre), static_cast<const __nv_bfloat16*>(dh),
                static_cast<__nv_bfloat16*>(d_pre), static_cast<__nv_bfloat16*>(d_pre_pad),
                static_cast<__nv_bfloat16*>(h_pad), a.offsets, a.E, a.f);
        else
            act_backward_pad_kernel<false><<<sms * 8, 256, 0, s>>>(
                static_cast<const __nv_bfloat16*>(pre), static_cast<const __nv_bfloat16*>(dh),
                static_cast<__nv_bfloat16*>(d_pre), static_cast<__nv_bfloat16*>(d_pre_pad),
                static_cast<__nv_bfloat16*>(h_pad), a.offsets, a.E, a.f);
    } else if (!tc) {
        act_backward_kernel<float><<<sms * 8, 256, 0, s>>>(
            static_cast<const float*>(pre), static_cast<const float*>(dh), static_cast<float*>(d_pre),
            static_cast<float*>(h), a.offsets, a.E, a.f, gated, a.rows_cap);
    } else {
        act_backward_kernel<__nv_bfloat16><<<sms * 8, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(pre), static_cast<const __nv_bfloat16*>(dh),
            static_cast<__nv_bfloat16*>(d_pre), nullptr, a.offsets, a.E, a.f, gated, a.rows_cap);
    }
    if ((e = noted_launch()) != cudaSuccess) return e;
    if (x3) {
        const Tf32SplitJob dp = job(DPRE, d_pre, a.rows_cap * up);
        if ((e = launch_tf32_split(&dp, 1, s)) != cudaSuccess) return e;
    }
    e = x3 ? gemm3(DPRE, WUT, a.d_xp, a.d, up)
           : gemm(d_pre, tc ? a.w_up : w_upT, a.d_xp, a.d, up, tc);  // 4
    if (e != cudaSuccess) return e;
    if (!wg) return cudaSuccess;
    // 5: weight gradients
    if (!tc) {
        if (a.d_w_down) {
            dim3 grid((a.f + 63) / 64, (a.d + 63) / 64, a.E);
            wgrad_simt_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(a.d_yp),
                                                   static_cast<const float*>(h),
                                                   static_cast<float*>(a.d_w_down), a.offsets, a.d, a.f);
            if ((e = noted_launch()) != cudaSuccess) return e;
        }
        if (a.d_w_up) {
            dim3 grid((a.d + 63) / 64, (up + 63) / 64, a.E);
            wgrad_simt_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(d_pre),
                                                   static_cast<const float*>(a.xp),
                                                   static_cast<float*>(a.d_w_up), a.offsets, up, a.d);
            if ((e = noted_launch()) != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    pad_rows_kernel<<<sms * 4, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.xp), static_cast<__nv_bfloat16*>(xp_pad),
        static_cast<const __nv_bfloat16*>(a.d_yp), static_cast<__nv_bfloat16*>(dyp_pad), a.offsets,
        a.E, a.d);
    if ((e = noted_launch()) != cudaSuccess) return e;
    // dW[e] = A_pad[K_e, :]^T . B_pad[K_e, :] over expert e's padded rows
    auto kgemm = [&](const void* A, const void* B, void* out, int M, int N) {
        GemmArgs g;
        g.A = A;      // [P, M]
        g.B = B;      // [P, N]
        g.out = out;  // [E, M, N]
        g.offsets = a.offsets;
        g.rows_cap = M;
        g.m_rows = 0;
        g.G = a.E;
        g.N = N;
        g.K = (int)P;
        g.epi = EPI_NONE;
        g.dtype = a.dtype;
        g.status = a.status;
        g.kgrouped = 1;
        return launch_gemm_tc(g, s);
    };
    if (a.d_w_down && (e = kgemm(dyp_pad, h_pad, a.d_w_down, a.d, a.f)) != cudaSuccess) return e;
    if (a.d_w_up && (e = kgemm(d_pre_pad, xp_pad, a.d_w_up, up, a.d)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace moe
