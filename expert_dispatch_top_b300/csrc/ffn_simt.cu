// ffn_simt.cu -- Step 3, Compute, for fp32 experts: an FFMA grouped GEMM.
//
// Ultralytics glossary "Expert Parallelism", "How Tokens Move Between GPUs",
// step 3: every expert processes the rows dispatched to it.  fp32 experts
// cannot use the bf16 tensor-core path (and tf32 would miss a 1e-4 relative
// accuracy budget), so they run as a tiled FFMA GEMM: 64 x 64 output tiles,
// K in chunks of 16 through shared memory, 4 x 4 outputs per thread.
//
// Groups are ragged: group g owns rows [offsets[g], offsets[g+1]) of A and
// out.  blockIdx.x enumerates (group, m-tile) pairs from the device-side
// offsets (no host synchronisation); blocks past the last tile exit.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int SBM = 64, SBN = 64, SBK = 16;

__device__ __forceinline__ float gelu_f(float v) {
    return 0.5f * v * (1.f + erff(v * 0.70710678118654752440f));
}
__device__ __forceinline__ float silu_f(float v) { return v / (1.f + expf(-v)); }

template <typename T, bool GATED>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a) {
    __shared__ __align__(16) float As[SBK][SBM];
    __shared__ __align__(16) float Bs[SBK][SBN];
    __shared__ __align__(16) float Us[GATED ? SBK : 1][GATED ? SBN : 1];
    __shared__ int s_g, s_row0, s_rows;
    const int tid = threadIdx.x;
    if (tid == 0) {
        // find (group, m-tile) of this block
        int rem = blockIdx.x, g = -1, row0 = 0, rows = 0;
        for (int q = 0; q < a.G; ++q) {
            const int lo = a.offsets ? a.offsets[q] : 0;
            const int hi = a.offsets ? a.offsets[q + 1] : (int)a.m_rows;
            const int mt = (hi - lo + SBM - 1) / SBM;
            if (rem < mt) {
                g = q;
                row0 = lo + rem * SBM;
                rows = hi - row0 < SBM ? hi - row0 : SBM;
                break;
            }
            rem -= mt;
        }
        s_g = g;
        s_row0 = row0;
        s_rows = rows;
    }
    __syncthreads();
    const int g = s_g;
    if (g < 0) return;
    const int row0 = s_row0, rows = s_rows;
    const int n0 = blockIdx.y * SBN;
    const int K = a.K, N = a.N;
    const int b_rows = GATED ? 2 * N : N;
    const T* A = static_cast<const T*>(a.A);
    const T* B = static_cast<const T*>(a.B) + (int64_t)g * b_rows * K;
    const int tx = tid & 15, ty = tid >> 4;

    float acc[4][4], accu[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = accu[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += SBK) {
        // 64 x 16 tiles: 1024 elements each, one element per thread per pass
        for (int i = tid; i < SBM * SBK; i += 256) {
            const int r = i / SBK, kk = i % SBK;
            const int gk = k0 + kk;
            As[kk][r] = (r < rows && gk < K) ? Elem<T>::to_f(A[(int64_t)(row0 + r) * K + gk]) : 0.f;
            const int n = n0 + r;
            Bs[kk][r] = (n < N && gk < K) ? Elem<T>::to_f(B[(int64_t)n * K + gk]) : 0.f;
            if (GATED)
                Us[kk][r] = (n < N && gk < K) ? Elem<T>::to_f(B[(int64_t)(N + n) * K + gk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SBK; ++kk) {
            const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float ar[4] = {av.x, av.y, av.z, av.w};
            const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
            if (GATED) {
                const float4 uv = *reinterpret_cast<const float4*>(&Us[kk][tx * 4]);
                const float ur[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) accu[i][j] = fmaf(ar[i], ur[j], accu[i][j]);
            }
        }
        __syncthreads();
    }
    T* out = static_cast<T*>(a.out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        if (r >= rows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[i][j];
            if (a.epi == EPI_GELU) v = gelu_f(v);
            else if (GATED) v = silu_f(v) * accu[i][j];
            out[(int64_t)(row0 + r) * N + n] = Elem<T>::from_f(v);
        }
    }
}

template <typename T>
cudaError_t launch_simt_typed(const GemmArgs& a, cudaStream_t s) {
    const int64_t rows_bound = a.offsets ? a.rows_cap : a.m_rows;
    const int64_t mtiles = (rows_bound + SBM - 1) / SBM + a.G;
    if (rows_bound == 0) return cudaSuccess;
    dim3 grid((unsigned)mtiles, (unsigned)((a.N + SBN - 1) / SBN));
    if (a.epi == EPI_SWIGLU)
        gemm_simt_kernel<T, true><<<grid, 256, 0, s>>>(a);
    else
        gemm_simt_kernel<T, false><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t s) {
    if (a.dtype == MOE_DTYPE_F32) return launch_simt_typed<float>(a, s);
    return launch_simt_typed<__nv_bfloat16>(a, s);
}

}  // namespace moe
