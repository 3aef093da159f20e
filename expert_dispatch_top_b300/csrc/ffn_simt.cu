// ffn_simt.cu -- Step 3, Compute, for fp32 experts: an FFMA grouped GEMM.
//
// Ultralytics glossary "Expert Parallelism", "How Tokens Move Between GPUs",
// step 3: every expert processes the rows dispatched to it.  fp32 experts
// cannot use the bf16 tensor-core path (and tf32 would miss a 1e-4 relative
// accuracy budget), so they run as a tiled FFMA GEMM:
//   out[rows of group g, :] = epi( A[rows, :K] . B[g]^T )
// 128 x 128 output tiles (SwiGLU: 128 x 64 gate columns and the matching 64
// up columns), K in steps of 8 through double-buffered shared memory with the
// next step's loads in registers, 8 x 8 outputs per thread split over rows
// {4ty.., 64+4ty..} and columns {4tx.., 64+4tx..} so that every shared-memory
// read is a conflict-free float4; the products run as paired FMAs (two
// columns per instruction).
//
// Groups are ragged: group g owns rows [offsets[g], offsets[g+1]) of A and
// out.  blockIdx.x enumerates (group, m-tile) pairs from the device-side
// offsets (no host synchronisation); blocks past the last tile exit.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int SBM = 128, SBN = 128, SBK = 8;


// Packed fp32 pairs (a .b64 register holding two floats) and the paired FMA
// of sm_100+: two IEEE single-precision FMAs per instruction, each rounded as
// fmaf rounds, so results are bit-identical to scalar FMAs while the FMA
// instructions a warp must issue halve.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

template <bool GATED>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a) {
    __shared__ __align__(16) float As[2][SBK][SBM];
    __shared__ __align__(16) float Bs[2][SBK][SBN];
    __shared__ int s_g, s_row0, s_rows;
    const int tid = threadIdx.x;
    pdl_wait();  // programmatic dependent launch: the previous kernel's writes
    if (tid == 0) {
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
    const int K = a.K, N = a.N;
    // output columns of this block: SBN plain, or SBN/2 gate + SBN/2 up
    const int ncol = GATED ? SBN / 2 : SBN;
    const int n0 = blockIdx.y * ncol;
    const int b_rows = GATED ? 2 * N : N;
    const float* A = static_cast<const float*>(a.A);
    const float* B = static_cast<const float*>(a.B) + (int64_t)g * b_rows * K;
    const int tx = tid & 15, ty = tid >> 4;

    // global -> register loads: one float4 of A and one of B per thread per k-step
    const int lr = tid >> 1;        // tile row 0..127
    const int lk = (tid & 1) * 4;   // k offset 0 or 4
    const bool a_ok = lr < rows;
    const float* a_src = A + (int64_t)(row0 + (a_ok ? lr : 0)) * K + lk;
    int brow;  // weight row feeding tile row lr
    if (GATED)
        brow = lr < 64 ? n0 + lr : N + n0 + (lr - 64);
    else
        brow = n0 + lr;
    const bool b_ok = GATED ? ((lr < 64 ? n0 + lr : n0 + lr - 64) < N) : (brow < N);
    const float* b_src = B + (int64_t)(b_ok ? brow : 0) * K + lk;

    // accumulators: row i, column pairs (2jp, 2jp+1) packed
    uint64_t acc2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) acc2[i][jp] = 0ull;

    auto load = [&](int k0, float4& ra, float4& rb) {
        const bool kin = k0 + lk < K;  // K % 4 == 0: a float4 is all in or all out
        ra = (a_ok && kin) ? *reinterpret_cast<const float4*>(a_src + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
        rb = (b_ok && kin) ? *reinterpret_cast<const float4*>(b_src + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto store = [&](int buf, const float4& ra, const float4& rb) {
        As[buf][lk + 0][lr] = ra.x;
        As[buf][lk + 1][lr] = ra.y;
        As[buf][lk + 2][lr] = ra.z;
        As[buf][lk + 3][lr] = ra.w;
        Bs[buf][lk + 0][lr] = rb.x;
        Bs[buf][lk + 1][lr] = rb.y;
        Bs[buf][lk + 2][lr] = rb.z;
        Bs[buf][lk + 3][lr] = rb.w;
    };

    float4 ra, rb;
    load(0, ra, rb);
    store(0, ra, rb);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += SBK) {
        const bool more = k0 + SBK < K;
        if (more) load(k0 + SBK, ra, rb);
#pragma unroll
        for (int kk = 0; kk < SBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint64_t bp[4] = {pack2(b0.x, b0.y), pack2(b0.z, b0.w), pack2(b1.x, b1.y),
                                    pack2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint64_t ai = pack2(ar[i], ar[i]);
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) acc2[i][jp] = ffma2(ai, bp[jp], acc2[i][jp]);
            }
        }
        if (more) store(buf ^ 1, ra, rb);
        __syncthreads();
        buf ^= 1;
    }
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) unpack2(acc2[i][jp], acc[i][2 * jp], acc[i][2 * jp + 1]);
    // epilogue: row r = {4ty + i, 64 + 4ty + i}; plain columns {4tx + j, 64 + 4tx + j};
    // gated: gate column 4tx + j pairs with up column (tile column 64 + 4tx + j)
    float* out = static_cast<float*>(a.out);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
        if (r >= rows) continue;
        float* orow = out + (int64_t)(row0 + r) * N;
        if (GATED) {
            const int n = n0 + tx * 4;
            if (n < N) {
                float4 o;
                o.x = silu_exact_f(acc[i][0]) * acc[i][4];
                o.y = silu_exact_f(acc[i][1]) * acc[i][5];
                o.z = silu_exact_f(acc[i][2]) * acc[i][6];
                o.w = silu_exact_f(acc[i][3]) * acc[i][7];
                *reinterpret_cast<float4*>(orow + n) = o;
            }
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = n0 + h * 64 + tx * 4;
                if (n >= N) continue;
                float4 o;
                o.x = acc[i][4 * h + 0];
                o.y = acc[i][4 * h + 1];
                o.z = acc[i][4 * h + 2];
                o.w = acc[i][4 * h + 3];
                if (a.epi == EPI_GELU) {
                    o.x = gelu_erf_f(o.x);
                    o.y = gelu_erf_f(o.y);
                    o.z = gelu_erf_f(o.z);
                    o.w = gelu_erf_f(o.w);
                }
                *reinterpret_cast<float4*>(orow + n) = o;
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t s) {
    if (a.dtype != MOE_DTYPE_F32) return cudaErrorInvalidValue;  // bf16 runs on the tensor cores
    if (a.K % 4 != 0 || a.N % 4 != 0) return cudaErrorInvalidValue;
    const int64_t rows_bound = a.offsets ? a.rows_cap : a.m_rows;
    if (rows_bound == 0) return cudaSuccess;
    const int64_t mtiles = (rows_bound + SBM - 1) / SBM + a.G;
    const bool gated = a.epi == EPI_SWIGLU;
    const int ncol = gated ? SBN / 2 : SBN;
    dim3 grid((unsigned)mtiles, (unsigned)((a.N + ncol - 1) / ncol));
    if (gated) return launch_pdl(gemm_simt_kernel<true>, grid, 256, 0, s, a);
    return launch_pdl(gemm_simt_kernel<false>, grid, 256, 0, s, a);
}

}  // namespace moe
