// ffn_tf32.cu -- Step 3, Compute, for fp32 experts: the grouped GEMM on the
// tensor cores, every fp32 product formed from three tf32 products.
//
// Ultralytics glossary "Expert Parallelism", "How Tokens Move Between GPUs",
// step 3: every expert processes the rows dispatched to it.
//
// tf32 keeps fp32's sign and 8-bit exponent and 10 of its 23 mantissa bits,
// so one tf32 product (up to 2^-11 relative error per operand) misses the
// 1e-4 relative budget of fp32 experts.  Each fp32 operand x is split into two
// tf32 numbers,
//     hi = rn_tf32(x),   lo = rn_tf32(x - hi)          (x - hi is exact),
// with |x - hi| <= 2^-11 |x| and |x - hi - lo| <= 2^-22 |x|, and
//     a . b  ~=  a_lo . b_hi  +  a_hi . b_lo  +  a_hi . b_hi
// drops only a_lo . b_lo and the two lo roundings, each at most 2^-22 |a b|:
// under 3 * 2^-22 relative per product, against fp32's own 2^-24 per rounding.
// The product of two tf32 numbers (11-bit significands) is exact in fp32; the
// accumulation rounds as an fp32 sum does.
//
// The split: launch_tf32_split writes hi and lo of the expert inputs and of
// both weight stacks into the workspace in one elementwise pass, and the up
// projection's epilogue writes h already split -- its tf32 high part into the
// caller's h (scratch), its low part into the workspace -- which the down
// projection reads.  Since the tensor cores only ever see numbers exact in
// tf32, the result does not depend on how the hardware treats the low 13 bits
// of an fp32 operand.
//
// Kernel: the structure of the bf16 grouped GEMM (ffn_tc.cu) -- persistent,
// one CTA per SM, warp 0 TMA producer, warp 1 TMEM allocator and single-lane
// MMA issuer, warps 2-9 epilogue (two per TMEM lane quarter, each on half of
// the tile's columns), two 256-column fp32 accumulators so the epilogue of one
// tile overlaps the MMAs of the next, the ragged tile schedule of
// gemm_tiles.cuh -- with a stage of A_hi, A_lo (128 x 16 fp32 each) and B_hi,
// B_lo (256 x 16 fp32 each), rows of 64 bytes with the 64-byte swizzle: 48 KB,
// four stages in 192 KB.  Per K step of 8 the issuer runs the three
// tcgen05.mma kind::tf32 above, the small terms first (M = 128, or 64 for a
// group's last tile of at most 64 rows; N = 256).  The epilogue applies the
// activation in fp32 (GELU in its erf form, SwiGLU = silu(gate) * up) and
// stores fp32 rows through a padded shared-memory transpose as coalesced
// 64-byte segments.  Every mbarrier
// wait is bounded (MOE_DEV_GEMM_TIMEOUT, abort flag, bounded MMA drain, TMEM
// freed before returning).
#include "gemm_tiles.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace tc;
using tiles::TileInfo;

constexpr int BM = 128, BN = 256;
// Eight epilogue warps: two per TMEM lane quarter, each taking half of a tile's
// output columns (with four, the up projection's epilogue -- the activation and
// two fp32 output streams per element -- outlasted the tile's MMAs).
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int STG_PITCH = 80;  // staged row: 16 fp32 (64 bytes) + 16 pad (conflict-free writes)
constexpr int STG_BYTES = EPI_WARPS * 32 * STG_PITCH;
constexpr int MAX_GROUPS = tiles::kMaxGroups;
constexpr int TABLE_BYTES = 128 + 4 * MAX_GROUPS * 4;  // barriers + flags, then 4 int tables
constexpr int RING_BYTES = 192 * 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr int HALF_M = 64;  // tail tiles: accumulator rows in TMEM lanes 32*(r/16) + r%16
constexpr uint32_t kIdesc = idesc_tf32(BM, BN);
constexpr uint32_t kIdesc64 = idesc_tf32(HALF_M, BN);
// K elements per stage: 16 fp32 (64-byte rows, 64-byte swizzle, 48 KB stages,
// four in the ring) keep more loads in flight than 32 (128-byte rows, 96 KB
// stages, two).
constexpr int kStageK = 16;

// Ring geometry for BK fp32 of K per stage (one swizzled shared-memory row).
template <int BK>
struct X3Ring {
    static constexpr int SPAN = BK * 4;                              // bytes per row
    static constexpr int A_TILE = BM * SPAN;                         // 8 or 16 KB
    static constexpr int B_TILE = BN * SPAN;                         // 16 or 32 KB
    static constexpr int STAGE_BYTES = 2 * A_TILE + 2 * B_TILE;      // A_hi A_lo B_hi B_lo
    static constexpr int STAGES = RING_BYTES / STAGE_BYTES;          // 4 or 2
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_BYTES + TABLE_BYTES;
    static_assert(BK == 16 || BK == 32, "64- or 128-byte rows");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
    static_assert(2 * STAGES + 5 <= 14, "barriers fit below the abort flag");
    __device__ static uint64_t desc(uint32_t saddr) {
        return BK == 32 ? sw128_desc(saddr) : sw64_desc(saddr);
    }
};

struct X3Params {
    const int32_t* offsets;
    int64_t m_rows;
    int G, N, K, epi;
    int num_kb;
    int n_tiles;
    int out_cols;   // output columns per tile (128 SwiGLU, 256 otherwise)
    int kg_M, band;  // tile decoder: row-offset mode without bands (both 0)
    uint64_t wait_ns;
    float* out;     // the output, or with out_lo its tf32 high part
    float* out_lo;  // non-null: the output's tf32 low part (the up projection's h)
    uint32_t* status;
};

// Round to nearest, ties to even, to tf32 (10 explicit mantissa bits).
// Non-finite values pass unchanged; a finite value that would round past the
// largest finite one is truncated instead.
__device__ __forceinline__ float rn_tf32(float x) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7f800000u) == 0x7f800000u) return x;
    uint32_t r = (u + 0xfffu + ((u >> 13) & 1u)) & 0xffffe000u;
    if ((r & 0x7f800000u) == 0x7f800000u) r = u & 0xffffe000u;
    return __uint_as_float(r);
}

__device__ __forceinline__ float tf32_lo(float x, float hi) {
    return isfinite(x) ? rn_tf32(x - hi) : 0.f;
}

__global__ void __launch_bounds__(256) tf32_split_kernel(Tf32SplitJob j0, Tf32SplitJob j1,
                                                         Tf32SplitJob j2) {
    pdl_wait();  // the inputs may be the previous kernel's output
    const int64_t n0 = j0.n / 4, n1 = j1.n / 4, n2 = j2.n / 4;
    const int64_t total = n0 + n1 + n2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const bool in0 = i < n0, in1 = !in0 && i < n0 + n1;
        const int64_t v = in0 ? i : in1 ? i - n0 : i - n0 - n1;
        const float* src = in0 ? j0.src : in1 ? j1.src : j2.src;
        float* hi = in0 ? j0.hi : in1 ? j1.hi : j2.hi;
        float* lo = in0 ? j0.lo : in1 ? j1.lo : j2.lo;
        const uint4 raw = ld_nc_v4(src + 4 * v);
        const float x[4] = {__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                            __uint_as_float(raw.w)};
        float h[4], l[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            h[c] = rn_tf32(x[c]);
            l[c] = tf32_lo(x[c], h[c]);
        }
        st_v4(hi + 4 * v, make_uint4(__float_as_uint(h[0]), __float_as_uint(h[1]),
                                     __float_as_uint(h[2]), __float_as_uint(h[3])));
        st_v4(lo + 4 * v, make_uint4(__float_as_uint(l[0]), __float_as_uint(l[1]),
                                     __float_as_uint(l[2]), __float_as_uint(l[3])));
    }
}

template <int BK>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_x3_kernel(const __grid_constant__ CUtensorMap tmAh,
                      const __grid_constant__ CUtensorMap tmAl,
                      const __grid_constant__ CUtensorMap tmBh,
                      const __grid_constant__ CUtensorMap tmBl, const X3Params p) {
    using R = X3Ring<BK>;
    constexpr int STAGES = R::STAGES, STAGE_BYTES = R::STAGE_BYTES;
    constexpr int A_TILE = R::A_TILE, B_TILE = R::B_TILE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* stg = smem + STAGES * STAGE_BYTES;
    uint8_t* tbl = stg + STG_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(tbl);  // full[] empty[] accf[2] acce[2] drain
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tbl + 112);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tbl + 116);
    int* total_s = reinterpret_cast<int*>(tbl + 120);
    int* tstart = reinterpret_cast<int*>(tbl + 128);  // [MAX_GROUPS]
    int* mt = tstart + MAX_GROUPS;                     // [MAX_GROUPS]
    int* rowoff = mt + MAX_GROUPS;                     // [MAX_GROUPS]
    int* grows = rowoff + MAX_GROUPS;                  // [MAX_GROUPS]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        prefetch_tmap(&tmAh);
        prefetch_tmap(&tmAl);
        prefetch_tmap(&tmBh);
        prefetch_tmap(&tmBl);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    // programmatic dependent launch: everything above touched no global data
    pdl_wait();
    if (warp == 2)
        tiles::build_tile_table<false, BM, BK>(p.offsets, p.m_rows, p.G, p.n_tiles, 0, lane, tstart,
                                               mt, rowoff, grows, total_s);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *total_s;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                const TileInfo ti =
                    tiles::decode_tile<false, BM>(tile, p.G, tstart, mt, rowoff, grows, p);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status,
                                   MOE_DEV_GEMM_TIMEOUT, p.wait_ns))
                        break;
                    const uint32_t fb = full0 + 8 * stage;
                    const uint32_t ah = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t al = ah + A_TILE, bh = ah + 2 * A_TILE, bl = bh + B_TILE;
                    const int k0 = kb * BK;
                    mbar_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(ah, &tmAh, k0, ti.row0, fb);
                    tma_load_2d(al, &tmAl, k0, ti.row0, fb);
                    if (p.epi == EPI_SWIGLU) {
                        // 128 gate rows, then the matching 128 up rows
                        const int r0 = ti.n_tile * 128;
                        tma_load_3d(bh, &tmBh, k0, r0, ti.g, fb);
                        tma_load_3d(bh + B_TILE / 2, &tmBh, k0, p.N + r0, ti.g, fb);
                        tma_load_3d(bl, &tmBl, k0, r0, ti.g, fb);
                        tma_load_3d(bl + B_TILE / 2, &tmBl, k0, p.N + r0, ti.g, fb);
                    } else {
                        tma_load_3d(bh, &tmBh, k0, ti.n_tile * BN, ti.g, fb);
                        tma_load_3d(bl, &tmBl, k0, ti.n_tile * BN, ti.g, fb);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1, abort_flag, p.status,
                               MOE_DEV_GEMM_TIMEOUT, p.wait_ns)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                const TileInfo ti =
                    tiles::decode_tile<false, BM>(tile, p.G, tstart, mt, rowoff, grows, p);
                const uint32_t idesc = ti.rows <= HALF_M ? kIdesc64 : kIdesc;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status,
                                   MOE_DEV_GEMM_TIMEOUT, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t ah = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t al = ah + A_TILE, bh = ah + 2 * A_TILE, bl = bh + B_TILE;
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint32_t o = (uint32_t)kk * 32;  // 8 fp32 of each row
                        mma_tf32(d_tmem, R::desc(al + o), R::desc(bh + o), idesc,
                                 (kb | kk) != 0 ? 1u : 0u);
                        mma_tf32(d_tmem, R::desc(ah + o), R::desc(bl + o), idesc, 1u);
                        mma_tf32(d_tmem, R::desc(ah + o), R::desc(bh + o), idesc, 1u);
                    }
                    commit(empty0 + 8 * stage);
                    if (++stage == STAGES) {
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
        // ---------------- epilogue ----------------
        const int q = warp & 3;               // TMEM lane quarter this warp may access
        const int ch = p.out_cols / 64;       // 32-column chunks per warp
        const int c0 = ((warp - 2) >> 2) * ch;  // first chunk: warps 2-5 the left half, 6-9 the right
        uint8_t* my_stg = stg + (warp - 2) * (32 * STG_PITCH);
        const bool split = p.out_lo != nullptr;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const TileInfo ti = tiles::decode_tile<false, BM>(tile, p.G, tstart, mt, rowoff, grows, p);
            // every lane waits, then the warp agrees, so the .sync.aligned TMEM loads
            // below always run converged
            const bool ok = __all_sync(0xffffffffu, mbar_wait(accf0 + 8 * acc, acc_phase, abort_flag,
                                                              p.status, MOE_DEV_GEMM_TIMEOUT,
                                                              p.wait_ns));
            if (!ok) break;
            fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const bool half = ti.rows <= HALF_M;  // M = 64: rows 16q + lane, lane < 16
            const int gc0 = ti.n_tile * p.out_cols + (lane & 3) * 4;
            for (int c = c0; c < c0 + ch; ++c) {
                float v[32];
                tmem_ld32(tbase + (uint32_t)(c * 32), v);
                if (p.epi == EPI_SWIGLU) {
                    float u[32];
                    tmem_ld32(tbase + (uint32_t)(128 + c * 32), u);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = silu_exact_f(v[i]) * u[i];
                } else if (p.epi == EPI_GELU) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = gelu_erf_f(v[i]);
                }
                for (int o = 0; o < (split ? 2 : 1); ++o) {
                    // o = 0: the value, or its tf32 high part; 1: its low part
                    float* dst = o == 0 ? p.out : p.out_lo;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {  // 16 columns at a time
                        uint8_t* srow = my_stg + lane * STG_PITCH;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t w[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float x = v[16 * part + 4 * i + j];
                                const float hi = rn_tf32(x);
                                w[j] = __float_as_uint(!split ? x : o == 0 ? hi : tf32_lo(x, hi));
                            }
                            *reinterpret_cast<uint4*>(srow + 16 * i) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        __syncwarp();
                        // 32 rows x 64 bytes: 4 lanes per row, 8 rows per pass
                        const int gc = gc0 + c * 32 + part * 16;
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int r = it * 8 + (lane >> 2);
                            // row inside the tile of staged row r (TMEM lane q*32 + r)
                            const int lr = half ? (r < 16 ? q * 16 + r : BM) : q * 32 + r;
                            if (lr < ti.rows && gc < p.N) {
                                const uint4 w = *reinterpret_cast<const uint4*>(
                                    my_stg + r * STG_PITCH + (lane & 3) * 16);
                                st_v4(dst + (int64_t)(ti.row0 + lr) * p.N + gc, w);
                            }
                        }
                        __syncwarp();
                    }
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * acc);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int gemm_x3_supported(const GemmArgs& a) {
    if (a.dtype != MOE_DTYPE_F32) return 1;
    if (a.K < kStageK || a.K % kStageK != 0 || a.N < 4 || a.N % 4 != 0) return 2;
    if (a.G < 1 || a.G > MAX_GROUPS) return 3;
    if (a.rows_cap >= (1ll << 31) || a.m_rows >= (1ll << 31) || a.K > (1 << 20) || a.N > (1 << 20))
        return 4;
    if (!al16(a.A) || !al16(a.A_lo) || !al16(a.B) || !al16(a.B_lo) || !al16(a.out) ||
        !al16(a.out_lo))
        return 5;
    if (a.b_mn || a.kgrouped || a.stall_kb >= 0) return 6;
    if (!a.A || !a.A_lo || !a.B || !a.B_lo || !a.out)
        return 7;
    return 0;
}

cudaError_t launch_gemm_x3(const GemmArgs& a, cudaStream_t s) {
    using R = X3Ring<kStageK>;
    if (gemm_x3_supported(a) != 0) return cudaErrorInvalidValue;
    const int64_t rows_cap = a.offsets ? a.rows_cap : a.m_rows;
    if (rows_cap <= 0) return cudaSuccess;
    const bool gated = a.epi == EPI_SWIGLU;
    const uint64_t b_rows = gated ? 2ull * a.N : (uint64_t)a.N;
    const int G = a.offsets ? a.G : 1;
    const uint32_t b_box = gated ? 128 : BN;
    CUtensorMap tmAh, tmAl, tmBh, tmBl;
    if (!make_tmap_f32(&tmAh, R::SPAN, a.A, (uint64_t)a.K, (uint64_t)rows_cap, 1, BM, 2) ||
        !make_tmap_f32(&tmAl, R::SPAN, a.A_lo, (uint64_t)a.K, (uint64_t)rows_cap, 1, BM, 2) ||
        !make_tmap_f32(&tmBh, R::SPAN, a.B, (uint64_t)a.K, b_rows, (uint64_t)G, b_box, 3) ||
        !make_tmap_f32(&tmBl, R::SPAN, a.B_lo, (uint64_t)a.K, b_rows, (uint64_t)G, b_box, 3))
        return cudaErrorInvalidValue;
    X3Params p;
    p.offsets = a.offsets;
    p.m_rows = a.m_rows;
    p.G = G;
    p.N = a.N;
    p.K = a.K;
    p.epi = a.epi;
    p.num_kb = a.K / kStageK;
    p.out_cols = gated ? 128 : BN;
    p.n_tiles = (a.N + p.out_cols - 1) / p.out_cols;
    p.kg_M = 0;
    p.band = 0;
    p.wait_ns = a.wait_ns ? a.wait_ns : kWaitTimeoutNs;
    p.out = static_cast<float*>(a.out);
    p.out_lo = static_cast<float*>(a.out_lo);
    p.status = a.status;

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles_bound = ((rows_cap + BM - 1) / BM + G) * p.n_tiles;
    int grid = (int)(tiles_bound < sms ? tiles_bound : sms);
    if (grid < 1) grid = 1;
    auto kern = tc_gemm_x3_kernel<kStageK>;
    // the shared-memory limit is a per-device function attribute: set it once per device
    constexpr int kDevs = 64;
    static bool attr_set[kDevs] = {};
    if (dev < 0 || dev >= kDevs || !attr_set[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, R::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kDevs) attr_set[dev] = true;
    }
    return launch_pdl(kern, dim3(grid), THREADS, (size_t)R::SMEM_BYTES, s, tmAh, tmAl, tmBh, tmBl, p);
}

cudaError_t launch_tf32_split(const Tf32SplitJob* jobs, int njobs, cudaStream_t s) {
    if (njobs < 0 || njobs > 3 || (njobs > 0 && !jobs)) return cudaErrorInvalidValue;
    Tf32SplitJob j[3];
    int64_t total = 0;
    for (int i = 0; i < njobs; ++i) {
        if (!jobs[i].src || jobs[i].n == 0) continue;
        if (jobs[i].n < 0 || jobs[i].n % 4 != 0 || !jobs[i].hi || !jobs[i].lo || !al16(jobs[i].src) ||
            !al16(jobs[i].hi) || !al16(jobs[i].lo))
            return cudaErrorInvalidValue;
        j[i] = jobs[i];
        total += jobs[i].n / 4;
    }
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    return launch_pdl(tf32_split_kernel, dim3(grid), 256, 0, s, j[0], j[1], j[2]);
}

}  // namespace moe
