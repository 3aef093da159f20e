// ffn_tc.cu -- Step 3, Compute, for bf16 experts: a tcgen05 grouped GEMM.
//
// Ultralytics glossary "Expert Parallelism", "How Tokens Move Between GPUs",
// step 3: every expert processes the rows dispatched to it.  The expert FFN
// is the only dense contraction of the layer, so it runs on the 5th-gen
// tensor cores:
//
//   out[rows of group g, :] = epi( A[rows, :K] . B[g]^T )
//
// with bf16 operands, fp32 accumulation in tensor memory (TMEM) and a fused
// epilogue (GELU, SwiGLU = silu(gate) * up, or none) that rounds to bf16 once.
//
// Persistent, warp-specialised kernel, one CTA per SM (192 threads):
//   warp 0     TMA producer: A tile 128 x 64 and B tile 256 x 64 (bf16,
//              128-byte swizzle) per stage into a 4-stage shared-memory ring;
//   warp 1     allocates 512 TMEM columns; one lane issues tcgen05.mma
//              (M=128, N=256, K=16, kind::f16) into one of two 256-column
//              accumulators and commits each stage back to the producer;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (each warp owns the
//              32 TMEM lanes its warp index allows), activation, bf16 pack,
//              a padded shared-memory transpose and coalesced 128-byte row
//              stores masked to the group's rows.  With two accumulators the
//              epilogue of tile i overlaps the MMAs of tile i+1.
//
// Ragged groups: tiles are enumerated from the device-side row offsets, group
// by group, n-tile by n-tile, m-tile fastest (the 148 concurrent tiles share
// one group's A rows and a few of its weight tiles through L2); when a group's
// rows of A are too large for that (the Mixtral-shaped down projection: 117 MB
// of h per expert), in bands of 8 n-tiles with the m-tile fastest in a band.  A tile that
// runs past its group's last row reads the next group's rows (or TMA's zero
// fill past the buffer); those output rows are computed and never stored.  A
// group's last tile with at most 64 rows issues M = 64 MMAs instead of M = 128
// (row-offset and MN-major modes).
// SwiGLU weights are [G, 2N, K] with the gate rows first: one B stage holds
// 128 gate rows and the matching 128 up rows, so the accumulator holds gate
// and up side by side and the epilogue writes 128 output columns per tile.
//
// MN-major B (input gradients of the backward): B is given as [G, K, N] with
// N contiguous, i.e. the forward's weights read without a transpose.  A stage
// holds four TMA boxes of 64 N-columns x 64 K-rows (128-byte swizzle), and the
// MMA reads B through MN-major descriptors (chunk stride 8 KB).  No epilogue.
//
// K-grouped mode (weight gradients): group g's output is a whole [M, N]
// matrix, out[g] = A[K_g, :]^T . B[K_g, :], where A [K, M] and B [K, N] are
// activation buffers whose rows are laid out so that each group's rows form a
// 64-aligned range K_g (zero rows pad each group to a multiple of 64).  Both
// operands are read MN-major, as stored: a stage holds two (A) and four (B)
// TMA boxes of 64 columns x 64 rows.  Tiles run over (group, n-tile, m-tile)
// as above, but every tile's K loop covers only its group's K blocks; the
// tiles of a group without rows issue no MMA and store zeros.
//
// Every mbarrier wait is bounded by %globaltimer: on timeout the kernel sets
// MOE_DEV_GEMM_TIMEOUT, raises an abort flag seen by the other roles, drains
// its own MMAs (bounded) and frees TMEM before returning.
#include "gemm_tiles.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

using namespace tc;
using tiles::TileInfo;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int EPI_WARPS = 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int STG_PITCH = 144;  // staged row: 128 data bytes + 16 pad (conflict-free)
constexpr int STG_BYTES = EPI_WARPS * 32 * STG_PITCH;
constexpr int MAX_GROUPS = tiles::kMaxGroups;
constexpr int TABLE_BYTES = 128 + 4 * MAX_GROUPS * 4;  // barriers + flags, then 4 int tables
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_BYTES + TABLE_BYTES;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t kIdesc = idesc_bf16(BM, BN);
constexpr uint32_t kIdescBmn = idesc_bf16_bmn(BM, BN);
// Tail tiles with at most 64 of their group's rows run M = 64 MMAs (half the
// tensor work).  Their accumulator rows land in TMEM lanes 32*(r/16) + r%16:
// lanes 0-15 of each warp's 32-lane quarter.
constexpr int HALF_M = 64;
constexpr uint32_t kIdesc64 = idesc_bf16(HALF_M, BN);
constexpr uint32_t kIdescBmn64 = idesc_bf16_bmn(HALF_M, BN);
constexpr uint32_t kIdescMn = idesc_bf16_bmn(BM, BN) | (1u << 15);  // A and B MN-major
constexpr int MN_CHUNK = 64 * BK * 2;  // one 64-column x 64-row box of an MN-major B: 8 KB
constexpr int kBandTiles = 8;                      // n-tiles per band of the banded tile order
constexpr int64_t kBandMinABytes = 64ll << 20;     // banded when a group's A exceeds this

struct TcParams {
    const int32_t* offsets;
    int64_t m_rows;
    int G, N, K, epi;
    int num_kb;
    int n_tiles;
    int out_cols;  // output columns per tile (128 SwiGLU, 256 otherwise)
    int kg_M;      // K-grouped mode: rows of each group's output matrix
    int stall_kb;  // failure-detection hook (-1: off)
    int band;      // > 0: tiles run in bands of `band` n-tiles, m-tile fastest inside a band
    uint64_t wait_ns;
    __nv_bfloat16* out;
    uint32_t* status;
};

// GELU in its tanh form with the hardware tanh: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))).
// It differs from the erf form by less than 5e-4 |v| (the form's own error plus
// the 2^-11 relative error of tanh.approx), below the bf16 rounding of h
// (2^-9 relative), and costs a handful of instructions instead of erff.
__device__ __forceinline__ float gelu_f(float v) {
    float t;
    const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(u));
    const float hv = 0.5f * v;
    return fmaf(hv, t, hv);
}
__device__ __forceinline__ float silu_f(float v) { return v / (1.f + __expf(-v)); }

template <bool KG, bool BMN>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* stg = smem + STAGES * STAGE_BYTES;
    uint8_t* tbl = stg + STG_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(tbl);  // full[4] empty[4] accf[2] acce[2] drain
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tbl + 112);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tbl + 116);
    int* total_s = reinterpret_cast<int*>(tbl + 120);
    int* tstart = reinterpret_cast<int*>(tbl + 128);           // [MAX_GROUPS]
    int* mt = tstart + MAX_GROUPS;                              // [MAX_GROUPS]
    int* rowoff = mt + MAX_GROUPS;                              // [MAX_GROUPS]
    int* grows = rowoff + MAX_GROUPS;                           // [MAX_GROUPS]

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
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    }
    // programmatic dependent launch: everything above touched no global data
    pdl_wait();
    if (warp == 2)
        tiles::build_tile_table<KG, BM, BK>(p.offsets, p.m_rows, p.G, p.n_tiles, p.kg_M, lane, tstart,
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
                const TileInfo ti = tiles::decode_tile<KG, BM>(tile, p.G, tstart, mt, rowoff, grows, p);
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status, MOE_DEV_GEMM_TIMEOUT, p.wait_ns)) break;
                    const uint32_t fb = full0 + 8 * stage;
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_STAGE;
                    const int k0 = (ti.kb0 + kb) * BK;
                    if (kb == p.stall_kb && tile == 0) {
                        // test hook: leave this stage unfilled; the MMA issuer's wait runs out
                    } else if (KG) {
                        mbar_expect_tx(fb, STAGE_BYTES);
#pragma unroll
                        for (int c = 0; c < BM / 64; ++c)
                            tma_load_2d(sa + c * MN_CHUNK, &tmA, ti.row0 + c * 64, k0, fb);
#pragma unroll
                        for (int c = 0; c < BN / 64; ++c)
                            tma_load_3d(sb + c * MN_CHUNK, &tmB, ti.n_tile * BN + c * 64, k0, 0, fb);
                    } else if (BMN) {
                        mbar_expect_tx(fb, STAGE_BYTES);
                        tma_load_2d(sa, &tmA, k0, ti.row0, fb);
#pragma unroll
                        for (int c = 0; c < BN / 64; ++c)
                            tma_load_3d(sb + c * MN_CHUNK, &tmB, ti.n_tile * BN + c * 64, k0, ti.g, fb);
                    } else if (p.epi == EPI_SWIGLU) {
                        mbar_expect_tx(fb, STAGE_BYTES);
                        tma_load_2d(sa, &tmA, k0, ti.row0, fb);
                        tma_load_3d(sb, &tmB, k0, ti.n_tile * 128, ti.g, fb);
                        tma_load_3d(sb + B_STAGE / 2, &tmB, k0, p.N + ti.n_tile * 128, ti.g, fb);
                    } else {
                        mbar_expect_tx(fb, STAGE_BYTES);
                        tma_load_2d(sa, &tmA, k0, ti.row0, fb);
                        tma_load_3d(sb, &tmB, k0, ti.n_tile * BN, ti.g, fb);
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
                if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1, abort_flag, p.status, MOE_DEV_GEMM_TIMEOUT, p.wait_ns)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                const TileInfo ti = tiles::decode_tile<KG, BM>(tile, p.G, tstart, mt, rowoff, grows, p);
                const int nkb = KG ? ti.nkb : p.num_kb;
                const bool half = !KG && ti.rows <= HALF_M;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status, MOE_DEV_GEMM_TIMEOUT, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_STAGE;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        if (KG)  // both operands MN-major: 16 K rows of 128 B per MMA
                            mma_bf16(d_tmem, sw128_mn_desc(sa + kk * 2048, MN_CHUNK),
                                     sw128_mn_desc(sb + kk * 2048, MN_CHUNK), kIdescMn,
                                     (kb | kk) != 0 ? 1u : 0u);
                        else if (BMN)  // 16 K rows of 128 B per MMA
                            mma_bf16(d_tmem, sw128_desc(sa + kk * 32),
                                     sw128_mn_desc(sb + kk * 2048, MN_CHUNK),
                                     half ? kIdescBmn64 : kIdescBmn, (kb | kk) != 0 ? 1u : 0u);
                        else
                            mma_bf16(d_tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32),
                                     half ? kIdesc64 : kIdesc, (kb | kk) != 0 ? 1u : 0u);
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
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint8_t* my_stg = stg + (warp - 2) * (32 * STG_PITCH);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const TileInfo ti = tiles::decode_tile<KG, BM>(tile, p.G, tstart, mt, rowoff, grows, p);
            __nv_bfloat16* obase = KG ? p.out + (int64_t)ti.g * p.kg_M * p.N : p.out;
            // every lane waits, then the warp agrees, so the .sync.aligned TMEM loads
            // below always run converged
            const bool ok = __all_sync(0xffffffffu, mbar_wait(accf0 + 8 * acc, acc_phase, abort_flag, p.status, MOE_DEV_GEMM_TIMEOUT, p.wait_ns));
            if (!ok) break;
            fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const int col0 = ti.n_tile * p.out_cols;
            const bool half = !KG && ti.rows <= HALF_M;  // M = 64: rows 16q + lane, lane < 16
            for (int c64 = 0; c64 < p.out_cols / 64; ++c64) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int col = c64 * 64 + h * 32;
                    float v[32];
                    if (KG && ti.nkb == 0) {  // warp-uniform: the group has no rows
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    } else {
                        tmem_ld32(tbase + (uint32_t)col, v);
                    }
                    if (p.epi == EPI_SWIGLU) {
                        float u[32];
                        tmem_ld32(tbase + (uint32_t)(128 + col), u);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = silu_f(v[i]) * u[i];
                    } else if (p.epi == EPI_GELU) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i]);
                    }
                    uint8_t* dst = my_stg + lane * STG_PITCH + h * 64;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 w;
                        w.x = Elem<__nv_bfloat16>::pack2(v[8 * i + 0], v[8 * i + 1]);
                        w.y = Elem<__nv_bfloat16>::pack2(v[8 * i + 2], v[8 * i + 3]);
                        w.z = Elem<__nv_bfloat16>::pack2(v[8 * i + 4], v[8 * i + 5]);
                        w.w = Elem<__nv_bfloat16>::pack2(v[8 * i + 6], v[8 * i + 7]);
                        *reinterpret_cast<uint4*>(dst + 16 * i) = w;
                    }
                }
                __syncwarp();
                // 32 rows x 128 bytes: 8 lanes per row, 4 rows per pass
                const int gc = col0 + c64 * 64 + (lane & 7) * 8;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int r = it * 4 + (lane >> 3);
                    // row inside the tile of staged row r (TMEM lane q*32 + r)
                    const int lr = half ? (r < 16 ? q * 16 + r : BM) : q * 32 + r;
                    if (lr < ti.rows && gc < p.N) {
                        const uint4 w = *reinterpret_cast<const uint4*>(my_stg + r * STG_PITCH +
                                                                        (lane & 7) * 16);
                        st_v4(obase + (int64_t)(ti.row0 + lr) * p.N + gc, w);
                    }
                }
                __syncwarp();
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
}  // namespace

int gemm_tc_supported(const GemmArgs& a) {
    if (a.dtype != MOE_DTYPE_BF16) return 1;
    if (a.K % BK != 0 || a.N % 64 != 0) return 2;
    if (a.G < 1 || a.G > MAX_GROUPS) return 3;
    if (a.rows_cap >= (1ll << 31) || a.K > (1 << 20)) return 4;
    if (a.b_mn && (a.kgrouped || a.epi != EPI_NONE)) return 6;
    if (a.kgrouped && (a.rows_cap % 64 != 0 || !a.offsets || a.epi != EPI_NONE)) return 7;
    if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B) |
         reinterpret_cast<uintptr_t>(a.out)) & 15)
        return 5;
    return 0;
}

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t s) {
    if (gemm_tc_supported(a) != 0) return cudaErrorInvalidValue;
    const int64_t rows_cap = a.offsets ? a.rows_cap : a.m_rows;
    if (rows_cap <= 0) return cudaSuccess;
    const bool kg = a.kgrouped != 0;
    const bool bmn = a.b_mn != 0;
    if (kg && (!a.offsets || a.epi != EPI_NONE)) return cudaErrorInvalidValue;
    const bool gated = a.epi == EPI_SWIGLU;
    const int b_rows = gated ? 2 * a.N : a.N;
    CUtensorMap tmA, tmB;
    // A is read with 2-D loads, the stacked weights with 3-D loads (group index;
    // a single [N, K] matrix in K-grouped mode).
    if (kg) {  // A [K, M] and B [K, N]: boxes of 64 columns x 64 K-rows
        if (!make_tmap_bf16(&tmA, a.A, (uint64_t)rows_cap, (uint64_t)a.K, 1, BK, 2) ||
            !make_tmap_bf16(&tmB, a.B, (uint64_t)a.N, (uint64_t)a.K, 1, BK, 3))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_bf16(&tmA, a.A, (uint64_t)a.K, (uint64_t)rows_cap, 1, BM, 2)) {
        return cudaErrorInvalidValue;
    } else if (bmn) {  // [G, K, N]: boxes of 64 N-columns x 64 K-rows
        if (!make_tmap_bf16(&tmB, a.B, (uint64_t)a.N, (uint64_t)a.K, (uint64_t)a.G, BK, 3))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_bf16(&tmB, a.B, (uint64_t)a.K, (uint64_t)b_rows, kg ? 1 : (uint64_t)a.G,
                               gated ? 128 : BN, 3)) {
        return cudaErrorInvalidValue;
    }
    TcParams p;
    p.offsets = a.offsets;
    p.m_rows = a.m_rows;
    p.G = a.offsets ? a.G : 1;
    p.N = a.N;
    p.K = a.K;
    p.epi = a.epi;
    p.num_kb = a.K / BK;
    p.out_cols = gated ? 128 : BN;
    p.n_tiles = (a.N + p.out_cols - 1) / p.out_cols;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.status = a.status;
    p.kg_M = kg ? (int)rows_cap : 0;
    p.stall_kb = a.stall_kb;
    // When one group's rows of A (the down projection's h) would not share L2 with
    // its weights, the concurrent tiles should form a near-square block of the
    // output so that both operands are re-read as little as possible: bands of
    // kBandTiles n-tiles, m-tile fastest inside each band (a wave of 148 tiles
    // then covers ~18 m-tiles x 8 n-tiles instead of every m-tile x ~4.6 n-tiles).
    p.band = 0;
    if (!kg && !bmn && a.offsets && a.G > 0 &&
        rows_cap / a.G * (int64_t)a.K * 2 > kBandMinABytes && p.n_tiles > kBandTiles)
        p.band = kBandTiles;
    p.wait_ns = a.wait_ns ? a.wait_ns : kWaitTimeoutNs;

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles_bound =
        kg ? (int64_t)p.G * ((rows_cap + BM - 1) / BM) * p.n_tiles
           : ((rows_cap + BM - 1) / BM + p.G) * p.n_tiles;
    int grid = (int)(tiles_bound < sms ? tiles_bound : sms);
    if (grid < 1) grid = 1;
    const int mode = kg ? 1 : bmn ? 2 : 0;
    auto kern = mode == 1 ? tc_gemm_kernel<true, false>
                          : mode == 2 ? tc_gemm_kernel<false, true> : tc_gemm_kernel<false, false>;
    // the shared-memory limit is a per-device function attribute: set it once per
    // device and kernel form (a repeated set from a racing thread is harmless)
    constexpr int kDevs = 64;
    static bool attr_set[kDevs][3] = {};
    if (dev < 0 || dev >= kDevs || !attr_set[dev][mode]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kDevs) attr_set[dev][mode] = true;
    }
    return launch_pdl(kern, dim3(grid), THREADS, (size_t)SMEM_BYTES, s, tmA, tmB, p);
}

}  // namespace moe
