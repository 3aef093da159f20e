// dispatch.cu -- Step 2, Dispatch, as one on-device permutation.
//
// Ultralytics glossary "Expert Parallelism", "How Tokens Move Between GPUs",
// step 2 (each token's hidden state goes to the owners of its experts) and
// "Load Balancing and Capacity" (each expert takes at most C tokens, the
// overflow skips it); ai360xpert "Expert Parallelism", "The All-to-All
// Bottleneck" (Scatter).  With every expert on this GPU, the exchange becomes
// a permutation into an expert-major buffer whose contiguous expert blocks
// are the virtual ranks (expert e on rank e / (E/R)); the send counts the
// all-to-all would have used are reported as rank_splits.
//
// Two kernels:
//   count_kernel  -- per-expert loads (block histogram in shared memory, one
//                    global atomic per expert and block); the last block to
//                    finish turns them into capacity-clipped counts and the
//                    expert offsets.  It also clears the scan state used by
//                    place_kernel.
//   place_kernel  -- 32, 64 or 128 tokens per block, blocks ordered by an atomic ticket.
//                    A per-expert decoupled look-back over the blocks gives
//                    each assignment its position among the same expert's
//                    assignments in token order; the position decides
//                    keep/drop against C and the row; then the block copies
//                    its tokens' rows with 16-byte vectors.
// The look-back only ever waits on blocks that drew an earlier ticket, which
// are already running, and every wait is bounded (status word on timeout).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kPlaceTokens = 32;  // smallest place_kernel block: one warp's worth of tokens
constexpr int kPlaceThreads = 256;
constexpr int kMaxRanks = 32;     // virtual ranks supported by the send-count accumulator
constexpr uint64_t kFlagAgg = 1ull << 32;   // descriptor holds the block's own count
constexpr uint64_t kFlagIncl = 2ull << 32;  // descriptor holds the inclusive prefix

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* scratch /* >= 32 ints */, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        int wv = lane < nw ? scratch[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < nw) scratch[lane] = wi - wv;
        if (lane == nw - 1) scratch[32] = wi;
    }
    __syncthreads();
    const int out = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return out;
}

__global__ void __launch_bounds__(256) count_kernel(DispatchArgs a, int64_t n_desc) {
    __shared__ int hist[256];
    __shared__ int scratch[33];
    __shared__ bool last;
    const int tid = threadIdx.x;
    for (int e = tid; e < a.E; e += blockDim.x) hist[e] = 0;
    // clear the look-back descriptors and the split accumulator for place_kernel
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < n_desc;
         i += (int64_t)gridDim.x * blockDim.x)
        a.desc[i] = 0ull;
    int32_t* splits = a.rank_splits ? a.rank_splits : a.splits_acc;
    if (blockIdx.x == 0)
        for (int i = tid; i < a.R * a.R; i += blockDim.x) splits[i] = 0;
    __syncthreads();
    const int64_t n = a.T * a.k;
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int e = a.idx[i];
        if ((unsigned)e < (unsigned)a.E)
            atomicAdd(&hist[e], 1);
        else
            bad = true;
    }
    if (bad) atomicOr(a.status, MOE_DEV_BAD_INDEX);
    __syncthreads();
    for (int e = tid; e < a.E; e += blockDim.x)
        if (hist[e]) atomicAdd(&a.counts[e], hist[e]);
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(a.done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    // Last block: capacity-clipped counts, offsets, per-rank receive counts.
    int cnt = 0, kept = 0;
    if (tid < a.E) {
        cnt = atomicAdd(&a.counts[tid], 0);
        kept = (a.C >= 0 && cnt > a.C) ? (int)a.C : cnt;
        a.expert_counts[tid] = cnt;
    }
    int total = 0;
    const int off = block_exclusive_scan(tid < a.E ? kept : 0, scratch, &total);
    if (tid < a.E) a.expert_offsets[tid] = off;
    if (tid == 0) {
        a.expert_offsets[a.E] = total;
        a.n_dropped[0] = (int32_t)(n - total);
    }
    __syncthreads();
    // rank r owns experts [r*E/R, (r+1)*E/R): a difference of offsets
    const int per = a.E / a.R;
    for (int r = tid; r < a.R; r += blockDim.x)
        a.rank_counts[r] = a.expert_offsets[(r + 1) * per] - a.expert_offsets[r * per];
}

// SUB sub-tiles of 32 tokens per block (TB = 32*SUB tokens): warp s < SUB
// ranks sub-tile s with per-expert lane bitmaps; larger blocks amortise the
// block's fixed costs (ticket, look-back, barriers) over more row copies.
template <typename T, int SUB>
__global__ void __launch_bounds__(kPlaceThreads) place_kernel(DispatchArgs a) {
    constexpr int TB = 32 * SUB;
    __shared__ uint32_t bits[SUB][256];  // per sub-tile and expert: lanes (tokens) that chose it
    __shared__ int wpre[SUB][256];       // per sub-tile and expert: assignments in earlier sub-tiles
    __shared__ int prefix[256];          // per expert: assignments in earlier blocks
    __shared__ int offs[256];
    __shared__ int rows[TB][8];
    __shared__ int split_acc[kMaxRanks * kMaxRanks];  // [src][dst] kept rows of this block
    __shared__ uint32_t blk_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) blk_s = atomicAdd(a.ticket, 1u);
    for (int e = tid; e < a.E; e += kPlaceThreads) {
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) bits[sb][e] = 0u;
        offs[e] = a.expert_offsets[e];
    }
    for (int i = tid; i < a.R * a.R; i += kPlaceThreads) split_acc[i] = 0;
    __syncthreads();
    const uint32_t blk = blk_s;
    const int64_t t0 = (int64_t)blk * TB;
    const int64_t t = t0 + warp * 32 + lane;  // meaningful for warps < SUB
    const bool live = warp < SUB && t < a.T;
    int my_e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) my_e[j] = -1;
    if (warp < SUB) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < a.k && live) {
                const int e = a.idx[t * a.k + j];
                if ((unsigned)e < (unsigned)a.E) {
                    my_e[j] = e;
                    atomicOr(&bits[warp][e], 1u << lane);
                }
            }
        }
    }
    __syncthreads();
    // Per-expert decoupled look-back over the preceding blocks.
    uint64_t* desc = a.desc + (int64_t)blk * a.E;
    for (int e = tid; e < a.E; e += kPlaceThreads) {
        int own = 0;
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
            wpre[sb][e] = own;
            own += __popc(bits[sb][e]);
        }
        const bool publish = (int)blk != a.stall_block;
        if (blk == 0) {
            if (publish) st_relaxed_u64(desc + e, kFlagIncl | (uint32_t)own);
            prefix[e] = 0;
            continue;
        }
        if (publish) st_relaxed_u64(desc + e, kFlagAgg | (uint32_t)own);
        int excl = 0;
        int64_t j = (int64_t)blk - 1;
        uint64_t t_start = 0;
        while (j >= 0) {
            const uint64_t v = ld_relaxed_u64(a.desc + j * a.E + e);
            const uint64_t flag = v & (3ull << 32);
            if (flag == 0) {
                if (t_start == 0) t_start = globaltimer_ns();
                else if (globaltimer_ns() - t_start > a.wait_ns) {
                    atomicOr(a.status, MOE_DEV_LOOKBACK_TIMEOUT);
                    break;
                }
                __nanosleep(32);
                continue;
            }
            excl += (int)(uint32_t)v;
            if (flag == kFlagIncl) break;
            --j;
            t_start = 0;
        }
        prefix[e] = excl;
        if (publish) st_relaxed_u64(desc + e, kFlagIncl | (uint32_t)(excl + own));
    }
    __syncthreads();
    // Positions, keep/drop, rows.
    if (warp < SUB) {
        const int per = a.E / a.R;
        const int64_t src_size = (a.T + a.R - 1) / a.R;
        const int src = live ? (int)(t / src_size) : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= a.k) break;
            int row = -1;
            const int e = my_e[j];
            if (e >= 0) {
                const int pos = prefix[e] + wpre[warp][e] + __popc(bits[warp][e] & lanemask_lt());
                if (a.C < 0 || pos < a.C) {
                    row = offs[e] + pos;
                    a.row_token[row] = (int32_t)t;
                    atomicAdd(&split_acc[src * a.R + e / per], 1);
                }
            }
            if (live) a.slot_row[t * a.k + j] = row;
            rows[warp * 32 + lane][j] = row;
        }
    }
    __syncthreads();
    // This block's send counts -> rank_splits (a few global atomics per block).
    {
        int32_t* splits = a.rank_splits ? a.rank_splits : a.splits_acc;
        for (int i = tid; i < a.R * a.R; i += kPlaceThreads) {
            const int v = split_acc[i];
            if (v) atomicAdd(&splits[i], v);
        }
    }
    // Row copies: x[t] -> xp[row] for every kept row, 16-byte vectors, eight
    // loads in flight per thread.  Rows of >= 256 chunks (4 KB): one warp per
    // token, lanes along the row.  Shorter rows: the block's 256 threads walk
    // the (token, chunk) space of its TB rows together, each stepping its pair
    // by 256 chunks, so short rows keep as many bytes in flight as long ones.
    const int nvec = a.d * (int)sizeof(T) / 16;
    const int64_t row_bytes = (int64_t)a.d * sizeof(T);
    const char* x = static_cast<const char*>(a.x);
    char* xp = static_cast<char*>(a.xp);
    const int ntok = (int)((a.T - t0) < TB ? (a.T - t0) : TB);
    if (nvec >= kPlaceThreads) {
        for (int tok = warp; tok < ntok; tok += kPlaceThreads / 32) {
            int r[8];
            int nk = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                r[j] = (j < a.k) ? rows[tok][j] : -1;
                nk += r[j] >= 0;
            }
            if (nk == 0) continue;
            const char* src = x + (t0 + tok) * row_bytes;
            for (int c0 = lane; c0 < nvec; c0 += 256) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c0 + 32 * u < nvec) v[u] = ld_nc_v4(src + (int64_t)(c0 + 32 * u) * 16);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= nvec) break;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (r[j] >= 0) st_v4(xp + (int64_t)r[j] * row_bytes + (int64_t)c * 16, v[u]);
                }
            }
        }
        return;
    }
    int tok = tid / nvec, c = tid - (tid / nvec) * nvec;
    while (tok < ntok) {
        uint4 v[8];
        int vt[8], vc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            vt[u] = tok;
            vc[u] = c;
            if (tok < ntok) v[u] = ld_nc_v4(x + (t0 + tok) * row_bytes + (int64_t)c * 16);
            c += kPlaceThreads;
            while (c >= nvec) {
                c -= nvec;
                ++tok;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (vt[u] >= ntok) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= a.k) break;
                const int r = rows[vt[u]][j];
                if (r >= 0) st_v4(xp + (int64_t)r * row_bytes + (int64_t)vc[u] * 16, v[u]);
            }
        }
    }
}

}  // namespace

int64_t dispatch_blocks(int64_t T) { return (T + kPlaceTokens - 1) / kPlaceTokens; }

namespace {
// Sub-tiles per place_kernel block: as large as keeps >= 2 blocks per SM.
int place_sub(int64_t T) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n32 = dispatch_blocks(T);
    if (n32 >= 4 * 2 * (int64_t)sms) return 4;
    if (n32 >= 2 * 2 * (int64_t)sms) return 2;
    return 1;
}

template <typename T>
void launch_place(const DispatchArgs& a, int sub, int64_t nblk, cudaStream_t s) {
    if (sub == 4)
        place_kernel<T, 4><<<(unsigned)nblk, kPlaceThreads, 0, s>>>(a);
    else if (sub == 2)
        place_kernel<T, 2><<<(unsigned)nblk, kPlaceThreads, 0, s>>>(a);
    else
        place_kernel<T, 1><<<(unsigned)nblk, kPlaceThreads, 0, s>>>(a);
}
}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
    const int sub = place_sub(a.T);
    const int64_t nblk = (a.T + 32 * sub - 1) / (32 * sub);
    const int64_t n_desc = nblk * a.E;
    const int64_t n = a.T * a.k;
    int64_t cb = (n + 256 * 8 - 1) / (256 * 8);
    const int64_t cb_desc = (n_desc + 256 * 4 - 1) / (256 * 4);
    if (cb_desc > cb) cb = cb_desc;
    if (cb < 1) cb = 1;
    if (cb > 296) cb = 296;
    count_kernel<<<(unsigned)cb, 256, 0, s>>>(a, n_desc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nblk == 0) return e;
    if (a.dtype == MOE_DTYPE_F32)
        launch_place<float>(a, sub, nblk, s);
    else
        launch_place<__nv_bfloat16>(a, sub, nblk, s);
    return cudaGetLastError();
}

}  // namespace moe
