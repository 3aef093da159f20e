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
//   place_kernel  -- 32 tokens per block, blocks ordered by an atomic ticket.
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

constexpr int kPlaceTokens = 32;  // tokens per place_kernel block (one warp's worth)
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

template <typename T>
__global__ void __launch_bounds__(kPlaceThreads) place_kernel(DispatchArgs a) {
    __shared__ uint32_t bits[256];      // per expert: lanes (tokens) of this block that chose it
    __shared__ int prefix[256];         // per expert: assignments in earlier blocks
    __shared__ int offs[256];
    __shared__ int rows[kPlaceTokens][8];
    __shared__ int split_acc[kMaxRanks * kMaxRanks];  // [src][dst] kept rows of this block
    __shared__ uint32_t blk_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) blk_s = atomicAdd(a.ticket, 1u);
    for (int e = tid; e < a.E; e += kPlaceThreads) {
        bits[e] = 0u;
        offs[e] = a.expert_offsets[e];
    }
    for (int i = tid; i < a.R * a.R; i += kPlaceThreads) split_acc[i] = 0;
    __syncthreads();
    const uint32_t blk = blk_s;
    const int64_t t0 = (int64_t)blk * kPlaceTokens;
    const int64_t t = t0 + lane;
    const bool live = t < a.T;
    int my_e[8];
    if (warp == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            my_e[j] = -1;
            if (j < a.k && live) {
                const int e = a.idx[t * a.k + j];
                if ((unsigned)e < (unsigned)a.E) {
                    my_e[j] = e;
                    atomicOr(&bits[e], 1u << lane);
                }
            }
        }
    }
    __syncthreads();
    // Per-expert decoupled look-back over the preceding blocks.
    uint64_t* desc = a.desc + (int64_t)blk * a.E;
    for (int e = tid; e < a.E; e += kPlaceThreads) {
        const int own = __popc(bits[e]);
        if (blk == 0) {
            st_relaxed_u64(desc + e, kFlagIncl | (uint32_t)own);
            prefix[e] = 0;
            continue;
        }
        st_relaxed_u64(desc + e, kFlagAgg | (uint32_t)own);
        int excl = 0;
        int64_t j = (int64_t)blk - 1;
        uint64_t t_start = 0;
        while (j >= 0) {
            const uint64_t v = ld_relaxed_u64(a.desc + j * a.E + e);
            const uint64_t flag = v & (3ull << 32);
            if (flag == 0) {
                if (t_start == 0) t_start = globaltimer_ns();
                else if (globaltimer_ns() - t_start > kWaitTimeoutNs) {
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
        st_relaxed_u64(desc + e, kFlagIncl | (uint32_t)(excl + own));
    }
    __syncthreads();
    // Positions, keep/drop, rows.
    if (warp == 0) {
        const int per = a.E / a.R;
        const int64_t src_size = (a.T + a.R - 1) / a.R;
        const int src = live ? (int)(t / src_size) : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= a.k) break;
            int row = -1;
            const int e = my_e[j];
            if (e >= 0) {
                const int pos = prefix[e] + __popc(bits[e] & lanemask_lt());
                if (a.C < 0 || pos < a.C) {
                    row = offs[e] + pos;
                    a.row_token[row] = (int32_t)t;
                    atomicAdd(&split_acc[src * a.R + e / per], 1);
                }
            }
            if (live) a.slot_row[t * a.k + j] = row;
            rows[lane][j] = row;
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
    // Row copies: x[t] -> xp[row] for every kept row, 16-byte vectors.
    const int nvec = a.d * (int)sizeof(T) / 16;
    const char* x = static_cast<const char*>(a.x);
    char* xp = static_cast<char*>(a.xp);
    for (int tok = warp; tok < kPlaceTokens; tok += kPlaceThreads / 32) {
        const int64_t tt = t0 + tok;
        if (tt >= a.T) break;
        int r[8];
        int nk = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            r[j] = (j < a.k) ? rows[tok][j] : -1;
            nk += r[j] >= 0;
        }
        if (nk == 0) continue;
        const char* src = x + tt * (int64_t)a.d * sizeof(T);
        for (int c = lane; c < nvec; c += 32) {
            const uint4 v = ld_nc_v4(src + (int64_t)c * 16);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r[j] >= 0) st_v4(xp + ((int64_t)r[j] * a.d * sizeof(T)) + (int64_t)c * 16, v);
        }
    }
}

}  // namespace

int64_t dispatch_blocks(int64_t T) { return (T + kPlaceTokens - 1) / kPlaceTokens; }

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
    const int64_t nblk = dispatch_blocks(a.T);
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
        place_kernel<float><<<(unsigned)nblk, kPlaceThreads, 0, s>>>(a);
    else
        place_kernel<__nv_bfloat16><<<(unsigned)nblk, kPlaceThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
