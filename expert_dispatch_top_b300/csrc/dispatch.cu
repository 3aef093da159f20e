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
// The tokens are cut into blocks of TB = 32, 64 or 128 tokens, and three
// kernels run on them:
//   count_kernel  -- one CTA per token block: its per-expert assignment counts
//                    (shared-memory histogram), stored expert-major.
//   scan_kernel   -- one CTA per expert: the exclusive prefix of that expert's
//                    counts over the blocks (its assignments in earlier
//                    blocks, i.e. in earlier tokens) and its total.
//   place_kernel  -- one CTA per token block: the capacity-clipped totals give
//                    the expert offsets (every CTA scans the E totals; CTA 0
//                    stores the metadata outputs); an assignment's position
//                    among its expert's assignments in token order is the
//                    block's prefix plus its rank inside the block, which
//                    decides keep/drop against C and the row; then the block
//                    copies its tokens' rows with 16-byte vectors.
// Nothing waits on another CTA: the order comes from the scan, not from a
// look-back chain, so no kernel here spins.  All three are launched as
// programmatic dependents of the kernel before them (pre-staged, started when
// it completes) and wait (griddepcontrol.wait) for its memory before reading
// its results.  place_kernel builds its per-block bitmaps from topk_idx before
// that wait: it starts only after scan_kernel has completed, which waited for
// count_kernel, which waited for the router that wrote topk_idx.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

using tc::mbar_expect_tx;
using tc::mbar_fence_init;
using tc::mbar_init;
using tc::mbar_try_wait;
using tc::smem_u32;

constexpr int kPlaceTokens = 32;  // smallest token block: one warp's worth of tokens
constexpr int kPlaceThreads = 256;
constexpr int kMaxRanks = 32;     // virtual ranks supported by the send-count accumulator
constexpr int kScanThreads = 256, kScanItems = 4;

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* scratch /* >= 33 ints */, int* total) {
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

// Per-block, per-expert assignment counts: hist[e * nblk + b].
__global__ void __launch_bounds__(256) count_kernel(DispatchArgs a, int tb, int nblk) {
    __shared__ int h[256];
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    for (int e = tid; e < a.E; e += blockDim.x) h[e] = 0;
    // The router's topk_idx (or whatever kernel ran before).  Dependents are
    // released only after this wait: place_kernel reads topk_idx before its own
    // wait, which is safe because no kernel of the chain lets its successor
    // start before its own predecessor has completed.
    pdl_wait();
    if (b == 0) {
        int32_t* splits = a.rank_splits ? a.rank_splits : a.splits_acc;
        for (int i = tid; i < a.R * a.R; i += blockDim.x) splits[i] = 0;
    }
    __syncthreads();
    const int64_t t0 = (int64_t)b * tb;
    const int64_t t1 = t0 + tb < a.T ? t0 + tb : a.T;
    const int64_t n = (t1 - t0) * a.k;
    const int32_t* idx = a.idx + t0 * a.k;
    bool bad = false;
    for (int64_t i = tid; i < n; i += blockDim.x) {
        const int e = idx[i];
        if ((unsigned)e < (unsigned)a.E)
            atomicAdd(&h[e], 1);
        else
            bad = true;
    }
    if (bad) atomicOr(a.status, MOE_DEV_BAD_INDEX);
    __syncthreads();
    if (b < nblk)
        for (int e = tid; e < a.E; e += blockDim.x) a.hist[(int64_t)e * nblk + b] = h[e];
}

// Expert e = blockIdx.x: prefix[e * nblk + b] = sum of hist[e * nblk + j] over
// j < b, and totals[e] = the sum over all blocks.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(DispatchArgs a, int nblk) {
    __shared__ int scratch[33];
    pdl_wait();  // count_kernel's histograms
    const int e = blockIdx.x;
    const int32_t* in = a.hist + (int64_t)e * nblk;
    int32_t* out = a.prefix + (int64_t)e * nblk;
    int carry = 0;
    for (int base = 0; base < nblk; base += kScanThreads * kScanItems) {
        const int i0 = base + threadIdx.x * kScanItems;
        int v[kScanItems];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < kScanItems; ++j) {
            v[j] = i0 + j < nblk ? in[i0 + j] : 0;
            sum += v[j];
        }
        int total = 0;
        int run = carry + block_exclusive_scan(sum, scratch, &total);
#pragma unroll
        for (int j = 0; j < kScanItems; ++j) {
            if (i0 + j < nblk) out[i0 + j] = run;
            run += v[j];
        }
        carry += total;
    }
    if (threadIdx.x == 0) a.totals[e] = carry;
}

// Bulk (TMA engine, untiled) copies between global and shared memory.  Both
// addresses 16-byte aligned, sizes multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bounded wait for phase `parity` of a shared-memory barrier.
__device__ __forceinline__ bool bar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

constexpr int kBulkLag = 6;           // store groups allowed to still read their slot
constexpr int kBulkMaxSlots = 16;
constexpr int kBulkRingBytes = 48 * 1024;  // with ~18 KB of static shared memory: 3 CTAs per SM

// SUB sub-tiles of 32 tokens per block (TB = 32*SUB tokens): warp s < SUB
// ranks sub-tile s with per-expert lane bitmaps; larger blocks amortise the
// block's fixed costs (offsets, barriers) over more row copies.
// nslot > 0: the row copies go through a ring of nslot shared-memory slots
// with bulk copies (dynamic shared memory: nslot * chunk bytes); 0: 16-byte
// vector loads and stores.
template <typename T, int SUB>
__global__ void __launch_bounds__(kPlaceThreads) place_kernel(DispatchArgs a, int nblk, int nslot) {
    constexpr int TB = 32 * SUB;
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t ring_bar[kBulkMaxSlots];
    __shared__ uint32_t bits[SUB][256];  // per sub-tile and expert: lanes (tokens) that chose it
    __shared__ int wpre[SUB][256];       // per sub-tile and expert: assignments in earlier sub-tiles
    __shared__ int prefix[256];          // per expert: assignments in earlier blocks
    __shared__ int offs[257];
    __shared__ int rows[TB][8];
    __shared__ int split_acc[kMaxRanks * kMaxRanks];  // [src][dst] kept rows of this block
    __shared__ int scratch[33];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int blk = blockIdx.x;
    // blockIdx.y: column chunk of the row copies; chunk 0 also writes the metadata
    const bool chunk0 = blockIdx.y == 0;
    for (int e = tid; e < a.E; e += kPlaceThreads) {
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) bits[sb][e] = 0u;
    }
    for (int i = tid; i < a.R * a.R; i += kPlaceThreads) split_acc[i] = 0;
    if (tid == 0 && nslot > 0) {
        for (int i = 0; i < nslot; ++i) mbar_init(smem_u32(&ring_bar[i]), 1);
        mbar_fence_init();
    }
    __syncthreads();
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
    for (int e = tid; e < a.E; e += kPlaceThreads) {
        int own = 0;
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb) {
            wpre[sb][e] = own;
            own += __popc(bits[sb][e]);
        }
    }
    // scan_kernel's prefixes and totals from here on
    pdl_wait();
    {
        const int e = tid;  // E <= 256 = blockDim.x
        int total = 0, kept = 0, pre = 0;
        if (e < a.E) {
            total = a.totals[e];
            kept = (a.C >= 0 && total > a.C) ? (int)a.C : total;
            pre = blk < nblk ? a.prefix[(int64_t)e * nblk + blk] : 0;
        }
        int sum = 0;
        const int off = block_exclusive_scan(kept, scratch, &sum);
        if (e < a.E) {
            offs[e] = off;
            prefix[e] = pre;
            if (blk == 0 && chunk0) {
                a.expert_counts[e] = total;
                a.expert_offsets[e] = off;
            }
        }
        if (tid == 0) {
            offs[a.E] = sum;
            if (blk == 0 && chunk0) {
                a.expert_offsets[a.E] = sum;
                a.n_dropped[0] = (int32_t)(a.T * a.k - sum);
            }
        }
    }
    __syncthreads();
    if (blk == 0 && chunk0) {
        // rank r owns experts [r*E/R, (r+1)*E/R): a difference of offsets
        const int per = a.E / a.R;
        for (int r = tid; r < a.R; r += kPlaceThreads)
            a.rank_counts[r] = offs[(r + 1) * per] - offs[r * per];
    }
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
                    if (kChecked && (int64_t)row >= (a.C < 0 || a.T * a.k < (int64_t)a.E * a.C
                                                        ? a.T * a.k : (int64_t)a.E * a.C)) {
                        atomicOr(a.status, MOE_DEV_BOUNDS);  // cannot happen: counts are exact
                        row = -1;
                    }
                }
                if (row >= 0) {
                    if (chunk0) {
                        a.row_token[row] = (int32_t)t;
                        atomicAdd(&split_acc[src * a.R + e / per], 1);
                    }
                }
            }
            if (live && chunk0) a.slot_row[t * a.k + j] = row;
            rows[warp * 32 + lane][j] = row;
        }
    }
    __syncthreads();
    // This block's send counts -> rank_splits (a few global atomics per block).
    if (chunk0) {
        int32_t* splits = a.rank_splits ? a.rank_splits : a.splits_acc;
        for (int i = tid; i < a.R * a.R; i += kPlaceThreads) {
            const int v = split_acc[i];
            if (v) atomicAdd(&splits[i], v);
        }
    }
    // Row copies: x[t] -> xp[row] for every kept row, 16-byte vectors, eight
    // loads in flight per thread; this CTA copies the row columns of its chunk,
    // 16-byte vectors [vlo, vhi).  Chunks of >= 256 vectors (4 KB): one warp per
    // token, lanes along the row.  Narrower chunks: the block's 256 threads walk
    // the (token, vector) space of its TB rows together, each stepping its pair
    // by 256 vectors, so short rows keep as many bytes in flight as long ones.
    const int nvec = a.d * (int)sizeof(T) / 16;
    const int vlo = (int)((int64_t)blockIdx.y * nvec / gridDim.y);
    const int vhi = (int)((int64_t)(blockIdx.y + 1) * nvec / gridDim.y);
    const int w = vhi - vlo;
    const int64_t row_bytes = (int64_t)a.d * sizeof(T);
    const char* x = static_cast<const char*>(a.x) + (int64_t)vlo * 16;
    char* xp = static_cast<char*>(a.xp) + (int64_t)vlo * 16;
    const int ntok = (int)((a.T - t0) < TB ? (a.T - t0) : TB);
    if (nslot > 0) {
        // One thread moves the rows: a bulk load of each token's chunk into a
        // ring slot, then one bulk store per kept row.  A slot is reloaded once
        // the store group that read it is done reading (kBulkLag groups behind).
        if (tid != 0) return;
        const uint32_t cb = (uint32_t)w * 16u;
        const uint32_t ring0 = smem_u32(ring);
        const uint32_t bar0 = smem_u32(ring_bar);
        int lt = 0, st = 0, loads = 0, groups = 0;
        auto kept = [&](int tok) {
            bool any = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) any |= j < a.k && rows[tok][j] >= 0;
            return any;
        };
        auto refill = [&]() {
            while (loads < groups - kBulkLag + nslot) {
                while (lt < ntok && !kept(lt)) ++lt;
                if (lt >= ntok) return;
                const int slot = loads % nslot;
                mbar_expect_tx(bar0 + 8 * slot, cb);
                bulk_load(ring0 + slot * cb, x + (t0 + lt) * row_bytes, cb, bar0 + 8 * slot);
                ++loads;
                ++lt;
            }
        };
        refill();
        bool ok = true;
        while (groups < loads) {
            while (!kept(st)) ++st;
            const int slot = groups % nslot;
            if (!bar_wait_bounded(bar0 + 8 * slot, (uint32_t)(groups / nslot) & 1u, kWaitTimeoutNs)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = j < a.k ? rows[st][j] : -1;
                if (r >= 0) bulk_store(xp + (int64_t)r * row_bytes, ring0 + slot * cb, cb);
            }
            bulk_commit();
            ++groups;
            ++st;
            bulk_wait_read<kBulkLag>();
            refill();
        }
        if (!ok) {
            // a load never landed: report it, and wait (bounded) for the loads
            // still in flight before the shared memory they target goes away
            atomicOr(a.status, MOE_DEV_COPY_TIMEOUT);
            for (int g = groups; g < loads; ++g)
                bar_wait_bounded(bar0 + 8 * (g % nslot), (uint32_t)(g / nslot) & 1u, kWaitTimeoutNs / 16);
        }
        bulk_wait_all();
        return;
    }
    if (w >= kPlaceThreads) {
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
            for (int c0 = lane; c0 < w; c0 += 256) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c0 + 32 * u < w) v[u] = ld_nc_v4(src + (int64_t)(c0 + 32 * u) * 16);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= w) break;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (r[j] >= 0) st_v4(xp + (int64_t)r[j] * row_bytes + (int64_t)c * 16, v[u]);
                }
            }
        }
        return;
    }
    int tok = tid / w, c = tid - (tid / w) * w;
    while (tok < ntok) {
        uint4 v[8];
        int vt[8], vc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            vt[u] = tok;
            vc[u] = c;
            if (tok < ntok) v[u] = ld_nc_v4(x + (t0 + tok) * row_bytes + (int64_t)c * 16);
            c += kPlaceThreads;
            while (c >= w) {
                c -= w;
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

// Column chunks per token block: enough CTAs for about four per SM, chunks of
// at least 64 vectors (1 KB).
int place_chunks(const DispatchArgs& a, int nblk, int elem_bytes) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (nblk <= 0) return 1;
    const int nvec = a.d * elem_bytes / 16;
    int S = (int)((4LL * sms + nblk - 1) / nblk);
    const int max_s = nvec / 64 > 1 ? nvec / 64 : 1;
    if (S > max_s) S = max_s;
    return S < 1 ? 1 : S;
}

template <typename T>
cudaError_t launch_place(const DispatchArgs& a, int sub, int nblk, cudaStream_t s) {
    // one CTA writes the metadata when T = 0
    const int S = place_chunks(a, nblk, (int)sizeof(T));
    const dim3 grid(nblk > 0 ? (unsigned)nblk : 1u, (unsigned)S);
    // Bulk copies through a shared-memory ring (as many chunk-sized slots as fit
    // kBulkRingBytes, more than kBulkLag) where they measured faster than the
    // vector copies: many destination rows per token (k >= 4), chunks of at
    // least 2 KB and batches of at most 16384 tokens (DeepSeek-shaped layer
    // 204 -> 191 us, 7168-wide rows at T = 4096 114 -> 111 us).  With k <= 2 or
    // short rows one issuing thread per CTA falls behind the vector copies
    // (Mixtral-shaped 75 -> 89 us, Switch-shaped 36 -> 105 us), and at
    // T = 131072 the two forms tie.
    const int nvec = a.d * (int)sizeof(T) / 16;
    const int64_t cb = (int64_t)((nvec + S - 1) / S) * 16;  // the widest chunk
    int nslot = (int)(kBulkRingBytes / cb);
    if (nslot > kBulkMaxSlots) nslot = kBulkMaxSlots;
    if (nslot < kBulkLag + 1 || a.k < 4 || cb < 2048 || a.T > 16384) nslot = 0;
    const size_t smem = (size_t)nslot * (size_t)cb;
    auto kern = sub == 4 ? place_kernel<T, 4> : sub == 2 ? place_kernel<T, 2> : place_kernel<T, 1>;
    if (smem > 0) {
        // the dynamic shared-memory limit is a per-device function attribute
        constexpr int kDevs = 64;
        static bool attr_set[kDevs][3] = {};
        const int form = sub == 4 ? 2 : sub == 2 ? 1 : 0;
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= kDevs || !attr_set[dev][form]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kBulkRingBytes);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < kDevs) attr_set[dev][form] = true;
        }
    }
    return launch_pdl(kern, grid, kPlaceThreads, smem, s, a, nblk, nslot);
}
}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
    if (a.E < 1 || a.E > 256 || a.k < 1 || a.k > 8 || a.R < 1 || a.R > kMaxRanks)
        return cudaErrorInvalidValue;
    const int sub = place_sub(a.T);
    const int64_t nblk64 = (a.T + 32 * sub - 1) / (32 * sub);
    if (nblk64 > (1 << 30)) return cudaErrorInvalidValue;
    const int nblk = (int)nblk64;
    cudaError_t e = launch_pdl(count_kernel, dim3(nblk > 0 ? (unsigned)nblk : 1u), 256, 0, s, a,
                               32 * sub, nblk);
    if (e != cudaSuccess) return e;
    e = launch_pdl(scan_kernel, dim3((unsigned)a.E), kScanThreads, 0, s, a, nblk);
    if (e != cudaSuccess) return e;
    if (a.dtype == MOE_DTYPE_F32) return launch_place<float>(a, sub, nblk, s);
    return launch_place<__nv_bfloat16>(a, sub, nblk, s);
}

}  // namespace moe
