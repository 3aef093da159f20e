// dispatch_noalloc.cu -- moe_dispatch_noalloc: the dispatch step with its
// scratch state kept in a fixed-size array inside the library.
//
// Some callers cannot call cudaMalloc: a plugin inside an inference engine
// that is handed only its input and output pointers, or a serving loop whose
// device memory was all reserved by another allocator at start-up.  They have
// no way to provide the workspace moe_dispatch needs.  This entry point runs
// the very same dispatch kernels, but points their scratch state (status
// word, per-expert totals, per-block counts and prefixes, send-count
// accumulator) at the file-scope device array below.
//
// The array is a static __device__ object: every GPU that loads the library
// holds kScratchBytes of it until the process exits.  Host code cannot use
// the array's name as a device address (in host code it names a host-side
// stand-in), so the first call in each CUDA context (with that context
// current) looks the address up with cudaGetSymbolAddress and caches it under
// the context's unique ID.  A context that is destroyed and created again
// (cudaDeviceReset, or an engine that manages its own contexts through the
// driver API) gets a new ID, and with it a fresh lookup: the library's module
// may load at another address in the new context.  Every call shares the one
// array and finds the previous call's contents in it; the kernels write every
// part they read before reading it.
// Calls that overlap on the GPU (different streams, or several host threads
// without ordering) race on the array.
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr size_t kAlignNA = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kScratchBytes];

std::mutex g_scratch_mu;
struct ScratchEntry {
    unsigned long long ctx_id;
    void* addr;
};
ScratchEntry g_scratch_cache[kMaxDevices] = {};
int g_scratch_next = 0;  // next entry to reuse once the cache is full

inline size_t up256(size_t v) { return (v + kAlignNA - 1) / kAlignNA * kAlignNA; }

// Unique ID of the current CUDA context (driver entry points through the
// runtime, so the library needs no -lcuda).  False if there is no current
// context or the driver cannot say.
bool current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (!get_current || !get_id) {
        void* p = nullptr;
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) !=
                cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) !=
                cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess)
            return false;
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(q);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context (looked up once
// per context).
cudaError_t scratch_address(void** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = 0;
    if (!current_context_id(&id)) {
        // no current context yet: the runtime call below makes the device's
        // primary context current, and the cache is keyed by that context
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess) return e;
        if (!current_context_id(&id)) {
            *out = p;
            return cudaSuccess;
        }
    }
    for (int i = 0; i < kMaxDevices; ++i)
        if (g_scratch_cache[i].addr != nullptr && g_scratch_cache[i].ctx_id == id) {
            *out = g_scratch_cache[i].addr;
            return cudaSuccess;
        }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_cache[g_scratch_next] = ScratchEntry{id, p};
    g_scratch_next = (g_scratch_next + 1) % kMaxDevices;
    *out = p;
    return cudaSuccess;
}

// Scratch layout: status | totals [E] | per-block counts [E, ceil(T/32)] |
// per-block prefixes [E, ceil(T/32)] | send-count accumulator [R, R].
struct NoAllocLayout {
    size_t totals, hist, prefix, splits, total;
};

NoAllocLayout noalloc_layout(const moe_config* c) {
    NoAllocLayout L;
    L.totals = kAlignNA;
    L.hist = up256(L.totals + (size_t)c->E * 4);
    L.prefix = up256(L.hist + (size_t)dispatch_blocks(c->T) * c->E * 4);
    L.splits = up256(L.prefix + (size_t)dispatch_blocks(c->T) * c->E * 4);
    L.total = up256(L.splits + (size_t)c->R * c->R * 4);
    return L;
}

inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline bool a4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* x,
                                           const int32_t* topk_idx, void* xp, int32_t* row_token,
                                           int32_t* slot_row, int32_t* expert_counts,
                                           int32_t* expert_offsets, int32_t* rank_counts,
                                           int32_t* rank_splits, int32_t* n_dropped,
                                           uint32_t* device_status, moe_stream_t stream) {
    NvtxRange range("moe_dispatch_noalloc");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (!expert_counts || !expert_offsets || !rank_counts || !n_dropped) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!x || !topk_idx || !xp || !row_token || !slot_row)) return MOE_ERR_INVALID_ARG;
    if (!a16(x) || !a16(xp) || !a4(topk_idx) || !a4(row_token) || !a4(slot_row) ||
        !a4(expert_counts) || !a4(expert_offsets) || !a4(rank_counts) || !a4(rank_splits) ||
        !a4(n_dropped) || !a4(device_status))
        return MOE_ERR_INVALID_ARG;
    const NoAllocLayout L = noalloc_layout(cfg);
    if (L.total > kScratchBytes) return MOE_ERR_INVALID_ARG;  // beyond the fixed scratch size

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
    char* s = static_cast<char*>(base);
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);

    DispatchArgs a;
    a.x = x;
    a.idx = topk_idx;
    a.xp = xp;
    a.row_token = row_token;
    a.slot_row = slot_row;
    a.expert_counts = expert_counts;
    a.expert_offsets = expert_offsets;
    a.rank_counts = rank_counts;
    a.rank_splits = rank_splits;
    a.n_dropped = n_dropped;
    a.status = device_status ? device_status : reinterpret_cast<uint32_t*>(s);
    a.totals = reinterpret_cast<int32_t*>(s + L.totals);
    a.hist = reinterpret_cast<int32_t*>(s + L.hist);
    a.prefix = reinterpret_cast<int32_t*>(s + L.prefix);
    a.splits_acc = reinterpret_cast<int32_t*>(s + L.splits);
    a.T = cfg->T;
    a.d = cfg->d;
    a.E = cfg->E;
    a.k = cfg->k;
    a.R = cfg->R;
    a.dtype = cfg->act_dtype;
    a.C = moe_capacity(cfg);
    return launch_dispatch(a, strm) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
