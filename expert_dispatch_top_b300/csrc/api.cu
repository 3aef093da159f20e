// api.cu -- the C ABI declared in include/moe.h: argument checks, workspace
// layout and the launch sequence of each step.  Host code only; every step of
// the layer runs in the library's own kernels on the caller's stream.
#include <math.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Kernel launches enqueued since the library loaded (all threads and devices).
std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxRanks = 32;

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

inline int elem_bytes(const moe_config* c) { return c->act_dtype == MOE_DTYPE_F32 ? 4 : 2; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

int64_t capacity_of(const moe_config* c) {
    if (c->capacity > 0) return c->capacity;
    if (c->capacity_factor > 0.f)
        return (int64_t)ceil((double)c->capacity_factor * (double)c->T * (double)c->k / (double)c->E);
    return -1;
}

int64_t max_rows_of(const moe_config* c) {
    const int64_t tk = (int64_t)c->T * c->k;
    const int64_t C = capacity_of(c);
    if (C < 0) return tk;
    const int64_t ec = (int64_t)c->E * C;
    return ec < tk ? ec : tk;
}

// Byte offsets of every workspace section.
struct Layout {
    size_t status = 0;
    size_t totals, hist, prefix, splits_acc, route_part, safe_offsets;
    size_t topk_idx, topk_gate, slot_row, row_token, expert_counts, offsets, rank_counts,
        rank_splits, n_dropped;
    // fp32 experts on the tensor cores: tf32 high and low parts of the GEMM operands
    size_t x3_a_hi, x3_a_lo, x3_wu_hi, x3_wu_lo, x3_wd_hi, x3_wd_lo, x3_h_lo;
    size_t total;
};

// fp32 experts whose contraction lengths (d for the up projection, d_ff for
// the down projection) are multiples of 16 -- the 3xTF32 kernel's K per stage
// -- run on the tensor cores as three tf32 products (ffn_tf32.cu); other fp32
// shapes run on FFMA (ffn_simt.cu).
inline bool ffn_uses_x3(const moe_config* c) {
    return c->act_dtype == MOE_DTYPE_F32 && c->act != MOE_ACT_IDENTITY && c->d % 16 == 0 &&
           c->d_ff % 16 == 0;
}

Layout layout_of(const moe_config* c) {
    Layout L;
    size_t o = kAlign;
    L.totals = o;
    o = align_up(o + (size_t)c->E * 4);
    L.hist = o;
    o = align_up(o + (size_t)dispatch_blocks(c->T) * c->E * 4);
    L.prefix = o;
    o = align_up(o + (size_t)dispatch_blocks(c->T) * c->E * 4);
    L.splits_acc = o;
    o = align_up(o + (size_t)c->R * c->R * 4);
    // partial top-k lists of a bf16 router that splits its experts (small T)
    L.route_part = o;
    if (c->act_dtype == MOE_DTYPE_BF16) o = align_up(o + (size_t)route_partial_bytes(c->T, c->E));
    // checked build: the sanitised copy of expert_offsets the FFN kernels read
    L.safe_offsets = o;
    o = align_up(o + (size_t)(c->E + 1) * 4);
    const size_t tk = (size_t)c->T * c->k;
    L.topk_idx = o;
    o = align_up(o + tk * 4);
    L.topk_gate = o;
    o = align_up(o + tk * 4);
    L.slot_row = o;
    o = align_up(o + tk * 4);
    L.row_token = o;
    o = align_up(o + (size_t)max_rows_of(c) * 4);
    L.expert_counts = o;
    o = align_up(o + (size_t)c->E * 4);
    L.offsets = o;
    o = align_up(o + (size_t)(c->E + 1) * 4);
    L.rank_counts = o;
    o = align_up(o + (size_t)c->R * 4);
    L.rank_splits = o;
    o = align_up(o + (size_t)c->R * c->R * 4);
    L.n_dropped = o;
    o = align_up(o + 4);
    L.x3_a_hi = L.x3_a_lo = L.x3_wu_hi = L.x3_wu_lo = L.x3_wd_hi = L.x3_wd_lo = L.x3_h_lo = o;
    if (ffn_uses_x3(c)) {
        // rows of A: the routed rows, or the shared expert's T rows (the passes
        // run one after the other and reuse these sections)
        const int64_t mr = max_rows_of(c);
        const size_t arows = (size_t)(c->n_shared == 1 && c->T > mr ? c->T : mr);
        const size_t up_rows = (size_t)(c->act == MOE_ACT_SWIGLU ? 2 : 1) * c->d_ff;
        const size_t a = arows * c->d * 4, wu = (size_t)c->E * up_rows * c->d * 4;
        const size_t wd = (size_t)c->E * c->d * c->d_ff * 4, h = arows * c->d_ff * 4;
        size_t* sec[7] = {&L.x3_a_hi, &L.x3_a_lo, &L.x3_wu_hi, &L.x3_wu_lo,
                          &L.x3_wd_hi, &L.x3_wd_lo, &L.x3_h_lo};
        const size_t len[7] = {a, a, wu, wu, wd, wd, h};
        for (int i = 0; i < 7; ++i) {
            *sec[i] = o;
            o = align_up(o + len[i]);
        }
    }
    L.total = o;
    return L;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_ffn_config(const moe_config* c) {
    if (c->act == MOE_ACT_IDENTITY) return c->n_shared == 0 ? MOE_OK : MOE_ERR_INVALID_ARG;
    if (c->d_ff < 1 || ((int64_t)c->d_ff * elem_bytes(c)) % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (c->act_dtype == MOE_DTYPE_BF16 && (c->d % 64 != 0 || c->d_ff % 64 != 0))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Each *_impl checks its arguments first and, unless check_only, enqueues its
// kernels.  moe_layer_forward runs every step's checks before the first
// launch, so an argument error never leaves part of the layer enqueued.
moe_status route_impl(const moe_config* c, const void* x, const void* w, const float* lb,
                      const float* sb, int32_t* idx, float* gate, void* ws, cudaStream_t s,
                      bool check_only = false) {
    if (c->T == 0) return MOE_OK;
    if (!x || !w || !idx || !gate || !ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned4(idx) || !aligned4(gate) || !aligned4(lb) ||
        !aligned4(sb))
        return MOE_ERR_INVALID_ARG;
    if (sb && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_UNSUPPORTED;
    const bool limited = c->max_ranks > 0 && c->max_ranks < c->R;
    if (check_only) return MOE_OK;
    const Layout L0 = layout_of(c);
    RouteArgs a;
    a.x = x;
    a.w = w;
    a.logit_bias = lb;
    a.sel_bias = sb;
    a.idx = idx;
    a.gate = gate;
    a.status = at<uint32_t>(ws, L0.status);
    a.T = c->T;
    a.d = c->d;
    a.E = c->E;
    a.k = c->k;
    a.score = c->score;
    a.renorm = c->renorm;
    a.dtype = c->act_dtype;
    a.R = c->R;
    a.max_ranks = limited ? c->max_ranks : 0;
    if (c->act_dtype == MOE_DTYPE_BF16 && route_partial_bytes(c->T, c->E) > 0)
        a.part = at<RoutePartial>(ws, L0.route_part);
    return cuda_status(launch_route(a, s));
}

moe_status dispatch_impl(const moe_config* c, const void* x, const int32_t* idx, void* xp,
                         int32_t* row_token, int32_t* slot_row, int32_t* counts, int32_t* offsets,
                         int32_t* rank_counts, int32_t* rank_splits, int32_t* n_dropped, void* ws,
                         cudaStream_t s, bool check_only = false) {
    if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !rank_counts || !n_dropped) return MOE_ERR_INVALID_ARG;
    if (c->T > 0 && (!x || !idx || !xp || !row_token || !slot_row)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xp) || !aligned4(idx) || !aligned4(row_token) ||
        !aligned4(slot_row) || !aligned4(counts) || !aligned4(offsets) || !aligned4(rank_counts) ||
        !aligned4(rank_splits) || !aligned4(n_dropped))
        return MOE_ERR_INVALID_ARG;
    if (check_only) return MOE_OK;
    const Layout L = layout_of(c);
    DispatchArgs a;
    a.x = x;
    a.idx = idx;
    a.xp = xp;
    a.row_token = row_token;
    a.slot_row = slot_row;
    a.expert_counts = counts;
    a.expert_offsets = offsets;
    a.rank_counts = rank_counts;
    a.rank_splits = rank_splits;
    a.n_dropped = n_dropped;
    a.status = at<uint32_t>(ws, L.status);
    a.totals = at<int32_t>(ws, L.totals);
    a.hist = at<int32_t>(ws, L.hist);
    a.prefix = at<int32_t>(ws, L.prefix);
    a.splits_acc = at<int32_t>(ws, L.splits_acc);
    a.T = c->T;
    a.d = c->d;
    a.E = c->E;
    a.k = c->k;
    a.R = c->R;
    a.dtype = c->act_dtype;
    a.C = capacity_of(c);
    return cuda_status(launch_dispatch(a, s));
}

moe_status ffn_impl(const moe_config* c, const void* xp, const int32_t* offsets, const void* w_up,
                    const void* w_down, void* h, void* yp, const void* shared_x,
                    const void* shared_up, const void* shared_down, void* shared_h,
                    void* shared_out, void* ws, cudaStream_t s, bool check_only = false) {
    if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    const int64_t rows = max_rows_of(c);
    const int eb = elem_bytes(c);
    if (c->act == MOE_ACT_IDENTITY) {
        if (!xp || !yp) return rows == 0 ? MOE_OK : MOE_ERR_INVALID_ARG;
        if (xp == yp || rows == 0 || check_only) return MOE_OK;
        return cuda_status(cudaMemcpyAsync(yp, xp, (size_t)rows * c->d * eb,
                                           cudaMemcpyDeviceToDevice, s));
    }
    if (!offsets || !w_up || !w_down || !aligned4(offsets) || !aligned16(w_up) || !aligned16(w_down))
        return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!xp || !h || !yp || !aligned16(xp) || !aligned16(h) || !aligned16(yp)))
        return MOE_ERR_INVALID_ARG;
    if (c->n_shared == 1 && c->T > 0) {
        if (!shared_x || !shared_up || !shared_down || !shared_h || !shared_out ||
            !aligned16(shared_x) || !aligned16(shared_up) || !aligned16(shared_down) ||
            !aligned16(shared_h) || !aligned16(shared_out))
            return MOE_ERR_INVALID_ARG;
    }
    const Layout L = layout_of(c);
    uint32_t* status = at<uint32_t>(ws, L.status);
    const bool tc = c->act_dtype == MOE_DTYPE_BF16;
    const bool x3 = ffn_uses_x3(c);
    if (kChecked && !check_only) {
        // checked build: the kernels read a copy made non-decreasing within the rows
        int32_t* safe = at<int32_t>(ws, L.safe_offsets);
        if (launch_sanitize_offsets(offsets, safe, c->E, rows, status, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        offsets = safe;
    }
    // One up/down pair per expert set: routed experts (device offsets), then the
    // shared expert over all T rows of shared_x.  Every pair is checked before
    // the first launch.
    const int npass = 1 + (c->n_shared == 1 ? 1 : 0);
    GemmArgs up[2], down[2];
    for (int pass = 0; pass < npass; ++pass) {
        const bool shared = pass == 1;
        GemmArgs& u = up[pass];
        u.A = shared ? shared_x : xp;
        u.B = shared ? shared_up : w_up;
        u.out = shared ? shared_h : h;
        u.offsets = shared ? nullptr : offsets;
        u.rows_cap = shared ? c->T : rows;
        u.m_rows = shared ? c->T : 0;
        u.G = shared ? 1 : c->E;
        u.N = c->d_ff;
        u.K = c->d;
        u.epi = c->act == MOE_ACT_SWIGLU ? EPI_SWIGLU : EPI_GELU;
        u.dtype = c->act_dtype;
        u.status = status;
        GemmArgs& dn = down[pass];
        dn = u;
        dn.A = shared ? shared_h : h;
        dn.B = shared ? shared_down : w_down;
        dn.out = shared ? shared_out : yp;
        dn.N = c->d;
        dn.K = c->d_ff;
        dn.epi = EPI_NONE;
        if (x3) {
            // both GEMMs read the tf32 split of their operands; the up projection
            // stores h split (high part in h, low part in the workspace), which the
            // down projection reads
            u.A = at<float>(ws, L.x3_a_hi);
            u.A_lo = at<float>(ws, L.x3_a_lo);
            u.B = at<float>(ws, L.x3_wu_hi);
            u.B_lo = at<float>(ws, L.x3_wu_lo);
            u.out_lo = at<float>(ws, L.x3_h_lo);
            dn.A_lo = u.out_lo;
            dn.B = at<float>(ws, L.x3_wd_hi);
            dn.B_lo = at<float>(ws, L.x3_wd_lo);
        }
        if (u.rows_cap > 0 && tc && (gemm_tc_supported(u) != 0 || gemm_tc_supported(dn) != 0))
            return MOE_ERR_UNSUPPORTED;
        if (u.rows_cap > 0 && x3 && (gemm_x3_supported(u) != 0 || gemm_x3_supported(dn) != 0))
            return MOE_ERR_UNSUPPORTED;
    }
    if (check_only) return MOE_OK;
    for (int pass = 0; pass < npass; ++pass) {
        if (up[pass].rows_cap == 0) continue;
        cudaError_t e;
        if (x3) {
            // this expert set's input rows and weights, split into the workspace
            const bool shared = pass == 1;
            const int64_t up_rows = (int64_t)(c->act == MOE_ACT_SWIGLU ? 2 : 1) * c->d_ff;
            Tf32SplitJob j[3];
            j[0].src = static_cast<const float*>(shared ? shared_x : xp);
            j[0].n = up[pass].rows_cap * c->d;
            j[1].src = static_cast<const float*>(shared ? shared_up : w_up);
            j[1].n = (int64_t)up[pass].G * up_rows * c->d;
            j[2].src = static_cast<const float*>(shared ? shared_down : w_down);
            j[2].n = (int64_t)up[pass].G * c->d * c->d_ff;
            const size_t hi[3] = {L.x3_a_hi, L.x3_wu_hi, L.x3_wd_hi};
            const size_t lo[3] = {L.x3_a_lo, L.x3_wu_lo, L.x3_wd_lo};
            for (int i = 0; i < 3; ++i) {
                j[i].hi = at<float>(ws, hi[i]);
                j[i].lo = at<float>(ws, lo[i]);
            }
            e = launch_tf32_split(j, 3, s);
            if (e == cudaSuccess) e = launch_gemm_x3(up[pass], s);
            if (e == cudaSuccess) e = launch_gemm_x3(down[pass], s);
        } else {
            e = tc ? launch_gemm_tc(up[pass], s) : launch_gemm_simt(up[pass], s);
            if (e == cudaSuccess) e = tc ? launch_gemm_tc(down[pass], s) : launch_gemm_simt(down[pass], s);
        }
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status combine_impl(const moe_config* c, const void* yp, const int32_t* slot_row,
                        const float* gate, const void* shared_out, const void* resid, void* y,
                        cudaStream_t s, bool check_only = false) {
    if (c->T == 0) return MOE_OK;
    if (!yp || !slot_row || !gate || !y) return MOE_ERR_INVALID_ARG;
    if (c->add_residual && !resid) return MOE_ERR_INVALID_ARG;
    if (c->n_shared == 1 && !shared_out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(yp) || !aligned16(y) || !aligned16(shared_out) || !aligned16(resid) ||
        !aligned4(slot_row) || !aligned4(gate))
        return MOE_ERR_INVALID_ARG;
    if (check_only) return MOE_OK;
    CombineArgs a;
    a.yp = yp;
    a.slot_row = slot_row;
    a.gate = gate;
    a.shared = c->n_shared == 1 ? shared_out : nullptr;
    a.resid = c->add_residual ? resid : nullptr;
    a.y = y;
    a.T = c->T;
    a.d = c->d;
    a.k = c->k;
    a.dtype = c->act_dtype;
    a.rows_cap = max_rows_of(c);
    return cuda_status(launch_combine(a, s));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: unsupported combination";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA call or launch failed";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait gave up";
        case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE: non-finite input";
        case MOE_ERR_BOUNDS: return "MOE_ERR_BOUNDS: index out of range";
    }
    return "unknown moe_status";
}

moe_status moe_check_config(const moe_config* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->d < 1 || c->d > 16384 || c->E < 1 || c->E > 256 || c->k < 1 || c->k > 8 ||
        c->k > c->E || c->R < 1 || c->R > kMaxRanks || c->E % c->R != 0)
        return MOE_ERR_INVALID_ARG;
    if ((int64_t)c->T * c->k >= (1ll << 30)) return MOE_ERR_INVALID_ARG;
    if (c->act_dtype != MOE_DTYPE_F32 && c->act_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (c->act != MOE_ACT_GELU && c->act != MOE_ACT_SWIGLU && c->act != MOE_ACT_IDENTITY)
        return MOE_ERR_INVALID_ARG;
    if ((c->renorm != 0 && c->renorm != 1) || (c->add_residual != 0 && c->add_residual != 1))
        return MOE_ERR_INVALID_ARG;
    if (c->n_shared < 0 || c->n_shared > 1) return MOE_ERR_INVALID_ARG;
    if (c->capacity < 0 || !(c->capacity_factor == c->capacity_factor)) return MOE_ERR_INVALID_ARG;
    if (c->max_ranks < 0 || c->max_ranks > c->R ||
        (c->max_ranks > 0 && (int64_t)c->max_ranks * (c->E / c->R) < c->k))
        return MOE_ERR_INVALID_ARG;
    if (((int64_t)c->d * elem_bytes(c)) % 16 != 0) return MOE_ERR_INVALID_ARG;
    return check_ffn_config(c);
}

size_t moe_workspace_size(const moe_config* cfg) {
    if (moe_check_config(cfg) != MOE_OK) return 0;
    return layout_of(cfg).total;
}

int64_t moe_capacity(const moe_config* cfg) {
    if (moe_check_config(cfg) != MOE_OK) return -1;
    return capacity_of(cfg);
}

int64_t moe_max_rows(const moe_config* cfg) {
    if (moe_check_config(cfg) != MOE_OK) return -1;
    return max_rows_of(cfg);
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* w_router,
                     const float* logit_bias, const float* sel_bias, int32_t* topk_idx,
                     float* topk_gate, void* ws, moe_stream_t stream) {
    NvtxRange range("moe_route");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    return route_impl(cfg, x, w_router, logit_bias, sel_bias, topk_idx, topk_gate, ws,
                      reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx, void* xp,
                        int32_t* row_token, int32_t* slot_row, int32_t* expert_counts,
                        int32_t* expert_offsets, int32_t* rank_counts, int32_t* rank_splits,
                        int32_t* n_dropped, void* ws, moe_stream_t stream) {
    NvtxRange range("moe_dispatch");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    return dispatch_impl(cfg, x, topk_idx, xp, row_token, slot_row, expert_counts, expert_offsets,
                         rank_counts, rank_splits, n_dropped, ws,
                         reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_test_expert_ffn_stall(const moe_config* cfg, const void* xp,
                                     const int32_t* expert_offsets, const void* w_up, void* h,
                                     int32_t stall_kb, uint32_t wait_limit_us, void* ws,
                                     moe_stream_t stream) {
    NvtxRange range("moe_test_expert_ffn_stall");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_ffn_config(cfg)) != MOE_OK) return st;
    if (cfg->act_dtype != MOE_DTYPE_BF16 || cfg->act == MOE_ACT_IDENTITY) return MOE_ERR_UNSUPPORTED;
    if (stall_kb < 0 || stall_kb >= cfg->d / 64 || wait_limit_us == 0 || wait_limit_us > 4000000u)
        return MOE_ERR_INVALID_ARG;
    const int64_t rows = max_rows_of(cfg);
    if (rows == 0 || !ws || !aligned16(ws) || !xp || !expert_offsets || !w_up || !h ||
        !aligned16(xp) || !aligned4(expert_offsets) || !aligned16(w_up) || !aligned16(h))
        return MOE_ERR_INVALID_ARG;
    GemmArgs g;
    g.A = xp;
    g.B = w_up;
    g.out = h;
    g.offsets = expert_offsets;
    g.rows_cap = rows;
    g.m_rows = 0;
    g.G = cfg->E;
    g.N = cfg->d_ff;
    g.K = cfg->d;
    g.epi = cfg->act == MOE_ACT_SWIGLU ? EPI_SWIGLU : EPI_GELU;
    g.dtype = cfg->act_dtype;
    g.status = at<uint32_t>(ws, layout_of(cfg).status);
    g.stall_kb = stall_kb;
    g.wait_ns = (uint64_t)wait_limit_us * 1000ull;
    if (gemm_tc_supported(g) != 0) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_gemm_tc(g, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* expert_offsets,
                          const void* w_up, const void* w_down, void* h, void* yp,
                          const void* shared_x, const void* shared_up, const void* shared_down,
                          void* shared_h, void* shared_out, void* ws, moe_stream_t stream) {
    NvtxRange range("moe_expert_ffn");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    return ffn_impl(cfg, xp, expert_offsets, w_up, w_down, h, yp, shared_x, shared_up, shared_down,
                    shared_h, shared_out, ws, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot_row,
                       const float* topk_gate, const void* shared_out, const void* x_residual,
                       void* y, moe_stream_t stream) {
    NvtxRange range("moe_combine");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    return combine_impl(cfg, yp, slot_row, topk_gate, shared_out, x_residual, y,
                        reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace moe {
namespace {

// The layer's four steps; with check_only, every step's argument checks and
// nothing else (so a caller can check before enqueueing anything of its own).
moe_status layer_impl(const moe_config* cfg, const void* x, const void* w_router,
                      const float* logit_bias, const float* sel_bias, const void* w_up,
                      const void* w_down, const void* shared_up, const void* shared_down,
                      const moe_buffers* buf, void* y, void* ws, cudaStream_t s, bool check_only) {
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (!buf || !ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    const Layout L = layout_of(cfg);
    int32_t* idx = buf->topk_idx ? buf->topk_idx : at<int32_t>(ws, L.topk_idx);
    float* gate = buf->topk_gate ? buf->topk_gate : at<float>(ws, L.topk_gate);
    int32_t* slot_row = buf->slot_row ? buf->slot_row : at<int32_t>(ws, L.slot_row);
    int32_t* row_token = buf->row_token ? buf->row_token : at<int32_t>(ws, L.row_token);
    int32_t* counts = buf->expert_counts ? buf->expert_counts : at<int32_t>(ws, L.expert_counts);
    int32_t* offsets = buf->expert_offsets ? buf->expert_offsets : at<int32_t>(ws, L.offsets);
    int32_t* rank_counts = buf->rank_counts ? buf->rank_counts : at<int32_t>(ws, L.rank_counts);
    int32_t* rank_splits = buf->rank_splits ? buf->rank_splits : at<int32_t>(ws, L.rank_splits);
    int32_t* n_dropped = buf->n_dropped ? buf->n_dropped : at<int32_t>(ws, L.n_dropped);
    const bool identity = cfg->act == MOE_ACT_IDENTITY;
    if (!buf->xp || (!identity && (!buf->h || !buf->yp))) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared == 1 && (!shared_up || !shared_down || !buf->shared_h || !buf->shared_out))
        return MOE_ERR_INVALID_ARG;
    if (!y || (cfg->T > 0 && !x)) return MOE_ERR_INVALID_ARG;

    // Every step's checks first: an argument error returns before any launch.
    const void* yp = identity ? buf->xp : buf->yp;
    for (int pass = 0; pass < (check_only ? 1 : 2); ++pass) {
        const bool check = pass == 0;
        st = route_impl(cfg, x, w_router, logit_bias, sel_bias, idx, gate, ws, s, check);
        if (st != MOE_OK) return st;
        st = dispatch_impl(cfg, x, idx, buf->xp, row_token, slot_row, counts, offsets, rank_counts,
                           rank_splits, n_dropped, ws, s, check);
        if (st != MOE_OK) return st;
        if (!identity) {
            st = ffn_impl(cfg, buf->xp, offsets, w_up, w_down, buf->h, buf->yp, x, shared_up,
                          shared_down, buf->shared_h, buf->shared_out, ws, s, check);
            if (st != MOE_OK) return st;
        }
        st = combine_impl(cfg, yp, slot_row, gate, buf->shared_out, x, y, s, check);
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_layer_forward(const moe_config* cfg, const void* x, const void* w_router,
                             const float* logit_bias, const float* sel_bias, const void* w_up,
                             const void* w_down, const void* shared_up, const void* shared_down,
                             const moe_buffers* buf, void* y, void* ws, moe_stream_t stream) {
    NvtxRange range("moe_layer_forward");
    return layer_impl(cfg, x, w_router, logit_bias, sel_bias, w_up, w_down, shared_up, shared_down,
                      buf, y, ws, reinterpret_cast<cudaStream_t>(stream), false);
}

moe_status moe_layer_forward_host(const moe_config* cfg, const void* x_host, void* x_dev,
                                  const void* w_router, const float* logit_bias,
                                  const float* sel_bias, const void* w_up, const void* w_down,
                                  const void* shared_up, const void* shared_down,
                                  const moe_buffers* buf, void* y_dev, void* y_host, void* ws,
                                  moe_stream_t stream) {
    NvtxRange range("moe_layer_forward_host");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (cfg->T > 0 && (!x_host || !y_host || !x_dev || !y_dev)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the layer's checks before the input copy is enqueued
    st = layer_impl(cfg, x_dev, w_router, logit_bias, sel_bias, w_up, w_down, shared_up,
                    shared_down, buf, y_dev, ws, s, true);
    if (st != MOE_OK) return st;
    const size_t bytes = (size_t)cfg->T * cfg->d * elem_bytes(cfg);
    if (bytes && cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    st = layer_impl(cfg, x_dev, w_router, logit_bias, sel_bias, w_up, w_down, shared_up,
                    shared_down, buf, y_dev, ws, s, false);
    if (st != MOE_OK) return st;
    if (bytes && cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_route_backward(const moe_config* cfg, const void* x, const void* w_router,
                              const float* logit_bias, const int32_t* topk_idx,
                              const float* d_gate, float* d_logits, void* dx, void* d_w_router,
                              float* d_logit_bias, moe_stream_t stream) {
    NvtxRange range("moe_route_backward");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) {
        // no tokens: the weight and bias gradients are zero
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d_w_router && !aligned16(d_w_router)) return MOE_ERR_INVALID_ARG;
        if (d_w_router && cudaMemsetAsync(d_w_router, 0, (size_t)cfg->E * cfg->d * elem_bytes(cfg),
                                          s) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (d_logit_bias && cudaMemsetAsync(d_logit_bias, 0, (size_t)cfg->E * 4, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!x || !w_router || !topk_idx || !d_gate || !d_logits) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(dx) || !aligned16(d_w_router) ||
        !aligned4(logit_bias) || !aligned4(topk_idx) || !aligned4(d_gate) || !aligned4(d_logits) ||
        !aligned4(d_logit_bias))
        return MOE_ERR_INVALID_ARG;
    RouteBwdArgs a;
    a.x = x;
    a.w = w_router;
    a.logit_bias = logit_bias;
    a.idx = topk_idx;
    a.d_gate = d_gate;
    a.d_logits = d_logits;
    a.dx = dx;
    a.d_w = d_w_router;
    a.d_logit_bias = d_logit_bias;
    a.T = cfg->T;
    a.d = cfg->d;
    a.E = cfg->E;
    a.k = cfg->k;
    a.score = cfg->score;
    a.renorm = cfg->renorm;
    a.dtype = cfg->act_dtype;
    return cuda_status(launch_route_backward(a, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_backward(const moe_config* cfg, const void* dy, const void* yp,
                                const int32_t* slot_row, const float* topk_gate, void* d_yp,
                                float* d_gate, moe_stream_t stream) {
    NvtxRange range("moe_combine_backward");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    if (!dy || !yp || !slot_row || !topk_gate || !d_yp || !d_gate) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(yp) || !aligned16(d_yp) || !aligned4(slot_row) ||
        !aligned4(topk_gate) || !aligned4(d_gate))
        return MOE_ERR_INVALID_ARG;
    CombineBwdArgs a;
    a.dy = dy;
    a.yp = yp;
    a.slot_row = slot_row;
    a.gate = topk_gate;
    a.d_yp = d_yp;
    a.d_gate = d_gate;
    a.T = cfg->T;
    a.d = cfg->d;
    a.k = cfg->k;
    a.dtype = cfg->act_dtype;
    a.rows_cap = max_rows_of(cfg);
    return cuda_status(launch_combine_backward(a, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_backward(const moe_config* cfg, const void* d_xp, const int32_t* slot_row,
                                 void* dx, moe_stream_t stream) {
    NvtxRange range("moe_dispatch_backward");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    if (!d_xp || !slot_row || !dx || !aligned16(d_xp) || !aligned16(dx) || !aligned4(slot_row))
        return MOE_ERR_INVALID_ARG;
    CombineArgs a;
    a.yp = d_xp;
    a.slot_row = slot_row;
    a.gate = nullptr;  // the plain sum of the token's kept rows
    a.shared = nullptr;
    a.resid = nullptr;
    a.y = dx;
    a.T = cfg->T;
    a.d = cfg->d;
    a.k = cfg->k;
    a.dtype = cfg->act_dtype;
    a.rows_cap = max_rows_of(cfg);
    return cuda_status(launch_combine(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_expert_ffn_backward_scratch_size(const moe_config* cfg, int weight_grads) {
    if (moe_check_config(cfg) != MOE_OK || check_ffn_config(cfg) != MOE_OK) return 0;
    if (cfg->act == MOE_ACT_IDENTITY) return 0;
    return ffn_backward_scratch_bytes(max_rows_of(cfg), cfg->E, cfg->d, cfg->d_ff,
                                      cfg->act == MOE_ACT_SWIGLU, elem_bytes(cfg), weight_grads != 0);
}

moe_status moe_expert_ffn_backward(const moe_config* cfg, const void* xp,
                                   const int32_t* expert_offsets, const void* w_up,
                                   const void* w_down, const void* d_yp, void* d_xp, void* d_w_up,
                                   void* d_w_down, void* scratch, size_t scratch_bytes, void* ws,
                                   moe_stream_t stream) {
    NvtxRange range("moe_expert_ffn_backward");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_ffn_config(cfg)) != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows = max_rows_of(cfg);
    const int eb = elem_bytes(cfg);
    if (cfg->act == MOE_ACT_IDENTITY) {
        // identity experts: d_xp = d_yp, no weights
        if (d_w_up || d_w_down) return MOE_ERR_INVALID_ARG;
        if (rows == 0) return MOE_OK;
        if (!d_yp || !d_xp) return MOE_ERR_INVALID_ARG;
        if (d_yp == d_xp) return MOE_OK;
        return cuda_status(
            cudaMemcpyAsync(d_xp, d_yp, (size_t)rows * cfg->d * eb, cudaMemcpyDeviceToDevice, s));
    }
    if (!ws || !aligned16(ws) || !expert_offsets || !aligned4(expert_offsets) || !w_up || !w_down ||
        !aligned16(w_up) || !aligned16(w_down) || !aligned16(d_w_up) || !aligned16(d_w_down))
        return MOE_ERR_INVALID_ARG;
    const bool wg = d_w_up || d_w_down;
    if (scratch_bytes < moe_expert_ffn_backward_scratch_size(cfg, wg) || !scratch ||
        (reinterpret_cast<uintptr_t>(scratch) & 255))
        return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!xp || !d_yp || !d_xp || !aligned16(xp) || !aligned16(d_yp) || !aligned16(d_xp)))
        return MOE_ERR_INVALID_ARG;
    if (cfg->act_dtype == MOE_DTYPE_BF16 && cfg->E > 256) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) {
        // no routed rows: the weight gradients are zero
        if (d_w_up && cudaMemsetAsync(d_w_up, 0, (size_t)cfg->E * (cfg->act == MOE_ACT_SWIGLU ? 2 : 1) *
                                                     cfg->d_ff * cfg->d * eb, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (d_w_down &&
            cudaMemsetAsync(d_w_down, 0, (size_t)cfg->E * cfg->d * cfg->d_ff * eb, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    uint32_t* status = at<uint32_t>(ws, layout_of(cfg).status);
    if (kChecked) {
        // checked build: the kernels read a copy made non-decreasing within the rows
        int32_t* safe = at<int32_t>(ws, layout_of(cfg).safe_offsets);
        if (launch_sanitize_offsets(expert_offsets, safe, cfg->E, rows, status, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        expert_offsets = safe;
    }
    FfnBwdArgs a;
    a.xp = xp;
    a.offsets = expert_offsets;
    a.w_up = w_up;
    a.w_down = w_down;
    a.d_yp = d_yp;
    a.d_xp = d_xp;
    a.d_w_up = d_w_up;
    a.d_w_down = d_w_down;
    a.scratch = scratch;
    a.status = status;
    a.rows_cap = rows;
    a.E = cfg->E;
    a.d = cfg->d;
    a.f = cfg->d_ff;
    a.epi = cfg->act == MOE_ACT_SWIGLU ? EPI_SWIGLU : EPI_GELU;
    a.dtype = cfg->act_dtype;
    return cuda_status(launch_ffn_backward(a, s));
}

moe_status moe_update_sel_bias(const moe_config* cfg, const int32_t* expert_counts, float* sel_bias,
                               float gamma, moe_stream_t stream) {
    NvtxRange range("moe_update_sel_bias");
    moe_status st = moe_check_config(cfg);
    if (st != MOE_OK) return st;
    if (!expert_counts || !sel_bias || !aligned4(expert_counts) || !aligned4(sel_bias))
        return MOE_ERR_INVALID_ARG;
    if (!(gamma >= 0.f) || gamma == INFINITY) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_update_sel_bias(expert_counts, sel_bias, cfg->E, cfg->T, cfg->k, gamma,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_read_device_status(const void* ws, uint32_t* out, moe_stream_t stream) {
    NvtxRange range("moe_read_device_status");
    if (!ws || !out) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(const_cast<void*>(ws), 0, 4, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = take_checked_status(&v, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *out = v;
    return MOE_OK;
}

int moe_build_checked(void) { return kChecked ? 1 : 0; }

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
