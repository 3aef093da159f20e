// kernels.h -- host-side launchers of the library's kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// One entry of a partial top-k list (router split over expert slices).
struct RoutePartial {
    float key;  // selection key
    float val;  // logit (softmax) or exact sigmoid score
    int32_t idx;
};
// The tensor-core router splits a tile's experts over up to kRouteSplitMax
// work units when T <= kRouteSplitMaxT and a partial-list buffer is given.
constexpr int kRouteSplitMax = 4;
constexpr int64_t kRouteSplitMaxT = 16384;
// Bytes of that buffer for T tokens and E experts (0: the router never splits).
int64_t route_partial_bytes(int64_t T, int E);

struct RouteArgs {
    const void* x;
    const void* w;
    const float* logit_bias;
    const float* sel_bias;
    int32_t* idx;
    float* gate;
    uint32_t* status;  // device status word (bounded-wait timeouts)
    int64_t T;
    int d, E, k, score, renorm, dtype;
    int R, max_ranks;  // rank-limited routing when 0 < max_ranks < R (tensor-core router)
    RoutePartial* part = nullptr;  // route_partial_bytes(T, E) bytes, or null: no split
};
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
// Tensor-core router (bf16, E <= 256): 0 if supported.
int route_tc_supported(const RouteArgs& a);
cudaError_t launch_route_tc(const RouteArgs& a, cudaStream_t s);

struct DispatchArgs {
    const void* x;
    const int32_t* idx;
    void* xp;
    int32_t* row_token;
    int32_t* slot_row;
    int32_t* expert_counts;
    int32_t* expert_offsets;
    int32_t* rank_counts;
    int32_t* rank_splits;  // may be null
    int32_t* n_dropped;
    // workspace pieces
    uint32_t* status;
    int32_t* totals;      // [E] assignments per expert (before capacity)
    int32_t* hist;        // [E, blocks] per-block assignment counts (blocks <= dispatch_blocks(T))
    int32_t* prefix;      // [E, blocks] exclusive per-expert prefixes over the blocks
    int32_t* splits_acc;  // [R*R] accumulation (used when rank_splits is null)
    int64_t T;
    int d, E, k, R, dtype;
    int64_t C;            // < 0: no limit
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s);
// Upper bound on the token blocks of one dispatch (sizes hist and prefix).
int64_t dispatch_blocks(int64_t T);

struct CombineArgs {
    const void* yp;
    const int32_t* slot_row;
    const float* gate;
    const void* shared;
    const void* resid;
    void* y;
    int64_t T;
    int d, k, dtype;
    int64_t rows_cap = 0;  // rows of yp (the checked build's range of a kept slot_row)
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);  // gate == null: unit gates

struct CombineBwdArgs {
    const void* dy;
    const void* yp;
    const int32_t* slot_row;
    const float* gate;
    void* d_yp;
    float* d_gate;
    int64_t T;
    int d, k, dtype;
    int64_t rows_cap = 0;  // rows of yp / d_yp (checked build)
};
cudaError_t launch_combine_backward(const CombineBwdArgs& a, cudaStream_t s);

// Checked build: copies offsets [G+1] to out, clamped to be non-decreasing
// within [0, rows_cap], and sets MOE_DEV_BOUNDS in *status if anything changed.
cudaError_t launch_sanitize_offsets(const int32_t* in, int32_t* out, int G, int64_t rows_cap,
                                    uint32_t* status, cudaStream_t s);
// Checked build: the library-wide bounds word of calls without a workspace,
// OR-ed into *out and cleared (after the stream's work); unchecked: nothing.
cudaError_t take_checked_status(uint32_t* out, cudaStream_t s);

// Epilogue of one grouped GEMM: out = epi(A . B^T).
enum Epilogue { EPI_NONE = 0, EPI_GELU = 1, EPI_SWIGLU = 2 };

struct GemmArgs {
    const void* A;          // [rows_cap, K] row-major
    const void* B;          // [G, b_rows, K] row-major (b_rows = N, or 2N for SwiGLU)
    void* out;              // [rows_cap, N]
    const int32_t* offsets; // [G+1] device row offsets, or null: one group of m_rows rows
    int64_t rows_cap;       // rows the A/out buffers hold
    int64_t m_rows;         // rows of the single group when offsets is null
    int G, N, K, epi, dtype;
    uint32_t* status;
    // K-grouped mode (tensor-core kernel only): out[g] [rows_cap, N] = A[:, Kg] . B[:, Kg]^T
    // where A is [rows_cap, K], B is [N, K] and group g owns the 64-aligned K range
    // that ceil((offsets[g+1]-offsets[g]) / 64) blocks take after the previous groups'.
    int kgrouped = 0;
    // MN-major B (tensor-core kernel, no epilogue): B is [G, K, N] row-major, i.e.
    // out = A . B[g] with the weights read as stored.
    int b_mn = 0;
    // Failure-detection hook: CTA 0 never loads K block stall_kb of its first
    // tile (-1: off); wait_ns bounds every pipeline wait (0: the 4 s default).
    int stall_kb = -1;
    uint64_t wait_ns = 0;
    // fp32 on the tensor cores (3xTF32 kernel): A and B are the tf32 high parts of
    // the fp32 operands and A_lo / B_lo their low parts (same shapes, see
    // launch_tf32_split).  out_lo non-null: the output is stored split, its tf32
    // high part in out and its low part in out_lo (the up projection's h, which
    // the down projection reads as its A and A_lo).
    const void* A_lo = nullptr;
    const void* B_lo = nullptr;
    void* out_lo = nullptr;
};
cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t s);
// Returns 0 if the tensor-core grouped GEMM supports the shape, else non-zero.
int gemm_tc_supported(const GemmArgs& a);
// fp32 grouped GEMM on the tensor cores as three tf32 products (ffn_tf32.cu):
// row-offset mode, K-major B, any epilogue.  0 if supported.
int gemm_x3_supported(const GemmArgs& a);
cudaError_t launch_gemm_x3(const GemmArgs& a, cudaStream_t s);
// Splits up to three fp32 arrays x (n elements each, n % 4 == 0, 16-byte
// aligned) into tf32 high and low parts: hi = rn_tf32(x), lo = rn_tf32(x - hi)
// (non-finite x: hi = x, lo = 0).  One launch; null src skips a job.
struct Tf32SplitJob {
    const float* src = nullptr;
    float* hi = nullptr;
    float* lo = nullptr;
    int64_t n = 0;
};
cudaError_t launch_tf32_split(const Tf32SplitJob* jobs, int njobs, cudaStream_t s);

// Backward through the expert FFNs (input gradient, optional weight gradients).
struct FfnBwdArgs {
    const void* xp;          // [rows_cap, d]
    const int32_t* offsets;  // [E+1] device
    const void* w_up;        // [E, up_rows, d]
    const void* w_down;      // [E, d, f]
    const void* d_yp;        // [rows_cap, d]
    void* d_xp;              // [rows_cap, d]
    void* d_w_up;            // [E, up_rows, d] or null
    void* d_w_down;          // [E, d, f] or null
    void* scratch;           // ffn_backward_scratch_bytes
    uint32_t* status;
    int64_t rows_cap;
    int E, d, f, epi, dtype;
};
size_t ffn_backward_scratch_bytes(int64_t rows_cap, int E, int d, int f, int gated, int eb,
                                  int weight_grads);
cudaError_t launch_ffn_backward(const FfnBwdArgs& a, cudaStream_t s);

// Backward of the router through its gates (route_bwd.cu).
struct RouteBwdArgs {
    const void* x;          // [T, d]
    const void* w;          // [E, d]
    const float* logit_bias;
    const int32_t* idx;     // [T, k]
    const float* d_gate;    // [T, k]
    float* d_logits;        // [T, E]
    void* dx;               // [T, d] or null
    void* d_w;              // [E, d] or null
    float* d_logit_bias;    // [E] or null
    int64_t T;
    int d, E, k, score, renorm, dtype;
};
cudaError_t launch_route_backward(const RouteBwdArgs& a, cudaStream_t s);

cudaError_t launch_update_sel_bias(const int32_t* counts, float* bias, int E, int64_t T, int k,
                                   float gamma, cudaStream_t s);

}  // namespace moe
