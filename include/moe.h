/*
 * moe.h -- C ABI of the B300 (sm_103a) mixture-of-experts layer hot path.
 *
 * One MoE layer forward pass in the four steps of the Ultralytics glossary
 * page "Expert Parallelism", section "How Tokens Move Between GPUs": Route,
 * Dispatch, Compute, Combine.  On one GPU the two all-to-all exchanges of
 * that section become on-device permutations: dispatch writes an
 * expert-major buffer whose contiguous expert blocks are the virtual
 * expert-parallel ranks (expert e lives on rank e / (E/R), the uniform
 * placement of mbrenndoerfer.com "Expert Parallelism > Summary"), and
 * combine gathers it back into token order.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers on the current CUDA device unless a
 *    parameter says otherwise; the caller owns every buffer.  The library
 *    never allocates or frees device memory and keeps no global state,
 *    except the fixed scratch array that moe_dispatch_noalloc uses.
 *  - Every pointer must be 16-byte aligned; tensors are dense and row-major.
 *  - Activations and expert/router weights share one storage type,
 *    cfg->act_dtype (fp32 or bf16).  Router logits, gates and every
 *    accumulation are fp32.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream).  No entry point synchronises the stream, except
 *    moe_read_device_status.
 *  - Argument errors are returned synchronously before anything is
 *    enqueued.  A failed launch returns MOE_ERR_CUDA.  Errors found on the
 *    device (a bounded wait that timed out, an index out of range) are
 *    recorded in the status word at the start of the workspace and read with
 *    moe_read_device_status.  No entry point traps, aborts or throws.
 *  - Calls on different streams need separate workspaces.
 *
 * Limits: 0 <= T, T*k < 2^30; 1 <= k <= min(E, 8); 1 <= E <= 256; 1 <= R <= 32
 * and E % R == 0; d <= 16384; d a multiple of 8 for bf16 (4 for fp32), and
 * with bf16 GELU or SwiGLU experts d and d_ff multiples of 64
 * (MOE_ERR_UNSUPPORTED otherwise).  moe_layer_forward checks the arguments of
 * all four steps before it enqueues the first one.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (binary-compatible typedef; no CUDA header needed). */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or limit */
    MOE_ERR_UNSUPPORTED = 2,  /* a valid combination this library does not run */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 4,      /* a bounded device wait gave up (status word) */
    MOE_ERR_NONFINITE = 5,    /* a non-finite router logit was seen (status word) */
    MOE_ERR_BOUNDS = 6        /* an index left its range (status word) */
} moe_status;

enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };
enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1, MOE_ACT_IDENTITY = 2 };

/* Bits of the device status word (first 4 bytes of the workspace). */
/* 0x1u: unused */
#define MOE_DEV_GEMM_TIMEOUT 0x2u     /* a tensor-core pipeline wait (expert GEMM or router) gave up */
#define MOE_DEV_BAD_INDEX 0x4u        /* an expert index outside [0, E) reached dispatch */
#define MOE_DEV_COPY_TIMEOUT 0x8u     /* a bulk row copy of dispatch did not land in time */
#define MOE_DEV_NONFINITE 0x10u       /* a router logit was NaN or +-inf (x or w_router holds one) */
#define MOE_DEV_BOUNDS 0x20u          /* checked build only: an index read from a caller's buffer
                                         (slot_row, expert_offsets) was out of range */

/*
 * Layer shape and method switches.
 *   T tokens, d = d_model, E routed experts, k experts per token, R virtual
 *   expert-parallel ranks (contiguous blocks of E/R experts), d_ff expert
 *   hidden size, n_shared always-on shared experts (0 or 1; gate 1, run on
 *   every token -- DeepSeek-V3-style).
 *   score: softmax or sigmoid router scores.  renorm: gates normalised over
 *   the chosen k; otherwise a gate is the full softmax probability or the
 *   plain sigmoid score.
 *   capacity: > 0 is an explicit per-expert capacity C; otherwise
 *   capacity_factor > 0 gives C = ceil(capacity_factor * T * k / E)
 *   (Ultralytics "Load Balancing and Capacity": at most a fixed number of
 *   tokens per expert, e.g. 1.25x the even share); otherwise no limit.
 *   Overflow is decided per (token, expert) assignment in token order.
 *   act: expert FFN form (GELU: down(gelu(up x)); SWIGLU: down(silu(gate x)
 *   * (up x)); IDENTITY: the expert returns its input).  No biases.
 *   add_residual: combine adds x to the MoE output, so a fully dropped token
 *   leaves the layer unchanged.
 *   max_ranks: rank-limited routing (Ultralytics "Load Balancing and
 *   Capacity": DeepSeek-V3 sends each token to experts on at most 4 nodes).
 *   A rank's score is the best selection key among its E/R experts; the
 *   max_ranks best ranks are kept (ties to the lower rank) and the top-k is
 *   taken among their experts.  Needs max_ranks <= R and max_ranks*(E/R) >= k.
 */
typedef struct moe_config {
    int32_t T;
    int32_t d;
    int32_t E;
    int32_t k;
    int32_t R;
    int32_t d_ff;
    int32_t n_shared;
    int32_t act_dtype;      /* MOE_DTYPE_* */
    int32_t score;          /* MOE_SCORE_* */
    int32_t renorm;         /* 0 or 1 */
    float capacity_factor;  /* <= 0: none (unless capacity > 0) */
    int32_t capacity;       /* > 0: explicit per-expert capacity */
    int32_t act;            /* MOE_ACT_* */
    int32_t add_residual;   /* 0 or 1 */
    int32_t max_ranks;      /* > 0: rank-limited routing (see below); 0: no limit */
} moe_config;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status s);

/* Checks cfg against the limits above; MOE_OK or the reason it fails. */
moe_status moe_check_config(const moe_config* cfg);

/* Workspace bytes for cfg (0 if cfg is invalid).  The workspace holds the
   device status word, the dispatch scan state and the default metadata
   arrays of moe_layer_forward, and for fp32 experts on the tensor cores the
   tf32 split of the expert GEMMs' operands (2 x 4 bytes per element of the
   input rows and both weight stacks, 4 bytes per element of h: about 134 MB
   for T = 4096, d = 512, E = 8, k = 2, d_ff = 1024).  Caller-allocated, 256-byte aligned; it need
   not be initialised, except that the status word should be zeroed once
   (moe_read_device_status does this). */
size_t moe_workspace_size(const moe_config* cfg);

/* Per-expert capacity C in force for cfg (-1: no limit). */
int64_t moe_capacity(const moe_config* cfg);

/* Rows the expert-major buffers (xp, h, yp) must hold: min(T*k, E*C), or
   T*k without a capacity limit. */
int64_t moe_max_rows(const moe_config* cfg);

/*
 * Step 1, Route (Ultralytics "How Tokens Move Between GPUs", step 1): every
 * token is scored against every expert and the k best experts are kept.
 *   x [T,d], w_router [E,d] (act dtype).  logit_bias [E] fp32 or NULL is
 *   added to each logit (it moves both the selection and the gates).
 *   sel_bias [E] fp32 or NULL is DeepSeek-V3's selection-only bias
 *   (Ultralytics "Load Balancing and Capacity", bias-based balancing):
 *   added to the fp32 sigmoid score for the selection only; sigmoid scores
 *   only (MOE_ERR_UNSUPPORTED with softmax).
 *   logit L[t,e] = fp32 sum_i x[t,i] * w_router[e,i] (+ logit_bias[e]).
 *   Selection key: L (softmax) or fp32(1/(1+exp(-L))) (+ sel_bias) (sigmoid).
 * Outputs: topk_idx [T,k] int32, experts in descending key order with ties
 * to the lower expert index; topk_gate [T,k] fp32.  ws: workspace.
 * Device-side: every logit is checked; a NaN or infinite one (from a
 * non-finite element of x or w_router, or an overflowing sum) sets
 * MOE_DEV_NONFINITE in the status word, and that token's choices are then
 * unspecified (other tokens are unaffected).
 */
moe_status moe_route(const moe_config* cfg, const void* x, const void* w_router,
                     const float* logit_bias, const float* sel_bias, int32_t* topk_idx,
                     float* topk_gate, void* ws, moe_stream_t stream);

/*
 * Step 2, Dispatch (Ultralytics step 2; ai360xpert "The All-to-All
 * Bottleneck", Scatter) as one on-device permutation.
 *   x [T,d]; topk_idx [T,k] (any valid choices, e.g. from moe_route).
 * Outputs:
 *   expert_counts [E]: assignments per expert before drops;
 *   expert_offsets [E+1]: exclusive prefix over experts of the kept counts
 *     min(count, C); expert e's kept rows are [offsets[e], offsets[e+1]);
 *   rank_counts [R]: kept rows per virtual rank (its receive count);
 *   rank_splits [R,R] or NULL: kept rows sent from source rank s (token t
 *     belongs to rank t / ceil(T/R)) to destination rank r, i.e. the send
 *     counts the all-to-all would use;
 *   slot_row [T,k]: row of assignment (t,j) in the expert-major buffer, or
 *     -1 if it overflowed its expert's capacity (in token order);
 *   row_token [max_rows]: token of each kept row (entries past
 *     offsets[E] are left untouched);
 *   xp [max_rows, d]: xp[slot_row[t,j]] = x[t], bit for bit; token order is
 *     kept inside every expert block;
 *   n_dropped [1]: T*k - offsets[E].
 * Device-side: an expert index outside [0,E) sets MOE_DEV_BAD_INDEX and the
 * assignment is treated as dropped.
 */
moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx, void* xp,
                        int32_t* row_token, int32_t* slot_row, int32_t* expert_counts,
                        int32_t* expert_offsets, int32_t* rank_counts, int32_t* rank_splits,
                        int32_t* n_dropped, void* ws, moe_stream_t stream);

/*
 * Failure-detection test hook (no counterpart on the pages): the up
 * projection of moe_expert_ffn (bf16 tensor-core path; h = act(xp . W_up^T))
 * with one pipeline stage left unfilled.  CTA 0 never loads K block stall_kb
 * (0 <= stall_kb < d/64) of its first tile, so the MMA issuer's wait on that
 * stage runs out after wait_limit_us (1..4,000,000; every pipeline wait of
 * the launch gets this bound).  The kernel then sets MOE_DEV_GEMM_TIMEOUT in
 * the status word, raises its abort flag, drains the MMAs it issued, frees its
 * tensor memory and returns, so the context stays usable; h is then
 * meaningless.  moe_expert_ffn itself uses a 4 s bound and never stalls.
 * MOE_ERR_UNSUPPORTED for fp32 or IDENTITY configs.
 */
moe_status moe_test_expert_ffn_stall(const moe_config* cfg, const void* xp,
                                     const int32_t* expert_offsets, const void* w_up, void* h,
                                     int32_t stall_kb, uint32_t wait_limit_us, void* ws,
                                     moe_stream_t stream);

/*
 * moe_dispatch without a workspace, for callers that cannot allocate device
 * memory (a plugin handed only its input and output pointers; a serving loop
 * whose memory was all reserved by another allocator).  The pages have no
 * counterpart: this is a deployment variant of moe_dispatch, not a step of
 * the method.
 *   Arguments and outputs are those of moe_dispatch, minus ws; results are
 *   identical to moe_dispatch's.  device_status (DEVICE pointer, nullable):
 *   the kernels OR their MOE_DEV_* bits into it; the caller zeroes it.
 *   Scratch state lives in one fixed 4 MiB device array inside the library
 *   (allocated when the library loads, on every GPU that loads it, until the
 *   process exits).  Limit: 256 + 4*E + 2 * 4*E*ceil(T/32) + 4*R*R bytes,
 *   each term rounded up to 256, must fit in 4 MiB (T*E <= ~16.7 million, e.g.
 *   T = 65536 with E = 128); larger shapes return MOE_ERR_INVALID_ARG before
 *   anything is enqueued.
 *   The first call in each CUDA context (with that context current) looks up
 *   the array's device address and caches it under the context's unique ID,
 *   so a context created anew (after cudaDeviceReset, or by an engine that
 *   manages its own contexts) is looked up again; make the first call in a
 *   context before any stream capture.
 *   Every call shares the array and writes each part of it before reading
 *   it; calls that overlap on the GPU (other streams, unordered host threads)
 *   race on it.  Allocates nothing: no cudaMalloc, no cudaFree.
 */
moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                void* xp, int32_t* row_token, int32_t* slot_row,
                                int32_t* expert_counts, int32_t* expert_offsets,
                                int32_t* rank_counts, int32_t* rank_splits, int32_t* n_dropped,
                                uint32_t* device_status, moe_stream_t stream);

/*
 * Step 3, Compute (Ultralytics step 3): each expert's FFN on its rows of xp.
 *   xp [max_rows, d]; expert_offsets [E+1] (device; read on the device, no
 *   host synchronisation).  w_up [E, d_ff, d] (GELU) or [E, 2*d_ff, d]
 *   (SwiGLU: the d_ff gate rows first, then the d_ff up rows); w_down
 *   [E, d, d_ff].  All weights are [out, in] row-major.
 *   h [max_rows, d_ff]: scratch for the hidden activations (act dtype; for
 *   fp32 experts on the tensor cores, the activations' tf32 high parts).
 *   yp [max_rows, d]: expert outputs, same row layout as xp.  Rows past
 *   offsets[E] are left untouched.
 *   Shared expert (cfg->n_shared == 1): shared_x [T,d] (normally x),
 *   shared_up / shared_down shaped like one expert's weights, shared_h
 *   [T, d_ff] scratch and shared_out [T,d] output; all NULL when
 *   n_shared == 0.
 * bf16 runs on the tensor cores (tcgen05, fp32 accumulation in tensor
 * memory, h rounded to bf16 once).  fp32 with d and d_ff multiples of 16 also
 * runs on the tensor cores: each operand x is split into tf32 numbers
 * hi = rn(x), lo = rn(x - hi) in the workspace (one elementwise pass over the
 * input rows and weights; h is stored split, hi in h and lo in the
 * workspace), and each product
 * is a_lo*b_hi + a_hi*b_lo + a_hi*b_hi (kind::tf32, fp32 accumulation),
 * within a few 2^-22 relative of the exact product; other fp32 shapes run as
 * an fp32 FFMA grouped GEMM.
 * IDENTITY copies xp to yp (nothing if they are the same buffer).
 */
moe_status moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* expert_offsets,
                          const void* w_up, const void* w_down, void* h, void* yp,
                          const void* shared_x, const void* shared_up, const void* shared_down,
                          void* shared_h, void* shared_out, void* ws, moe_stream_t stream);

/*
 * Step 4, Combine (Ultralytics step 4; ai360xpert Gather): back to token
 * order, weighted by the gates and summed.
 *   y[t] = sum over kept j, in slot order, of topk_gate[t,j] *
 *   yp[slot_row[t,j]] (+ shared_out[t]) (+ x_residual[t] if
 *   cfg->add_residual), accumulated in fp32 and rounded once to the act
 *   dtype.  A token with every slot dropped gets exactly 0 (or exactly x).
 *   shared_out [T,d] or NULL; x_residual [T,d] (required iff add_residual).
 */
moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot_row,
                       const float* topk_gate, const void* shared_out, const void* x_residual,
                       void* y, moe_stream_t stream);

/*
 * Backward of Step 1 (training: topicspectrum "Training teaches both experts
 * and router").  Which experts a token picks is piecewise constant in the
 * logits, so no gradient flows through the selection (nor into the
 * selection-only bias, nor through rank limiting); it flows through the gates.
 * For a token with chosen experts e_j, gates g_j and dg_j = dL/dtopk_gate:
 *   softmax, renorm:  dlogit[e_j] = g_j (dg_j - sum_i g_i dg_i), 0 elsewhere;
 *   softmax, full:    dlogit[e] = p_e (dg_e - sum_j p_(e_j) dg_j) for every e
 *                     (p: softmax over all experts; dg_e = 0 off the choice);
 *   sigmoid, renorm:  dlogit[e_j] = (dg_j - sum_i g_i dg_i) / (sum_i s_i)
 *                     * s_j (1 - s_j), s = sigmoid(logit);
 *   sigmoid:          dlogit[e_j] = dg_j s_j (1 - s_j).
 * Then dx[t] = sum_e dlogit[t,e] w_router[e], d_w_router[e] = sum_t
 * dlogit[t,e] x[t], d_logit_bias[e] = sum_t dlogit[t,e].
 *   x [T,d], w_router [E,d], logit_bias [E] or NULL: the forward's inputs (the
 *   needed logits are recomputed); topk_idx [T,k]: the forward's choices
 *   (an index outside [0,E) is read as expert 0 with no gradient);
 *   d_gate [T,k] fp32, e.g. from moe_combine_backward.
 * Outputs (overwritten): d_logits [T,E] fp32, required; dx [T,d] and
 * d_w_router [E,d] (act dtype, one rounding of fp32 sums) and d_logit_bias
 * [E] fp32, each NULL to skip.  The weight gradient sums the tokens in order
 * (deterministic).
 */
moe_status moe_route_backward(const moe_config* cfg, const void* x, const void* w_router,
                              const float* logit_bias, const int32_t* topk_idx,
                              const float* d_gate, float* d_logits, void* dx, void* d_w_router,
                              float* d_logit_bias, moe_stream_t stream);

/*
 * Backward of Step 4 (the reverse of the combine exchange).  Combine is
 * linear in the expert outputs and in the gates, so for dy = dL/dy [T,d]:
 *   d_yp[slot_row[t,j]] = topk_gate[t,j] * dy[t] for every kept slot (one
 *     rounding to the act dtype; rows no slot points to are left untouched);
 *   d_gate[t,j] = sum_c dy[t,c] * yp[slot_row[t,j], c] (fp32), 0 if dropped.
 * The residual and shared-expert terms pass dy through unchanged (no call
 * needed).  dy [T,d], yp [max_rows,d], d_yp [max_rows,d]; d_gate [T,k] fp32.
 */
moe_status moe_combine_backward(const moe_config* cfg, const void* dy, const void* yp,
                                const int32_t* slot_row, const float* topk_gate, void* d_yp,
                                float* d_gate, moe_stream_t stream);

/*
 * Backward of Step 2 (the reverse of the dispatch exchange): every kept row
 * of xp is a copy of its token, so dx[t] = sum over kept j of
 * d_xp[slot_row[t,j]] (fp32 accumulation in slot order, one rounding; 0 for a
 * fully dropped token).  d_xp [max_rows,d], dx [T,d] (act dtype).
 */
moe_status moe_dispatch_backward(const moe_config* cfg, const void* d_xp, const int32_t* slot_row,
                                 void* dx, moe_stream_t stream);

/*
 * Backward of Step 3 (training: topicspectrum "Training teaches both experts
 * and router").  For each expert e and each of its rows r (forward:
 * pre = xp[r] W_up[e]^T, h = act(pre), yp[r] = h W_down[e]^T) and
 * d_yp = dL/dyp:
 *   dh = d_yp[r] W_down[e];  d_pre = act'(pre) * dh  (SwiGLU: d_gate =
 *   dh*u*silu'(g), d_up = dh*silu(g); GELU: dh*(Phi(a) + a*phi(a)));
 *   d_xp[r] = d_pre W_up[e];
 *   d_w_down[e] = sum over e's rows of d_yp[r]^T h;
 *   d_w_up[e]   = sum over e's rows of d_pre^T xp[r].
 * xp, d_yp, d_xp [max_rows, d]; expert_offsets [E+1] (device); weights and
 * weight gradients shaped like moe_expert_ffn's weights.  d_w_up and
 * d_w_down are outputs (overwritten, not accumulated); either may be NULL to
 * skip it.  Rows of d_xp past offsets[E] are left untouched.  Routed experts
 * only: the shared expert's backward is this call with a one-expert config
 * (E = 1, k = 1) over its T rows.
 * scratch: device memory of at least
 * moe_expert_ffn_backward_scratch_size(cfg, weight_grads) bytes, 256-byte
 * aligned, owned by the caller (weight_grads non-zero when either weight
 * gradient is asked for).  ws supplies the device status word.
 * bf16: pre, dh and d_pre are rounded to bf16 once each; the three
 * contractions and the weight gradients run on the tensor cores with fp32
 * accumulation (each weight gradient rounded to bf16 once).  fp32: the three
 * contractions on the tensor cores as three tf32 products per product when d
 * and d_ff are multiples of 16 (their operands split into tf32 parts in the
 * scratch), else FFMA; the weight gradients on FFMA.
 * IDENTITY: d_xp = d_yp (weight gradients must be NULL, scratch unused).
 */
size_t moe_expert_ffn_backward_scratch_size(const moe_config* cfg, int weight_grads);
moe_status moe_expert_ffn_backward(const moe_config* cfg, const void* xp,
                                   const int32_t* expert_offsets, const void* w_up,
                                   const void* w_down, const void* d_yp, void* d_xp, void* d_w_up,
                                   void* d_w_down, void* scratch, size_t scratch_bytes, void* ws,
                                   moe_stream_t stream);

/*
 * Buffers of moe_layer_forward.  xp, yp, h (and shared_h, shared_out when
 * n_shared == 1) are required.  Any metadata pointer may be NULL; the
 * library then keeps that array in the workspace.  For IDENTITY experts,
 * yp and h may be NULL (combine reads xp).
 */
typedef struct moe_buffers {
    int32_t* topk_idx;       /* [T,k] */
    float* topk_gate;        /* [T,k] */
    int32_t* slot_row;       /* [T,k] */
    int32_t* row_token;      /* [max_rows] */
    int32_t* expert_counts;  /* [E] */
    int32_t* expert_offsets; /* [E+1] */
    int32_t* rank_counts;    /* [R] */
    int32_t* rank_splits;    /* [R,R] */
    int32_t* n_dropped;      /* [1] */
    void* xp;                /* [max_rows, d] */
    void* h;                 /* [max_rows, d_ff] */
    void* yp;                /* [max_rows, d] */
    void* shared_h;          /* [T, d_ff] */
    void* shared_out;        /* [T, d] */
} moe_buffers;

/* The whole layer: route, dispatch, expert compute, combine, enqueued on
   one stream with no host synchronisation.  y [T,d] (act dtype). */
moe_status moe_layer_forward(const moe_config* cfg, const void* x, const void* w_router,
                             const float* logit_bias, const float* sel_bias, const void* w_up,
                             const void* w_down, const void* shared_up, const void* shared_down,
                             const moe_buffers* buf, void* y, void* ws, moe_stream_t stream);

/*
 * The whole layer with HOST input and output, for a caller that holds x and
 * wants y in host memory: enqueues on `stream` the copy of x_host [T,d] into
 * x_dev, moe_layer_forward on x_dev (y into y_dev), and the copy of y_dev
 * into y_host [T,d].  x_host and y_host are HOST pointers (page-locked memory
 * keeps the copies asynchronous; pageable memory makes them synchronous);
 * x_dev and y_dev are caller-owned device buffers of T*d elements.  Nothing is
 * allocated.  All of moe_layer_forward's argument checks run before the first
 * copy is enqueued; y_host holds the result once the stream has reached the
 * end of the call.  Two calls may overlap on two streams only with separate
 * buffers, workspaces and staging buffers.
 */
moe_status moe_layer_forward_host(const moe_config* cfg, const void* x_host, void* x_dev,
                                  const void* w_router, const float* logit_bias,
                                  const float* sel_bias, const void* w_up, const void* w_down,
                                  const void* shared_up, const void* shared_down,
                                  const moe_buffers* buf, void* y_dev, void* y_host, void* ws,
                                  moe_stream_t stream);

/*
 * Bias-based balancing (Ultralytics "Load Balancing and Capacity": DeepSeek-V3
 * lowers the selection bias of overloaded experts and raises it for idle ones
 * after each step).  For each expert e: if expert_counts[e] * E > T * k (load
 * above the even share) sel_bias[e] -= gamma; if below, sel_bias[e] += gamma;
 * if equal, unchanged.  The comparison is exact (64-bit integers); the update
 * is one fp32 add.  expert_counts [E] (device, e.g. moe_dispatch's output,
 * counted before drops); sel_bias [E] fp32 (device, updated in place);
 * gamma >= 0 and finite (the pages give no step size).  Enqueued on stream.
 */
moe_status moe_update_sel_bias(const moe_config* cfg, const int32_t* expert_counts, float* sel_bias,
                               float gamma, moe_stream_t stream);

/* Copies the device status word of `ws` to *out (HOST pointer), waiting for
   `stream`, then clears it.  MOE_OK with *out == 0 means no device error.
   In a checked build (below) it also reports, and clears, the bounds bit that
   calls without a workspace (moe_combine, moe_combine_backward,
   moe_dispatch_backward) record in a library-wide word. */
moe_status moe_read_device_status(const void* ws, uint32_t* out, moe_stream_t stream);

/*
 * 1 if this library was built with MOE_CHECKED (libmoe_b300_checked.so), else
 * 0.  A checked build is a debugging aid standing in for a memory checker: it
 * range-checks every index the kernels read from a caller's buffer --
 * slot_row entries in combine and in the two exchange backwards (kept rows
 * must lie in [0, moe_max_rows)), the rows dispatch computes, and
 * expert_offsets in the expert FFN and its backward (non-decreasing, within
 * [0, moe_max_rows]; a sanitised copy in the workspace is what the kernels
 * then read).  A violation sets MOE_DEV_BOUNDS and the access is skipped (a
 * bad slot counts as dropped, a bad expert range as empty).  The release
 * build performs none of these checks: such inputs are undefined there.
 */
int moe_build_checked(void);

/*
 * Kernel launches this library has enqueued since it was loaded, over all
 * threads, streams and devices (each successful launch counts one; a call
 * that fails its argument checks launches nothing).  The difference of two
 * readings around a region counts the library's kernels enqueued in it, e.g.
 * the launches one moe_layer_forward makes for a configuration (route 1, or 2
 * when a batch's expert slices take more than one wave; dispatch 3; FFN 2 per
 * expert set, 3 for fp32 experts on the tensor cores; combine 1).  Host-side;
 * no synchronisation.
 */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
