/*
 * etmoe.h -- C ABI of libetmoe.so, the Event-Tensor MoE megakernel library
 * for GB300 (sm_103a).
 *
 * What the library computes is the plain definition of each layer; what it
 * changes is the schedule.  Sources (restated, not quoted):
 *  - "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
 *    Kernels" (episode summary of "Event Tensor: A Unified Abstraction for
 *    Compiling Dynamic Megakernel"): dependencies between tiled tasks are
 *    tracked by events instead of kernel boundaries; split-K partial sums are
 *    combined through events; a batch size kept symbolic lets one compiled
 *    kernel serve every token count; MoE routing produces data-dependent
 *    event counters and triggers tasks from the router output; static
 *    scheduling suits dense, predictable work and dynamic scheduling suits
 *    irregular MoE work.
 *  - "Megakernels ch. 5 - Event Tensor et le dynamisme", section 5.5:
 *    obstacle 1 (a waiter spins until its counter reaches a target; with
 *    dynamism that target must be computed on the GPU at run time, before
 *    the wait) and obstacle 3 (unpredictable task sizes need an online,
 *    atomic work queue).
 *
 * Conventions for every call:
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *    stated otherwise.  The library never allocates device memory and never
 *    synchronises in the compute calls; work is enqueued on `stream` (a
 *    cudaStream_t passed as void*; NULL is the legacy default stream).
 *  - bf16 tensors are row-major IEEE bfloat16; weights use the Linear layout
 *    [out_features, in_features] (the inner dimension is contiguous), except
 *    the router weight, which is [H, E] (hidden-major) as it is given.
 *  - Each call needs a caller-owned workspace of *_workspace_bytes(...)
 *    bytes, 256-byte aligned and ZEROED ONCE when it is allocated.  The
 *    kernels return every counter in it to zero before they exit, so a
 *    workspace can be reused by any number of later calls on one stream.
 *    Two calls that run concurrently must not share a workspace.
 *  - Return codes: ET_OK, or a synchronous validation error (nothing was
 *    launched).  Errors found on the device (a bounded wait that ran out, a
 *    device token count above its maximum) are recorded in a sticky status
 *    word inside the workspace; read it with et_status().
 *  - Token counts stay symbolic: pass d_T (a device int32) to have the kernel
 *    read the count at run time, so that one launch -- or one captured CUDA
 *    graph -- serves every count 0 <= T <= T_max without host involvement.
 *    With d_T == NULL the host value T is used.
 *
 * Supported shapes: H and F multiples of 128; 1 <= k <= min(E, 8);
 * 1 <= E <= 256; 0 <= T <= T_max.  Anything else returns ET_ERR_UNSUPPORTED
 * or ET_ERR_INVALID.  T == 0 launches nothing and leaves `out` untouched.
 */
#ifndef ETMOE_H
#define ETMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum et_status_code {
    ET_OK = 0,
    ET_ERR_INVALID = 1,     /* null pointer, negative size, T > T_max, k > E ... */
    ET_ERR_WORKSPACE = 2,   /* workspace missing, too small or misaligned */
    ET_ERR_UNSUPPORTED = 3, /* shape outside the supported tiling */
    ET_ERR_CUDA = 4,        /* a CUDA runtime call failed (see et_last_error_string) */
    ET_ERR_TIMEOUT = 5,     /* device: a bounded event or barrier wait ran out */
    ET_ERR_BOUNDS = 6       /* device: the device-side count exceeded its maximum */
};

/* Optional knobs; pass NULL for the defaults. */
typedef struct et_opts {
    uint32_t timeout_us; /* bound on every device-side wait; 0 = 200000 us */
    uint32_t trace_cap;  /* records the trace buffer holds (0 = no trace) */
    int32_t fault_mode;  /* test hook, 0 = off; 1 = the producer task chosen by
                            fault_arg skips its event release, so that its
                            consumers must time out cleanly */
    int32_t fault_arg;
    void* trace;         /* optional DEVICE buffer of 32 + 32*trace_cap bytes,
                            zeroed by the caller: the MoE calls, et_splitk_gemm
                            and et_mlp_chain write one record per task and
                            role (and one per ring fill) -- {int32 type |
                            role<<8, a, b, cta; uint64 t_begin, t_end}
                            (%globaltimer ns) -- after a 32-byte header; each
                            CTA owns trace_cap / grid consecutive records and
                            drops what does not fit; unused records stay zero.
                            NULL = no trace.  A diagnostic beyond the
                            computation: it changes no result. */
} et_opts;

/* ------------------------------------------------------------------------
 * MoE layer: router top-k -> per-expert counts -> SwiGLU expert FFN ->
 * weighted combine, in one persistent cooperative launch.
 *
 * Source: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
 * Kernels", the MoE discussion: routing yields data-dependent per-expert
 * counters on the device, and those counters trigger the expert tasks from
 * the router's output within one megakernel; "Megakernels ch. 5 - Event
 * Tensor et le dynamisme", section 5.1 (MoE routing as a source of data
 * dependence) and section 5.5, obstacles 1 and 3 (counter targets computed
 * on the GPU from this call's routing; an online atomic work queue).
 *
 *   logits[t,e] = sum_h x[t,h] * w_router[h,e] (+ router_bias[e]), fp32 in a
 *                 fixed order (32 strided partial sums, then a halving tree),
 *                 so routing is reproducible bit for bit;
 *   idx[t,:]    = the k largest logits, ties to the lower expert index;
 *   w[t,:]      = softmax over those k logits;
 *   h           = bf16( silu(x Wg[e]^T) * (x Wu[e]^T) ),  y = bf16( h Wd[e]^T );
 *   out[t]      = bf16( sum_j w[t,j] * y[t,j] ).
 *
 * x bf16 [T,H]; w_router bf16 [H,E]; router_bias fp32 [E] or NULL;
 * w_gate, w_up bf16 [E,F,H]; w_down bf16 [E,H,F]; out bf16 [T,H].
 * Optional outputs (NULL to skip): topk_idx int32 [T,k], topk_w fp32 [T,k],
 * expert_counts int32 [E], perm int32 [T*k] (perm[off[e]+r] = t*k+j for the
 * r-th token, ascending, routed to e; off = exclusive prefix sum of counts).
 * T is the token count (used when d_T is NULL); d_T an optional device int32
 * read by the kernel at run time (0 <= *d_T <= T_max; above that the kernel
 * records ET_ERR_BOUNDS and does nothing); T_max sizes the workspace and the
 * row buffers.  opts may be NULL.  Errors: ET_ERR_INVALID (a NULL or
 * misaligned tensor, T outside [0, T_max]), ET_ERR_UNSUPPORTED (shape),
 * ET_ERR_WORKSPACE, ET_ERR_CUDA; nothing is launched on any of them.
 * ---------------------------------------------------------------------- */
size_t et_moe_workspace_bytes(int T_max, int H, int F, int E, int k);

int et_moe_layer(const void* x, const void* w_router, const float* router_bias,
                 const void* w_gate, const void* w_up, const void* w_down, void* out,
                 int32_t* topk_idx, float* topk_w, int32_t* expert_counts, int32_t* perm,
                 int T, const int32_t* d_T, int T_max, int H, int F, int E, int k,
                 void* workspace, size_t workspace_bytes, const et_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * Fused MoE block: RMSNorm before the router, the routed experts, an optional
 * shared SwiGLU expert, and the residual add after the combine -- the layers
 * either side of the MoE layers the episode "Prompt Boundary-Aware Scheduling
 * with Event Tensors for Dynamic Kernels" discusses, joined to them in the
 * same launch.  All of it is one persistent cooperative launch: RMSNorm
 * tasks release an event the router and the shared expert's gate/up tiles
 * wait on; the shared expert's tiles carry no routing dependency and run
 * beside the router; the combine waits for both the routed and the shared
 * output tiles.
 *
 *   x_hat[t]  = bf16( (x[t] * r_t) * gamma ),  r_t = 1 / sqrt(ss_t / H + eps),
 *               ss_t = sum_h x[t,h]^2 in the router's fp32 order, and each
 *               step one IEEE-rounded fp32 operation;
 *   routing, h and y as et_moe_layer, with x_hat in place of x;
 *   ys[t]     = bf16( bf16( silu(x_hat Wsg^T) * (x_hat Wsu^T) ) Wsd^T )  (Fs > 0);
 *   out[t]    = bf16( x[t] + sum_j w[t,j] * y[t,j] + ys[t] ),  fp32 sum in
 *               that order, one rounding.
 *
 * gamma bf16 [H]; eps > 0; ws_gate, ws_up bf16 [Fs,H]; ws_down bf16 [H,Fs]
 * (NULL when Fs == 0); Fs a multiple of 128, or 0 for no shared expert.
 * x_hat: optional bf16 [T_max,H] output of the normalised rows (NULL = kept
 * in the workspace).  Other arguments as et_moe_layer.  Additionally
 * (k + 2) * H * 2 bytes must fit in the stage ring (ET_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------- */
size_t et_moe_block_workspace_bytes(int T_max, int H, int F, int E, int k, int Fs);

int et_moe_block(const void* x, const void* gamma, float eps, const void* w_router,
                 const float* router_bias, const void* w_gate, const void* w_up,
                 const void* w_down, const void* ws_gate, const void* ws_up,
                 const void* ws_down, int Fs, void* out, void* x_hat, int32_t* topk_idx,
                 float* topk_w, int32_t* expert_counts, int32_t* perm, int T,
                 const int32_t* d_T, int T_max, int H, int F, int E, int k, void* workspace,
                 size_t workspace_bytes, const et_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * Chained MoE layers in one launch.  Megakernels gain by letting the next
 * layer's work start where the previous layer's tail leaves SMs idle
 * ("Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
 * Kernels": events replace kernel boundaries; "Megakernels ch. 5 - Event
 * Tensor et le dynamisme", section 5.3: one megakernel for the model).
 *
 * Layer l + 1 takes layer l's output as its input.  Its first tasks for a
 * 16-token tile (RMSNorm in a fused block, else the router) wait on a
 * per-tile counter that layer l's combine raises by the rows it stored; the
 * layers' task lists are laid end to end in one task index space, so no
 * kernel boundary separates them.
 *
 * Each layer is described by one et_moe_layer_desc: gamma != NULL makes it a
 * fused MoE block (et_moe_block's definition: RMSNorm, routed experts,
 * optional shared expert of width Fs, residual), gamma == NULL a plain MoE
 * layer (et_moe_layer's definition; Fs must be 0).  All layers share
 * H, F, E, k and the token count.  out (bf16 [T_max, H], required) is the
 * layer's output; the optional outputs are as in et_moe_layer / et_moe_block.
 * 1 <= n_layers <= 4.  The workspace holds one region per layer (its size
 * depends on each layer's kind and Fs).  Errors: as et_moe_layer; the status
 * word is in the first layer's region (et_status(workspace)).
 * ---------------------------------------------------------------------- */
typedef struct et_moe_layer_desc {
    const void* gamma;         /* bf16 [H], or NULL for a plain MoE layer */
    float eps;                 /* RMSNorm epsilon (> 0) when gamma != NULL */
    const void* w_router;      /* bf16 [H, E] */
    const float* router_bias;  /* fp32 [E] or NULL */
    const void* w_gate;        /* bf16 [E, F, H] */
    const void* w_up;          /* bf16 [E, F, H] */
    const void* w_down;        /* bf16 [E, H, F] */
    const void* ws_gate;       /* bf16 [Fs, H] (fused block with Fs > 0) */
    const void* ws_up;         /* bf16 [Fs, H] */
    const void* ws_down;       /* bf16 [H, Fs] */
    int Fs;                    /* shared expert width, multiple of 128, or 0 */
    void* out;                 /* bf16 [T_max, H]: output, the next layer's input */
    void* x_hat;               /* optional bf16 [T_max, H] (fused block) */
    int32_t* topk_idx;         /* optional int32 [T_max, k] */
    float* topk_w;             /* optional fp32 [T_max, k] */
    int32_t* expert_counts;    /* optional int32 [E] */
    int32_t* perm;             /* optional int32 [T_max * k] */
} et_moe_layer_desc;

size_t et_moe_chain_workspace_bytes(int n_layers, const et_moe_layer_desc* layers, int T_max,
                                    int H, int F, int E, int k);

int et_moe_chain(int n_layers, const et_moe_layer_desc* layers, const void* x, int T,
                 const int32_t* d_T, int T_max, int H, int F, int E, int k, void* workspace,
                 size_t workspace_bytes, const et_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * Split-K GEMM with event-counter reduction:
 *   Y[M,N] = bf16( sum_{s<split} X[:,K_s] Wt[:,K_s]^T ),  K_s = s-th of `split`
 * equal K chunks.
 *
 * Source: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
 * Kernels", the split-K example: the tiles of each K chunk produce partial
 * sums, and the reduction of a tile starts when an event over its producing
 * tiles completes, not at a kernel boundary; the batch size M stays
 * symbolic, so one compiled kernel serves every M.
 *
 * Each (row tile, column tile, split) is one task; REDUCE tasks wait until a
 * tile's counter reaches `split`, then sum its fp32 partials in split order
 * and store Y.  X bf16 [M_max,K] (rows >= M are never read into Y); Wt bf16
 * [N,K] (the weight transposed, K contiguous); Y bf16 [M_max,N], rows >= M
 * untouched.  N % 128 == 0, K % (64*split) == 0, 1 <= split <= 16.  M is used
 * when d_M is NULL, else the device int32 *d_M (0 <= *d_M <= M_max, else
 * ET_ERR_BOUNDS on the device).  Errors as et_moe_layer.
 * ---------------------------------------------------------------------- */
size_t et_splitk_workspace_bytes(int M_max, int N, int K, int split);

int et_splitk_gemm(const void* X, const void* Wt, void* Y, int M, const int32_t* d_M, int M_max,
                   int N, int K, int split, void* workspace, size_t workspace_bytes,
                   const et_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * The same split-K GEMM with Blackwell's Cluster Launch Control as the work
 * queue ("Megakernels ch. 5 - Event Tensor et le dynamisme", section 5.5: a
 * running CTA can take over the work of a CTA that has not started).
 *
 * One CTA per tile task (ceil(M_max/256) * N/128 * split CTAs); each running
 * CTA cancels not-yet-launched CTAs (clusterlaunchcontrol.try_cancel) and
 * runs their tasks itself, so the hardware balances the work and no
 * cooperative launch is needed.  The task that completes a tile's counter
 * sums the tile's partials in split order (the last arriver).  Arguments,
 * workspace (et_splitk_workspace_bytes), results and errors as et_splitk_gemm;
 * the two calls may share a workspace, not concurrently.
 * ---------------------------------------------------------------------- */
int et_splitk_gemm_clc(const void* X, const void* Wt, void* Y, int M, const int32_t* d_M,
                       int M_max, int N, int K, int split, void* workspace,
                       size_t workspace_bytes, const et_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * Split-K GEMM that allocates nothing (the source paper has no counterpart;
 * this entry point exists for callers that cannot allocate).
 *
 * Same result as et_splitk_gemm with d_M = NULL and M_max = M, but without a
 * caller workspace: the scratch (status word, tile counters, fp32 partial
 * sums) lives in one device array of ET_SPLITK_NOALLOC_SCRATCH_BYTES inside
 * the library, held by every GPU that loads the library until the process
 * exits.  Meant for callers that cannot call cudaMalloc -- e.g. a plugin or
 * custom-op interface that only passes input and output buffers, or a code
 * path where allocating could synchronise the device or break a fixed
 * memory plan.  The caller still passes X, Wt and Y.
 *  - No cudaMalloc, cudaFree or other allocating call is made.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process, like the library's other per-device state: after
 *    cudaDeviceReset the process must be restarted.
 *  - Each call first clears the status word and tile counters of the array
 *    on `stream` (cudaMemsetAsync), then runs the split-K kernel.
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other host threads) race on it and must be serialised.
 *  - Shapes whose scratch (et_splitk_workspace_bytes(M, N, K, split)) exceeds
 *    the array are rejected with ET_ERR_WORKSPACE before anything is
 *    launched; other argument rules are those of et_splitk_gemm.
 *  - A device-side error of the last call (a bounded wait that ran out) is
 *    read with et_splitk_noalloc_status before the next call clears it.
 * ---------------------------------------------------------------------- */
#define ET_SPLITK_NOALLOC_SCRATCH_BYTES (16u << 20)

int et_splitk_gemm_noalloc(const void* X, const void* Wt, void* Y, int M, int N, int K, int split,
                           void* stream);

/* Device status of the last et_splitk_gemm_noalloc call on the current
 * device: synchronises `stream` (cudaStream_t as void*), then copies the
 * status word of the built-in scratch array to *code_out / *detail_out (host
 * pointers; detail_out may be NULL).  Allocates nothing.  Returns ET_OK, or
 * ET_ERR_INVALID / ET_ERR_CUDA when the status could not be read. */
int et_splitk_noalloc_status(void* stream, int32_t* code_out, int32_t* detail_out);

/* ------------------------------------------------------------------------
 * Dense dependent MLP chain, statically scheduled (tasks bound to CTAs):
 *   xhat = bf16( x / sqrt(mean(x^2) + eps) * gamma )
 *   out  = bf16( bf16( silu(xhat Wg^T) * (xhat Wu^T) ) Wd^T )
 *
 * Source: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
 * Kernels", static versus dynamic scheduling: for dense, predictable work a
 * static assignment of tasks to SMs is the better choice (no queue), while
 * events still order the dependent tiles in place of kernel boundaries.
 *
 * x bf16 [B_max,H]; gamma bf16 [H]; eps >= 0; w_gate, w_up bf16 [F,H];
 * w_down bf16 [H,F]; out bf16 [B_max,H] (rows >= B untouched).  RMSNorm
 * tasks release an event the gate/up tiles wait on; down tiles wait on
 * per-chunk event counters of the gate/up tiles.  B is used when d_B is
 * NULL, else the device int32 *d_B (0 <= *d_B <= B_max).  H and F multiples
 * of 128.  Errors as et_moe_layer.
 * ---------------------------------------------------------------------- */
size_t et_mlp_workspace_bytes(int B_max, int H, int F);

int et_mlp_chain(const void* x, const void* gamma, float eps, const void* w_gate,
                 const void* w_up, const void* w_down, void* out, int B, const int32_t* d_B,
                 int B_max, int H, int F, void* workspace, size_t workspace_bytes,
                 const et_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * Status of the device side.  Synchronises `stream`, then copies the sticky
 * status word of `workspace` to *code_out / *detail_out (host pointers).
 * detail identifies where a wait ran out.  For tests and diagnostics only.
 * et_reset_status clears the word (enqueued on `stream`, no sync).
 * ---------------------------------------------------------------------- */
int et_status(const void* workspace, void* stream, int32_t* code_out, int32_t* detail_out);
int et_reset_status(void* workspace, void* stream);

/* Message for the last error returned on this host thread ("" if none). */
const char* et_last_error_string(void);

/* Library version (major*10000 + minor*100 + patch). */
int et_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ETMOE_H */
