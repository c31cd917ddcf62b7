/* moe.h — C ABI of the GB300 decode-step Mixture-of-Experts block.
 *
 * The block (Qwen3-style routed MoE with a shared expert), per token t:
 *
 *   logits[e] = x . Wr[e]                                   router GEMV
 *   ids       = top-k of logits, ranked by (logit desc, index asc)
 *   w[j]      = softmax(logits)[ids[j]], renormalised over the k (norm_topk)
 *   gu        = W13[ids[j]] x      (rows [0,I) gate, rows [I,2I) up)
 *   act       = silu(gu[0:I]) * gu[I:2I]                    SiluAndMul
 *   y_j       = W2[ids[j]] act                              down GEMV
 *   out       = sum_j w[j] y_j  +  g * shared(x)            combine + shared
 *   g         = sigmoid(x . wg) if a shared gate is given, else 1
 *
 * Sources: "BI-V100 inference work log" (kernel_worklog): Part 3 (the MoE
 * fallback path: gate, topk, softmax, index_select, linear, SiluAndMul, bmm,
 * weighted sum, shared expert), Part 4 and Part 10 (the direct-routed W13
 * and W2 kernels that index W13[expert_ids[k], row, :] and
 * W2[expert_ids[k], h, :] in place instead of copying the selected experts);
 * "Decode throughput analysis report" (decode_analysis_report), code-level
 * profiling section (T > 1 tokens: the T*k (token, expert) pairs, grouped per
 * expert instead of a host-synchronised per-expert loop).  The tie-break,
 * the renormalisation and the sigmoid gate follow the plainest reading of
 * the pages (they do not spell them out).
 *
 * Conventions shared by every call
 * --------------------------------
 *  * All tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous, 16-byte aligned.  The library keeps no pointer after a call
 *    returns and allocates no device memory at run time (the allocation-free
 *    entry's scratch array below is a fixed module symbol).
 *  * Shapes: x [T, H]; router_w [E, H]; w13 [E, 2I, H] (gate rows then up
 *    rows); w2 [E, H, I]; shared_w13 [2Is, H]; shared_w2 [H, Is];
 *    shared_gate_w [H]; out [T, H] in cfg->out_dtype; topk.ids [T, k] int32;
 *    topk.weights [T, k] fp32; slot j of a token holds its rank-j expert.
 *  * Every input tensor has element type cfg->dtype (fp16 or bf16).  All sums
 *    are accumulated in fp32; intermediates (gate/up, activation, routing
 *    weights) stay fp32.
 *  * `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous: they validate their arguments on the host, enqueue work on
 *    the stream and return.  No call synchronises except moe_query_status.
 *  * The workspace is caller-owned device memory of moe_workspace_bytes()
 *    bytes, 256-byte aligned.  It carries state between calls (a launch epoch
 *    and a device status word), so it must be zero-filled once before its
 *    first use (moe_workspace_init, or any zeroing allocation), and it must
 *    not be shared by calls that can run at the same time.
 *  * Errors: every call returns a moe_status_t.  Host-detected errors
 *    (invalid argument, unsupported shape, small workspace, launch failure)
 *    are returned immediately and described by moe_last_error() (per
 *    thread).  Device-detected errors (a bounded wait that ran out, an
 *    out-of-range expert id) never trap: the kernel records the first one in
 *    the workspace status word and returns; moe_query_status reports it.
 *    After MOE_ERR_TIMEOUT the workspace must be re-initialised.
 */
#ifndef MOE_DECODE_GB300_H
#define MOE_DECODE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Element types. */
enum { MOE_F16 = 1, MOE_BF16 = 2, MOE_F32 = 3 };

/* Status codes. */
typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* NULL/unaligned pointer, bad size or flag          */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (shape, dtype, limits) */
  MOE_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required          */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed             */
  MOE_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up               */
  MOE_ERR_DEVICE = 6        /* a device-side check failed (e.g. expert id)      */
} moe_status_t;

/* Shape and numeric options of one MoE block.
 * Limits: H, I, Is multiples of 8; 1 <= k <= 32; k <= E <= 1024;
 * has_shared_gate requires shared_inter > 0. */
typedef struct moe_cfg {
  int32_t hidden;          /* H                                                */
  int32_t n_experts;       /* E                                                */
  int32_t top_k;           /* k                                                */
  int32_t inter;           /* I, per routed expert                             */
  int32_t shared_inter;    /* Is, 0 = no shared expert                         */
  int32_t dtype;           /* MOE_F16 or MOE_BF16: every input tensor          */
  int32_t out_dtype;       /* same as dtype, or MOE_F32                        */
  int32_t norm_topk;       /* 1: renormalise the k weights to sum 1; 0: keep
                              the full-softmax probabilities                    */
  int32_t has_shared_gate; /* 1: shared output scaled by sigmoid(x . wg)       */
  int32_t flags;           /* MOE_FLAG_* bits below (0 = defaults)             */
} moe_cfg_t;

/* cfg->flags bits selecting the T > 1 path (at most one of SIMT, TC and
 * SINGLE).  With none of them the library picks: the single-launch kernel
 * when the shape allows it (E <= 256, top_k <= 8, H a multiple of 256 up to
 * 2048, I and Is multiples of 16) for 2 <= T <= 8 (T <= 3 when I < 256), and
 * for T <= 16 when the tcgen05 kernels are not available; else the tcgen05
 * kernels when the shape allows (H % 128 == 0, I and Is multiples of 64);
 * else the CUDA-core kernels. */
#define MOE_FLAG_GROUPED_SIMT 1  /* T > 1 on the CUDA-core grouped kernels      */
#define MOE_FLAG_GROUPED_TC 2    /* T > 1 on the tcgen05 grouped kernels;
                                    MOE_ERR_UNSUPPORTED if the shape does not allow it */
#define MOE_FLAG_STATIC_WEIGHTS 4 /* promise: no work still in flight on the stream
                                    when the call is enqueued writes any weight
                                    tensor (fixed inference weights).  The T = 1
                                    kernel may then start reading its
                                    routing-independent weights (router rows,
                                    shared expert) before it waits for the
                                    preceding kernel; x is always read after. */
#define MOE_FLAG_RESIDUAL 8      /* out = x + block(x): the residual add of the
                                    decoder layer fused into the output write
                                    (x exact in fp32, added after the block's
                                    sum, one rounding to out_dtype), so a stack
                                    of layers chains out -> x with no extra
                                    kernel.  Both the T = 1 and T > 1 paths. */
#define MOE_FLAG_GROUPED_SINGLE 16 /* 2 <= T <= 16 in one launch: the T = 1
                                    kernel's design, the tokens as the
                                    tensor-core steps' B columns and the
                                    selected experts' union streamed once;
                                    MOE_ERR_UNSUPPORTED if T or the shape does
                                    not allow it */

/* Caller-owned routing outputs, [T, k] each (device memory). */
typedef struct moe_topk {
  int32_t* ids;
  float* weights;
} moe_topk_t;

/* Counters of which code path ran (process-wide, host side). */
typedef struct moe_stats {
  uint64_t decode_fused_calls;   /* T == 1 single-launch decode kernel          */
  uint64_t router_calls;         /* moe_router_topk                            */
  uint64_t grouped_calls;        /* T > 1 grouped path (either kind)            */
  uint64_t grouped_tc_calls;     /* ... of which on the tcgen05 kernels         */
  uint64_t kernels_launched;     /* every kernel this library enqueued          */
  uint64_t decode_general_calls; /* T == 1 calls on the all-paths decode kernel
                                    (shapes outside the specialised ones)       */
} moe_stats_t;

/* ABI version of the loaded library (MOE_ABI_VERSION it was built with). */
MOE_API int32_t moe_abi_version(void);

/* Bytes of workspace the calls below need for `T` tokens of `cfg`
 * (0 if cfg is invalid).  One workspace sized for the largest T serves every
 * smaller T of the same cfg. */
MOE_API size_t moe_workspace_bytes(const moe_cfg_t* cfg, int32_t T);

/* Zero-fill `ws` (ws_bytes bytes) on `stream`.  Needed once after the
 * workspace is allocated, and after a MOE_ERR_TIMEOUT. */
MOE_API moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Router GEMV, fp32 softmax and top-k for T >= 1 tokens.
 * ("BI-V100 inference work log", Part 3: gate, topk, softmax; the pages'
 * "Decode throughput analysis report" notes the fused topk_softmax is missing
 * on its hardware.)
 *   x [T, H], router_w [E, H] -> topk.ids [T, k], topk.weights [T, k];
 *   logits (optional, may be NULL) [T, E] fp32 receives the raw router logits.
 * Ranking key: fp32 logit, descending; equal logits rank the lower expert
 * index first.  Weights: fp32 softmax over all E, then renormalised over the
 * k when cfg->norm_topk.  T == 0 validates cfg only and enqueues nothing. */
MOE_API moe_status_t moe_router_topk(const moe_cfg_t* cfg, const void* x, const void* router_w, int32_t T,
                             moe_topk_t topk, float* logits, void* ws, size_t ws_bytes, void* stream);

/* One decode step (T = 1) of the whole block in a single kernel launch.
 * ("BI-V100 inference work log", Parts 3, 4, 9 and 10: direct-routed W13,
 * SiluAndMul fused in, W2 with the weighted sum, shared expert.)
 *   x [1, H] -> out [1, H]; topk receives the chosen ids and weights [1, k].
 * shared_w13 / shared_w2 must be NULL iff cfg->shared_inter == 0;
 * shared_gate_w must be NULL iff cfg->has_shared_gate == 0.
 * The launch uses one CTA per SM (at most) whose CTAs exchange the router
 * logits and the activations through the workspace with bounded waits, so all
 * of them must be resident at once: a launch the occupancy calculator says
 * the device cannot hold is refused with MOE_ERR_UNSUPPORTED (a device whose
 * SMs are partly taken by other work is only caught by the wait limit); it is
 * enqueued with programmatic dependent launch so a following call on the same
 * stream can start its prologue early.  `out` must not alias any input. */
MOE_API moe_status_t moe_decode_forward(const moe_cfg_t* cfg, const void* x, const void* router_w,
                                const void* w13, const void* w2, const void* shared_w13,
                                const void* shared_w2, const void* shared_gate_w, moe_topk_t topk,
                                void* out, void* ws, size_t ws_bytes, void* stream);

/* The block for T >= 1 tokens.  T == 1 runs the single-launch decode kernel;
 * T > 1 groups the T*k (token, expert) pairs by expert on the device (no host
 * synchronisation) so each selected expert's weights stream from HBM once per
 * tile of its tokens, then combines per token in slot order.
 * ("Decode throughput analysis report", code-level profiling section.)
 * Arguments as moe_decode_forward, with x [T, H], out [T, H], topk [T, k].
 * T == 0 validates cfg only and enqueues nothing (the per-token buffers may
 * then be NULL). */
MOE_API moe_status_t moe_grouped_forward(const moe_cfg_t* cfg, const void* x, const void* router_w,
                                 const void* w13, const void* w2, const void* shared_w13,
                                 const void* shared_w2, const void* shared_gate_w, moe_topk_t topk,
                                 void* out, void* ws, size_t ws_bytes, int32_t T, void* stream);

/* Allocation-free variant of moe_decode_forward (T = 1).  The pages have no
 * counterpart; this entry exists for callers that cannot allocate device
 * memory and so cannot hand over the workspace moe_decode_forward needs:
 * code running inside a fixed device-memory pool reserved at start-up, where a
 * new cudaMalloc fails or is not allowed, or a plugin that only receives input
 * and output pointers from its host framework.  The scratch (the control block
 * and the words the CTAs exchange) lives in one fixed device array inside the
 * library, MOE_NOALLOC_SCRATCH_BYTES long, which every GPU that loads the
 * library keeps until the process exits.  A cfg whose workspace
 * (moe_workspace_bytes(cfg, 1)) is larger is rejected with
 * MOE_ERR_UNSUPPORTED.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  Every argument is validated before
 * anything is enqueued.  Each call then zero-fills the part of the array it
 * uses on `stream` (all but the device status word) and enqueues the same
 * kernel as moe_decode_forward; it allocates nothing.  All calls share the one
 * array, so calls that can overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller.  The device status word
 * is in that array and survives later calls: moe_query_status(NULL, stream)
 * reads and clears it.  Host-side errors are returned as for every other
 * call.  Arguments as moe_decode_forward, minus the workspace. */
#define MOE_NOALLOC_SCRATCH_BYTES (512u * 1024u)
MOE_API moe_status_t moe_decode_forward_noalloc(const moe_cfg_t* cfg, const void* x, const void* router_w,
                                                const void* w13, const void* w2, const void* shared_w13,
                                                const void* shared_w2, const void* shared_gate_w,
                                                moe_topk_t topk, void* out, void* stream);

/* Sum of per-shard partial outputs, for tensor-parallel use ("BI-V100
 * inference work log", Part 2: TP = 4 splits each expert's intermediate size I
 * = 512 into 128 per GPU; Part 9 and the "Decode throughput analysis report",
 * module profiling: one all-reduce of the MoE output per layer).  Shard r of
 * G holds W13 rows [r*I/G, (r+1)*I/G) of the gate and of the up block, W2
 * columns [r*I/G, (r+1)*I/G), the same slices of the shared expert, and the
 * full router and shared-gate vector; a decode or grouped call on it with
 * cfg->inter = I/G, cfg->shared_inter = Is/G and out_dtype = MOE_F32 gives a
 * partial output whose sum over the shards is the block's output.
 *   partials [n_parts, n] fp32 (device), summed in part order;
 *   residual [n] (optional, may be NULL) of residual_dtype (MOE_F16/MOE_BF16)
 *   added after the sum (the decoder layer's residual add);
 *   out [n] of out_dtype (MOE_F16, MOE_BF16 or MOE_F32), one rounding.
 * n must be a multiple of 8 and every pointer 16-byte aligned.  Across GPUs,
 * all-reduce the fp32 partials first and call this with n_parts = 1.
 * Enqueued with programmatic dependent launch; `out` must not alias the
 * partials. */
MOE_API moe_status_t moe_sum_partials(const float* partials, int32_t n_parts, int64_t n, const void* residual,
                                      int32_t residual_dtype, void* out, int32_t out_dtype, void* stream);

/* Synchronise `stream`, then read and clear the device status word of `ws`
 * (ws == NULL: the word in the built-in array of moe_decode_forward_noalloc on
 * the current device).  Returns MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE (or
 * MOE_ERR_CUDA if the synchronisation failed); moe_last_error() then names the
 * check that fired. */
MOE_API moe_status_t moe_query_status(void* ws, void* stream);

/* Text for the last error returned on this thread ("" if none). */
MOE_API const char* moe_last_error(void);

/* Copy the process-wide path counters into *stats. */
MOE_API moe_status_t moe_get_stats(moe_stats_t* stats);
MOE_API void moe_reset_stats(void);

/* Upper bound, in nanoseconds of GPU global time, on every device-side wait
 * of later launches (default 2e9 = 2 s).  Values below 1000 are refused. */
MOE_API moe_status_t moe_set_wait_timeout_ns(uint64_t ns);

/* Test hook for the failure path: enqueues one kernel that waits, with the
 * current time limit, on a workspace flag that nothing ever sets, then
 * records MOE_ERR_TIMEOUT in the status word and returns (no trap). */
MOE_API moe_status_t moe_test_wait_timeout(void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_GB300_H */
