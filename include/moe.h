/*
 * moe.h - C ABI of libmoe, the forward pass of a top-k Mixture-of-Experts FFN layer on one
 * NVIDIA B300 (sm_103a).
 *
 * The layer (page "8.6 - Mixture of Experts (MoE)", section 2, and section 4.1 for the
 * shared expert):
 *
 *     l      = x W_g (+ logit_bias)                          router logits, float32
 *     s      = softmax(l) over all E   |  sigmoid(l)         scores
 *     I      = the k experts with the largest l (+ sel_bias)  top-k, descending
 *     g_j    = s_{I_j} / sum_{j'} s_{I_j'}                    gates over the chosen k
 *     f_e(x) = ((x W1_e) * SiLU(x W2_e)) W3_e                 SwiGLU expert
 *     y      = sum_j g_j f_{I_j}(x) + sum_s f_shared_s(x)
 *
 * The calls follow the pages' four moves of one MoE layer - route, dispatch, compute,
 * combine (page "Mixture-of-Experts, from the router to the all-to-all", section "Expert
 * parallelism and the all-to-all"; page "Mixture of Experts: What Actually Happens When a
 * Token Hits the Router", Step 3: sort tokens by expert into contiguous blocks, one matmul
 * per expert, scatter back) - and moe_forward chains them.
 *
 * Conventions for every call
 *  - Pointers named x, W_g, W1, W2, W3, Ws1, Ws2, Ws3, y, x_perm, y_perm, topk_*, counts,
 *    offsets, perm_tok, inv_pos, logit_bias, sel_bias and ws are DEVICE pointers on the
 *    current CUDA device; `cfg` is a host pointer.  The caller owns all memory.  The
 *    library allocates and frees nothing; scratch comes from the caller's workspace `ws`
 *    of `ws_bytes` bytes (moe_workspace_bytes gives a size that is enough for any call).
 *  - All arrays are dense and row-major.  dtype (cfg->dtype) applies to x, W_g, the expert
 *    weights, x_perm and y.  Biases, gates, logits, y_perm and all accumulation are float32.
 *    Weights use the pages' x W orientation: W1, W2 are [E][d][d_ff], W3 is [E][d_ff][d],
 *    W_g is [d][E]; shared weights Ws1, Ws2 are [n_shared][d][d_ff_shared], Ws3 is
 *    [n_shared][d_ff_shared][d].
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and never synchronise, except moe_get_device_error and moe_forward_host.
 *    Calls on different streams need distinct workspaces.
 *  - Errors: every call returns a moe_status and never aborts.  The configuration and
 *    pointers are checked on the host before anything is launched (MOE_ERR_INVALID_ARG,
 *    MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE); a failed launch gives MOE_ERR_CUDA.
 *    Conditions that only the device can see (an expert id out of range in moe_dispatch's
 *    input, a pipeline wait that timed out) set a device error word that
 *    moe_get_device_error reports.
 *  - T = 0 is valid: the calls launch nothing and return MOE_OK.
 *
 * Limits: 1 <= k <= min(E, 32), E <= 1024, d, d_ff >= 1.  For bfloat16, d, d_ff, E (when
 * E > 32) and d_ff_shared must be multiples of 8 and every pointer 16-byte aligned
 * (the tensor-core path reads them through TMA).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same handle as cudaStream_t */
typedef struct CUevent_st* moe_event_t;   /* same handle as cudaEvent_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad sizes, k > E, null required pointer, misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2, /* valid MoE, but outside the shapes this library implements */
  MOE_ERR_WORKSPACE = 3,   /* ws is NULL or ws_bytes is too small for this call */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_DEVICE = 5       /* the device flagged an error (see moe_get_device_error) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  /* softmax over all E, top-k, renormalise over the chosen k (page "Mixture-of-Experts
     Internals: A Systems Engineer's Field Manual", section 2.1) */
  MOE_SOFTMAX_TOPK_RENORM = 0,
  /* sigmoid per expert, top-k, normalise among the chosen k (page "Mixture-of-Experts,
     from the router to the all-to-all", section "The router", DeepSeek-V3) */
  MOE_SIGMOID_TOPK_NORM = 1,
  /* softmax over all E, top-k, gates = the softmax probabilities themselves, not
     renormalised; with k = 1 this is the Switch Transformer's y = p_i(x) E_i(x) (page
     "Mixture-of-Experts, from the router to the all-to-all", section "The router") */
  MOE_SOFTMAX_TOPK_PLAIN = 2,
  /* expert choice: softmax over the E experts of each token's logits; every expert takes the
     m tokens with the largest score for it, m = ceil(T*k*c/E) (c = capacity_factor, 1 when
     0; at most T), and weights its output for token t by that score; a token may be taken by
     any number of experts (page "Mixture-of-Experts Internals: A Systems Engineer's Field
     Manual", section 5.1; page "Mixture-of-Experts, from the router to the all-to-all", "Load
     balancing").  k is the average number of experts per token.  moe_forward,
     moe_route_expert_choice, moe_experts and moe_combine_expert_choice take it; moe_route,
     moe_dispatch, moe_dispatch_static and moe_combine return MOE_ERR_UNSUPPORTED for it. */
  MOE_EXPERT_CHOICE = 3
} moe_scoring;

typedef struct {
  int32_t T;           /* tokens */
  int32_t d;           /* model width */
  int32_t d_ff;        /* routed expert width */
  int32_t E;           /* routed experts */
  int32_t k;           /* experts chosen per token */
  int32_t dtype;       /* moe_dtype */
  int32_t scoring;     /* moe_scoring */
  int32_t n_shared;    /* always-on shared experts (0 = none) */
  int32_t d_ff_shared; /* shared expert width */
  /* Capacity factor c (0 = no capacity: nothing is dropped).  With c > 0 every expert has
     ceil(T*k*c/E) slots and keeps its first pairs in token order; the pairs beyond are dropped
     and contribute nothing to the output (page "8.6 - Mixture of Experts (MoE)", section 3.2;
     page "Mixture-of-Experts, from the router to the all-to-all", "Capacity and token
     dropping").  Finite and >= 0. */
  float capacity_factor;
} moe_config;

/* Stages recorded by moe_forward_profiled: route, dispatch, experts (W1/W2 + SwiGLU),
   experts (W3), shared experts, combine. */
#define MOE_NUM_STAGES 6

/* Workspace size in bytes that is enough for every call below with this configuration
   (including moe_forward_host's device copies of x and y).  0 for an invalid config. */
size_t moe_workspace_bytes(const moe_config* cfg);

/* Route: logits -> scores -> top-k -> gates, for each token.
   Page "8.6 - Mixture of Experts (MoE)", section 2 (router x W_g, top-k by largest logit,
   gates normalised over the chosen k); page "Mixture-of-Experts Internals: A Systems
   Engineer's Field Manual", sections 2.1 (softmax, top-k, renormalise) and 3.3 (bias used
   for selection only); page "Mixture-of-Experts, from the router to the all-to-all",
   section "The router" (sigmoid variant).
     x          [T][d] dtype            W_g [d][E] dtype
     logit_bias [E] float32 or NULL: added to the logits (enters scores and selection)
     sel_bias   [E] float32 or NULL: a bias used for choosing only; gates stay unbiased.
                The top-k is taken over logit + sel_bias for softmax routing, and over
                sigmoid(logit) + sel_bias for sigmoid routing (the second page adds the bias
                to DeepSeek-V3's sigmoid scores).  moe_update_sel_bias adjusts it.
     topk_idx   [T][k] int32 out: chosen experts in descending key order, ties -> lower id
     topk_gate  [T][k] float32 out
   ws: needs T*E*4 bytes (+ alignment) when E > 32, else may be NULL. */
moe_status moe_route(const moe_config* cfg, const void* x, const void* W_g,
                     const float* logit_bias, const float* sel_bias, int32_t* topk_idx,
                     float* topk_gate, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Forward load statistics of one batch.
   Page "8.6 - Mixture of Experts (MoE)", section 3.1, and page "Mixture-of-Experts
   Internals: A Systems Engineer's Field Manual", section 3.2 (the Switch balancing loss);
   page "T2.6 What MoE changes", "Routing creates an assignment problem" and "In practice"
   (per-expert counts and maximum-to-mean load are what to monitor).
     x, W_g, logit_bias  the router's inputs, as for moe_route (the scores are recomputed)
     counts     [E] int32 in: the batch's per-expert assignment counts (moe_dispatch output)
     alpha      weight of the balancing loss
     f          [E] float32 out: f_e = counts[e] / T, the fraction of tokens routed to e
     P          [E] float32 out: P_e = mean over the T tokens of the score s_e (the softmax
                over all E for the softmax scorings, the sigmoid for MOE_SIGMOID_TOPK_NORM)
     summary    [2] float32 out: L_aux = alpha * E * sum_e f_e P_e, and max_e counts[e] / (T*k/E)
   Needs T >= 1.  Sums are float32 in a fixed order (identical results from run to run).
   ws: T*E*4 bytes for the logits plus a small per-block table (moe_workspace_bytes covers it). */
moe_status moe_load_stats(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                          const int32_t* counts, float alpha, float* f, float* P, float* summary, void* ws,
                          size_t ws_bytes, moe_stream_t stream);

/* Auxiliary-loss-free balancing: one step of the selection-bias controller.
   Page "Mixture-of-Experts Internals: A Systems Engineer's Field Manual", section 3.3, and
   page "Mixture-of-Experts, from the router to the all-to-all", "Load balancing": after each
   batch, an expert that received more than its share of the assignments has its bias
   lowered by gamma, one that received less has it raised by gamma; an expert at exactly its
   share keeps its bias.  The share is T*k/E, compared in integers (counts[e]*E against T*k).
     counts   [E] int32 in: the last batch's per-expert assignment counts (moe_dispatch's
              counts, or moe_forward's counts_out), for a batch of cfg->T tokens
     gamma    step size (finite, >= 0)
     sel_bias [E] float32 in/out: updated in place, in float32
   One tiny kernel on `stream`; no workspace. */
moe_status moe_update_sel_bias(const moe_config* cfg, const int32_t* counts, float gamma, float* sel_bias,
                               moe_stream_t stream);

/* Dispatch: per-expert histogram, exclusive prefix sum, stable permutation, row gather.
   Page "Mixture of Experts: What Actually Happens When a Token Hits the Router", Step 3
   (sort tokens by assigned expert into contiguous blocks); page "T2.6 What MoE changes",
   "Routing creates an assignment problem" (per-expert assignment counts).
     topk_idx [T][k] int32 in (every id in [0, E); an id out of range sets the device
              error word and that pair is skipped)
     x        [T][d] dtype in
     counts   [E] int32 out: pairs (t, j) routed to each expert (its load, before any dropping)
     offsets  [E+1] int32 out: exclusive prefix sum of the pairs each expert keeps:
              counts[e], or min(counts[e], slots) with a capacity factor; offsets[E] = pairs
              kept (T*k without a capacity factor)
     perm_tok [T*k] int32 out: token of the p-th kept pair in expert order, p < offsets[E];
              pairs of one expert keep ascending flattened index t*k + j; entries from
              offsets[E] on are not written
     inv_pos  [T][k] int32 out: position p of pair (t, j), or -1 if it was dropped
     x_perm   [T*k][d] dtype out: x_perm[p] = x[perm_tok[p]] for p < offsets[E]
   Deterministic: no atomics; identical inputs give identical outputs. */
moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                        int32_t* counts, int32_t* offsets, int32_t* perm_tok,
                        int32_t* inv_pos, void* x_perm, void* ws, size_t ws_bytes,
                        moe_stream_t stream);

/* Experts: for each expert e, over its block rows offsets[e]..offsets[e+1] of x_perm,
   y_perm = ((X W1_e) * SiLU(X W2_e)) W3_e.  Page "8.6 - Mixture of Experts (MoE)",
   section 2 (SwiGLU expert); page "Mixture-of-Experts, from the router to the all-to-all",
   section "Expert parallelism and the all-to-all" (one grouped matrix multiply per expert).
     x_perm  [T*k][d] dtype ([E*m][d] under expert choice)   offsets [E+1] int32
             (non-decreasing, offsets[0] = 0, offsets[E] <= the rows of x_perm; as written by
             moe_dispatch or moe_route_expert_choice)
     W1, W2  [E][d][d_ff] dtype     W3 [E][d_ff][d] dtype
     y_perm  [T*k][d] float32 out
   The intermediate h = (X W1) * SiLU(X W2) is kept in ws in dtype (bfloat16 for the
   bfloat16 path). Experts with no rows are skipped and their weights are not read.
   Rows of y_perm from offsets[E] on are not written. */
moe_status moe_experts(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                       const void* W1, const void* W2, const void* W3, float* y_perm,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* Combine: y[t] = sum_{j<k} topk_gate[t][j] * y_perm[inv_pos[t][j]] + sum_s f_shared_s(x[t]),
   summed in float32 in slot order j = 0..k-1 and rounded once to dtype.
   Page "8.6 - Mixture of Experts (MoE)", sections 2 (gate-weighted sum) and 4.1 (shared
   expert, gate 1); page "Mixture of Experts: What Actually Happens When a Token Hits the
   Router", Step 3 (scatter back).
     y_perm [T*k][d] float32   inv_pos [T][k] int32 (-1: a dropped pair, adds nothing)
     topk_gate [T][k] float32
     x [T][d] dtype, Ws1/Ws2/Ws3 as above: read only when cfg->n_shared > 0 (else may be NULL)
     y [T][d] dtype out */
moe_status moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* inv_pos,
                       const float* topk_gate, const void* x, const void* Ws1,
                       const void* Ws2, const void* Ws3, void* y, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Expert-choice route (cfg->scoring == MOE_EXPERT_CHOICE): logits -> per-token softmax ->
   every expert's m tokens, m = ceil(T*k*c/E) as described at MOE_EXPERT_CHOICE.  Each expert
   takes the m tokens with the largest float32 score; equal scores go to the lower token id.
     x [T][d], W_g [d][E], logit_bias [E] or NULL: as for moe_route
     offsets  [E+1] int32 out: e*m (every expert exactly m rows)
     perm_tok [E*m] int32 out: expert e's tokens at e*m .. e*m+m-1, in ascending token order
     gate     [E*m] float32 out: the score s[t][e] of the token at each position
     pos_of   [T][E] int32 out: the position of (t, e), or -1 if expert e did not take t
   ws: T*E*4 bytes (the scores).  Limits: T <= 51200 (an expert's T scores sit in shared
   memory); for float32 layers d must be a multiple of 4.  Then gather x rows with perm_tok
   (x_perm[p] = x[perm_tok[p]]), run moe_experts with offsets, and combine. */
moe_status moe_route_expert_choice(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                                   int32_t* offsets, int32_t* perm_tok, float* gate, int32_t* pos_of, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* Expert-choice combine: y[t] = sum over the experts e that took t, in expert order, of
   gate[p] * y_perm[p] with p = pos_of[t][e], summed in float32 and rounded once to dtype
   (+ the shared experts as in moe_combine).  A token no expert took gets only the shared
   experts (0 without them).
     y_perm [E*m][d] float32 (moe_experts output)   gate [E*m]   pos_of [T][E] */
moe_status moe_combine_expert_choice(const moe_config* cfg, const float* y_perm, const float* gate,
                                     const int32_t* pos_of, const void* x, const void* Ws1, const void* Ws2,
                                     const void* Ws3, void* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole layer: route -> dispatch -> experts -> combine (+ shared experts), on one
   stream, with every intermediate in ws.  Page "8.6 - Mixture of Experts (MoE)", section 2
   (MoE(x) = sum over TopK of g_e(x) f_e(x)) and section 4.1 (plus f_shared(x)).
   topk_idx_out [T][k] int32 and counts_out [E] int32 are optional copies of the routing.
   With MOE_EXPERT_CHOICE the layer runs expert-choice routing (route, gather, experts,
   combine as above); sel_bias, topk_idx_out and counts_out must then be NULL. */
moe_status moe_forward(const moe_config* cfg, const void* x, const void* W_g,
                       const float* logit_bias, const float* sel_bias, const void* W1,
                       const void* W2, const void* W3, const void* Ws1, const void* Ws2,
                       const void* Ws3, void* y, int32_t* topk_idx_out, int32_t* counts_out,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_forward that also records events[0..MOE_NUM_STAGES] on `stream` at the stage
   boundaries (route | dispatch | W1/W2 | W3 | shared | combine); events[i+1] - events[i]
   is stage i's device time (0 for a stage with no work).  `events` is a host array of
   MOE_NUM_STAGES + 1 events created by the caller; NULL entries are skipped. */
moe_status moe_forward_profiled(const moe_config* cfg, const void* x, const void* W_g,
                                const float* logit_bias, const float* sel_bias,
                                const void* W1, const void* W2, const void* W3,
                                const void* Ws1, const void* Ws2, const void* Ws3, void* y,
                                int32_t* topk_idx_out, int32_t* counts_out, void* ws,
                                size_t ws_bytes, moe_stream_t stream, moe_event_t* events);

/* moe_forward with x and y in HOST memory (pinned memory gives the fastest copies):
   copies x_host to the device, runs the layer and copies y back into y_host, all on
   `stream`, then waits for the stream.  Weights, biases and ws are device pointers. */
moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const void* W_g,
                            const float* logit_bias, const float* sel_bias, const void* W1,
                            const void* W2, const void* W3, const void* Ws1, const void* Ws2,
                            const void* Ws3, void* y_host, void* ws, size_t ws_bytes,
                            moe_stream_t stream);

/* moe_forward_host without the final wait: the copy of x_host, the layer and the copy back
   into y_host are enqueued on `stream` and the call returns.  y_host holds the result once the
   stream has reached that point (an event or a stream synchronisation), and x_host and y_host
   must stay valid until then.  With pinned host buffers, calls on two streams (each with its
   own workspace) overlap one call's copies with the other call's kernels. */
moe_status moe_forward_host_async(const moe_config* cfg, const void* x_host, const void* W_g,
                                  const float* logit_bias, const float* sel_bias, const void* W1,
                                  const void* W2, const void* W3, const void* Ws1, const void* Ws2,
                                  const void* Ws3, void* y_host, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* Waits for `stream`, then reads and clears the device error word of the current device.
   Returns MOE_OK, MOE_ERR_DEVICE (and the raw word in *word when word != NULL), or
   MOE_ERR_CUDA when the wait itself failed.  Bits of the word:
     1 << 0  an expert id outside [0, E) in moe_dispatch's input (that pair was skipped)
     1 << 1  grouped GEMM: offsets decreasing or beyond the rows of x_perm (clamped)
     1 << 2, 1 << 3, 1 << 4  a pipeline wait of the TMA producer / MMA issuer / epilogue timed out
     1 << 5  router: a non-finite logit
     1 << 6  bounds-checking build only (libmoe_debug.so, compiled with MOE_DEBUG_BOUNDS): an
             index read from offsets, perm_tok, inv_pos or pos_of was out of range (the access
             was skipped; the normal build skips it silently) */
moe_status moe_get_device_error(moe_stream_t stream, uint32_t* word);

/* Testing aid for the failure detection of the pipelined GEMM kernels (the pages have no
   counterpart): the next grouped tensor-core GEMM that this process launches gets a TMA
   producer that issues no copies, and every pipeline wait of that launch gives up after
   wait_limit_ns (1 .. 2e9) instead of 2 s.  Its waits then run out one after another, the
   kernel sets the device error word (MMA and epilogue wait bits), frees its tensor memory and
   returns; nothing faults and the CUDA context stays usable.  The results of that launch are
   garbage.  Later launches are unaffected. */
moe_status moe_test_pipeline_fault(uint64_t wait_limit_ns);

/* Number of kernels the last call on this host thread launched. */
int32_t moe_last_launch_count(void);

/* Static description of a status code. */
const char* moe_status_string(moe_status status);

/* Size of the library's own device scratch for moe_dispatch_static (bytes, per device). */
#define MOE_DISPATCH_STATIC_SCRATCH_BYTES (1u << 20)

/* moe_dispatch without a workspace: the same outputs as moe_dispatch, bit for bit, with its
   scratch (the per-chunk count and position tables) taken from a fixed 1 MiB array that the
   library keeps in device memory instead of from a caller-provided buffer.  The pages have
   no counterpart for this call: it exists for callers that cannot allocate device memory
   themselves, for example a plug-in whose host framework owns all device memory and hands
   it no scratch, or a latency-critical path that must not call cudaMalloc (which can
   synchronise the device).
     Arguments and outputs are those of moe_dispatch minus ws/ws_bytes.
     Size limit: ceil(T*k / 256) * E <= 131072 (the two tables fill at most 1 MiB), e.g.
     T*k <= 131072 pairs with E = 256, or T*k <= 4194304 with E = 8.  Larger sizes return
     MOE_ERR_UNSUPPORTED before anything is launched.
     Allocation: none, on any call.  The array is part of the library's device image, so
     every GPU that loads the library holds the 1 MiB until the process exits.  The first
     call on each device looks up the array's device address (cudaGetSymbolAddress, with
     that device current) and caches it; make that first call before any stream capture.
     Sharing: every call on a device uses the same array, and a call overwrites what the
     previous one left there before reading it.  Calls whose kernels overlap on the GPU
     (different streams, no ordering between them) race on the array and give wrong
     results: order them, or use moe_dispatch with separate workspaces. */
moe_status moe_dispatch_static(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                               int32_t* counts, int32_t* offsets, int32_t* perm_tok,
                               int32_t* inv_pos, void* x_perm, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
