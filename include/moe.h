/*
 * moe.h -- C ABI of libmoe.so: the forward pass of a sparse
 * Mixture-of-Experts FFN layer on one NVIDIA B300 (sm_103a).
 *
 * The method (sources are the study-note pages this library follows):
 *   router     "MoE notes" (chiang97912.github.io), sections Expert selection
 *              and KeepTopK: logits x.Wg, optional trainable noise
 *              H = x.Wg + StandardNormal() * Softplus(x.Wnoise), KeepTopK,
 *              G(x) = Softmax(KeepTopK(H, k)).
 *              heavensheep.xyz MoE notes, section Training: softmax with the
 *              maximum subtracted, exponentials in fp32.
 *              ld246.com MoE Q3: loss-free balance, a per-expert bias added to
 *              the softmax scores for the Top-K choice only.
 *   capacity   "MoE notes", section Expert capacity: capacity =
 *              (tokens per batch / number of experts) * capacity factor;
 *              mkbk-pku.cn MoE notes, load-balance section: a token beyond
 *              capacity is dropped (its output is zero; the caller's residual
 *              connection carries it).
 *   dispatch   mkbk-pku.cn MoE notes, communication section: tokens bucketed
 *              by expert and packed contiguously (here an in-HBM permutation).
 *   experts    mkbk-pku.cn MoE notes, section on experts and the grouped-GEMM
 *              optimisation: each expert is a two-layer FFN; all experts run as
 *              one grouped GEMM.
 *   combine    "MoE notes": y = sum_i G(x)_i E_i(x); shared experts
 *              (ld246.com Q4, heavensheep.xyz) are always on, weight 1.
 *   statistics heavensheep.xyz MoE notes, section Training (Switch aux loss
 *              from f_i and P_i); "MoE notes", section Auxiliary loss
 *              (Importance, CV, L_importance).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless stated; the caller allocates and
 *     owns all memory, including the workspace `ws`. The library never
 *     allocates, frees or synchronises, except moe_read_device_error.
 *   - All work is enqueued on `stream` in order; functions return after
 *     enqueueing. They hold no state between calls and are re-entrant as long
 *     as concurrent calls use different workspaces.
 *   - Layouts are row-major. "dtype" below is cfg->dtype: float32 or bf16
 *     (raw 16-bit storage). Pointers passed to the library must be 16-byte
 *     aligned; d_model and d_ff must be multiples of 8.
 *   - Host-side argument errors return before anything is enqueued.
 *     A failed launch returns MOE_ERR_CUDA. Conditions found on the device
 *     (non-finite values, out-of-range ids, a barrier wait that ran out) are
 *     recorded in the workspace status word and reported by
 *     moe_read_device_error. Kernels never trap.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Same handle as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* bad size, NULL required pointer, k > E ...  */
    MOE_ERR_UNSUPPORTED = 2, /* valid but not implemented (alignment, sizes) */
    MOE_ERR_WORKSPACE = 3,   /* ws_bytes below moe_workspace_size          */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed        */
    MOE_ERR_NONFINITE = 5,   /* device: NaN/Inf in router scores or output  */
    MOE_ERR_TIMEOUT = 6,     /* device: a pipeline wait exceeded its limit  */
    MOE_ERR_DEVICE_ARG = 7   /* device: expert id / offsets out of range    */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_RELU = 0, MOE_GELU = 1, MOE_SWIGLU = 2 } moe_act;
/* Who chooses ("MoE notes" / heavensheep.xyz, Routing Function): tokens pick
 * their top-k experts, or each expert picks its C most probable tokens. */
typedef enum { MOE_TOKEN_CHOICE = 0, MOE_EXPERT_CHOICE = 1 } moe_routing;
/* Order in which token-choice assignments claim expert capacity: token by
 * token (each token's candidates in rank order), or rank by rank (every
 * token's first choice before any second choice). */
typedef enum { MOE_PRIORITY_TOKEN = 0, MOE_PRIORITY_RANK = 1 } moe_priority;
/* MOE_COMBINE_IN_GEMM: the down GEMM's epilogue adds each token's rows once
 * the last of them is stored (no combine launch; each row is still read back
 * once, to keep the fixed order of the sum). MOE_COMBINE_KERNEL: the separate
 * combine kernel after the down GEMM. MOE_COMBINE_AUTO: the separate kernel,
 * which measured as fast or faster on every workload of this library. */
typedef enum { MOE_COMBINE_AUTO = 0, MOE_COMBINE_IN_GEMM = 1, MOE_COMBINE_KERNEL = 2 } moe_combine_mode;

/* Problem statement of one MoE layer call. */
typedef struct {
    int32_t T;               /* tokens in the batch, >= 1                      */
    int32_t d_model;         /* d, multiple of 8                               */
    int32_t n_experts;       /* E routed experts, 1..1024                      */
    int32_t top_k;           /* k, 1..min(E, 32)                               */
    int32_t d_ff;            /* F, expert hidden size, multiple of 8           */
    int32_t n_shared;        /* S always-on shared experts, 0..64              */
    float capacity_factor;   /* C = ceil(T * cf / E); cf <= 0 means C = T      */
    int32_t renorm_topk;     /* 1: gates p_j / sum_chosen p; 0: gates p_j      */
    int32_t dtype;           /* moe_dtype of x, weights, h, expert outputs, y  */
    int32_t act;             /* moe_act; SwiGLU = silu(gate) * up              */
    float importance_weight; /* w in L_importance = w * CV^2                   */
    /* Overflow policy ("MoE notes", Expert capacity: a full expert sends the
     * token to its next candidate; mkbk-pku.cn MoE notes: drop, second-choice
     * re-routing, or padding to capacity). Zero-initialised fields give the
     * default: drop, token order, packed rows, token choice. */
    int32_t reroute;         /* r >= 0 extra candidates a token tries, in rank
                                order, when a choice is full; 0 = drop.
                                n_cand = k + r <= min(E, 32)                   */
    int32_t priority;        /* moe_priority                                   */
    int32_t pad_to_capacity; /* 1: expert e owns rows e*C .. e*C+C-1, unused
                                ones zero, and the expert GEMMs run on all
                                E*C rows (fixed shapes, wasted FLOPs)          */
    int32_t routing;         /* moe_routing                                    */
    /* Noisy router draws ("MoE notes", KeepTopK: StandardNormal()). 0: the
     * caller passes them as the noise tensor. 1: the library draws eps[t,e]
     * itself, as moe_draw_noise does, and the noise pointer must be NULL.   */
    int32_t noise_draw;
    uint64_t noise_seed;     /* generator key (noise_draw = 1)                 */
    uint64_t noise_counter;  /* stream number, e.g. the training step          */
    /* Where moe_layer_fwd combines the expert outputs (bf16 layers with packed
     * rows; fp32 and padded layers always use the separate combine kernel,
     * top-1 layers without shared experts always scatter gate * output from
     * the down GEMM). The result is the same bit for bit either way.        */
    int32_t combine_mode;    /* moe_combine_mode                               */
} moe_config;

/* Terms used below: n_cand = top_k + reroute candidates per token. R_max =
 * E*C when pad_to_capacity or expert choice, else min(T*k, E*C). */

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status status);

/* Capacity C and the row bound R_max of the expert-sorted buffers (xp, yp,
 * row_token). Host only. */
MOE_API moe_status moe_capacity(const moe_config* cfg, int32_t* capacity, int32_t* rows_max);

/* Bytes of workspace any entry point below needs for this configuration.
 * One workspace sized this way serves every entry point. Host only. */
MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Zero the parts of the workspace that must read zero between calls: the
 * status word and the counters the statistics, capacity and expert-GEMM
 * kernels reset after each use (enqueued on stream). Call once on a new
 * workspace before its first use, or allocate the workspace zero-filled. */
MOE_API moe_status moe_workspace_reset(const moe_config* cfg, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

/* The noisy router's standard-normal draws for (noise_seed, noise_counter),
 * the same values the layer and moe_route use with noise_draw = 1. The pages
 * name no generator: eps[t,e] comes from the counter-based Philox4x32-10
 * (Salmon, Moraes, Dror and Shaw, SC 2011) with counter words (e, t,
 * noise_counter low, high) and key (noise_seed low, high); of its first two
 * output words r0, r1, u1 = ((r0 >> 8) + 1) / 2^24 and u2 = (r1 >> 8) / 2^24,
 * and eps = sqrt(-2 ln u1) cos(2 pi u2) (Box and Muller, 1958), in float32.
 *   noise  out  [T,E] float32
 * Device-ordered on the stream; no workspace. */
MOE_API moe_status moe_draw_noise(const moe_config* cfg, float* noise, moe_stream_t stream);

/* Router ("MoE notes", Expert selection + KeepTopK; heavensheep.xyz softmax
 * numerics; ld246.com Q3 selection bias).
 *   x            [T,d] dtype
 *   Wg           [d,E] dtype
 *   Wnoise       [d,E] dtype or NULL   noisy router: H = z + noise*softplus(x.Wnoise)
 *   noise        [T,E] float32 or NULL  standard-normal draws, supplied by the caller
 *                                       (NULL with noise_draw = 1: drawn in the
 *                                       selection kernel, see moe_draw_noise)
 *   logit_offset [E] float32 or NULL    added to the logits
 *   sel_bias     [E] float32 or NULL    added to softmax p for the top-k choice only
 *   logits  out  [T,E] float32          z = x.Wg (+ offset), fp32 accumulation
 *   probs   out  [T,E] float32          p = softmax(H), max subtracted, fp32
 *   sel_scores   [T,E] float32 or NULL  out: the scores top-k ranked (H, or p + bias)
 *   topk_ids out [T,n_cand] int32       descending score, lower index wins ties;
 *                                       the first k are the top-k choice, the
 *                                       rest the re-route candidates in order
 *   topk_w   out [T,n_cand] float32     gates from the unbiased p: p_j / (sum of
 *                                       p over the first k) with renorm_topk,
 *                                       else p_j; capacity never changes them
 * from_scores = 1 skips the logits: top-k is taken on the caller's sel_scores
 * (input) and gates on the caller's probs (input); x, Wg, logits are unused.
 * With routing = MOE_EXPERT_CHOICE topk_ids and topk_w may be NULL (the
 * probabilities are what moe_expert_choice_dispatch needs). */
MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const void* Wg,
                             const void* Wnoise, const float* noise, const float* logit_offset,
                             const float* sel_bias, float* logits, float* probs,
                             float* sel_scores, int32_t* topk_ids, float* topk_w,
                             int32_t from_scores, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Capacity and dispatch ("MoE notes", Expert capacity; mkbk-pku.cn MoE notes,
 * bucketize + contiguous packing, capacity section).
 * Candidates are visited in the priority order (cfg->priority); a visit by a
 * token that still needs an expert succeeds if the expert holds fewer than C
 * rows, and the candidate takes the expert's next row; after a failed visit
 * the token moves on to its next candidate (reroute > 0), and a token that
 * runs out of candidates keeps fewer than k experts. With reroute = 0 and
 * token priority this is plain dropping in token order: the first C
 * assignments of each expert are kept.
 *   x         [T,d] dtype, topk_ids [T,n_cand] int32 (distinct per token, in [0,E))
 *   counts    out [E] int32    top-k choices (first k candidates) per expert,
 *                              before capacity
 *   kept      out [E] int32    rows taken by each expert (min(counts, C) when
 *                              reroute = 0)
 *   offsets   out [E+1] int32  exclusive prefix sum of kept, or e*C with
 *                              pad_to_capacity; R = offsets[E]
 *   slot      out [T,n_cand] int32  row of a kept candidate in xp, -1 otherwise
 *   xp        out [R_max,d] dtype  xp[slot[t,j]] = x[t]; with pad_to_capacity
 *                              the unused rows of each block are zeroed,
 *                              otherwise rows >= R are untouched
 *   row_token out [R_max] int32    token of each kept row
 * Re-routing or rank priority supports E <= 512 and T <= 131072 and returns
 * MOE_ERR_UNSUPPORTED beyond; its device loop is bounded and records
 * MOE_ERR_TIMEOUT if it ever fails to settle. */
MOE_API moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                                int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot,
                                void* xp, int32_t* row_token, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* Expert FFNs as one grouped GEMM pair (mkbk-pku.cn MoE notes: experts, grouped
 * GEMM). Rows offsets[e]..offsets[e+1]-1 of xp go through expert e:
 *   ReLU/GELU: yp = act(xp W1[e]^T) W2[e]^T,   W1 [E,F,d]
 *   SwiGLU   : yp = (silu(xp W1[e][0:F]^T) * (xp W1[e][F:2F]^T)) W2[e]^T,  W1 [E,2F,d]
 *   W2 [E,d,F]. The hidden activations are stored in the workspace in dtype.
 * Shared experts (S > 0) run the same way on all T rows of x:
 *   W1s [S,F1,d], W2s [S,d,F], ys out [S,T,d]; x, W1s, W2s, ys may be NULL if S = 0.
 *   yp out [R_max,d] dtype (rows >= offsets[E] untouched). */
MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* offsets,
                                  const void* W1, const void* W2, const void* x,
                                  const void* W1s, const void* W2s, void* yp, void* ys,
                                  void* ws, size_t ws_bytes, moe_stream_t stream);

/* Combine back to token order ("MoE notes": y = sum_i G(x)_i E_i(x)):
 *   y[t] = sum over j with slot[t,j] >= 0 of topk_w[t,j] * yp[slot[t,j]]
 *        + sum_s ys[s,t]
 * accumulated in fp32 in a fixed order (deterministic), stored in dtype.
 * Dropped assignments add nothing and the gates are not renormalised.
 *   yp [R_max,d], slot [T,n_cand], topk_w [T,n_cand], ys [S,T,d] or NULL,
 *   y out [T,d]. */
MOE_API moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot,
                               const float* topk_w, const void* ys, void* y, void* ws,
                               size_t ws_bytes, moe_stream_t stream);

/* Load-balance statistics (heavensheep.xyz MoE notes, Switch aux loss;
 * "MoE notes", Auxiliary loss):
 *   f[e] = #{(t,j): topk_ids[t,j] = e} / (T k)     (before capacity)
 *   P[e] = mean_t probs[t,e]
 *   importance[e] = sum of topk_w over assignments to e
 *   out3 = { aux = E * sum_e f[e] P[e],
 *            cv2 = (population std of importance / its mean)^2,
 *            L_imp = importance_weight * cv2 }
 * f, P, importance: out [E] float32 or NULL; out3: out [3] float32.
 * topk_ids / topk_w are [T,n_cand]; only the first k columns are used.
 * Reduction order is fixed (deterministic). */
MOE_API moe_status moe_aux_stats(const moe_config* cfg, const float* probs,
                                 const int32_t* topk_ids, const float* topk_w, float* f,
                                 float* P, float* importance, float* out3, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* Loss-free bias update (heavensheep.xyz notes on DeepSeek-V3; ld246.com Q3):
 *   bias[e] -= rate if counts[e] > T k / E;  += rate if below;  unchanged if equal.
 * counts [E] int32 (from moe_dispatch), bias [E] float32 in/out. fp32 arithmetic. */
MOE_API moe_status moe_bias_update(const moe_config* cfg, const int32_t* counts, float* bias,
                                   float rate, moe_stream_t stream);

/* The whole layer: route -> dispatch -> expert FFN -> combine -> statistics.
 * Inputs as in moe_route and moe_expert_ffn. Outputs:
 *   y         [T,d] dtype
 *   topk_ids  [T,n_cand] int32 or NULL, topk_w [T,n_cand] float32 or NULL
 *   counts    [E] int32 or NULL (before capacity)
 *   aux_vecs  [3,E] float32 or NULL: rows f, P, importance
 *   out3      [3] float32 or NULL: aux, cv2, L_imp
 * With routing = MOE_EXPERT_CHOICE the layer runs moe_expert_choice_dispatch
 * and moe_expert_choice_combine instead; topk_ids, topk_w, counts, aux_vecs
 * and out3 must then be NULL (the token-choice statistics do not apply).
 * Intermediates (logits, probs, slots, xp, h, yp, ys) live in ws. */
MOE_API moe_status moe_layer_fwd(const moe_config* cfg, const void* x, const void* Wg,
                                 const void* Wnoise, const float* noise,
                                 const float* logit_offset, const float* sel_bias,
                                 const void* W1, const void* W2, const void* W1s,
                                 const void* W2s, void* y, int32_t* topk_ids, float* topk_w,
                                 int32_t* counts, float* aux_vecs, float* out3, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* Expert-choice routing (heavensheep.xyz MoE notes, Routing Function: experts
 * choose tokens, which balances the load; xutianle.me CS336-04, section 3).
 * Expert e takes the C tokens with the largest probs[t,e] (the lower token
 * index first among equal values). Its rows are e*C .. e*C+C-1 and hold its
 * chosen tokens in increasing token order; the gate of a row is
 * probs[token,e]. A token may be chosen by several experts or by none.
 *   x         [T,d] dtype;  probs [T,E] float32 (from moe_route)
 *   offsets   out [E+1] int32   e*C (for moe_expert_ffn)
 *   row_token out [E*C] int32   token of each row
 *   row_w     out [E*C] float32 gate of each row
 *   tok_row   out [T,E] int32   row of (t,e), -1 if e did not choose t
 *   xp        out [E*C,d] dtype xp[r] = x[row_token[r]]
 * Supports T <= 32768 (MOE_ERR_UNSUPPORTED beyond). */
MOE_API moe_status moe_expert_choice_dispatch(const moe_config* cfg, const void* x,
                                              const float* probs, int32_t* offsets,
                                              int32_t* row_token, float* row_w,
                                              int32_t* tok_row, void* xp, void* ws,
                                              size_t ws_bytes, moe_stream_t stream);

/* Expert-choice combine:
 *   y[t] = sum over experts e that chose t, in increasing e, of
 *          probs[t,e] * yp[tok_row[t,e]]  +  sum_s ys[s,t]
 * in fp32 (deterministic), stored in dtype; a token no expert chose gets the
 * shared experts only (zero without them).
 *   yp [E*C,d] dtype, tok_row [T,E], probs [T,E], ys [S,T,d] or NULL, y out [T,d]. */
MOE_API moe_status moe_expert_choice_combine(const moe_config* cfg, const void* yp,
                                             const int32_t* tok_row, const float* probs,
                                             const void* ys, void* y, void* ws, size_t ws_bytes,
                                             moe_stream_t stream);

/* Sequence-level balance statistics (heavensheep.xyz MoE notes, Training: the
 * batch balance term taken inside each sequence, so that no single sequence
 * is skewed). Sequence q holds tokens seq_offsets[q] .. seq_offsets[q+1]-1
 * (T_q of them):
 *   f_seq[q,e] = (top-k choices of its tokens naming e) / (T_q k)
 *   P_seq[q,e] = mean over its tokens of probs[t,e]
 *   aux_seq[q] = E * sum_e f_seq[q,e] P_seq[q,e]   (0 for an empty sequence)
 *   aux_mean   = mean of aux_seq over the non-empty sequences (0 if none)
 * probs [T,E] float32, topk_ids [T,n_cand] (first k columns used),
 * seq_offsets [n_seq+1] int32 device, non-decreasing from 0 to T (device
 * check: MOE_ERR_DEVICE_ARG); 1 <= n_seq <= T + 1 (MOE_ERR_UNSUPPORTED
 * above); f_seq, P_seq [n_seq,E] float32 or NULL; aux_seq [n_seq] float32;
 * aux_mean [1] float32. Deterministic (integer fixed-point sums). */
MOE_API moe_status moe_seq_aux_stats(const moe_config* cfg, const float* probs,
                                     const int32_t* topk_ids, const int32_t* seq_offsets,
                                     int32_t n_seq, float* f_seq, float* P_seq, float* aux_seq,
                                     float* aux_mean, void* ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* Statistics without a workspace. The pages have no counterpart to this call.
 *
 * Same inputs, outputs and results as moe_aux_stats, for callers that cannot
 * hand the library any device memory of their own: for instance a plugin
 * running inside a host framework that owns every allocation and gives its
 * plugins no workspace, or code on a path where allocating (and the implicit
 * synchronisation that can come with it) is not allowed. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Its scratch (the fixed-point accumulators) is a file-scope device array
 * inside libmoe.so sized for at most 512 experts (10,256 bytes); every GPU
 * that loads the library holds one copy until the process exits. n_experts
 * above 512 returns MOE_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up that array's device address (with
 *     the device current) and caches it together with the current CUDA
 *     context; make that first call before any stream capture. A call made
 *     in another context of that device (after cudaDeviceReset destroyed the
 *     primary context and the runtime made a new one) looks it up again, so
 *     the first call after a reset should also come before any capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     each call clears it on its stream before use. Calls whose work overlaps
 *     on the GPU (other streams, other threads) race on it: serialise them. */
MOE_API moe_status moe_aux_stats_noalloc(const moe_config* cfg, const float* probs,
                                         const int32_t* topk_ids, const float* topk_w,
                                         float* f, float* P, float* importance, float* out3,
                                         moe_stream_t stream);

/* Limits of the library's bounded device waits, and a switch that makes one
 * of them run out on purpose. Settings of the process, read when a kernel is
 * enqueued, so they apply to every call made after this one, on every thread
 * and device.
 *   wait_ns        time limit of each pipeline wait of the tensor-core GEMM
 *                  kernels (the router and expert GEMMs); 0 restores the
 *                  default of 2 s. A wait that runs out records
 *                  MOE_ERR_TIMEOUT; the kernel then lets its own copies and
 *                  matrix operations in flight finish (with a fixed limit of
 *                  0.25 s), frees its tensor memory and returns, leaving its
 *                  outputs incomplete.
 *   policy_passes  pass limit of the fixed-point loop of capacity with
 *                  re-routing or rank priority (moe_dispatch); 0 restores the
 *                  default of 4096; if the loop has not settled by then it
 *                  records MOE_ERR_TIMEOUT and writes the slots of its last
 *                  pass (every row index still in range).
 *   hold_first_accumulator
 *                  1: in every CTA of the tensor-core GEMM kernels the thread
 *                  issuing the matrix operations withholds the signal that
 *                  the first tile's accumulator is ready, so the epilogue's
 *                  wait for it can only end by running out after wait_ns:
 *                  a way to exercise the failure path without a fault. 0 for
 *                  normal operation.
 * Negative or out-of-range values return MOE_ERR_INVALID_ARG. No device work:
 * the defaults never run out on a working GPU. Host only. */
MOE_API moe_status moe_set_wait_limits(uint64_t wait_ns, int32_t policy_passes,
                                       int32_t hold_first_accumulator);

/* Synchronise `stream`, read and clear the workspace status word, and map it
 * to MOE_OK, MOE_ERR_NONFINITE, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_ARG (the
 * first set, in that order of precedence: TIMEOUT, DEVICE_ARG, NONFINITE). */
MOE_API moe_status moe_read_device_error(const moe_config* cfg, void* ws, size_t ws_bytes,
                                         moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
