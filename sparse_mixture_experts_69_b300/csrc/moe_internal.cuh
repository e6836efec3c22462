// Internal declarations shared by the CUDA sources of libmoe.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- status word
// Bits OR-ed by kernels into the first int of the workspace.
enum : int { DEV_TIMEOUT = 1, DEV_NONFINITE = 2, DEV_BAD_ARG = 4 };
// Bits above DEV_BAD_ARG name the check that set it (a row index out of
// range, an expert id out of range, ...); moe_read_device_error reports
// them all as MOE_ERR_DEVICE_ARG.
enum : int {
    DEV_SITE_PERMUTE_ROW = 1 << 8,
    DEV_SITE_POLICY_ROW = 1 << 10,
    DEV_SITE_POLICY_ID = 1 << 11,
    DEV_SITE_POLICY_RANK = 1 << 12,
    DEV_SITE_POLICY_SMEM = 1 << 13,
};

// ------------------------------------------------------------- shape helpers
struct Shape {
    int T, d, E, k, F, S;
    int F1;       // rows of one expert's W1: 2F for SwiGLU, else F
    int C;        // capacity
    int R_max;    // rows of xp / yp / row_token: min(T k, E C), or E C when padded / expert choice
    int nc;       // candidates per token: k + reroute
    int priority; // MOE_PRIORITY_TOKEN / MOE_PRIORITY_RANK
    int pad;      // pad every expert's row block to C
    int routing;  // MOE_TOKEN_CHOICE / MOE_EXPERT_CHOICE
    int dtype;    // MOE_F32 / MOE_BF16
    int act;
    int renorm;
    float w_imp;
    int esize;    // bytes per element of dtype
    int noise_draw;                    // 1: the router draws its noise (moe_draw_noise)
    unsigned long long noise_seed;     // generator key
    unsigned long long noise_counter;  // stream number
    int combine_mode;                  // moe_combine_mode
};

// Workspace layout (byte offsets, each 256-aligned). One layout serves every
// entry point so the stages can be called separately on the same buffer.
struct WsLayout {
    // regions that must read zero between calls come first (moe_workspace_reset)
    size_t status;     // int32 status word (+ padding)
    size_t aux_acc;    // statistics accumulators (aux_acc_bytes(E, kAuxGroups))
    size_t blk_hist;   // [E][nblk] i32 capacity histogram counters
    size_t cap_ticket; // u32 ticket of the fused scan + slot kernel
    size_t fold_cnt;   // [T][down-GEMM column tiles] i32 arrivals of the folded combine
    size_t seq_ticket; // u32 ticket of the sequence-statistics kernel
    size_t tile_ctr;   // [2][2] i32 tile counters of the CTA-pair expert GEMMs (up, down)
    size_t zero_end;   // end of the zero-between-calls prefix
    size_t zn;         // [T,E] f32 noise logits x.Wnoise
    size_t rpart;      // K parts of a split router GEMM (router_plan), bf16 only
    size_t wgT;        // [Nr,d] dtype: Wg^T (rows 0..E-1) and Wnoise^T (E..2E-1)
    size_t logits;     // [T,E] f32 (layer only)
    size_t probs;      // [T,E] f32 (layer only)
    size_t ids;        // [T,nc] i32 (layer only)
    size_t w;          // [T,nc] f32 (layer only)
    size_t slot;       // [T,nc] i32 (layer only)
    size_t tok_row;    // [T,E] i32 (expert choice, layer only)
    size_t row_w;      // [R_max] f32 (expert choice, layer only)
    size_t seq_acc;    // sequence statistics accumulators for up to T + 1 sequences
    size_t counts;     // [E] i32 (layer only)
    size_t kept;       // [E] i32 (layer only)
    size_t offsets;    // [E+1] i32 (layer only)
    size_t row_token;  // [R_max] i32 (layer only)
    size_t tok_need;   // [T] i32 kept choices per token (layer, folded combine)
    size_t blk_base;   // [E][nblk] i32
    size_t xp;         // [R_max,d] dtype (layer only)
    size_t h;          // [R_max + S T, F] dtype
    size_t yp;         // [R_max,d] dtype (layer only)
    size_t ys;         // [S T, d] dtype (layer only)
    size_t aux_vecs;   // [3E] f32 (layer only)
    size_t out3;       // [4] f32 (layer only)
    size_t total;
};

constexpr int kCapBlockTokens = 256;  // tokens per block of the capacity kernels
constexpr int kAuxBlockTokens = 64;   // tokens per block of the statistics kernel

WsLayout ws_layout(const Shape& s);

// --------------------------------------------------------------- launchers
// Each returns a cudaError_t from the launch (cudaGetLastError).

// Router: Wg [d,E] (+ Wnoise) -> WgT [Nr,d]
cudaError_t launch_transpose_router_w(const Shape& s, const void* Wg, const void* Wnoise,
                                      void* wgT, cudaStream_t st);
// Router GEMM for float32 inputs (SIMT), reading Wg / Wnoise [d,E] in place:
// cols < E -> logits (+offset), cols >= E -> zn
cudaError_t launch_router_gemm_f32(const Shape& s, int Nr, const float* x, const float* Wg,
                                   const float* Wnoise, const float* offset, float* logits,
                                   float* zn, cudaStream_t st);
// Router GEMM for bf16 inputs (tcgen05). router_plan gives its column tile
// width, K split, whether it runs on CTA pairs and the rows of its tiles
// (pair and tile_rows may be NULL); with a
// split (ksplit > 1) the kernel writes the raw parts to part [ksplit][T][Nr]
// and logits, zn and offset are left to the selection kernel, otherwise it
// writes logits (+ offset) and zn itself.
void router_plan(int T, int d, int Nr, int* bn, int* ksplit, int* pair = nullptr,
                 int* tile_rows = nullptr);
// The selection's outputs when the router GEMM's epilogue selects
// (router_sel_in_gemm: bf16, no noise, E <= 32, nc <= 8, one K part): as
// launch_router_select writes them, plus, on the layer path, the capacity
// histogram and the statistics sums of launch_router_select_fused.
struct RouterSelOut {
    const float* bias;  // [E] or NULL
    float* probs;       // [T,E]
    float* sel;         // [T,E] or NULL
    int32_t* ids;       // [T,nc] or NULL (then w is NULL too)
    float* w;           // [T,nc]
    int32_t* blk_hist;  // capacity histogram or NULL
    void* acc_mem;      // statistics accumulators or NULL
    int late_trigger;   // 1 when no kernel of the call follows (moe_route): signal
                        // dependents only after the last accumulator
};
bool router_sel_in_gemm(const Shape& s, bool noisy);
cudaError_t launch_router_gemm_bf16(const Shape& s, int Nr, const void* x, const void* wgT,
                                    const float* offset, float* logits, float* zn, float* part,
                                    int* status, cudaStream_t st,
                                    const RouterSelOut* so = nullptr);
// The router's standard-normal draws for (s.noise_seed, s.noise_counter), [T,E]
cudaError_t launch_draw_noise(const Shape& s, float* noise, cudaStream_t st);

// The router GEMM's output as the selection kernels read it: logits and zn,
// or (nsplit > 1) the K parts part [nsplit][T][Nr] of [logits | zn] without
// the offset, which the selection kernel adds up in order and then adds the
// offset to.
struct RouterLogits {
    const float* logits;  // [T,E] (nsplit <= 1)
    const float* zn;      // [T,E] or NULL (nsplit <= 1)
    const float* part;    // [nsplit][T][Nr] (nsplit > 1)
    int nsplit, Nr;
    const float* offset;  // [E] or NULL (added when nsplit > 1)
};

// Noise, softmax, selection bias, top-k, gates. logits_out (or NULL) receives
// the logits when the selection kernel forms them from K parts.
cudaError_t launch_router_select(const Shape& s, const RouterLogits& rl, float* logits_out,
                                 const float* noise, const float* bias, float* probs,
                                 float* sel, int32_t* ids, float* w, int from_scores,
                                 const float* sel_in, const float* probs_in, int* status,
                                 cudaStream_t st);

// Layer path: selection + capacity histogram + statistics in one kernel
// defer_final: only add the statistics sums; a later kernel of the layer (the
// up GEMM) turns them into f, P, importance, aux and CV^2.
cudaError_t launch_router_select_fused(const Shape& s, const RouterLogits& rl,
                                       const float* noise, const float* bias, float* probs,
                                       int32_t* ids, float* w, int* status, int32_t* blk_hist,
                                       void* acc_mem, float* f, float* P, float* I, float* out3,
                                       bool defer_final, cudaStream_t st);

// Capacity: histogram -> scan -> slots; then the permute of x rows into xp
// hist_ready: blk_hist already holds the per-block histograms (the fused router
// kernel counted them), so only the scan and slot kernels run.
cudaError_t launch_capacity(const Shape& s, const int32_t* ids, int32_t* blk_hist,
                            unsigned int* cap_ticket, int32_t* blk_base, int32_t* counts,
                            int32_t* kept, int32_t* offsets, int32_t* slot, int32_t* row_token,
                            int* status, bool hist_ready, cudaStream_t st);
// y_zero (layers whose combine is done by the down GEMM and that have no
// shared experts): the output row of a token whose every assignment was
// dropped is zeroed here. tok_need (or NULL): each token's kept choices.
// Capacity with re-routing and/or rank priority: one thread-block cluster
// (see policy.cu). ids [T,nc]; slot [T,nc]; offsets e*C when s.pad.
cudaError_t launch_capacity_policy(const Shape& s, const int32_t* ids, int32_t* counts,
                                   int32_t* kept, int32_t* offsets, int32_t* slot,
                                   int32_t* row_token, int* status, cudaStream_t st);
// Expert choice (expert_choice.cu)
cudaError_t launch_expert_choice_select(const Shape& s, const float* probs, int32_t* offsets,
                                        int32_t* row_token, float* row_w, int32_t* tok_row,
                                        int* status, cudaStream_t st);
cudaError_t launch_gather_rows(const Shape& s, int rows, const void* x, const int32_t* row_token,
                               void* xp, cudaStream_t st);
cudaError_t launch_expert_choice_combine(const Shape& s, const void* yp, const int32_t* tok_row,
                                         const float* probs, const void* ys, void* y,
                                         cudaStream_t st);
// Sequence-level statistics (seq_stats.cu)
// scratch: seq_aux_scratch_bytes(E, n_seq) bytes of workspace, cleared on the stream
size_t seq_aux_scratch_bytes(int E, int n_seq);
cudaError_t launch_seq_aux(const Shape& s, const float* probs, const int32_t* ids,
                           const int32_t* seq_offsets, int n_seq, float* f_seq, float* P_seq,
                           float* aux_seq, float* aux_mean, void* scratch, unsigned int* ticket,
                           int* status, cudaStream_t st);
cudaError_t launch_permute(const Shape& s, const void* x, const int32_t* slot, void* xp,
                           void* y_zero, int32_t* tok_need, int* status, cudaStream_t st);
// Column tile width of the down projection's output (d), which the folded
// combine counts arrivals per.
constexpr int kDownTileN = 256;

// Grouped expert GEMMs. Up: h = act(A W1^T); down: out = h W2^T.
struct GroupedGemm {
    // routed groups e < E: rows offsets[e] .. offsets[e+1]-1 of A0, out0
    const int32_t* offsets;
    int E;
    // shared groups s < S: rows a1_row0 + s*a1_stride .. + T of A1; out1 rows s*T ..
    int S, T;
    int a1_row0, a1_stride;
    int rows_a0;        // rows of the A0 matrix
    int max_rows0;      // bound of offsets[E] (R_max): rows of out0
    int rows_a1;        // rows of A1
    int N;              // output columns
    int K;              // reduction length
    int b_rows_group;   // rows of one expert's B matrix (F1 or d)
    int glu;            // SwiGLU: B rows [0,N) gate, [N,2N) up
    int act;            // -1 none, MOE_RELU, MOE_GELU (ignored when glu)
    const void* A0; const void* A1;  // A matrices [rows, K] dtype
    const void* B0; const void* B1;  // B matrices [groups * b_rows_group, K] dtype
    void* out0; void* out1;          // [rows, N] dtype
    // top-1 layers without shared experts (tcgen05 only): routed output row r goes
    // to row scatter_rows[r] (its token) of scatter_out, times scatter_scale[token]
    const int32_t* scatter_rows;
    const float* scatter_scale;
    void* scatter_out;
    // combine folded into the down projection (tcgen05 only; fold_cnt != NULL):
    // after a warp has stored its rows of a tile (routed rows to out0, shared
    // rows to out1), each row counts itself in fold_cnt[token][column tile];
    // the arrival that completes a token's fold_need[token] + S rows sums
    // them, y[t] = sum_j fold_w[t,j] out0[fold_slot[t,j]] + sum_s out1[s T + t]
    // in fp32 in that order, into fold_y, and clears the counter.
    int32_t* fold_cnt;           // [T][ceil(N / column tile)], zero between calls
    const int32_t* fold_need;    // [T] kept choices of each token
    const int32_t* fold_rows;    // [rows of out0] token of each routed row
    const int32_t* fold_slot;    // [T][fold_nc] row of each choice, -1 if dropped
    const float* fold_w;         // [T][fold_nc] gates
    int fold_nc;
    void* fold_y;                // [T][N]
    // layer path (tcgen05 only): statistics accumulators the previous kernels
    // filled; CTA 0's epilogue warps finalise them while waiting for their first
    // accumulator (fin_acc_mem == NULL: nothing to do)
    void* fin_acc_mem;
    float* fin_f;
    float* fin_P;
    float* fin_I;
    float* fin_out3;
    int fin_k;
    float fin_w_imp;
    int* status;
    // 1: when the launch is made the offsets are final and B0 / B1 are not
    // written by any kernel still running, so the tcgen05 kernel builds its tile
    // table and loads its first B tiles before it waits for the preceding
    // kernel. Every tcgen05 launch signals its dependents only after that wait,
    // which makes this hold for the down projection that follows an up
    // projection.
    int early;
    // 1: the output is read back soon and fits in L2 (the up projection's h
    // of a small layer): store it with an evict-last L2 policy (tcgen05 only)
    int out_l2_keep;
    // 1: every group has at most one row tile, so each weight tile is read
    // once per launch: weights get an evict-first L2 policy and leave L2
    // before the activations (tcgen05 only; set for T <= 128)
    int b_evict_first;
    // 1: 256-row tiles on CTA pairs (tcgen05 pair MMA, clusters of two CTAs),
    // for groups of many rows (tcgen05 only)
    int pair;
    // row tiles per block of the tile order (group_table.cuh); 0: one block
    int row_block;
    // only groups of rows_lo .. rows_hi rows take part (0: no bound)
    int rows_lo, rows_hi;
    // CTA-pair kernel: [2] launch-wide tile counter and finished-pair count
    // (zero before the launch, zero again after it) for a dynamic tile order;
    // NULL: static order
    int* tile_ctr;
};
cudaError_t launch_grouped_gemm(const Shape& s, const GroupedGemm& g, cudaStream_t st);

// Combine, statistics, bias
cudaError_t launch_combine(const Shape& s, const void* yp, const int32_t* slot, const float* w,
                           const void* ys, void* y, int* status, cudaStream_t st);
// acc_groups: interleaved copies of the statistics accumulators in acc_mem
// (aux_acc_bytes(E, acc_groups) bytes, zero between calls)
cudaError_t launch_aux(const Shape& s, const float* probs, const int32_t* ids, const float* w,
                       void* acc_mem, int acc_groups, float* f, float* P, float* I, float* out3,
                       cudaStream_t st);
cudaError_t launch_bias_update(const Shape& s, const int32_t* counts, float* bias, float rate,
                               cudaStream_t st);

int num_sms();

// Limits of the bounded device waits (moe_set_wait_limits): the time limit of
// each tcgen05 pipeline mbarrier wait, the pass limit of the capacity
// policy's fixed-point loop, and the test switch that makes the tcgen05
// kernels withhold their first "accumulator ready" signal. Read at launch time.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
constexpr int kDefaultPolicyPasses = 4096;
unsigned long long wait_limit_ns();
int policy_max_passes();
int hold_first_accumulator();

// ------------------------------------------------- programmatic dependent launch
// Every kernel is launched with programmatic stream serialisation: it may be
// scheduled while the previous kernel on the stream is still running.
// pdl_wait() returns when the previous kernel has completed and its writes are
// visible; pdl_trigger() lets the next kernel start launching once every block
// of this one has called it (or exited). The rules every kernel here keeps:
//  - every block calls pdl_wait() before it exits, so a kernel completes only
//    after the kernel before it has, and completion follows stream order;
//  - global memory that an earlier kernel may still write, or still read, is
//    touched only after pdl_wait(). The exceptions read inputs that no kernel
//    of this library writes, and each argues why at the kernel: the router
//    weight copy (transpose_router_w_kernel) and the expert GEMMs launched
//    with GroupedGemm::early;
//  - the kernels those exceptions rely on call pdl_trigger() only after
//    pdl_wait(): the selection kernels (the router GEMM before them is then
//    complete), the permute and gather kernels (the capacity or selection
//    kernel that wrote the offsets is then complete) and the tcgen05 GEMM;
//    a router GEMM that selects itself and ends moe_route triggers in each
//    CTA only once that CTA's last accumulator is complete (all its copies of
//    the router weights have landed), so the next call's weight copy cannot
//    overwrite them while they are read.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------ device helpers
// Sorts N (a power of two, at most 8) 64-bit keys into descending order with
// a bitonic network of compile-time compare-exchanges (registers only).
template <int N>
__device__ __forceinline__ void sort_desc64(unsigned long long (&k)[N]) {
#pragma unroll
    for (int size = 2; size <= N; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    // within each bitonic block of `size`, the first half of
                    // the blocks sorts descending, the second ascending
                    const bool desc = ((i & size) == 0) || size == N;
                    const unsigned long long hi = k[i] > k[j] ? k[i] : k[j];
                    const unsigned long long lo = k[i] > k[j] ? k[j] : k[i];
                    k[i] = desc ? hi : lo;
                    k[j] = desc ? lo : hi;
                }
            }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ void flag_status(int* status, int bit) {
    if (status) atomicOr(status, bit);
}

}  // namespace moe
