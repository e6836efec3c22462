// Capacity with an overflow policy: re-routing to the next candidate and/or
// rank-major priority, optionally with every expert padded to C rows.
//
// Method: "MoE notes" (chiang97912.github.io), section Expert capacity (a
// full expert sends later tokens to their next candidate; a token whose
// candidates are all full skips the layer); mkbk-pku.cn MoE notes, capacity
// section (drop, second-choice re-routing, padding to capacity).
//
// The definition is sequential: candidates are visited one at a time in the
// priority order (token order: token by token, each token's candidates in
// rank order; rank order: rank by rank, each rank's tokens in token order),
// and a visit by a token that still needs an expert takes the expert's next
// row if it holds fewer than C. Whether token t tries its candidate j
// depends on earlier visits, so the slots cannot come from one prefix count
// as in the plain dropping path (capacity.cu).
//
// Parallel form used here. Give each visit its position v in the priority
// order. Each expert e has a fill position tau_e: the position of the visit
// that takes its last (C-th) row, or "never". A visit (t,j) to expert e
// succeeds iff v(t,j) <= tau_e. Given all tau, every token's tries follow
// from its own candidates alone (try in rank order until k succeed), and
// given every token's tries, tau_e is the position of the C-th try of e.
// Start from tau = never and alternate the two steps until tau stops
// changing. Each step can only move fill positions earlier, and the
// sequential assignment is the only consistent point. So the loop ends
// there, in a handful of passes on the workloads measured (the oracle's pins
// check this algorithm against the sequential walk).
//
// One CTA of 1024 threads runs it, one token per thread in chunks of 1024
// in token order. A pass ranks every try per expert in priority order: per
// round (one in token order, one per candidate rank in rank order) and chunk,
// rank = tries of the expert in earlier rounds and chunks + tries by lower
// lanes and warps of the chunk (lane bitmasks per warp and expert). A
// token's tries are recomputed from tau wherever they are needed, so shared
// memory holds only per-expert arrays and the masks.
#include "moe_internal.cuh"

namespace moe {

namespace {
constexpr int kPolThreads = 1024;
constexpr int kPolWarps = kPolThreads / 32;
constexpr int kPolMaxPasses = 4096;

struct PolArgs {
    int T, k, nc, E, C, priority, pad, rows;  // rows: R_max
    const int32_t* ids;  // [T,nc]
    int32_t* counts;     // [E]
    int32_t* kept;       // [E]
    int32_t* offsets;    // [E+1]
    int32_t* slot;       // [T,nc]; holds ranks between passes
    int32_t* row_token;  // [R_max]
    int* status;
};

__device__ __forceinline__ unsigned lanemask_lt_pol() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Shared-memory layout of cap_policy_kernel, in 4-byte words: tau, tau_new,
// total, first [E] each, offs [E+1], then the lane masks [warps][E]. The
// host sizes the allocation and the kernel checks it with this one function.
__host__ __device__ constexpr size_t policy_smem_words(int E) {
    return (size_t)5 * E + 1 + (size_t)kPolWarps * E;
}

__device__ __forceinline__ unsigned dynamic_smem_bytes() {
    unsigned v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}

__device__ __forceinline__ int visit_pos(const PolArgs& a, int t, int j) {
    return a.priority == MOE_PRIORITY_TOKEN ? t * a.nc + j : j * a.T + t;
}

// Bit j set: token t tries candidate j under the fill positions tau (in
// rank order until k tries succeed). Out-of-range ids are never tried.
__device__ __forceinline__ unsigned tries_of(const PolArgs& a, const int* tau, int t) {
    const int32_t* row = a.ids + (size_t)t * a.nc;
    int need = a.k;
    unsigned m = 0;
    for (int j = 0; j < a.nc && need > 0; ++j) {
        const int e = row[j];
        if (e < 0 || e >= a.E) continue;
        m |= 1u << j;
        if (visit_pos(a, t, j) <= tau[e]) --need;
    }
    return m;
}
}  // namespace

__global__ void __launch_bounds__(kPolThreads, 1) cap_policy_kernel(PolArgs a) {
    pdl_trigger();
    pdl_wait();
    const int T = a.T, E = a.E, nc = a.nc, C = a.C;
    // the allocation must hold the layout below (uniform exit before any barrier)
    if (dynamic_smem_bytes() < sizeof(int) * policy_smem_words(E)) {
        if (threadIdx.x == 0) flag_status(a.status, DEV_BAD_ARG | DEV_SITE_POLICY_SMEM);
        return;
    }
    extern __shared__ int sm[];
    int* tau = sm;             // [E] fill positions of this pass
    int* tau_new = tau + E;    // [E] fill positions found in this pass
    int* total = tau_new + E;  // [E] tries of e in earlier rounds and chunks of this pass
    int* first = total + E;    // [E] tries of the first pass = top-k choices
    int* offs = first + E;     // [E+1]
    unsigned* mask = reinterpret_cast<unsigned*>(offs + E + 1);  // [warps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = lanemask_lt_pol();
    const int never = T * nc;  // later than every visit position
    for (int e = tid; e < E; e += kPolThreads) {
        tau[e] = never;
        tau_new[e] = never;
    }
    // ids must be in range and distinct per token; a bad one is never tried
    bool bad = false;
    for (int t = tid; t < T; t += kPolThreads) {
        const int32_t* row = a.ids + (size_t)t * nc;
        for (int j = 0; j < nc; ++j) {
            const int e = row[j];
            if (e < 0 || e >= E) bad = true;
            for (int q = 0; q < j; ++q)
                if (row[q] == e) bad = true;
        }
    }
    if (bad) flag_status(a.status, DEV_BAD_ARG | DEV_SITE_POLICY_ID);
    __syncthreads();

    const int rounds = a.priority == MOE_PRIORITY_TOKEN ? 1 : nc;
    bool settled = false;
    for (int pass = 0; pass < kPolMaxPasses; ++pass) {
        for (int e = tid; e < E; e += kPolThreads) total[e] = 0;
        __syncthreads();
        for (int rd = 0; rd < rounds; ++rd) {
            const unsigned round_bits = rounds == 1 ? 0xffffffffu : (1u << rd);
            for (int c0 = 0; c0 < T; c0 += kPolThreads) {
                for (int i = tid; i < kPolWarps * E; i += kPolThreads) mask[i] = 0;
                __syncthreads();
                const int t = c0 + tid;
                const unsigned mine = t < T ? tries_of(a, tau, t) & round_bits : 0u;
                const int32_t* row = a.ids + (size_t)(t < T ? t : 0) * nc;
                for (unsigned m = mine; m; m &= m - 1)
                    atomicOr(&mask[warp * E + row[__ffs(m) - 1]], 1u << lane);
                __syncthreads();
                for (unsigned m = mine; m; m &= m - 1) {
                    const int j = __ffs(m) - 1;
                    const int e = row[j];
                    int r = total[e] + __popc(mask[warp * E + e] & lt);
                    for (int w = 0; w < warp; ++w) r += __popc(mask[w * E + e]);
                    a.slot[(size_t)t * nc + j] = r;
                    if (r == C - 1) tau_new[e] = visit_pos(a, t, j);  // the one try with rank C-1
                }
                __syncthreads();
                for (int e = tid; e < E; e += kPolThreads) {
                    int add = 0;
                    for (int w = 0; w < kPolWarps; ++w) add += __popc(mask[w * E + e]);
                    total[e] += add;
                }
                __syncthreads();
            }
        }
        if (pass == 0)
            for (int e = tid; e < E; e += kPolThreads) first[e] = total[e];
        int changed = 0;
        for (int e = tid; e < E; e += kPolThreads) changed |= tau_new[e] != tau[e];
        if (!__syncthreads_or(changed)) {
            settled = true;
            break;
        }
        for (int e = tid; e < E; e += kPolThreads) {
            tau[e] = tau_new[e];
            tau_new[e] = never;
        }
        __syncthreads();
    }
    if (!settled && tid == 0) flag_status(a.status, DEV_TIMEOUT);

    // rows: kept = min(tries, C), offsets = scan of kept (or e*C when padded)
    if (tid == 0) {
        offs[0] = 0;
        for (int e = 0; e < E; ++e)
            offs[e + 1] = a.pad ? (e + 1) * C : offs[e] + min(total[e], C);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kPolThreads) {
        a.counts[e] = first[e];
        a.kept[e] = min(total[e], C);
        a.offsets[e] = offs[e];
    }
    if (tid == 0) a.offsets[E] = offs[E];
    for (int t = tid; t < T; t += kPolThreads) {
        const unsigned m = tries_of(a, tau, t);  // the tries of the last pass
        for (int j = 0; j < nc; ++j) {
            const size_t ai = (size_t)t * nc + j;
            int out = -1;
            if ((m >> j) & 1u) {
                const int r = a.slot[ai];  // this thread's own rank from the last pass
                const int e = a.ids[ai];
                if (r >= 0 && r < C) {
                    out = offs[e] + r;
                    if (out < 0 || out >= a.rows) {
                        flag_status(a.status, DEV_BAD_ARG | DEV_SITE_POLICY_ROW);
                        out = -1;
                    } else {
                        a.row_token[out] = t;
                    }
                }
            }
            a.slot[ai] = out;
        }
    }
}

cudaError_t launch_capacity_policy(const Shape& s, const int32_t* ids, int32_t* counts,
                                   int32_t* kept, int32_t* offsets, int32_t* slot,
                                   int32_t* row_token, int* status, cudaStream_t st) {
    PolArgs a;
    a.T = s.T;
    a.k = s.k;
    a.nc = s.nc;
    a.E = s.E;
    a.C = s.C;
    a.priority = s.priority;
    a.pad = s.pad;
    a.rows = s.R_max;
    a.ids = ids;
    a.counts = counts;
    a.kept = kept;
    a.offsets = offsets;
    a.slot = slot;
    a.row_token = row_token;
    a.status = status;
    const size_t smem = sizeof(int) * policy_smem_words(s.E);
    cudaError_t err = cudaFuncSetAttribute(cap_policy_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_k(cap_policy_kernel, dim3(1), dim3(kPolThreads), smem, st, a);
}

}  // namespace moe
