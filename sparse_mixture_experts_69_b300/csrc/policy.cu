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
// One thread-block cluster of 8 CTAs x 1024 threads runs it; CTA c owns a
// contiguous block of tokens. Per pass and per round (one round in token
// order, one per candidate rank in rank order) each CTA counts its tries per
// expert, reads the other CTAs' counts through distributed shared memory,
// and ranks its own tries from per-warp lane bitmasks (chunks of 1024
// tokens). The CTA whose try gets rank C-1 writes tau_e into every CTA's
// shared memory. The decision to stop is posted by every CTA into CTA 0 and
// read back from there, so all CTAs leave the loop together. Every barrier
// between CTAs is a cluster barrier, preceded by a CTA barrier.
#include <cooperative_groups.h>

#include "moe_internal.cuh"

namespace cg = cooperative_groups;

namespace moe {

namespace {
constexpr int kPolCtas = 8;
constexpr int kPolThreads = 1024;
constexpr int kPolWarps = kPolThreads / 32;

struct PolArgs {
    int T, k, nc, E, C, priority, pad, rows;  // rows: R_max
    const int32_t* ids;  // [T,nc]
    int32_t* counts;     // [E]
    int32_t* kept;       // [E]
    int32_t* offsets;    // [E+1]
    int32_t* slot;       // [T,nc]; holds ranks between passes
    int32_t* row_token;  // [R_max]
    int* status;
    int max_passes;      // bound of the fixed-point loop (DEV_TIMEOUT when it is reached)
};

__device__ __forceinline__ unsigned lanemask_lt_pol() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__host__ __device__ constexpr int policy_tokens_per_cta(int T) { return (T + kPolCtas - 1) / kPolCtas; }

// Shared-memory layout of cap_policy_kernel, in 4-byte words: tau, tau_new,
// cnt[2], base, run, total, first ([E] each, cnt two of them), offs [E+1],
// the lane masks [warps][E], then the tries of each owned token [tokens per
// CTA]. The host sizes the allocation and the kernel checks it with this one
// function.
__host__ __device__ constexpr size_t policy_smem_words(int E, int T) {
    return (size_t)9 * E + 1 + (size_t)kPolWarps * E + (size_t)policy_tokens_per_cta(T);
}

__device__ __forceinline__ unsigned dynamic_smem_bytes() {
    unsigned v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}

__device__ __forceinline__ int visit_pos(const PolArgs& a, int t, int j) {
    return a.priority == MOE_PRIORITY_TOKEN ? t * a.nc + j : j * a.T + t;
}

// CTA barrier (warps converged), then the cluster barrier
__device__ __forceinline__ void cluster_barrier(cg::cluster_group& cl) {
    __syncthreads();
    cl.sync();
}
}  // namespace

__global__ void __launch_bounds__(kPolThreads, 1) cap_policy_kernel(PolArgs a) {
    pdl_trigger();
    pdl_wait();
    const int T = a.T, E = a.E, nc = a.nc, C = a.C;
    // every CTA of the cluster sees the same size, so this exit is uniform
    if (dynamic_smem_bytes() < sizeof(int) * policy_smem_words(E, T)) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            flag_status(a.status, DEV_BAD_ARG | DEV_SITE_POLICY_SMEM);
        return;
    }
    cg::cluster_group cl = cg::this_cluster();
    const int c = (int)cl.block_rank();
    const int Tc = policy_tokens_per_cta(T);
    const int t_lo = min(T, c * Tc), t_hi = min(T, t_lo + Tc);
    const int nown = t_hi - t_lo;
    extern __shared__ int sm[];
    int* tau = sm;               // [E] fill positions of this pass
    int* tau_new = tau + E;      // [E] written by whichever CTA holds the C-th try
    int* cnt = tau_new + E;      // [2][E] this CTA's tries per expert (alternating rounds)
    int* base = cnt + 2 * E;     // [E] tries at e before this CTA's, in this round
    int* run = base + E;         // [E] this CTA's tries at e in earlier chunks
    int* total = run + E;        // [E] tries at e in earlier rounds of this pass
    int* first = total + E;      // [E] tries of the first pass = top-k choices
    int* offs = first + E;       // [E+1]
    unsigned* mask = reinterpret_cast<unsigned*>(offs + E + 1);  // [warps][E]
    unsigned* att = mask + kPolWarps * E;                        // [Tc] tries of each token
    __shared__ int s_flag[kPolCtas];  // CTA 0's copy: each CTA's "still changing" flag
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = lanemask_lt_pol();
    const int never = T * nc;  // later than every visit position
    for (int e = tid; e < E; e += kPolThreads) {
        tau[e] = never;
        tau_new[e] = never;
        cnt[e] = 0;
        cnt[E + e] = 0;
    }
    // ids must be in range and distinct per token; a bad one is never tried
    bool bad = false;
    for (int tl = tid; tl < nown; tl += kPolThreads) {
        const int32_t* row = a.ids + (size_t)(t_lo + tl) * nc;
        for (int j = 0; j < nc; ++j) {
            const int e = row[j];
            if (e < 0 || e >= E) bad = true;
            for (int q = 0; q < j; ++q)
                if (row[q] == e) bad = true;
        }
    }
    if (bad) flag_status(a.status, DEV_BAD_ARG | DEV_SITE_POLICY_ID);
    cluster_barrier(cl);  // every CTA's tau_new is initialised before anyone writes into it

    const int rounds = a.priority == MOE_PRIORITY_TOKEN ? 1 : nc;
    bool settled = false;
    for (int pass = 0; pass < a.max_passes; ++pass) {
        // each owned token's tries under the current fill positions
        for (int tl = tid; tl < nown; tl += kPolThreads) {
            const int t = t_lo + tl;
            const int32_t* row = a.ids + (size_t)t * nc;
            int need = a.k;
            unsigned m = 0;
            for (int j = 0; j < nc && need > 0; ++j) {
                const int e = row[j];
                if (e < 0 || e >= E) continue;
                m |= 1u << j;
                if (visit_pos(a, t, j) <= tau[e]) --need;
            }
            att[tl] = m;
        }
        for (int e = tid; e < E; e += kPolThreads) total[e] = 0;
        __syncthreads();
        for (int rd = 0; rd < rounds; ++rd) {
            const unsigned round_bits = rounds == 1 ? 0xffffffffu : (1u << rd);
            int* buf = cnt + (rd & 1) * E;
            if (nown <= kPolThreads) {
                // one chunk: the lane masks of this round give the counts too
                for (int i = tid; i < kPolWarps * E; i += kPolThreads) mask[i] = 0;
                __syncthreads();
                const unsigned mine = tid < nown ? att[tid] & round_bits : 0u;
                const int t = t_lo + (tid < nown ? tid : 0);
                const int32_t* row = a.ids + (size_t)t * nc;
                for (unsigned m = mine; m; m &= m - 1)
                    atomicOr(&mask[warp * E + row[__ffs(m) - 1]], 1u << lane);
                __syncthreads();
                for (int e = tid; e < E; e += kPolThreads) {
                    int n = 0;
                    for (int w = 0; w < kPolWarps; ++w) n += __popc(mask[w * E + e]);
                    buf[e] = n;
                }
                cluster_barrier(cl);  // (A) every CTA's counts of this round are complete
                for (int e = tid; e < E; e += kPolThreads) {
                    int v[kPolCtas];  // the eight remote loads issued together
#pragma unroll
                    for (int r = 0; r < kPolCtas; ++r) v[r] = *cl.map_shared_rank(buf + e, r);
                    int before = 0, all = 0;
#pragma unroll
                    for (int r = 0; r < kPolCtas; ++r) {
                        all += v[r];
                        if (r < c) before += v[r];
                    }
                    base[e] = total[e] + before;
                    total[e] += all;
                }
                __syncthreads();
                for (unsigned m = mine; m; m &= m - 1) {
                    const int j = __ffs(m) - 1;
                    const int e = row[j];
                    int r = base[e] + __popc(mask[warp * E + e] & lt);
                    for (int w = 0; w < warp; ++w) r += __popc(mask[w * E + e]);
                    a.slot[(size_t)t * nc + j] = r;
                    if (r == C - 1) {  // the one try with rank C-1: publish the fill position
                        const int v = visit_pos(a, t, j);
                        for (int q = 0; q < kPolCtas; ++q) *cl.map_shared_rank(tau_new + e, q) = v;
                    }
                }
                __syncthreads();  // the masks are cleared again by the next round
                continue;
            }
            for (int e = tid; e < E; e += kPolThreads) buf[e] = 0;
            __syncthreads();
            for (int tl = tid; tl < nown; tl += kPolThreads) {
                const int32_t* row = a.ids + (size_t)(t_lo + tl) * nc;
                for (unsigned m = att[tl] & round_bits; m; m &= m - 1)
                    atomicAdd(&buf[row[__ffs(m) - 1]], 1);
            }
            cluster_barrier(cl);  // (A) every CTA's counts of this round are complete
            for (int e = tid; e < E; e += kPolThreads) {
                int before = 0, all = 0;
                for (int r = 0; r < kPolCtas; ++r) {
                    const int v = *cl.map_shared_rank(buf + e, r);
                    all += v;
                    if (r < c) before += v;
                }
                base[e] = total[e] + before;
                total[e] += all;
                run[e] = 0;
            }
            __syncthreads();
            for (int cs = 0; cs < nown; cs += kPolThreads) {
                for (int i = tid; i < kPolWarps * E; i += kPolThreads) mask[i] = 0;
                __syncthreads();
                const int tl = cs + tid;
                const int t = t_lo + (tl < nown ? tl : 0);
                const unsigned mine = tl < nown ? att[tl] & round_bits : 0u;
                const int32_t* row = a.ids + (size_t)t * nc;
                for (unsigned m = mine; m; m &= m - 1)
                    atomicOr(&mask[warp * E + row[__ffs(m) - 1]], 1u << lane);
                __syncthreads();
                for (unsigned m = mine; m; m &= m - 1) {
                    const int j = __ffs(m) - 1;
                    const int e = row[j];
                    int r = base[e] + run[e] + __popc(mask[warp * E + e] & lt);
                    for (int w = 0; w < warp; ++w) r += __popc(mask[w * E + e]);
                    a.slot[(size_t)t * nc + j] = r;
                    if (r == C - 1) {  // the one try with rank C-1: publish the fill position
                        const int v = visit_pos(a, t, j);
                        for (int q = 0; q < kPolCtas; ++q) *cl.map_shared_rank(tau_new + e, q) = v;
                    }
                }
                __syncthreads();
                for (int e = tid; e < E; e += kPolThreads) {
                    int add = 0;
                    for (int w = 0; w < kPolWarps; ++w) add += __popc(mask[w * E + e]);
                    run[e] += add;
                }
                __syncthreads();
            }
        }
        cluster_barrier(cl);  // (B) every fill position of this pass has landed everywhere
        if (pass == 0)
            for (int e = tid; e < E; e += kPolThreads) first[e] = total[e];
        int changed = 0;
        for (int e = tid; e < E; e += kPolThreads) changed |= tau_new[e] != tau[e];
        changed = __syncthreads_or(changed);
        if (tid == 0) *cl.map_shared_rank(s_flag + c, 0) = changed;
        cluster_barrier(cl);  // (C) every CTA's flag is in CTA 0
        int any = 0;
        for (int r = 0; r < kPolCtas; ++r) any |= *cl.map_shared_rank(s_flag + r, 0);
        if (!any) {
            settled = true;
            break;
        }
        // nobody writes tau_new or s_flag again before barrier (A) of the next pass
        for (int e = tid; e < E; e += kPolThreads) {
            tau[e] = tau_new[e];
            tau_new[e] = never;
        }
        __syncthreads();
    }
    if (!settled && c == 0 && tid == 0) flag_status(a.status, DEV_TIMEOUT);

    // rows: kept = min(tries, C), offsets = scan of kept (or e*C when padded)
    if (tid == 0) {
        offs[0] = 0;
        for (int e = 0; e < E; ++e)
            offs[e + 1] = a.pad ? (e + 1) * C : offs[e] + min(total[e], C);
    }
    __syncthreads();
    if (c == 0) {
        for (int e = tid; e < E; e += kPolThreads) {
            a.counts[e] = first[e];
            a.kept[e] = min(total[e], C);
            a.offsets[e] = offs[e];
        }
        if (tid == 0) a.offsets[E] = offs[E];
    }
    for (int tl = tid; tl < nown; tl += kPolThreads) {
        const int t = t_lo + tl;
        const unsigned m = att[tl];
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
    cluster_barrier(cl);  // no CTA exits while another might still address its shared memory
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
    a.max_passes = policy_max_passes();
    const size_t smem = sizeof(int) * policy_smem_words(s.E, s.T);
    cudaError_t err = cudaFuncSetAttribute(cap_policy_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kPolCtas);
    cfg.blockDim = dim3(kPolThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPolCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cap_policy_kernel, a);
}

}  // namespace moe
