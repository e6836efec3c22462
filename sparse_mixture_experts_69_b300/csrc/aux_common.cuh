// Load-balance statistics shared by the standalone statistics kernel and the
// fused router kernel of the layer path.
//
// Per-expert totals are kept as integers: the sum of probs and the sum of gates
// in 32.32 fixed point (uint64), and the assignment count (uint32). Integer
// addition is associative, so the totals are the same whatever order blocks
// add them in. The last block to finish (ticket counter) turns them into
// f, P, importance, aux = E sum f P and CV^2 with fixed-order reductions,
// then zeroes the accumulators and the ticket for the next call.
// Method: heavensheep.xyz MoE notes, section Training (Switch aux loss);
// "MoE notes" (chiang97912.github.io), section Auxiliary loss.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Totals are kept in `groups` interleaved copies ([groups][E] each); block b
// adds into copy b % groups, which spreads the global atomics of many blocks
// over more addresses. The last block sums the copies in a fixed order.
struct AuxAcc {
    unsigned long long* P;  // [groups][E]
    unsigned long long* I;  // [groups][E]
    unsigned int* cnt;      // [groups][E]
    unsigned int* ticket;   // [1]
    int groups;
};

constexpr int kAuxGroups = 8;  // copies used with a caller workspace

__host__ __device__ inline size_t aux_acc_bytes(int E, int groups) { return (size_t)groups * E * 20 + 16; }

struct AuxOut {
    float* f;      // [E] or NULL
    float* P;      // [E] or NULL
    float* I;      // [E] or NULL
    float* out3;   // [3]
    float w_imp;
};

// acc_mem layout: [groups][E] u64 P, [groups][E] u64 I, [groups][E] u32 count, u32 ticket
__host__ __device__ inline AuxAcc aux_acc_at(void* acc_mem, int E, int groups) {
    AuxAcc a;
    a.groups = groups;
    a.P = static_cast<unsigned long long*>(acc_mem);
    a.I = a.P + (size_t)groups * E;
    a.cnt = reinterpret_cast<unsigned int*>(a.I + (size_t)groups * E);
    a.ticket = a.cnt + (size_t)groups * E;
    return a;
}

// v (a probability or gate, in [0, 1]) as 32.32 fixed point, truncated. Built
// from the float's bits with integer shifts: float -> 64-bit integer
// conversion runs on the FP64 pipe, which is slow on this part.
static __device__ __forceinline__ unsigned long long to_fix(float v) {
    if (!(v > 0.f)) return 0ull;
    const unsigned bits = __float_as_uint(v);
    const int ex = (int)(bits >> 23);             // biased exponent
    if (ex == 0) return 0ull;                     // subnormal: below 2^-126
    const unsigned long long m = (bits & 0x7FFFFFu) | 0x800000u;  // 24-bit significand
    const int sh = ex - 127 - 23 + 32;            // v * 2^32 = m * 2^sh
    if (sh >= 0) return sh > 39 ? ~0ull : m << sh;
    return sh <= -24 ? 0ull : m >> (-sh);
}

// Totals of expert e over the group copies (exact integer sums). With the
// usual group count every load is issued before the first add.
static __device__ __forceinline__ void aux_fold(const AuxAcc& acc, int E, int e,
                                                unsigned long long& pe, unsigned long long& ie,
                                                unsigned int& ce) {
    pe = 0;
    ie = 0;
    ce = 0;
    if (acc.groups == kAuxGroups) {
        unsigned long long vp[kAuxGroups], vi[kAuxGroups];
        unsigned int vc[kAuxGroups];
#pragma unroll
        for (int g = 0; g < kAuxGroups; ++g) {
            vp[g] = __ldcg(&acc.P[(size_t)g * E + e]);
            vi[g] = __ldcg(&acc.I[(size_t)g * E + e]);
            vc[g] = __ldcg(&acc.cnt[(size_t)g * E + e]);
        }
#pragma unroll
        for (int g = 0; g < kAuxGroups; ++g) {
            pe += vp[g];
            ie += vi[g];
            ce += vc[g];
        }
    } else {
        for (int g = 0; g < acc.groups; ++g) {
            pe += __ldcg(&acc.P[(size_t)g * E + e]);
            ie += __ldcg(&acc.I[(size_t)g * E + e]);
            ce += __ldcg(&acc.cnt[(size_t)g * E + e]);
        }
    }
}

// Adds a block's shared-memory totals (final: after a barrier) into its group
// copy of the global accumulators. Integer atomics: order does not matter.
static __device__ __forceinline__ void aux_publish(int E, const AuxAcc& acc,
                                                   const unsigned long long* sP,
                                                   const unsigned long long* sI,
                                                   const unsigned int* sC) {
    const size_t g = (size_t)(blockIdx.x % acc.groups) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (sP[e]) atomicAdd(&acc.P[g + e], sP[e]);
        if (sI[e]) atomicAdd(&acc.I[g + e], sI[e]);
        if (sC[e]) atomicAdd(&acc.cnt[g + e], sC[e]);
    }
}

// Turns the global totals into f, P, importance, aux and CV^2, then zeroes the
// accumulators and the ticket. Run by `nthreads` threads (local ids tid,
// whole warps) of one block, synchronised by `bar`, after every contribution
// is visible.
// It avoids FP64 (slow on this part): with I_e the integer gate sums and
// N = sum_e I_e, the importance deviations E I_e - N are exact in int64, so
// CV^2 = sum_e (E I_e - N)^2 / (E N^2) loses nothing to cancellation, and
// aux = E / (T^2 k 2^32) * sum_e count_e * P_e (fixed point) is a sum of
// positive terms. Each thread keeps its first expert's totals in registers,
// so there is one round of loads when E <= nthreads.
// Not inlined: it runs in one block, and inlined it would raise the register
// count, and so lower the occupancy, of every kernel that calls it.
template <typename Bar>
static __device__ __noinline__ void aux_finalize(int T, int E, int k, const AuxAcc& acc,
                                                 const AuxOut& out, int tid, int nthreads,
                                                 Bar bar) {
    __shared__ long long s_n[32];
    __shared__ float s_a[32], s_b[32];
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
    unsigned long long pe0 = 0, ie0 = 0;
    unsigned int ce0 = 0;
    if (tid < E) aux_fold(acc, E, tid, pe0, ie0, ce0);
    long long nloc = (long long)ie0;
    for (int e = tid + nthreads; e < E; e += nthreads) {
        unsigned long long pe, ie;
        unsigned int ce;
        aux_fold(acc, E, e, pe, ie, ce);
        nloc += (long long)ie;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) nloc += __shfl_xor_sync(0xffffffffu, nloc, o);
    if (lane == 0) s_n[warp] = nloc;
    bar();
    long long N = 0;
    for (int w = 0; w < nwarps; ++w) N += s_n[w];  // same order in every thread
    const float inv_fix = 2.3283064365386963e-10f;  // 2^-32
    const float invT = 1.f / (float)T, invTk = 1.f / ((float)T * (float)k);
    float s_fp = 0.f, s_dev = 0.f;
    for (int e = tid; e < E; e += nthreads) {
        unsigned long long pe = pe0, ie = ie0;
        unsigned int ce = ce0;
        if (e >= nthreads) aux_fold(acc, E, e, pe, ie, ce);
        const float p = (float)pe * inv_fix * invT;
        if (out.f) out.f[e] = (float)ce * invTk;
        if (out.P) out.P[e] = p;
        if (out.I) out.I[e] = (float)ie * inv_fix;
        s_fp += (float)ce * invTk * p;
        const float dev = (float)((long long)ie * E - N);
        s_dev += dev * dev;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        s_fp += __shfl_xor_sync(0xffffffffu, s_fp, o);
        s_dev += __shfl_xor_sync(0xffffffffu, s_dev, o);
    }
    if (lane == 0) {
        s_a[warp] = s_fp;
        s_b[warp] = s_dev;
    }
    bar();
    if (tid == 0) {
        float sum_fp = 0.f, sum_dev = 0.f;
        for (int w = 0; w < nwarps; ++w) {
            sum_fp += s_a[w];
            sum_dev += s_b[w];
        }
        const float n = (float)N;
        const float cv2 = sum_dev / ((float)E * n * n);
        out.out3[0] = sum_fp * (float)E;
        out.out3[1] = cv2;
        out.out3[2] = out.w_imp * cv2;
        *acc.ticket = 0;
    }
    // every load of the accumulators is done (the barrier above): clear them
    for (int i = tid; i < acc.groups * E; i += nthreads) {
        acc.P[i] = 0;
        acc.I[i] = 0;
        acc.cnt[i] = 0;
    }
}

struct BlockBar {
    __device__ void operator()() const { __syncthreads(); }
};

// Publish, then the last of the `participants` blocks (default: the whole
// grid, counted with the ticket) finalises. Every thread of every
// participating block calls this once the shared-memory totals are final.
static __device__ __noinline__ void aux_publish_and_finalize(int T, int E, int k, AuxAcc acc,
                                                             AuxOut out,
                                                             const unsigned long long* sP,
                                                             const unsigned long long* sI,
                                                             const unsigned int* sC,
                                                             int participants = -1) {
    __shared__ int is_last;
    aux_publish(E, acc, sP, sI, sC);
    __threadfence();
    __syncthreads();
    const unsigned n_part = participants > 0 ? (unsigned)participants : gridDim.x;
    if (threadIdx.x == 0) is_last = atomicAdd(acc.ticket, 1u) == n_part - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    aux_finalize(T, E, k, acc, out, threadIdx.x, blockDim.x, BlockBar{});
}

}  // namespace moe
