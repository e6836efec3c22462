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

struct AuxAcc {
    unsigned long long* P;  // [E]
    unsigned long long* I;  // [E]
    unsigned int* cnt;      // [E]
    unsigned int* ticket;   // [1]
};

struct AuxOut {
    float* f;      // [E] or NULL
    float* P;      // [E] or NULL
    float* I;      // [E] or NULL
    float* out3;   // [3]
    float w_imp;
};

// acc_mem layout: [E] u64 P, [E] u64 I, [E] u32 count, u32 ticket
inline AuxAcc aux_acc_at(void* acc_mem, int E) {
    AuxAcc a;
    a.P = static_cast<unsigned long long*>(acc_mem);
    a.I = a.P + E;
    a.cnt = reinterpret_cast<unsigned int*>(a.I + E);
    a.ticket = a.cnt + E;
    return a;
}

static __device__ __forceinline__ unsigned long long to_fix(float v) {
    // v in [0, 1]; v * 2^32 is exact in fp32, then rounded to an integer
    return v > 0.f ? __float2ull_rn(v * 4294967296.0f) : 0ull;
}

// Sum of one double per thread, in a fixed order. scratch: 33 doubles.
static __device__ double block_sum_fixed(double v, double* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += scratch[w];
        scratch[32] = tot;
    }
    __syncthreads();
    const double tot = scratch[32];
    __syncthreads();
    return tot;
}

// Called by every thread of every block once the block's shared-memory totals
// sP/sI/sC are final (after a __syncthreads). Adds them to the global
// accumulators; the last block computes the statistics and resets.
static __device__ void aux_publish_and_finalize(int T, int E, int k, AuxAcc acc, AuxOut out,
                                                const unsigned long long* sP,
                                                const unsigned long long* sI,
                                                const unsigned int* sC) {
    __shared__ double red[33];
    __shared__ int is_last;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (sP[e]) atomicAdd(&acc.P[e], sP[e]);
        if (sI[e]) atomicAdd(&acc.I[e], sI[e]);
        if (sC[e]) atomicAdd(&acc.cnt[e], sC[e]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(acc.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const double inv_fix = 1.0 / 4294967296.0;
    double s_fp = 0.0, s_i = 0.0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double pe = (double)__ldcg(&acc.P[e]) * inv_fix / (double)T;
        const double ie = (double)__ldcg(&acc.I[e]) * inv_fix;
        const double fe = (double)__ldcg(&acc.cnt[e]) / ((double)T * (double)k);
        if (out.f) out.f[e] = (float)fe;
        if (out.P) out.P[e] = (float)pe;
        if (out.I) out.I[e] = (float)ie;
        s_fp += fe * pe;
        s_i += ie;
    }
    const double sum_fp = block_sum_fixed(s_fp, red);
    const double mean = block_sum_fixed(s_i, red) / (double)E;
    double s_v = 0.0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double dv = (double)__ldcg(&acc.I[e]) * inv_fix - mean;
        s_v += dv * dv;
    }
    const double var = block_sum_fixed(s_v, red) / (double)E;
    if (threadIdx.x == 0) {
        const double cv2 = var / (mean * mean);
        out.out3[0] = (float)(sum_fp * (double)E);
        out.out3[1] = (float)cv2;
        out.out3[2] = (float)((double)out.w_imp * cv2);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        acc.P[e] = 0;
        acc.I[e] = 0;
        acc.cnt[e] = 0;
    }
    if (threadIdx.x == 0) *acc.ticket = 0;
}

}  // namespace moe
