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

// Sum of one float per thread, in a fixed order. scratch: 33 floats.
static __device__ float block_sum_fixed(float v, float* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += scratch[w];
        scratch[32] = tot;
    }
    __syncthreads();
    const float tot = scratch[32];
    __syncthreads();
    return tot;
}

// Called by every thread of every block once the block's shared-memory totals
// sP/sI/sC are final (after a __syncthreads). Adds them to the global
// accumulators; the last block computes the statistics and resets.
// The last block avoids FP64 (slow on this part): with I_e the integer gate
// sums and N = sum_e I_e, the importance deviations E I_e - N are exact in
// int64, so CV^2 = sum_e (E I_e - N)^2 / (E N^2) loses nothing to
// cancellation, and aux = E / (T^2 k 2^32) * sum_e count_e * P_e (fixed
// point) is a sum of positive terms.
static __device__ void aux_publish_and_finalize(int T, int E, int k, AuxAcc acc, AuxOut out,
                                                const unsigned long long* sP,
                                                const unsigned long long* sI,
                                                const unsigned int* sC) {
    __shared__ float red[33];
    __shared__ long long s_nsum[32];
    __shared__ long long s_n;
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
    const float inv_fix = 2.3283064365386963e-10f;  // 2^-32
    const float invT = 1.f / (float)T, invTk = 1.f / ((float)T * (float)k);
    // N = sum of the gate sums (exact, int64), fixed-order reduction
    long long nloc = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) nloc += (long long)__ldcg(&acc.I[e]);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) nloc += __shfl_xor_sync(0xffffffffu, nloc, o);
    if (lane == 0) s_nsum[warp] = nloc;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long n = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) n += s_nsum[w];
        s_n = n;
    }
    __syncthreads();
    const long long N = s_n;
    float s_fp = 0.f, s_dev = 0.f;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const unsigned long long pe_fix = __ldcg(&acc.P[e]);
        const unsigned long long ie_fix = __ldcg(&acc.I[e]);
        const unsigned int ce = __ldcg(&acc.cnt[e]);
        const float pe = (float)pe_fix * inv_fix * invT;
        if (out.f) out.f[e] = (float)ce * invTk;
        if (out.P) out.P[e] = pe;
        if (out.I) out.I[e] = (float)ie_fix * inv_fix;
        s_fp += (float)ce * invTk * pe;
        const float dev = (float)((long long)ie_fix * E - N);
        s_dev += dev * dev;
    }
    const float sum_fp = block_sum_fixed(s_fp, red);
    const float sum_dev = block_sum_fixed(s_dev, red);
    if (threadIdx.x == 0) {
        const float n = (float)N;
        const float cv2 = sum_dev / ((float)E * n * n);
        out.out3[0] = sum_fp * (float)E;
        out.out3[1] = cv2;
        out.out3[2] = out.w_imp * cv2;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        acc.P[e] = 0;
        acc.I[e] = 0;
        acc.cnt[e] = 0;
    }
    if (threadIdx.x == 0) *acc.ticket = 0;
}

}  // namespace moe
