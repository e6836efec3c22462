// Combine back to token order, load-balance statistics, bias update.
//
// Method: "MoE notes" (chiang97912.github.io): y = sum_i G(x)_i E_i(x),
// section Auxiliary loss (Importance(X) = sum_x G(x), CV = sigma / mu,
// L = w CV^2); heavensheep.xyz MoE notes, section Training (Switch aux loss
// from f_i and P_i; DeepSeek-V3 per-expert bias adjusted online by load);
// ld246.com MoE Q3/Q4 (bias direction; shared experts always used).
#include "moe_internal.cuh"

namespace moe {

// ------------------------------------------------------------------ combine
template <typename Tv>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const void* p, float* f) {
        float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ static void store(void* p, const float* f) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void* p, float* f) {
        uint4 v = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ static void store(void* p, const float* f) {
        uint4 v;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = v;
    }
};

// One warp per token. y[t] = sum_{kept j} w[t,j] yp[slot[t,j]] + sum_s ys[s,t],
// fp32 accumulation in the fixed order j = 0..k-1, then s = 0..S-1.
template <typename Tv>
__global__ void __launch_bounds__(256) combine_kernel(int T, int d, int k, int S,
                                                      const Tv* __restrict__ yp,
                                                      const int32_t* __restrict__ slot,
                                                      const float* __restrict__ w,
                                                      const Tv* __restrict__ ys, Tv* __restrict__ y,
                                                      int* status) {
    constexpr int VN = Vec<Tv>::N;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int my_slot = lane < k ? slot[(size_t)t * k + lane] : -1;
    const float my_w = lane < k ? w[(size_t)t * k + lane] : 0.f;
    const unsigned live = __ballot_sync(0xffffffffu, my_slot >= 0);
    const int nvec = d / VN;
    bool bad = false;
    for (int v0 = 0; v0 < nvec; v0 += 32) {
        const int v = v0 + lane;
        const bool ok = v < nvec;
        float acc[VN];
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] = 0.f;
        unsigned m = live;
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            const int r = __shfl_sync(0xffffffffu, my_slot, j);
            const float g = __shfl_sync(0xffffffffu, my_w, j);
            if (ok) {
                float val[VN];
                Vec<Tv>::load(yp + (size_t)r * d + (size_t)v * VN, val);
#pragma unroll
                for (int i = 0; i < VN; ++i) acc[i] = fmaf(g, val[i], acc[i]);
            }
        }
        if (ok) {
            for (int s = 0; s < S; ++s) {
                float val[VN];
                Vec<Tv>::load(ys + ((size_t)s * T + t) * d + (size_t)v * VN, val);
#pragma unroll
                for (int i = 0; i < VN; ++i) acc[i] += val[i];
            }
#pragma unroll
            for (int i = 0; i < VN; ++i) bad |= !isfinite(acc[i]);
            Vec<Tv>::store(y + (size_t)t * d + (size_t)v * VN, acc);
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, DEV_NONFINITE);
}

cudaError_t launch_combine(const Shape& s, const void* yp, const int32_t* slot, const float* w,
                           const void* ys, void* y, int* status, cudaStream_t st) {
    dim3 grid((s.T + 7) / 8), block(256);
    if (s.dtype == MOE_BF16)
        combine_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(
            s.T, s.d, s.k, ys ? s.S : 0, (const __nv_bfloat16*)yp, slot, w,
            (const __nv_bfloat16*)ys, (__nv_bfloat16*)y, status);
    else
        combine_kernel<float><<<grid, block, 0, st>>>(s.T, s.d, s.k, ys ? s.S : 0,
                                                      (const float*)yp, slot, w,
                                                      (const float*)ys, (float*)y, status);
    return cudaGetLastError();
}

// --------------------------------------------------------------- statistics
// One launch. Each block takes kAuxBlockTokens tokens and adds, per expert e,
//   sum_t probs[t,e]           as 32.32 fixed point (uint64)
//   sum of gates assigned to e as 32.32 fixed point (uint64)
//   number of assignments to e (uint32)
// into the workspace accumulators with integer atomics. Integer addition is
// associative, so the totals do not depend on the order blocks run in. The
// last block to finish (ticket counter) turns the totals into f, P,
// importance, aux and CV^2 with a fixed-order tree, then zeroes the
// accumulators for the next call. Quantisation: 2^-32 per term.
struct AuxAcc {
    unsigned long long* P;  // [E]
    unsigned long long* I;  // [E]
    unsigned int* cnt;      // [E]
    unsigned int* ticket;   // [1]
};

constexpr float kFix = 4294967296.0f;  // 2^32

__device__ __forceinline__ unsigned long long to_fix(float v) {
    // v in [0, 1]; v * 2^32 is exact in fp32, then rounded to an integer
    return v > 0.f ? __float2ull_rn(v * kFix) : 0ull;
}

// fixed-order sum over a block of doubles (one value per thread)
__device__ double block_sum_fixed(double v, double* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    double tot = 0.0;
    if (threadIdx.x == 0) {
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += scratch[w];
        scratch[32] = tot;
    }
    __syncthreads();
    tot = scratch[32];
    __syncthreads();
    return tot;
}

__global__ void __launch_bounds__(256) aux_kernel(int T, int E, int k, int nblk, float w_imp,
                                                  const float* __restrict__ probs,
                                                  const int32_t* __restrict__ ids,
                                                  const float* __restrict__ w, AuxAcc acc,
                                                  float* f, float* P, float* I, float* out3) {
    extern __shared__ unsigned long long sm64[];
    unsigned long long* sP = sm64;
    unsigned long long* sI = sm64 + E;
    unsigned int* sC = reinterpret_cast<unsigned int*>(sm64 + 2 * E);
    __shared__ double red[33];
    __shared__ int is_last;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        sP[e] = 0;
        sI[e] = 0;
        sC[e] = 0;
    }
    __syncthreads();
    const int t0 = blockIdx.x * kAuxBlockTokens;
    const int nt = min(kAuxBlockTokens, T - t0);
    // column sums of probs: thread -> (column e, every rstep-th row)
    const int rstep = E <= (int)blockDim.x ? (int)blockDim.x / E : 1;
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + (int)threadIdx.x % min(E, (int)blockDim.x);
        const int r0 = E <= (int)blockDim.x ? (int)threadIdx.x / E : 0;
        if (e < E && r0 < rstep) {
            unsigned long long acc_p = 0;
            for (int r = r0; r < nt; r += rstep) acc_p += to_fix(probs[(size_t)(t0 + r) * E + e]);
            atomicAdd(&sP[e], acc_p);
        }
        if (E <= (int)blockDim.x) break;
    }
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
        const int e = ids[(size_t)t0 * k + i];
        if (e < 0 || e >= E) continue;
        atomicAdd(&sI[e], to_fix(w[(size_t)t0 * k + i]));
        atomicAdd(&sC[e], 1u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (sP[e]) atomicAdd(&acc.P[e], sP[e]);
        if (sI[e]) atomicAdd(&acc.I[e], sI[e]);
        if (sC[e]) atomicAdd(&acc.cnt[e], sC[e]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(acc.ticket, 1u) == (unsigned)(nblk - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // last block: totals -> statistics (fixed-order reductions), then reset
    const double inv_fix = 1.0 / 4294967296.0;
    double s_fp = 0.0, s_i = 0.0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double pe = (double)__ldcg(&acc.P[e]) * inv_fix / (double)T;
        const double ie = (double)__ldcg(&acc.I[e]) * inv_fix;
        const double fe = (double)__ldcg(&acc.cnt[e]) / ((double)T * (double)k);
        if (f) f[e] = (float)fe;
        if (P) P[e] = (float)pe;
        if (I) I[e] = (float)ie;
        s_fp += fe * pe;
        s_i += ie;
    }
    const double sum_fp = block_sum_fixed(s_fp, red);
    const double mean = block_sum_fixed(s_i, red) / (double)E;
    double s_v = 0.0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double d = (double)__ldcg(&acc.I[e]) * inv_fix - mean;
        s_v += d * d;
    }
    const double var = block_sum_fixed(s_v, red) / (double)E;
    if (threadIdx.x == 0) {
        const double cv2 = var / (mean * mean);
        out3[0] = (float)(sum_fp * (double)E);
        out3[1] = (float)cv2;
        out3[2] = (float)((double)w_imp * cv2);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        acc.P[e] = 0;
        acc.I[e] = 0;
        acc.cnt[e] = 0;
    }
    if (threadIdx.x == 0) *acc.ticket = 0;
}

cudaError_t launch_aux(const Shape& s, const float* probs, const int32_t* ids, const float* w,
                       void* acc_mem, float* f, float* P, float* I, float* out3,
                       cudaStream_t st) {
    const int nblk = (s.T + kAuxBlockTokens - 1) / kAuxBlockTokens;
    AuxAcc acc;
    acc.P = static_cast<unsigned long long*>(acc_mem);
    acc.I = acc.P + s.E;
    acc.cnt = reinterpret_cast<unsigned int*>(acc.I + s.E);
    acc.ticket = acc.cnt + s.E;
    const size_t smem = (size_t)s.E * (2 * sizeof(unsigned long long) + sizeof(unsigned int)) + 8;
    aux_kernel<<<nblk, 256, smem, st>>>(s.T, s.E, s.k, nblk, s.w_imp, probs, ids, w, acc, f, P,
                                        I, out3);
    return cudaGetLastError();
}

// -------------------------------------------------------------- bias update
__global__ void bias_update_kernel(int T, int E, int k, const int32_t* __restrict__ counts,
                                   float* __restrict__ bias, float rate) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const long long diff = (long long)counts[e] * E - (long long)T * k;
    float b = bias[e];
    if (diff > 0) b = b - rate;
    if (diff < 0) b = b + rate;
    bias[e] = b;
}

cudaError_t launch_bias_update(const Shape& s, const int32_t* counts, float* bias, float rate,
                               cudaStream_t st) {
    bias_update_kernel<<<(s.E + 255) / 256, 256, 0, st>>>(s.T, s.E, s.k, counts, bias, rate);
    return cudaGetLastError();
}

}  // namespace moe
