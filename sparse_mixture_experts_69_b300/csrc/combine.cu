// Combine back to token order, load-balance statistics, bias update.
//
// Method: "MoE notes" (chiang97912.github.io): y = sum_i G(x)_i E_i(x),
// section Auxiliary loss (Importance(X) = sum_x G(x), CV = sigma / mu,
// L = w CV^2); heavensheep.xyz MoE notes, section Training (Switch aux loss
// from f_i and P_i; DeepSeek-V3 per-expert bias adjusted online by load);
// ld246.com MoE Q3/Q4 (bias direction; shared experts always used).
#include "aux_common.cuh"

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

#ifndef MOE_COMBINE_ROWS
#define MOE_COMBINE_ROWS 1  // combine_rows_kernel for bf16 layers with 2 < k <= 8
#endif

// One warp per token. y[t] = sum_{kept j} w[t,j] yp[slot[t,j]] + sum_s ys[s,t],
// fp32 accumulation in the fixed order j = 0..k-1, then s = 0..S-1. Each lane
// covers up to VPL 16-byte vectors per pass and issues their loads together.
template <typename Tv, int VPL>
__global__ void __launch_bounds__(256, 4) combine_kernel(int T, int d, int k, int S,
                                                      const Tv* __restrict__ yp,
                                                      const int32_t* __restrict__ slot,
                                                      const float* __restrict__ w,
                                                      const Tv* __restrict__ ys, Tv* __restrict__ y,
                                                      int* status) {
    pdl_trigger();
    constexpr int VN = Vec<Tv>::N;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    pdl_wait();
    const int my_slot = lane < k ? slot[(size_t)t * k + lane] : -1;
    const float my_w = lane < k ? w[(size_t)t * k + lane] : 0.f;
    const unsigned live = __ballot_sync(0xffffffffu, my_slot >= 0);
    const int nvec = d / VN;
    bool bad = false;
    for (int v0 = 0; v0 < nvec; v0 += 32 * VPL) {
        float acc[VPL][VN];
#pragma unroll
        for (int q = 0; q < VPL; ++q)
#pragma unroll
            for (int i = 0; i < VN; ++i) acc[q][i] = 0.f;
        unsigned m = live;
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            const int r = __shfl_sync(0xffffffffu, my_slot, j);
            const float g = __shfl_sync(0xffffffffu, my_w, j);
            uint4 raw[VPL];
#pragma unroll
            for (int q = 0; q < VPL; ++q) {
                const int v = v0 + q * 32 + lane;
                if (v < nvec)
                    raw[q] = __ldg(reinterpret_cast<const uint4*>(yp + (size_t)r * d) + v);
            }
#pragma unroll
            for (int q = 0; q < VPL; ++q) {
                if (v0 + q * 32 + lane < nvec) {
                    float val[VN];
                    Vec<Tv>::load(&raw[q], val);
#pragma unroll
                    for (int i = 0; i < VN; ++i) acc[q][i] = fmaf(g, val[i], acc[q][i]);
                }
            }
        }
        for (int s = 0; s < S; ++s) {
#pragma unroll
            for (int q = 0; q < VPL; ++q) {
                const int v = v0 + q * 32 + lane;
                if (v < nvec) {
                    float val[VN];
                    const uint4 raw =
                        __ldg(reinterpret_cast<const uint4*>(ys + ((size_t)s * T + t) * d) + v);
                    Vec<Tv>::load(&raw, val);
#pragma unroll
                    for (int i = 0; i < VN; ++i) acc[q][i] += val[i];
                }
            }
        }
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int v = v0 + q * 32 + lane;
            if (v < nvec) {
#pragma unroll
                for (int i = 0; i < VN; ++i) bad |= !isfinite(acc[q][i]);
                Vec<Tv>::store(y + (size_t)t * d + (size_t)v * VN, acc[q]);
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, DEV_NONFINITE);
}

// The same sums for k <= KMAX, with every kept row's loads of a pass issued
// together before any is added (in the order j = 0..k-1, then the shared
// experts, as above): a warp keeps k times as many bytes in flight. A warp
// takes `npass` consecutive passes of one token (32 VPL vectors each); small
// token counts give each pass its own warp.
template <typename Tv, int VPL, int KMAX>
__global__ void __launch_bounds__(256, 2) combine_rows_kernel(int T, int d, int k, int S,
                                                             int npass,
                                                             const Tv* __restrict__ yp,
                                                             const int32_t* __restrict__ slot,
                                                             const float* __restrict__ w,
                                                             const Tv* __restrict__ ys,
                                                             Tv* __restrict__ y, int* status) {
    pdl_trigger();
    constexpr int VN = Vec<Tv>::N;
    const int lane = threadIdx.x & 31;
    const int nvec = d / VN;
    const int per_tok = (nvec + 32 * VPL * npass - 1) / (32 * VPL * npass);  // warps a token
    const long long wi = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int t = (int)(wi / per_tok);
    if (t >= T) return;
    const int v_begin = (int)(wi - (long long)t * per_tok) * 32 * VPL * npass;
    const int v_end = min(nvec, v_begin + 32 * VPL * npass);
    pdl_wait();
    const int my_slot = lane < k ? slot[(size_t)t * k + lane] : -1;
    const float my_w = lane < k ? w[(size_t)t * k + lane] : 0.f;
    unsigned m = __ballot_sync(0xffffffffu, my_slot >= 0);
    const int nlive = __popc(m);
    // the kept rows in order j = 0..k-1
    const Tv* rows[KMAX];
    float g[KMAX];
#pragma unroll
    for (int jj = 0; jj < KMAX; ++jj) {
        const int j = m ? __ffs(m) - 1 : 0;
        m &= m - 1;
        const int r = __shfl_sync(0xffffffffu, my_slot, j);
        g[jj] = __shfl_sync(0xffffffffu, my_w, j);
        rows[jj] = yp + (size_t)(r < 0 ? 0 : r) * d;
    }
    bool bad = false;
    for (int v0 = v_begin; v0 < v_end; v0 += 32 * VPL) {
        uint4 raw[KMAX][VPL];
#pragma unroll
        for (int jj = 0; jj < KMAX; ++jj)
#pragma unroll
            for (int q = 0; q < VPL; ++q) {
                const int v = v0 + q * 32 + lane;
                if (jj < nlive && v < v_end)
                    raw[jj][q] = __ldg(reinterpret_cast<const uint4*>(rows[jj]) + v);
            }
        float acc[VPL][VN];
#pragma unroll
        for (int q = 0; q < VPL; ++q)
#pragma unroll
            for (int i = 0; i < VN; ++i) acc[q][i] = 0.f;
#pragma unroll
        for (int jj = 0; jj < KMAX; ++jj)
#pragma unroll
            for (int q = 0; q < VPL; ++q)
                if (jj < nlive && v0 + q * 32 + lane < v_end) {
                    float val[VN];
                    Vec<Tv>::load(&raw[jj][q], val);
#pragma unroll
                    for (int i = 0; i < VN; ++i) acc[q][i] = fmaf(g[jj], val[i], acc[q][i]);
                }
        for (int s = 0; s < S; ++s) {
#pragma unroll
            for (int q = 0; q < VPL; ++q) {
                const int v = v0 + q * 32 + lane;
                if (v < v_end) {
                    float val[VN];
                    const uint4 raw1 =
                        __ldg(reinterpret_cast<const uint4*>(ys + ((size_t)s * T + t) * d) + v);
                    Vec<Tv>::load(&raw1, val);
#pragma unroll
                    for (int i = 0; i < VN; ++i) acc[q][i] += val[i];
                }
            }
        }
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int v = v0 + q * 32 + lane;
            if (v < v_end) {
#pragma unroll
                for (int i = 0; i < VN; ++i) bad |= !isfinite(acc[q][i]);
                Vec<Tv>::store(y + (size_t)t * d + (size_t)v * VN, acc[q]);
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, DEV_NONFINITE);
}

cudaError_t launch_combine(const Shape& s, const void* yp, const int32_t* slot, const float* w,
                           const void* ys, void* y, int* status, cudaStream_t st) {
    dim3 grid((s.T + 7) / 8), block(256);
#if MOE_COMBINE_ROWS
    // k <= 2 keeps the one-row-at-a-time kernel: its 64 registers give twice
    // the resident warps, and with two rows that wins (Mixtral-shaped combine
    // 82 us against 89 us, Switch-shaped 6.4 against 8.5 us, in the layer bench)
    if (s.dtype == MOE_BF16 && s.nc > 2 && s.nc <= 8) {
        // passes of a token per warp: all of them, unless the tokens are too
        // few to fill the GPU with warps (decode), then one
        const int passes = (s.d / 8 + 63) / 64;
        const int npass = (long long)s.T * 4 < (long long)num_sms() * 16 ? 1 : passes;
        const int per_tok = (passes + npass - 1) / npass;
        const dim3 g((unsigned)(((long long)s.T * per_tok + 7) / 8));
        return launch_k(combine_rows_kernel<__nv_bfloat16, 2, 8>, g, block, 0, st, s.T, s.d,
                        s.nc, ys ? s.S : 0, npass, (const __nv_bfloat16*)yp, slot, w,
                        (const __nv_bfloat16*)ys, (__nv_bfloat16*)y, status);
    }
#endif
    if (s.dtype == MOE_BF16)
        return launch_k(combine_kernel<__nv_bfloat16, 2>, grid, block, 0, st, s.T, s.d, s.nc,
                        ys ? s.S : 0, (const __nv_bfloat16*)yp, slot, w, (const __nv_bfloat16*)ys,
                        (__nv_bfloat16*)y, status);
    return launch_k(combine_kernel<float, 2>, grid, block, 0, st, s.T, s.d, s.nc, ys ? s.S : 0,
                    (const float*)yp, slot, w, (const float*)ys, (float*)y, status);
}

// --------------------------------------------------------------- statistics
// One launch; each block takes kAuxBlockTokens tokens, sums them per expert in
// shared memory (integers, see aux_common.cuh) and publishes; the last block
// finalises.
// ids and w hold `stride` columns per token; the first k are the top-k choice.
__global__ void __launch_bounds__(256) aux_kernel(int T, int E, int k, int stride, int vec4,
                                                  const float* __restrict__ probs,
                                                  const int32_t* __restrict__ ids,
                                                  const float* __restrict__ w, AuxAcc acc,
                                                  AuxOut out) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ unsigned long long sm64[];
    unsigned long long* sP = sm64;
    unsigned long long* sI = sm64 + E;
    unsigned int* sC = reinterpret_cast<unsigned int*>(sm64 + 2 * E);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        sP[e] = 0;
        sI[e] = 0;
        sC[e] = 0;
    }
    __syncthreads();
    const int t0 = blockIdx.x * kAuxBlockTokens;
    const int nt = min(kAuxBlockTokens, T - t0);
    // column sums of probs. With E a multiple of 4 whose quads divide the
    // block, each thread keeps one column quad (float4 loads) over every
    // (blockDim / (E/4))-th row in registers, then adds once to shared memory.
    const int E4 = E >> 2;
    if (vec4 && E4 <= (int)blockDim.x && (int)blockDim.x % E4 == 0) {
        const int q = (int)threadIdx.x % E4, r0 = (int)threadIdx.x / E4;
        const int rstep = (int)blockDim.x / E4;
        unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
        const float4* p4 = reinterpret_cast<const float4*>(probs);
#pragma unroll 4
        for (int r = r0; r < nt; r += rstep) {
            const float4 v = __ldg(&p4[(size_t)(t0 + r) * E4 + q]);
            a0 += to_fix(v.x);
            a1 += to_fix(v.y);
            a2 += to_fix(v.z);
            a3 += to_fix(v.w);
        }
        if (r0 < nt) {
            atomicAdd(&sP[4 * q], a0);
            atomicAdd(&sP[4 * q + 1], a1);
            atomicAdd(&sP[4 * q + 2], a2);
            atomicAdd(&sP[4 * q + 3], a3);
        }
    } else {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            unsigned long long acc_p = 0;
            for (int r = 0; r < nt; ++r) acc_p += to_fix(__ldg(&probs[(size_t)(t0 + r) * E + e]));
            atomicAdd(&sP[e], acc_p);
        }
    }
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
        const size_t a = (size_t)(t0 + i / k) * stride + i % k;
        const int e = ids[a];
        if (e < 0 || e >= E) continue;
        atomicAdd(&sI[e], to_fix(w[a]));
        atomicAdd(&sC[e], 1u);
    }
    __syncthreads();
    aux_publish_and_finalize(T, E, k, acc, out, sP, sI, sC);
}

cudaError_t launch_aux(const Shape& s, const float* probs, const int32_t* ids, const float* w,
                       void* acc_mem, int acc_groups, float* f, float* P, float* I, float* out3,
                       cudaStream_t st) {
    const int nblk = (s.T + kAuxBlockTokens - 1) / kAuxBlockTokens;
    const AuxOut out{f, P, I, out3, s.w_imp};
    const size_t smem = (size_t)s.E * (2 * sizeof(unsigned long long) + sizeof(unsigned int)) + 8;
    // float4 loads need 16-byte aligned rows
    const int vec4 = (s.E % 4 == 0) && (reinterpret_cast<uintptr_t>(probs) % 16 == 0);
    return launch_k(aux_kernel, dim3(nblk), dim3(256), smem, st, s.T, s.E, s.k, s.nc, vec4, probs,
                    ids, w, aux_acc_at(acc_mem, s.E, acc_groups), out);
}

// -------------------------------------------------------------- bias update
__global__ void bias_update_kernel(int T, int E, int k, const int32_t* __restrict__ counts,
                                   float* __restrict__ bias, float rate) {
    pdl_trigger();
    pdl_wait();
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
    return launch_k(bias_update_kernel, dim3((s.E + 255) / 256), dim3(256), 0, st, s.T, s.E, s.k,
                    counts, bias, rate);
}

}  // namespace moe
