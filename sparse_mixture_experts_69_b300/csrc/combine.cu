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
// Pass 1: per block of kAuxBlockTokens tokens, per expert e (thread e):
//   part[b][e]      = sum_t probs[t,e]
//   part[b][E+e]    = sum of gates of assignments to e
//   part[b][2E+e]   = number of assignments to e
// sums run over tokens in order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(256) aux_partial_kernel(int T, int E, int k,
                                                          const float* __restrict__ probs,
                                                          const int32_t* __restrict__ ids,
                                                          const float* __restrict__ w,
                                                          float* __restrict__ part) {
    extern __shared__ unsigned char sm[];
    int32_t* sid = reinterpret_cast<int32_t*>(sm);
    float* sw = reinterpret_cast<float*>(sm + sizeof(int32_t) * kAuxBlockTokens * k);
    const int t0 = blockIdx.x * kAuxBlockTokens;
    const int nt = min(kAuxBlockTokens, T - t0);
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
        sid[i] = ids[(size_t)t0 * k + i];
        sw[i] = w[(size_t)t0 * k + i];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float P = 0.f, I = 0.f;
        int c = 0;
        for (int t = 0; t < nt; ++t) P += probs[(size_t)(t0 + t) * E + e];
        for (int i = 0; i < nt * k; ++i)
            if (sid[i] == e) {
                I += sw[i];
                ++c;
            }
        float* pb = part + (size_t)blockIdx.x * 3 * E;
        pb[e] = P;
        pb[E + e] = I;
        pb[2 * E + e] = (float)c;
    }
}

// Pass 2 (one block): totals over blocks in block order (double), then
// f = count / (T k), P = sum p / T, aux = E sum f P, CV^2 of importance.
__global__ void __launch_bounds__(1024) aux_final_kernel(int T, int E, int k, int nblk,
                                                         float w_imp,
                                                         const float* __restrict__ part,
                                                         float* f, float* P, float* I,
                                                         float* out3) {
    __shared__ double sfp[1024], simp[1024];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        double sp = 0.0, si = 0.0, sc = 0.0;
        for (int b = 0; b < nblk; ++b) {
            const float* pb = part + (size_t)b * 3 * E;
            sp += pb[e];
            si += pb[E + e];
            sc += pb[2 * E + e];
        }
        const double fe = sc / ((double)T * (double)k);
        const double Pe = sp / (double)T;
        if (f) f[e] = (float)fe;
        if (P) P[e] = (float)Pe;
        if (I) I[e] = (float)si;
        sfp[e] = fe * Pe;
        simp[e] = si;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double aux = 0.0, mean = 0.0;
        for (int e = 0; e < E; ++e) {
            aux += sfp[e];
            mean += simp[e];
        }
        mean /= (double)E;
        double var = 0.0;
        for (int e = 0; e < E; ++e) var += (simp[e] - mean) * (simp[e] - mean);
        var /= (double)E;
        const double cv2 = var / (mean * mean);
        out3[0] = (float)(aux * (double)E);
        out3[1] = (float)cv2;
        out3[2] = (float)((double)w_imp * cv2);
    }
}

cudaError_t launch_aux(const Shape& s, const float* probs, const int32_t* ids, const float* w,
                       float* part, float* f, float* P, float* I, float* out3,
                       cudaStream_t st) {
    const int nblk = (s.T + kAuxBlockTokens - 1) / kAuxBlockTokens;
    const size_t smem = (size_t)kAuxBlockTokens * s.k * (sizeof(int32_t) + sizeof(float));
    aux_partial_kernel<<<nblk, 256, smem, st>>>(s.T, s.E, s.k, probs, ids, w, part);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    aux_final_kernel<<<1, 1024, 0, st>>>(s.T, s.E, s.k, nblk, s.w_imp, part, f, P, I, out3);
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
