// Expert-choice routing: each expert chooses its C most probable tokens.
//
// Method: heavensheep.xyz MoE notes, Routing Function ("expert choose token"
// gives a balanced load); xutianle.me CS336-04, section 3 (routing can be
// reversed so that experts select tokens). Expert e takes the C tokens with
// the largest probs[t,e], the lower token index first among equal values.
// Its rows e*C .. e*C+C-1 hold those tokens in increasing token order, each
// gated by probs[t,e]; a token's output sums its experts in increasing e.
//
// Selection, one CTA per expert: the column probs[:,e] is staged in shared
// memory as float bit patterns (for p >= 0 the unsigned order of the bits
// is the numeric order), a 4-digit radix select finds the C-th largest value
// thr and how many of the tokens equal to it are taken, and ordered passes
// over contiguous per-warp token ranges (warp ballots, scans over warps) take
// every token above thr and the first such tokens equal to it, assigning
// rows in token order.
#include "moe_internal.cuh"

namespace moe {

namespace {
constexpr int kEcThreads = 1024;
constexpr int kEcWarps = kEcThreads / 32;

__device__ __forceinline__ unsigned lanemask_lt_ec() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive prefix sum over the warps of the block of one value per warp
// (every lane of a warp passes the same v); all threads call it. Uses
// wsum[kEcWarps + 1] in shared memory.
__device__ __forceinline__ int warp_exclusive_scan_over_block(int v, int* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int x = lane < kEcWarps ? wsum[lane] : 0;
        int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane < kEcWarps) wsum[lane] = incl - x;
    }
    __syncthreads();
    const int r = wsum[warp];
    __syncthreads();  // wsum is reused by the next call
    return r;
}
}  // namespace

__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(int T, int E, int C,
                                                               const float* __restrict__ probs,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ row_token,
                                                               float* __restrict__ row_w,
                                                               int32_t* __restrict__ tok_row,
                                                               int* status) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ unsigned col[];  // [T] value bits of probs[:,e]
    __shared__ int hist[256];
    __shared__ int wsum[kEcWarps + 1];
    __shared__ unsigned s_digit;
    __shared__ int s_left;
    const int e = blockIdx.x;
    bool nonfinite = false;
    for (int t = threadIdx.x; t < T; t += kEcThreads) {
        const float p = probs[(size_t)t * E + e];
        unsigned bits = __float_as_uint(p);
        if (!(p > 0.f)) {  // zero, negative zero, NaN or negative: lowest value
            if (p != 0.f) nonfinite = true;
            bits = 0u;
        } else if (isinf(p)) {
            nonfinite = true;
        }
        col[t] = bits;
    }
    if (__syncthreads_or(nonfinite) && threadIdx.x == 0) flag_status(status, DEV_NONFINITE);
    // radix select of the C-th largest value, 8 bits at a time from the top
    unsigned prefix = 0u, pmask = 0u;
    int left = C;  // how many still to take among values matching the prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kEcThreads) hist[i] = 0;
        __syncthreads();
        // most probabilities share their top bits: aggregate equal digits within
        // the warp so each distinct digit costs one shared-memory atomic per warp
        for (int t0 = 0; t0 < T; t0 += kEcThreads) {
            const int t = t0 + threadIdx.x;
            const unsigned v = t < T ? col[t] : 0u;
            const bool in = t < T && (v & pmask) == prefix;
            const unsigned dg = in ? (v >> shift) & 255u : 256u;  // 256: not counted
            const unsigned same = __match_any_sync(0xffffffffu, dg);
            if (in && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[dg], __popc(same));
        }
        __syncthreads();
        // warp 0 finds the digit: lane l holds bins 255-8l .. 248-8l (descending),
        // a suffix sum over lanes gives each bin the count of values above it
        if (threadIdx.x < 32) {
            const int l = threadIdx.x;
            int h[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = hist[255 - 8 * l - i];
                sum += h[i];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (l >= o) incl += n;
            }
            int above = incl - sum;  // values in the bins of lower lanes (larger digits)
            int found = -1, above_found = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (found < 0 && above + h[i] >= left) {
                    found = 255 - 8 * l - i;
                    above_found = above;
                }
                above += h[i];
            }
            // the largest digit whose cumulative count reaches `left` is in the
            // lowest lane that found one
            const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
            const int src = hit ? __ffs(hit) - 1 : 31;
            const int dsel = __shfl_sync(0xffffffffu, found, src);
            const int ab = __shfl_sync(0xffffffffu, above_found, src);
            if (l == 0) {
                s_digit = (unsigned)(dsel < 0 ? 0 : dsel);
                s_left = left - ab;
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= 255u << shift;
        left = s_left;
        __syncthreads();
    }
    // tokens above thr are all taken; of those equal to it, the first `left` in
    // token order. Warp w owns the contiguous tokens [w*L, (w+1)*L): it counts
    // its ties, then (after a scan over warps gives each warp its tie base)
    // its takes, then (after a second scan) writes its rows in token order.
    const unsigned thr = prefix;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt_ec();
    const int L = (T + kEcWarps - 1) / kEcWarps;
    const int w0 = min(T, warp * L), w1 = min(T, w0 + L);
    int nties = 0;
    for (int t0 = w0; t0 < w1; t0 += 32) {
        const int t = t0 + lane;
        nties += __popc(__ballot_sync(0xffffffffu, t < w1 && col[t] == thr));
    }
    const int tie_base0 = warp_exclusive_scan_over_block(nties, wsum);
    int tie_base = tie_base0;
    int ntake = 0;
    for (int t0 = w0; t0 < w1; t0 += 32) {
        const int t = t0 + lane;
        const unsigned v = t < w1 ? col[t] : 0u;
        const bool tie = t < w1 && v == thr;
        const unsigned tb = __ballot_sync(0xffffffffu, tie);
        const bool take = t < w1 && (v > thr || (tie && tie_base + __popc(tb & lt) < left));
        tie_base += __popc(tb);
        ntake += __popc(__ballot_sync(0xffffffffu, take));
    }
    tie_base = tie_base0;
    int row_base = warp_exclusive_scan_over_block(ntake, wsum);
    for (int t0 = w0; t0 < w1; t0 += 32) {
        const int t = t0 + lane;
        const unsigned v = t < w1 ? col[t] : 0u;
        const bool tie = t < w1 && v == thr;
        const unsigned tb = __ballot_sync(0xffffffffu, tie);
        const bool take = t < w1 && (v > thr || (tie && tie_base + __popc(tb & lt) < left));
        tie_base += __popc(tb);
        const unsigned kb = __ballot_sync(0xffffffffu, take);
        if (t < w1) {
            if (take) {
                const int r = e * C + row_base + __popc(kb & lt);
                row_token[r] = t;
                row_w[r] = __uint_as_float(v);
                tok_row[(size_t)t * E + e] = r;
            } else {
                tok_row[(size_t)t * E + e] = -1;
            }
        }
        row_base += __popc(kb);
    }
    if (threadIdx.x == 0) {
        offsets[e] = e * C;
        if (e == E - 1) offsets[E] = E * C;
    }
}

cudaError_t launch_expert_choice_select(const Shape& s, const float* probs, int32_t* offsets,
                                        int32_t* row_token, float* row_w, int32_t* tok_row,
                                        int* status, cudaStream_t st) {
    const size_t smem = sizeof(unsigned) * (size_t)s.T;
    cudaError_t err = cudaFuncSetAttribute(ec_select_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_k(ec_select_kernel, dim3(s.E), dim3(kEcThreads), smem, st, s.T, s.E, s.C, probs,
                    offsets, row_token, row_w, tok_row, status);
}

// xp[r] = x[row_token[r]] for r < rows: one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(int rows, int nvec,
                                                          const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ row_token,
                                                          uint4* __restrict__ xp) {
    // the expert GEMM that follows reads the offsets before its own wait, so
    // dependents launch only after this kernel's wait (the selection kernel
    // that wrote them is then complete)
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int t = row_token[r];
    const uint4* src = x + (size_t)t * nvec;
    for (int v = lane; v < nvec; v += 32) xp[(size_t)r * nvec + v] = __ldg(src + v);
}

cudaError_t launch_gather_rows(const Shape& s, int rows, const void* x, const int32_t* row_token,
                               void* xp, cudaStream_t st) {
    const int nvec = s.d * s.esize / 16;
    return launch_k(gather_rows_kernel, dim3((rows + 7) / 8), dim3(256), 0, st, rows, nvec,
                    (const uint4*)x, row_token, (uint4*)xp);
}

// y[t] = sum over experts e choosing t (increasing e) of probs[t,e] yp[row]
//        + sum_s ys[s,t]; one warp per token, fp32 accumulation, each lane
// owning the 16-byte vectors lane, lane+32, ... of the row.
template <typename Tv>
struct EcVec;
template <>
struct EcVec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float* p, float* o) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
    __device__ static void store(float* p, const float* o) {
        *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
    }
};
template <>
struct EcVec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16* p, float* o) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            o[2 * i] = f.x;
            o[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(__nv_bfloat16* p, const float* o) {
        uint4 v;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = v;
    }
};

template <typename Tv>
__global__ void __launch_bounds__(256) ec_combine_kernel(int T, int d, int E, int S,
                                                         const Tv* __restrict__ yp,
                                                         const int32_t* __restrict__ tok_row,
                                                         const float* __restrict__ probs,
                                                         const Tv* __restrict__ ys,
                                                         Tv* __restrict__ y) {
    pdl_trigger();
    constexpr int VN = EcVec<Tv>::N;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    pdl_wait();
    const int nvec = d / VN;
    for (int v0 = 0; v0 < nvec; v0 += 32) {
        const int v = v0 + lane;
        float acc[VN];
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] = 0.f;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int my_r = e < E ? tok_row[(size_t)t * E + e] : -1;
            const float my_g = my_r >= 0 ? probs[(size_t)t * E + e] : 0.f;
            unsigned m = __ballot_sync(0xffffffffu, my_r >= 0);
            while (m) {
                const int j = __ffs(m) - 1;
                m &= m - 1;
                const int r = __shfl_sync(0xffffffffu, my_r, j);
                const float g = __shfl_sync(0xffffffffu, my_g, j);
                if (v < nvec) {
                    float o[VN];
                    EcVec<Tv>::load(yp + (size_t)r * d + (size_t)v * VN, o);
#pragma unroll
                    for (int i = 0; i < VN; ++i) acc[i] = fmaf(g, o[i], acc[i]);
                }
            }
        }
        if (v < nvec) {
            for (int s2 = 0; s2 < S; ++s2) {
                float o[VN];
                EcVec<Tv>::load(ys + ((size_t)s2 * T + t) * d + (size_t)v * VN, o);
#pragma unroll
                for (int i = 0; i < VN; ++i) acc[i] += o[i];
            }
            EcVec<Tv>::store(y + (size_t)t * d + (size_t)v * VN, acc);
        }
    }
}

cudaError_t launch_expert_choice_combine(const Shape& s, const void* yp, const int32_t* tok_row,
                                         const float* probs, const void* ys, void* y,
                                         cudaStream_t st) {
    dim3 grid((s.T + 7) / 8), block(256);
    if (s.dtype == MOE_BF16)
        return launch_k(ec_combine_kernel<__nv_bfloat16>, grid, block, 0, st, s.T, s.d, s.E,
                        ys ? s.S : 0, (const __nv_bfloat16*)yp, tok_row, probs,
                        (const __nv_bfloat16*)ys, (__nv_bfloat16*)y);
    return launch_k(ec_combine_kernel<float>, grid, block, 0, st, s.T, s.d, s.E, ys ? s.S : 0,
                    (const float*)yp, tok_row, probs, (const float*)ys, (float*)y);
}

}  // namespace moe
