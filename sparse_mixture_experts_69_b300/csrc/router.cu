// Router kernels: the transposed copy of the router weights for the tensor-core
// GEMM, the float32 (SIMT) router GEMM, and the per-token selection kernel
// (noise, max-subtracted softmax, selection bias, top-k, gates).
//
// Method: "MoE notes" (chiang97912.github.io), sections Expert selection and
// KeepTopK; heavensheep.xyz MoE notes, section Training (softmax numerics);
// ld246.com MoE Q3 (bias on the softmax scores, for the top-k choice only).
#include <float.h>

#include <algorithm>

#include "aux_common.cuh"

namespace moe {

// ------------------------------------------------------------------ transpose
// WgT[n, i] = Wg[i, n] for n < E; WgT[E + n, i] = Wnoise[i, n]. 32x32 tiles.
// The router weights are inputs no kernel of this library writes, and the only
// reader of WgT, the router GEMM, is complete whenever a later kernel launches
// (the selection kernel after it signals its dependents only after its own
// wait). So the copy runs before the wait for the preceding kernel, under that
// kernel's tail; the wait at the end keeps the completion order.
template <typename Tv>
__global__ void transpose_router_w_kernel(int d, int E, const Tv* __restrict__ Wg,
                                          const Tv* __restrict__ Wn, Tv* __restrict__ wgT) {
    pdl_trigger();
    __shared__ Tv tile[32][33];
    const Tv* src = blockIdx.z == 0 ? Wg : Wn;
    const int i0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        int i = i0 + r, n = n0 + threadIdx.x;
        if (i < d && n < E) tile[r][threadIdx.x] = src[(size_t)i * E + n];
    }
    __syncthreads();
    Tv* dst = wgT + (size_t)blockIdx.z * E * d;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        int n = n0 + r, i = i0 + threadIdx.x;
        if (i < d && n < E) dst[(size_t)n * d + i] = tile[threadIdx.x][r];
    }
    pdl_wait();
}

cudaError_t launch_transpose_router_w(const Shape& s, const void* Wg, const void* Wnoise,
                                      void* wgT, cudaStream_t st) {
    dim3 grid((s.E + 31) / 32, (s.d + 31) / 32, Wnoise ? 2 : 1), block(32, 8);
    if (s.dtype == MOE_BF16)
        return launch_k(transpose_router_w_kernel<uint16_t>, grid, block, 0, st, s.d, s.E,
                        (const uint16_t*)Wg, (const uint16_t*)Wnoise, (uint16_t*)wgT);
    else
        return launch_k(transpose_router_w_kernel<float>, grid, block, 0, st, s.d, s.E,
                        (const float*)Wg, (const float*)Wnoise, (float*)wgT);
}

// ------------------------------------------------------- float32 router GEMM
// z[t, n] = sum_i x[t, i] W[i, n], W = [Wg | Wnoise] read in place ([d,E] each).
// 64x64 output tile per block, 16-deep k slices, 4x4 per thread, fp32 FMA.
__global__ void __launch_bounds__(256) router_gemm_f32_kernel(
    int T, int d, int E, int Nr, const float* __restrict__ x, const float* __restrict__ Wg,
    const float* __restrict__ Wn, const float* __restrict__ offset, float* __restrict__ logits,
    float* __restrict__ zn) {
    pdl_trigger();
    pdl_wait();
    __shared__ float As[16][64 + 1];
    __shared__ float Bs[16][64 + 1];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            int r = i / 16, kk = i % 16, t = m0 + r, kx = k0 + kk;
            As[kk][r] = (t < T && kx < d) ? x[(size_t)t * d + kx] : 0.f;
        }
        for (int i = threadIdx.x; i < 16 * 64; i += 256) {
            int kk = i / 64, c = i % 64, n = n0 + c, kx = k0 + kk;
            float v = 0.f;
            if (kx < d && n < Nr) v = n < E ? Wg[(size_t)kx * E + n] : Wn[(size_t)kx * E + (n - E)];
            Bs[kk][c] = v;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int t = m0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int n = n0 + tx * 4 + j;
            if (n >= Nr) continue;
            if (n < E)
                logits[(size_t)t * E + n] = acc[i][j] + (offset ? offset[n] : 0.f);
            else
                zn[(size_t)t * E + (n - E)] = acc[i][j];
        }
    }
}

cudaError_t launch_router_gemm_f32(const Shape& s, int Nr, const float* x, const float* Wg,
                                   const float* Wnoise, const float* offset, float* logits,
                                   float* zn, cudaStream_t st) {
    dim3 grid((Nr + 63) / 64, (s.T + 63) / 64);
    return launch_k(router_gemm_f32_kernel, grid, dim3(256), 0, st, s.T, s.d, s.E, Nr, x, Wg,
                    Wnoise, offset, logits, zn);
}

// ------------------------------------------------------------------ selection
struct SelectArgs {
    int T, E, k, nc, renorm, from_scores;  // nc >= k candidates are written
    RouterLogits rl;       // z = x.Wg (+ offset) and zn = x.Wnoise, or their K parts
    float* logits_out;     // [T,E] or NULL: z, written when formed from K parts
    const float* noise;    // [T,E] or NULL
    int draw;              // 1: noise drawn from (seed, ctr) instead of read
    unsigned long long seed, ctr;
    const float* bias;     // [E] or NULL
    const float* sel_in;   // from_scores: [T,E]
    const float* probs_in; // from_scores: [T,E]
    float* probs;          // out [T,E]
    float* sel;            // out [T,E] or NULL
    int32_t* ids;          // out [T,nc]
    float* w;              // out [T,nc]
    int* status;
};

// softplus(u) = log(1 + e^u) = max(u, 0) + log(1 + e^-|u|), with the fast
// exponential and logarithm (a few ulp: far inside the 1e-4 relative tolerance
// the probabilities are held to).
__device__ __forceinline__ float softplus_f(float u) {
    return fmaxf(u, 0.f) + __logf(1.f + __expf(-fabsf(u)));
}

// ------------------------------------------------------------- drawn noise
// The noisy router's StandardNormal() draw eps[t,e] for the stream (seed, ctr):
// the counter-based Philox4x32-10 (Salmon, Moraes, Dror and Shaw, SC 2011;
// ten rounds of two 32x32 -> 64-bit products by 0xD2511F53 and 0xCD9E8D57,
// key bumped by 0x9E3779B9 and 0xBB67AE85) with counter words (e, t, ctr low,
// ctr high) and key (seed low, seed high); the top 24 bits of its first two
// words give u1 in (0, 1] and u2 in [0, 1), and the Box-Muller transform
// sqrt(-2 ln u1) cos(2 pi u2) the draw.
__device__ __forceinline__ float draw_eps(unsigned long long seed, unsigned long long ctr, int t,
                                          int e) {
    uint32_t c0 = (uint32_t)e, c1 = (uint32_t)t, c2 = (uint32_t)ctr, c3 = (uint32_t)(ctr >> 32);
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    const float u1 = (float)((c0 >> 8) + 1u) * 0x1p-24f;  // exact: 24-bit integers
    const float u2 = (float)(c1 >> 8) * 0x1p-24f;
    return sqrtf(-2.f * logf(u1)) * cospif(2.f * u2);
}

// One thread per (t, e), row-major [T,E].
__global__ void __launch_bounds__(256) draw_noise_kernel(int T, int E, unsigned long long seed,
                                                         unsigned long long ctr,
                                                         float* __restrict__ noise) {
    pdl_trigger();
    pdl_wait();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * E) return;
    noise[i] = draw_eps(seed, ctr, (int)(i / E), (int)(i % E));
}

cudaError_t launch_draw_noise(const Shape& s, float* noise, cudaStream_t st) {
    const long long n = (long long)s.T * s.E;
    return launch_k(draw_noise_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, s.T,
                    s.E, s.noise_seed, s.noise_counter, noise);
}

// One token's inputs for the lanes of a warp: lane l holds experts l, l+32, ...
template <int EPL>
struct TokenRegs {
    float z[EPL];    // logits (from_scores: selection scores)
    float zn[EPL];   // noise logits x.Wnoise (from_scores: probabilities)
    float eps[EPL];  // standard-normal noise
};

// PARTS: the logits come as K parts of the router GEMM (a.rl.nsplit > 1).
template <int EPL, bool PARTS>
__device__ __forceinline__ void load_token(const SelectArgs& a, int t, TokenRegs<EPL>& r) {
    const int lane = threadIdx.x & 31;
    const size_t row = (size_t)t * a.E;
    const bool noisy = a.rl.zn && (a.noise || a.draw);
    const RouterLogits& rl = a.rl;
    if constexpr (PARTS) {
        // the K parts of [z | zn], added in part order, then the offset
        const size_t plane = (size_t)a.T * rl.Nr;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            r.z[i] = 0.f;
            r.zn[i] = 0.f;
        }
        for (int q = 0; q < rl.nsplit; ++q) {
            const float* pr = rl.part + q * plane + (size_t)t * rl.Nr;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < a.E) {
                    r.z[i] += pr[e];
                    if (noisy) r.zn[i] += pr[a.E + e];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (!a.draw) r.eps[i] = 0.f;
            if (e < a.E) {
                if (rl.offset) r.z[i] += rl.offset[e];
                if (a.logits_out) a.logits_out[row + e] = r.z[i];
                if (noisy && !a.draw) r.eps[i] = a.noise[row + e];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            const bool in = e < a.E;
            if (!a.draw) r.eps[i] = 0.f;  // drawn noise: already in r (draw_token_eps)
            if (a.from_scores) {
                r.z[i] = in ? a.sel_in[row + e] : 0.f;
                r.zn[i] = in ? a.probs_in[row + e] : 0.f;
            } else {
                r.z[i] = in ? rl.logits[row + e] : 0.f;
                r.zn[i] = in && noisy ? rl.zn[row + e] : 0.f;
                if (in && noisy && !a.draw) r.eps[i] = a.noise[row + e];
            }
        }
    }
}

// Drawn noise of token t (a.draw). It reads no global memory, so the selection
// kernels make the draws before they wait for the router GEMM, under its run.
template <int EPL>
__device__ __forceinline__ void draw_token_eps(const SelectArgs& a, int t, TokenRegs<EPL>& r) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        r.eps[i] = e < a.E ? draw_eps(a.seed, a.ctr, t, e) : 0.f;
    }
}

// Selection for token t from its loaded inputs. On return pr[] holds this
// lane's probabilities (also stored to sp[0..E), the warp's row of shared
// memory, when sp is not NULL; E <= 256 needs it), and lanes j < nc hold the
// j-th candidate (my_id) and its gate (my_w): p_j over the sum of p of the
// first k candidates (renorm), else p_j.
template <int EPL>
__device__ __forceinline__ void select_regs(const SelectArgs& a, int t, const TokenRegs<EPL>& r,
                                            float (&pr)[EPL], float* sp, int& my_id,
                                            float& my_w) {
    const int lane = threadIdx.x & 31;
    const int E = a.E;
    const size_t row = (size_t)t * E;
    // Scores become unsigned keys in the same order (sign flip of the float's
    // bits; -0 is first made +0 so the two compare equal, as floats do).
    unsigned key[EPL];
    bool nonfinite = false;
    auto to_key = [](float v) {
        const unsigned b = __float_as_uint(__fadd_rn(v, 0.f));
        return b ^ ((b >> 31) ? 0xFFFFFFFFu : 0x80000000u);
    };
    if (a.from_scores) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            key[i] = e < E ? to_key(r.z[i]) : 0u;
            pr[i] = e < E ? r.zn[i] : 0.f;
            if (e < E && !isfinite(r.z[i])) nonfinite = true;
        }
    } else {
        const bool noisy = a.rl.zn && (a.noise || a.draw);
        float H[EPL];
        float m = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            float h = -FLT_MAX;
            if (e < E) {
                h = r.z[i];
                if (noisy) h = h + r.eps[i] * softplus_f(r.zn[i]);
                if (!isfinite(h)) nonfinite = true;
                m = fmaxf(m, h);
            }
            H[i] = h;
        }
        m = warp_max(m);
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            pr[i] = e < E ? __expf(H[i] - m) : 0.f;
            part += pr[i];
        }
        // the largest term is e^0 = 1, so the sum is at least 1; the
        // reciprocal is correctly rounded, as 1 / sum would be
        const float inv = __frcp_rn(warp_sum(part));
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            key[i] = 0u;
            if (e < E) {
                pr[i] = pr[i] * inv;
                a.probs[row + e] = pr[i];
                const float sc = a.bias ? pr[i] + a.bias[e] : H[i];
                if (a.sel) a.sel[row + e] = sc;
                key[i] = to_key(sc);
            }
        }
    }
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0) flag_status(a.status, DEV_NONFINITE);
    if (sp) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) sp[e] = pr[i];
        }
    }

    // top-nc: nc rounds of a warp arg-max ordered by (score desc, index asc).
    float my_p = 0.f;
    my_id = 0;
    if (EPL <= 8) {
        // One 64-bit key per expert: the score key, and below it the
        // complement of the expert index, so that the unsigned order is
        // (score desc, index asc) and every key is distinct (0: no expert).
        // Each lane sorts its keys once; a round is then the warp maximum of
        // the lanes' first keys (high word, then low word among the lanes
        // holding that high word) and a shift of the winning lane's list.
        unsigned long long k64[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            k64[i] = e < E ? ((unsigned long long)key[i] << 32) | (unsigned)~e : 0ull;
        }
        sort_desc64<EPL>(k64);
        for (int j = 0; j < a.nc; ++j) {
            const unsigned hi = (unsigned)(k64[0] >> 32), lo = (unsigned)k64[0];
            const unsigned top = __reduce_max_sync(0xffffffffu, hi);
            const int win = (int)~__reduce_max_sync(0xffffffffu, hi == top ? lo : 0u);
            if (lane == (win & 31)) {
#pragma unroll
                for (int i = 0; i + 1 < EPL; ++i) k64[i] = k64[i + 1];
                k64[EPL - 1] = 0ull;
            }
            if (lane == j) my_id = win;
        }
        __syncwarp();  // every lane's sp[] stores are visible
        if (lane < a.nc) my_p = sp[my_id];
    } else {
        // a lane-local scan per round over the candidates not yet taken
        unsigned taken = 0;
        for (int j = 0; j < a.nc; ++j) {
            unsigned bk = 0;
            int be = -1;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (be < 0 || key[i] > bk)) {
                    bk = key[i];
                    be = e;
                }
            }
            const unsigned top = __reduce_max_sync(0xffffffffu, be >= 0 ? bk : 0u);
            const int win = (int)__reduce_min_sync(
                0xffffffffu, (be >= 0 && bk == top) ? (unsigned)be : 0x7FFFFFFFu);
            const int owner = win & 31, slot_i = win >> 5;
            float mine = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i == slot_i) mine = pr[i];
            if (lane == owner) taken |= 1u << slot_i;
            const float pj = __shfl_sync(0xffffffffu, mine, owner);
            if (lane == j) {
                my_id = win;
                my_p = pj;
            }
        }
    }
    // the gates' denominator: the first k candidates' probabilities, summed
    // over the warp in a fixed order
    const float psum = warp_sum(lane < a.k ? my_p : 0.f);
    my_w = a.renorm ? my_p / psum : my_p;
    if (lane < a.nc && a.ids) {
        a.ids[(size_t)t * a.nc + lane] = my_id;
        a.w[(size_t)t * a.nc + lane] = my_w;
    }
}

// One token per warp: at the token counts of a layer call nearly the whole
// grid is resident at once, so the selection takes about one token's latency
// chain (giving a warp several tokens made that chain several times longer).
constexpr int kSelWarps = 8;

// Standalone selection.
template <int EPL, bool PARTS>
__global__ void __launch_bounds__(32 * kSelWarps, EPL <= 4 ? 4 : EPL == 8 ? 5 : 1) router_select_kernel(SelectArgs a) {
    const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
    TokenRegs<EPL> r;
    if (a.draw && t < a.T) draw_token_eps<EPL>(a, t, r);
    // dependents launch after this wait: the router GEMM before this kernel is
    // then complete, so the next router-weight copy may overwrite WgT
    pdl_wait();
    pdl_trigger();
    if (t >= a.T) return;
    load_token<EPL, PARTS>(a, t, r);
    // the warp's probabilities, where the candidates' gates are looked up
    __shared__ float s_prob[EPL <= 8 ? kSelWarps * 32 * EPL : 1];
    float pr[EPL];
    int id;
    float w;
    select_regs<EPL>(a, t, r, pr, EPL <= 8 ? s_prob + (threadIdx.x >> 5) * 32 * EPL : nullptr, id,
                     w);
}

static int sel_blocks(int T) { return (T + kSelWarps - 1) / kSelWarps; }

cudaError_t launch_router_select(const Shape& s, const RouterLogits& rl, float* logits_out,
                                 const float* noise, const float* bias, float* probs,
                                 float* sel, int32_t* ids, float* w, int from_scores,
                                 const float* sel_in, const float* probs_in, int* status,
                                 cudaStream_t st) {
    SelectArgs a;
    a.T = s.T; a.E = s.E; a.k = s.k; a.nc = s.nc; a.renorm = s.renorm;
    a.from_scores = from_scores;
    a.rl = rl; a.logits_out = logits_out; a.noise = noise; a.bias = bias;
    a.draw = rl.zn && !noise && s.noise_draw; a.seed = s.noise_seed; a.ctr = s.noise_counter;
    a.sel_in = sel_in; a.probs_in = probs_in;
    a.probs = probs; a.sel = sel; a.ids = ids; a.w = w; a.status = status;
#define MOE_SEL(EPL)                                                                       \
    return a.rl.nsplit > 1 && !from_scores                                                 \
               ? launch_k(router_select_kernel<EPL, true>, dim3(sel_blocks(s.T)),          \
                          dim3(32 * kSelWarps), 0, st, a)                                   \
               : launch_k(router_select_kernel<EPL, false>, dim3(sel_blocks(s.T)),         \
                          dim3(32 * kSelWarps), 0, st, a)
    if (s.E <= 32) MOE_SEL(1);
    if (s.E <= 64) MOE_SEL(2);
    if (s.E <= 128) MOE_SEL(4);
    if (s.E <= 256) MOE_SEL(8);
    if (s.E <= 512) MOE_SEL(16);
    MOE_SEL(32);
#undef MOE_SEL
}

// Layer path: selection fused with the capacity histogram and the
// load-balance statistics, one token per warp. Each warp leaves its token's
// probabilities in shared memory and thread e of the block adds expert e's
// column (fp32, in warp order) and turns the sum into 32.32 fixed point for
// the order-free global total; each chosen (token, expert) adds 1 to
// blk_hist[e][token / kCapBlockTokens] (the scan kernel zeroes those counters
// after reading them) and its gate to the block's importance sum.
// For E <= 128, 32 registers a thread (eight blocks an SM) keep every warp of a
// T = 8192 grid resident at once.
template <int EPL, bool PARTS>
__global__ void __launch_bounds__(32 * kSelWarps, EPL <= 4 ? 8 : EPL == 8 ? 5 : 1) router_select_fused_kernel(
    SelectArgs a, int32_t* blk_hist, int nblk_cap, AuxAcc acc, AuxOut out, int defer_final) {
    const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
    TokenRegs<EPL> r;
    if (a.draw && t < a.T) draw_token_eps<EPL>(a, t, r);
    pdl_wait();
    pdl_trigger();  // after the wait, as in router_select_kernel
    extern __shared__ unsigned long long sm64[];
    const int E = a.E;
    unsigned long long* sP = sm64;
    unsigned long long* sI = sm64 + E;
    unsigned int* sC = reinterpret_cast<unsigned int*>(sm64 + 2 * E);
    float* sProb = reinterpret_cast<float*>(sC + E);  // [kSelWarps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (t < a.T) load_token<EPL, PARTS>(a, t, r);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        sI[e] = 0;
        sC[e] = 0;
    }
    __syncthreads();
    float* mine = sProb + warp * E;
    if (t < a.T) {
        float pr[EPL];
        int id;
        float w;
        select_regs<EPL>(a, t, r, pr, mine, id, w);
        if (lane < a.k) {
            atomicAdd(&sI[id], to_fix(w));
            atomicAdd(&sC[id], 1u);
            if (blk_hist) atomicAdd(&blk_hist[(size_t)id * nblk_cap + t / kCapBlockTokens], 1);
        }
    } else {
        for (int e = lane; e < E; e += 32) mine[e] = 0.f;
    }
    __syncthreads();
    // the block's probability sum of expert e: fp32 in warp order (fixed),
    // then one fixed-point conversion, so the total over blocks is exact
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < kSelWarps; ++q) v += sProb[q * E + e];
        sP[e] = to_fix(v);
    }
    __syncthreads();
    if (defer_final)  // a later kernel finalises the statistics
        aux_publish(E, acc, sP, sI, sC);
    else
        aux_publish_and_finalize(a.T, E, a.k, acc, out, sP, sI, sC);
}

cudaError_t launch_router_select_fused(const Shape& s, const RouterLogits& rl,
                                       const float* noise, const float* bias, float* probs,
                                       int32_t* ids, float* w, int* status, int32_t* blk_hist,
                                       void* acc_mem, float* f, float* P, float* I, float* out3,
                                       bool defer_final, cudaStream_t st) {
    SelectArgs a;
    a.T = s.T; a.E = s.E; a.k = s.k; a.nc = s.nc; a.renorm = s.renorm; a.from_scores = 0;
    a.rl = rl; a.logits_out = nullptr; a.noise = noise; a.bias = bias;
    a.draw = rl.zn && !noise && s.noise_draw; a.seed = s.noise_seed; a.ctr = s.noise_counter;
    a.sel_in = nullptr; a.probs_in = nullptr;
    a.probs = probs; a.sel = nullptr; a.ids = ids; a.w = w; a.status = status;
    const int nblk_cap = (s.T + kCapBlockTokens - 1) / kCapBlockTokens;
    const AuxAcc acc = aux_acc_at(acc_mem, s.E, kAuxGroups);
    const AuxOut out{f, P, I, out3, s.w_imp};
    // sP, sI (u64), sC (u32) and the warps' probabilities (f32) per expert
    const size_t smem = (size_t)s.E * (2 * sizeof(unsigned long long) + sizeof(unsigned int) +
                                       kSelWarps * sizeof(float)) + 8;
    if (smem > 48 * 1024) {
        for (auto fn : {router_select_fused_kernel<32, false>, router_select_fused_kernel<32, true>}) {
            cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
            if (err != cudaSuccess) return err;
        }
    }
#define MOE_SEL_FUSED(EPL)                                                                 \
    return a.rl.nsplit > 1                                                                 \
               ? launch_k(router_select_fused_kernel<EPL, true>, dim3(sel_blocks(s.T)),    \
                          dim3(32 * kSelWarps), smem, st, a, blk_hist, nblk_cap, acc, out,  \
                          defer_final ? 1 : 0)                                              \
               : launch_k(router_select_fused_kernel<EPL, false>, dim3(sel_blocks(s.T)),   \
                          dim3(32 * kSelWarps), smem, st, a, blk_hist, nblk_cap, acc, out,  \
                          defer_final ? 1 : 0)
    if (s.E <= 32) MOE_SEL_FUSED(1);
    if (s.E <= 64) MOE_SEL_FUSED(2);
    if (s.E <= 128) MOE_SEL_FUSED(4);
    if (s.E <= 256) MOE_SEL_FUSED(8);
    if (s.E <= 512) MOE_SEL_FUSED(16);
    MOE_SEL_FUSED(32);
#undef MOE_SEL_FUSED
}

}  // namespace moe
