// Capacity assignment and dispatch.
//
// Method: "MoE notes" (chiang97912.github.io), section Expert capacity
// (capacity = tokens per batch / experts * capacity factor); mkbk-pku.cn MoE
// notes, load-balance section (a token beyond capacity is dropped) and the
// grouped-GEMM section (tokens bucketed by expert, packed contiguously).
//
// Token-order priority without any inter-block waiting, in three steps:
//   1. hist : per block of 256 tokens, assignments per expert (cap_hist_kernel,
//             or the layer's fused selection kernel)
//   2. scan : per expert, exclusive prefix over blocks (block base); totals
//             give counts, kept = min(counts, C), offsets = scan of kept
//   3. slot : within a block, the rank of (t, e) among earlier tokens of the
//             block that chose e, from per-warp lane bitmasks; slot = base + rank
// Steps 2 and 3 are one launch (cap_scan_slot_kernel, every block reading the
// histograms itself) up to kMaxFusedCapBlocks blocks, two beyond. Then a
// permute copies each token's row to its kept rows.
#include "moe_internal.cuh"

namespace moe {

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// blk_hist is expert-major: [E][nblk]; written whole here (no atomics into it)
__global__ void __launch_bounds__(kCapBlockTokens) cap_hist_kernel(
    int T, int k, int E, int nblk, const int32_t* __restrict__ ids, int32_t* __restrict__ blk_hist,
    int* status) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * kCapBlockTokens + threadIdx.x;
    bool bad = false;
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            if (e >= 0 && e < E) {
                atomicAdd(&hist[e], 1);
                for (int q = 0; q < j; ++q)
                    if (ids[(size_t)t * k + q] == e) bad = true;  // ids must be distinct
            } else {
                bad = true;
            }
        }
    }
    if (bad) flag_status(status, DEV_BAD_ARG);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        blk_hist[(size_t)e * nblk + blockIdx.x] = hist[e];
}

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// One block of 1024 threads. Warp w scans experts w, w+32, ...
__global__ void __launch_bounds__(1024) cap_scan_kernel(
    int nblk, int E, int C, int pad, int32_t* __restrict__ blk_hist, int32_t* __restrict__ blk_base,
    int32_t* __restrict__ counts, int32_t* __restrict__ kept, int32_t* __restrict__ offsets) {
    pdl_trigger();
    pdl_wait();
    __shared__ int kp[1024];
    __shared__ int wsum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = warp; e < E; e += 32) {
        int running = 0;
        for (int b0 = 0; b0 < nblk; b0 += 32) {
            int b = b0 + lane;
            int v = 0;
            if (b < nblk) {
                v = blk_hist[(size_t)e * nblk + b];
                blk_hist[(size_t)e * nblk + b] = 0;  // counters start at zero for the next call
            }
            int incl = warp_incl_scan(v);
            if (b < nblk) blk_base[(size_t)e * nblk + b] = running + incl - v;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            counts[e] = running;
            int kv = running < C ? running : C;
            kept[e] = kv;
            kp[e] = kv;
        }
    }
    __syncthreads();
    // exclusive scan of kept over experts (E <= 1024)
    const int e = threadIdx.x;
    int v = e < E ? kp[e] : 0;
    int incl = warp_incl_scan(v);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = wsum[lane];
        int si = warp_incl_scan(s);
        wsum[lane] = si - s;
    }
    __syncthreads();
    if (e < E) offsets[e] = pad ? e * C : wsum[warp] + incl - v;
    if (e == E - 1) offsets[E] = pad ? E * C : wsum[warp] + incl;
}

// Dynamic smem: mask[8][E] lane bitmasks (bit l of mask[w][e]: lane l of warp w chose e)
__global__ void __launch_bounds__(kCapBlockTokens) cap_slot_kernel(
    int T, int k, int E, int C, int nblk, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ slot, int32_t* __restrict__ row_token) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ unsigned mask[];
    constexpr int W = kCapBlockTokens / 32;
    for (int i = threadIdx.x; i < W * E; i += blockDim.x) mask[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kCapBlockTokens + threadIdx.x;
    if (t < T)
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            if (e >= 0 && e < E) atomicOr(&mask[warp * E + e], 1u << lane);
        }
    __syncthreads();
    if (t >= T) return;
    const unsigned lt = lanemask_lt();
    for (int j = 0; j < k; ++j) {
        const size_t a = (size_t)t * k + j;
        int e = ids[a];
        int out = -1;
        if (e >= 0 && e < E) {
            int r = __popc(mask[warp * E + e] & lt);
            for (int w = 0; w < warp; ++w) r += __popc(mask[w * E + e]);
            int sl = blk_base[(size_t)e * nblk + blockIdx.x] + r;
            if (sl < C) {
                out = offsets[e] + sl;
                row_token[out] = t;
            }
        }
        slot[a] = out;
    }
}

// Scan and slots in one launch, for up to kMaxFusedCapBlocks token blocks.
// Every block reads the histogram rows itself: counts[e] = sum over blocks,
// its own base = sum over earlier blocks, offsets = exclusive scan of
// kept = min(counts, C) over experts (block 0 writes counts, kept, offsets).
// Then the lane-bitmask ranks of cap_slot_kernel. The last block to finish
// reading (ticket) zeroes the histogram counters and the ticket.
constexpr int kMaxFusedCapBlocks = 256;

__global__ void __launch_bounds__(kCapBlockTokens) cap_scan_slot_kernel(
    int T, int k, int E, int C, int pad, int nblk, const int32_t* __restrict__ ids,
    int32_t* __restrict__ blk_hist, unsigned int* __restrict__ ticket,
    int32_t* __restrict__ counts, int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
    int32_t* __restrict__ slot, int32_t* __restrict__ row_token) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ unsigned mask[];                  // [8][E]
    int* s_base = reinterpret_cast<int*>(mask + (kCapBlockTokens / 32) * E);  // [E]
    int* s_off = s_base + E;                             // [E+1]
    __shared__ int wsum[kCapBlockTokens / 32];
    __shared__ int s_last;
    constexpr int W = kCapBlockTokens / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = blockIdx.x;
    for (int i = threadIdx.x; i < W * E; i += blockDim.x) mask[i] = 0;
    // per expert: base (earlier blocks) and total. Warp w takes experts w, w+W,
    // ... kE at a time, lane q block q (32 blocks a round), so the loads of
    // all its experts are in flight together.
    constexpr int kE = 8;
    for (int e0 = warp; e0 < E; e0 += W * kE) {
        int total[kE], before[kE];
#pragma unroll
        for (int i = 0; i < kE; ++i) total[i] = before[i] = 0;
        for (int q0 = 0; q0 < nblk; q0 += 32) {
            const int q = q0 + lane;
            int v[kE];
#pragma unroll
            for (int i = 0; i < kE; ++i) {
                const int e = e0 + i * W;
                v[i] = (e < E && q < nblk) ? __ldcg(blk_hist + (size_t)e * nblk + q) : 0;
            }
#pragma unroll
            for (int i = 0; i < kE; ++i) {
                total[i] += v[i];
                before[i] += q < b ? v[i] : 0;
            }
        }
#pragma unroll
        for (int i = 0; i < kE; ++i) {
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                total[i] += __shfl_xor_sync(0xffffffffu, total[i], o);
                before[i] += __shfl_xor_sync(0xffffffffu, before[i], o);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < kE; ++i) {
                const int e = e0 + i * W;
                if (e >= E) break;
                s_base[e] = before[i];
                s_off[e] = total[i] < C ? total[i] : C;  // kept, scanned below
                if (b == 0) {
                    counts[e] = total[i];
                    kept[e] = s_off[e];
                }
            }
        }
    }
    __syncthreads();
    // this block no longer needs the histogram: the last one to get here clears it
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(ticket, 1u) == (unsigned)(nblk - 1);
    }
    // exclusive scan of kept over experts: each thread scans a contiguous run
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * per, hi = min(E, lo + per);
    int run = 0;
    for (int e = lo; e < hi; ++e) run += s_off[e];
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += wsum[w];
    int acc = wbase + incl - run;
    for (int e = lo; e < hi; ++e) {
        const int kv = s_off[e];
        s_off[e] = pad ? e * C : acc;
        acc += kv;
    }
    if (threadIdx.x == blockDim.x - 1) s_off[E] = pad ? E * C : acc;
    __syncthreads();
    if (b == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
    if (s_last) {
        __threadfence();
        for (int i = threadIdx.x; i < E * nblk; i += blockDim.x) blk_hist[i] = 0;
        if (threadIdx.x == 0) *ticket = 0u;
    }
    // slots (as in cap_slot_kernel)
    const int t = b * kCapBlockTokens + threadIdx.x;
    if (t < T)
        for (int j = 0; j < k; ++j) {
            const int e = ids[(size_t)t * k + j];
            if (e >= 0 && e < E) atomicOr(&mask[warp * E + e], 1u << lane);
        }
    __syncthreads();
    if (t >= T) return;
    const unsigned lt = lanemask_lt();
    for (int j = 0; j < k; ++j) {
        const size_t a = (size_t)t * k + j;
        const int e = ids[a];
        int out = -1;
        if (e >= 0 && e < E) {
            int r = __popc(mask[warp * E + e] & lt);
            for (int w = 0; w < warp; ++w) r += __popc(mask[w * E + e]);
            const int sl = s_base[e] + r;
            if (sl < C) {
                out = s_off[e] + sl;
                row_token[out] = t;
            }
        }
        slot[a] = out;
    }
}

cudaError_t launch_capacity(const Shape& s, const int32_t* ids, int32_t* blk_hist,
                            unsigned int* cap_ticket, int32_t* blk_base, int32_t* counts,
                            int32_t* kept, int32_t* offsets, int32_t* slot, int32_t* row_token,
                            int* status, bool hist_ready, cudaStream_t st) {
    const int nblk = (s.T + kCapBlockTokens - 1) / kCapBlockTokens;
    cudaError_t err;
    if (!hist_ready) {
        err = launch_k(cap_hist_kernel, dim3(nblk), dim3(kCapBlockTokens), s.E * sizeof(int), st,
                       s.T, s.k, s.E, nblk, ids, blk_hist, status);
        if (err != cudaSuccess) return err;
    }
    if (nblk <= kMaxFusedCapBlocks) {
        const size_t smem = (size_t)(kCapBlockTokens / 32) * s.E * sizeof(unsigned) +
                            (size_t)(2 * s.E + 1) * sizeof(int);
        return launch_k(cap_scan_slot_kernel, dim3(nblk), dim3(kCapBlockTokens), smem, st, s.T,
                        s.k, s.E, s.C, s.pad, nblk, ids, blk_hist, cap_ticket, counts, kept,
                        offsets, slot, row_token);
    }
    err = launch_k(cap_scan_kernel, dim3(1), dim3(1024), 0, st, nblk, s.E, s.C, s.pad, blk_hist,
                   blk_base, counts, kept, offsets);
    if (err != cudaSuccess) return err;
    const size_t smem = (size_t)(kCapBlockTokens / 32) * s.E * sizeof(unsigned);
    return launch_k(cap_slot_kernel, dim3(nblk), dim3(kCapBlockTokens), smem, st, s.T, s.k, s.E,
                    s.C, nblk, ids, (const int32_t*)blk_base, (const int32_t*)offsets, slot,
                    row_token);
}

// ---------------------------------------------------------------- permute
// One warp per token: read the row once (16-byte vectors), write it to each of
// the token's kept rows. Algorithmic bytes: T d b read + R d b written.
#ifndef MOE_PERMUTE_VPL
#define MOE_PERMUTE_VPL 16
#endif
constexpr int kPermuteVpl = MOE_PERMUTE_VPL;  // 16-byte vectors a lane loads per pass

__global__ void __launch_bounds__(256) permute_kernel(int T, int k, int nvec, int rows,
                                                      const uint4* __restrict__ x,
                                                      const int32_t* __restrict__ slot,
                                                      uint4* __restrict__ xp,
                                                      uint4* __restrict__ y_zero,
                                                      int32_t* __restrict__ tok_need,
                                                      int* status) {
    // the expert GEMM that follows reads the offsets before its own wait, so
    // dependents launch only after this kernel's wait (the capacity kernel
    // that wrote them is then complete)
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_slot = lane < k ? slot[(size_t)t * k + lane] : -1;
    if (my_slot >= rows) {  // never produced by the capacity kernels: skip and report
        flag_status(status, DEV_BAD_ARG | DEV_SITE_PERMUTE_ROW);
        my_slot = -1;
    }
    unsigned live = __ballot_sync(0xffffffffu, my_slot >= 0);
    if (tok_need && lane == 0) tok_need[t] = __popc(live);
    if (y_zero && !live) {  // dropped everywhere: its output row is zero
        for (int v = lane; v < nvec; v += 32) y_zero[(size_t)t * nvec + v] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* src = x + (size_t)t * nvec;
    // the loop bound is warp-uniform so every shuffle has all lanes present;
    // each lane loads up to kPermuteVpl vectors before storing them
    constexpr int kV = kPermuteVpl;
    for (int v0 = 0; v0 < nvec; v0 += 32 * kV) {
        uint4 val[kV];
#pragma unroll
        for (int q = 0; q < kV; ++q) {
            const int v = v0 + 32 * q + lane;
            if (v < nvec) val[q] = __ldcs(src + v);
        }
        unsigned m = live;
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            const int r = __shfl_sync(0xffffffffu, my_slot, j);
#pragma unroll
            for (int q = 0; q < kV; ++q) {
                const int v = v0 + 32 * q + lane;
                if (v < nvec) xp[(size_t)r * nvec + v] = val[q];
            }
        }
    }
}

cudaError_t launch_permute(const Shape& s, const void* x, const int32_t* slot, void* xp,
                           void* y_zero, int32_t* tok_need, int* status, cudaStream_t st) {
    const int nvec = s.d * s.esize / 16;
    return launch_k(permute_kernel, dim3((s.T + 7) / 8), dim3(256), 0, st, s.T, s.nc, nvec,
                    s.R_max, (const uint4*)x, slot, (uint4*)xp, (uint4*)y_zero, tok_need,
                    status);
}

}  // namespace moe
