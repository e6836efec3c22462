// Sequence-level balance statistics.
//
// Method: heavensheep.xyz MoE notes, section Training: next to the batch
// balance term, DeepSeek adds one computed inside each sequence so that no
// single sequence routes lopsidedly. Here that is the Switch aux loss of
// the batch restricted to the tokens of one sequence: f = top-k choices per
// expert / (T_q k), P = mean probability, aux_q = E sum_e f P, and the mean
// of aux_q over the non-empty sequences.
//
// Two launches after the accumulators are cleared:
//   1. seq_accumulate_kernel: each warp walks 8 consecutive tokens of the
//      batch (so the whole batch is read once, by many CTAs) and sums the
//      probabilities of each expert column while the tokens belong to one
//      sequence, then adds the run to that sequence's accumulator. The sums
//      are 32.32 fixed-point integers, so the totals do not depend on the
//      order of the atomics; choice counts are integer atomics.
//   2. seq_finalize_kernel: one CTA per sequence forms f, P and aux_q from its
//      accumulators in a fixed order; the last CTA (ticket) averages aux over
//      the sequences in sequence order and resets the ticket.
#include "aux_common.cuh"

namespace moe {

namespace {
constexpr int kSeqWarpTokens = 8;
constexpr int kSeqAccThreads = 128;  // 4 warps: 32 tokens per CTA
constexpr int kSeqBatch = 8;         // probabilities loaded together before they are added
constexpr int kSeqFinThreads = 256;
}  // namespace

// Sequence of token t: the largest q with seq_offsets[q] <= t (offsets are
// non-decreasing; empty sequences are skipped over).
__device__ __forceinline__ int seq_of(const int32_t* seq_offsets, int n_seq, int t) {
    int lo = 0, hi = n_seq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seq_offsets[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kSeqAccThreads) seq_accumulate_kernel(
    int T, int E, int k, int nc, const float* __restrict__ probs, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ seq_offsets, int n_seq, unsigned long long* __restrict__ accP,
    unsigned int* __restrict__ accC, int* status) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    // tokens outside [seq_offsets[0], seq_offsets[n_seq]) belong to no sequence
    const int first = max(0, seq_offsets[0]), last = min(T, seq_offsets[n_seq]);
    const int t0 = max(first, (blockIdx.x * (kSeqAccThreads / 32) + (threadIdx.x >> 5)) *
                                  kSeqWarpTokens);
    const int t1 = min(last, (blockIdx.x * (kSeqAccThreads / 32) + (threadIdx.x >> 5) + 1) *
                                 kSeqWarpTokens);
    if (t0 >= t1) return;
    const int q0 = seq_of(seq_offsets, n_seq, t0);
    // choice counts: lane j < k of the token's row, token by token
    bool bad = false;
    {
        int q = q0;
        for (int t = t0; t < t1; ++t) {
            while (q + 1 < n_seq && seq_offsets[q + 1] <= t) ++q;
            if (lane < k) {
                const int e = ids[(size_t)t * nc + lane];
                if (e >= 0 && e < E) atomicAdd(&accC[(size_t)q * E + e], 1u);
                else bad = true;
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, DEV_BAD_ARG);
    // probability sums, 32 experts (one per lane) at a time; kSeqBatch tokens'
    // values are loaded together, then added token by token
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        int q = q0;
        unsigned long long run = 0;
        for (int tb = t0; tb < t1; tb += kSeqBatch) {
            float v[kSeqBatch];
#pragma unroll
            for (int u = 0; u < kSeqBatch; ++u)
                v[u] = (e < E && tb + u < t1) ? __ldg(&probs[(size_t)(tb + u) * E + e]) : 0.f;
#pragma unroll
            for (int u = 0; u < kSeqBatch; ++u) {
                const int t = tb + u;
                if (t >= t1) break;
                if (q + 1 < n_seq && seq_offsets[q + 1] <= t) {  // the run's sequence ended
                    if (e < E && run) atomicAdd(&accP[(size_t)q * E + e], run);
                    run = 0;
                    while (q + 1 < n_seq && seq_offsets[q + 1] <= t) ++q;
                }
                run += to_fix(v[u]);
            }
        }
        if (e < E && run) atomicAdd(&accP[(size_t)q * E + e], run);
    }
}

__global__ void __launch_bounds__(kSeqFinThreads) seq_finalize_kernel(
    int T, int E, int k, const int32_t* __restrict__ seq_offsets, int n_seq,
    const unsigned long long* __restrict__ accP, const unsigned int* __restrict__ accC,
    float* __restrict__ f_seq, float* __restrict__ P_seq, float* __restrict__ aux_seq,
    float* __restrict__ aux_mean, unsigned int* __restrict__ ticket, int* status) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[kSeqFinThreads / 32];
    __shared__ int s_last;
    const int q = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int t0 = seq_offsets[q], t1 = seq_offsets[q + 1];
    if (t0 < 0 || t1 < t0 || t1 > T) {
        if (tid == 0) flag_status(status, DEV_BAD_ARG);
        t0 = t1 = 0;  // treated as empty
    }
    const int Tq = t1 - t0;
    float prod = 0.f;
    for (int e = tid; e < E; e += kSeqFinThreads) {
        float f = 0.f, P = 0.f;
        if (Tq > 0) {
            f = (float)accC[(size_t)q * E + e] / ((float)Tq * (float)k);
            P = (float)((double)accP[(size_t)q * E + e] * (1.0 / 4294967296.0)) / (float)Tq;
        }
        if (f_seq) f_seq[(size_t)q * E + e] = f;
        if (P_seq) P_seq[(size_t)q * E + e] = P;
        prod += f * P;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) prod += __shfl_xor_sync(0xffffffffu, prod, o);
    if (lane == 0) red[warp] = prod;
    __syncthreads();
    if (tid == 0) {
        float a = 0.f;
        for (int r = 0; r < kSeqFinThreads / 32; ++r) a += red[r];
        aux_seq[q] = Tq > 0 ? (float)E * a : 0.f;
        __threadfence();
        s_last = atomicAdd(ticket, 1u) == (unsigned)(n_seq - 1);
    }
    __syncthreads();
    if (s_last && tid == 0) {
        __threadfence();
        float total = 0.f;
        int nonempty = 0;
        for (int i = 0; i < n_seq; ++i) {
            const int a0 = seq_offsets[i], a1 = seq_offsets[i + 1];
            if (a0 < 0 || a1 < a0 || a1 > T) continue;
            if (a1 > a0) {
                total += __ldcg(&aux_seq[i]);
                ++nonempty;
            }
        }
        *aux_mean = nonempty ? total / (float)nonempty : 0.f;
        *ticket = 0u;
    }
}

size_t seq_aux_scratch_bytes(int E, int n_seq) {
    return (size_t)n_seq * E * (sizeof(unsigned long long) + sizeof(unsigned int));
}

cudaError_t launch_seq_aux(const Shape& s, const float* probs, const int32_t* ids,
                           const int32_t* seq_offsets, int n_seq, float* f_seq, float* P_seq,
                           float* aux_seq, float* aux_mean, void* scratch, unsigned int* ticket,
                           int* status, cudaStream_t st) {
    unsigned long long* accP = static_cast<unsigned long long*>(scratch);
    unsigned int* accC = reinterpret_cast<unsigned int*>(accP + (size_t)n_seq * s.E);
    cudaError_t err = cudaMemsetAsync(scratch, 0, seq_aux_scratch_bytes(s.E, n_seq), st);
    if (err != cudaSuccess) return err;
    const int warps = (s.T + kSeqWarpTokens - 1) / kSeqWarpTokens;
    const int per = kSeqAccThreads / 32;
    err = launch_k(seq_accumulate_kernel, dim3((warps + per - 1) / per), dim3(kSeqAccThreads), 0,
                   st, s.T, s.E, s.k, s.nc, probs, ids, seq_offsets, n_seq, accP, accC, status);
    if (err != cudaSuccess) return err;
    return launch_k(seq_finalize_kernel, dim3(n_seq), dim3(kSeqFinThreads), 0, st, s.T, s.E, s.k,
                    seq_offsets, n_seq, (const unsigned long long*)accP,
                    (const unsigned int*)accC, f_seq, P_seq, aux_seq, aux_mean, ticket, status);
}

}  // namespace moe
