// Sequence-level balance statistics.
//
// Method: heavensheep.xyz MoE notes, section Training: next to the batch
// balance term, DeepSeek adds one computed inside each sequence so that no
// single sequence routes lopsidedly. Here that is the Switch aux loss of
// the batch restricted to the tokens of one sequence: f = top-k choices per
// expert / (T_q k), P = mean probability, aux_q = E sum_e f P, and the mean
// of aux_q over the non-empty sequences.
//
// One CTA per sequence, 1024 threads. Counts are integer atomics in shared
// memory. The probability sums give each thread a fixed set of tokens
// (every 32nd) for one expert column, added in a fixed order, so the result
// does not depend on scheduling. The last CTA to finish (ticket) averages
// aux over the sequences in sequence order and resets the ticket.
#include "moe_internal.cuh"

namespace moe {

namespace {
constexpr int kSeqThreads = 1024;
constexpr int kSeqRows = kSeqThreads / 32;
}  // namespace

__global__ void __launch_bounds__(kSeqThreads) seq_aux_kernel(
    int T, int E, int k, int nc, const float* __restrict__ probs, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ seq_offsets, int n_seq, float* __restrict__ f_seq,
    float* __restrict__ P_seq, float* __restrict__ aux_seq, float* __restrict__ aux_mean,
    unsigned int* __restrict__ ticket, int* status) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int sm_seq[];
    int* cnt = sm_seq;                                      // [E]
    float* psum = reinterpret_cast<float*>(cnt + E);        // [E]
    __shared__ float part[kSeqRows][33];
    __shared__ float red[kSeqThreads / 32];
    __shared__ int s_last;
    const int q = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, row = tid >> 5;
    int t0 = seq_offsets[q], t1 = seq_offsets[q + 1];
    if (t0 < 0 || t1 < t0 || t1 > T) {
        if (tid == 0) flag_status(status, DEV_BAD_ARG);
        t0 = t1 = 0;  // treated as empty
    }
    const int Tq = t1 - t0;
    for (int e = tid; e < E; e += kSeqThreads) cnt[e] = 0;
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < Tq * k; i += kSeqThreads) {
        const int e = ids[(size_t)(t0 + i / k) * nc + i % k];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else bad = true;
    }
    if (bad) flag_status(status, DEV_BAD_ARG);
    // probability column sums, 32 experts at a time
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        float acc = 0.f;
        if (e < E)
            for (int t = t0 + row; t < t1; t += kSeqRows) acc += __ldg(&probs[(size_t)t * E + e]);
        part[row][lane] = acc;
        __syncthreads();
        if (row == 0 && e < E) {
            float sum = 0.f;
            for (int r = 0; r < kSeqRows; ++r) sum += part[r][lane];
            psum[e] = sum;
        }
        __syncthreads();
    }
    // f, P and the per-expert products, reduced in a fixed tree
    float prod = 0.f;
    for (int e = tid; e < E; e += kSeqThreads) {
        float f = 0.f, P = 0.f;
        if (Tq > 0) {
            f = (float)cnt[e] / ((float)Tq * (float)k);
            P = psum[e] / (float)Tq;
        }
        if (f_seq) f_seq[(size_t)q * E + e] = f;
        if (P_seq) P_seq[(size_t)q * E + e] = P;
        prod += f * P;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) prod += __shfl_xor_sync(0xffffffffu, prod, o);
    if (lane == 0) red[row] = prod;
    __syncthreads();
    if (tid == 0) {
        float a = 0.f;
        for (int r = 0; r < kSeqThreads / 32; ++r) a += red[r];
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
            int a0 = seq_offsets[i], a1 = seq_offsets[i + 1];
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

cudaError_t launch_seq_aux(const Shape& s, const float* probs, const int32_t* ids,
                           const int32_t* seq_offsets, int n_seq, float* f_seq, float* P_seq,
                           float* aux_seq, float* aux_mean, unsigned int* ticket, int* status,
                           cudaStream_t st) {
    const size_t smem = (size_t)s.E * (sizeof(int) + sizeof(float));
    return launch_k(seq_aux_kernel, dim3(n_seq), dim3(kSeqThreads), smem, st, s.T, s.E, s.k, s.nc,
                    probs, ids, seq_offsets, n_seq, f_seq, P_seq, aux_seq, aux_mean, ticket,
                    status);
}

}  // namespace moe
