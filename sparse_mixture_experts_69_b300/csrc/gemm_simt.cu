// Grouped expert GEMM for float32 layers (SIMT FFMA). The tensor cores have
// no float32 x float32 -> float32 mode of the needed accuracy (TF32 keeps 10
// mantissa bits), so the float32 configuration runs here.
//
// Method: mkbk-pku.cn MoE notes, sections on experts (two linear maps around an
// activation) and MoE optimisation (grouped GEMM over expert-contiguous rows).
#include "group_table.cuh"

namespace moe {

namespace {
constexpr int SB = 64;  // tile rows and output columns
constexpr int SK = 16;  // k slice

__device__ __forceinline__ float act_f32(int act, float u) {
    if (act == MOE_RELU) return fmaxf(u, 0.f);
    if (act == MOE_GELU) return 0.5f * u * erfcf(-u * 0.70710678118654752f);
    return u;
}
}  // namespace

// out[r, n] = act(sum_k A[r, k] B[n, k]); GLU: silu(A B_gate^T) * (A B_up^T)
template <bool GLU>
__global__ void __launch_bounds__(256) grouped_gemm_simt_kernel(GroupedGemm p) {
    extern __shared__ int mt_start[];
    __shared__ float As[SK][SB + 4];
    __shared__ float Bs[SK][SB + 4];
    __shared__ float Bu[GLU ? SK : 1][SB + 4];
    pdl_trigger();
    pdl_wait();
    build_tile_table(p, SB, mt_start);
    __syncthreads();
    const int G = p.E + p.S;
    const int nt = (p.N + SB - 1) / SB;
    const int total = mt_start[G] * nt;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const GroupTile gt = decode_tile(p, mt_start, nt, SB, tile);
        const bool routed = gt.g < p.E;
        const float* A = static_cast<const float*>(routed ? p.A0 : p.A1);
        const float* B = static_cast<const float*>(routed ? p.B0 : p.B1);
        float* O = static_cast<float*>(routed ? p.out0 : p.out1);
        const int rows = min(SB, gt.rows);
        const int n0 = gt.n_tile * SB;
        float acc[4][4] = {}, accu[4][4] = {};
        for (int k0 = 0; k0 < p.K; k0 += SK) {
            for (int i = threadIdx.x; i < SB * SK; i += 256) {
                const int r = i / SK, kk = i % SK, kx = k0 + kk;
                As[kk][r] = (r < rows && kx < p.K) ? A[(size_t)(gt.a_row + r) * p.K + kx] : 0.f;
                const int n = n0 + r;
                const bool nb = n < p.N && kx < p.K;
                Bs[kk][r] = nb ? B[(size_t)(gt.b_row + n) * p.K + kx] : 0.f;
                if (GLU) Bu[kk][r] = nb ? B[(size_t)(gt.b_row + p.N + n) * p.K + kx] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < SK; ++kk) {
                float a[4], b[4], u[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    b[j] = Bs[kk][tx * 4 + j];
                    if (GLU) u[j] = Bu[kk][tx * 4 + j];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                        if (GLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
                    }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= rows) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (n >= p.N) continue;
                float v;
                if (GLU) {
                    const float g = acc[i][j];
                    v = g / (1.f + expf(-g)) * accu[i][j];
                } else {
                    v = act_f32(p.act, acc[i][j]);
                }
                O[(size_t)(gt.out_row + r) * p.N + n] = v;
            }
        }
    }
}

cudaError_t launch_grouped_gemm_simt(const Shape& s, const GroupedGemm& g, cudaStream_t st) {
    const int G = g.E + g.S;
    const size_t smem = sizeof(int) * (size_t)(G + 1);
    const long long nt = (g.N + SB - 1) / SB;
    long long mt = (long long)g.max_rows0 / SB + g.E + (long long)g.S * ((g.T + SB - 1) / SB);
    long long bound = mt * nt;
    if (bound < 1) bound = 1;
    const int grid = (int)(bound < 4LL * num_sms() ? bound : 4LL * num_sms());
    if (g.glu) return launch_k(grouped_gemm_simt_kernel<true>, dim3(grid), dim3(256), smem, st, g);
    return launch_k(grouped_gemm_simt_kernel<false>, dim3(grid), dim3(256), smem, st, g);
}

}  // namespace moe
