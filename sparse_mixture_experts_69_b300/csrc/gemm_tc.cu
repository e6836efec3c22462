// Grouped GEMM on the 5th-generation tensor cores (tcgen05, sm_103a), bf16 in,
// fp32 accumulation in tensor memory, used for
//   - the expert FFN up projection with a fused ReLU / GELU / SwiGLU epilogue,
//   - the expert FFN down projection,
//   - the router logits (one group, fp32 output split into logits and noise logits).
//
// Method: mkbk-pku.cn MoE notes, section on MoE optimisation (all experts' GEMMs
// merged into one grouped schedule over expert-contiguous rows).
//
// Structure (one persistent CTA per SM, 6 warps):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [BN x 64] per stage,
//               128-byte swizzle, completion on a per-stage mbarrier
//   warp 1      owns the tensor-memory allocation; lane 0 issues tcgen05.mma
//               (M=128, or M=64 for tiles of at most 64 rows; N=BN, K=16 per
//               instruction) and commits stage releases and finished
//               accumulators to mbarriers
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4) .. +31 = tile rows), activation, bf16 pack, stores
//               through a shared-memory tile
// Two accumulator buffers in TMEM let the epilogue of one tile overlap the
// main loop of the next. Launched early (GroupedGemm::early), a CTA builds its
// tile table and issues its first B tiles before waiting for the preceding
// kernel. Every mbarrier wait is bounded in time; on expiry the CTA records
// DEV_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits. The
// limit is 2 s unless moe_set_wait_limits changed it.
#include <algorithm>
#include <cfloat>
#include <mutex>

#include "aux_common.cuh"
#include "group_table.cuh"

// Compile-time tuning knobs (defaults are the measured best on B300).
#ifndef MOE_TC_KH
#define MOE_TC_KH 1  // 64-wide K halves per pipeline stage (1 or 2)
#endif
#ifndef MOE_TC_PROMO
#define MOE_TC_PROMO 2  // L2 promotion of TMA loads: 0 none, 1 128 B, 2 256 B
#endif
#ifndef MOE_TC_BN_ACT
#define MOE_TC_BN_ACT 256  // output tile width of the ReLU/GELU/plain expert GEMMs
#endif
#ifndef MOE_TC_SMEM
#define MOE_TC_SMEM (192 * 1024)  // shared memory for the pipeline stages
#endif
#ifndef MOE_TC_MAX_STAGES
#define MOE_TC_MAX_STAGES 8
#endif
#ifndef MOE_TC_L2_HINTS
#define MOE_TC_L2_HINTS 1  // L2 eviction policies (b_evict_first, out_l2_keep)
#endif

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int KH = MOE_TC_KH;
constexpr int BKH = 64;      // 64 bf16 = 128 bytes = one swizzle atom row
constexpr int BK = BKH * KH; // K per pipeline stage
constexpr int kThreads = 192;
// Waits of a CTA that is aborting, for its own copies and MMAs already in
// flight, keep this fixed limit whatever the limit of the pipeline waits is
// (moe_set_wait_limits): those operations finish in microseconds, and shared
// memory and TMEM must not be released under them.
constexpr unsigned long long kDrainNs = 250000000ull;

enum Epi : int { EPI_ACT = 0, EPI_GLU = 1, EPI_ROUTER = 2 };

// Selection in the router GEMM's epilogue: with one K part and at most 32
// router columns (no noise), each epilogue thread holds one token's whole row
// of logits and does that token's softmax, top-nc and gates itself, in place
// of the one-warp-per-token selection kernel. Same outputs as that kernel; the
// layer path also counts the capacity histogram and the statistics sums.
struct RouterSel {
    int on;
    int k, nc, renorm;
    const float* bias;  // [E] or NULL: selection scores p + bias
    float* probs;       // [T,E]
    float* sel;         // [T,E] or NULL
    int32_t* ids;       // [T,nc]
    float* w;           // [T,nc]
    int32_t* blk_hist;  // [E][nblk_cap] or NULL
    int nblk_cap;
    void* acc_mem;      // statistics accumulators (aux_common.cuh) or NULL
    // 1: no pdl_trigger at the start. No selection kernel follows to order the
    // next router-weight copy after this GEMM's reads of the copy, so each
    // CTA signals only once its last accumulator is complete (every copy it
    // issued has landed), from one epilogue thread; the next kernel may then
    // overwrite the weight copy during the epilogue
    int late_trigger;
};

struct TcArgs {
    GroupedGemm p;
    const float* offset;  // router: [E] or NULL
    float* logits;        // router: [T,E]
    float* zn;            // router: [T,E] or NULL
    int E_router;         // router: columns < E_router are logits
    // router with its K range split over ksplit CTAs per output tile: CTA part
    // s writes its raw fp32 sums to part[s][T][N] (logits, zn, offset unused);
    // the selection kernel adds the parts in order s = 0, 1, ...
    int ksplit;
    float* part;
    // router: rows of a tile (at most BM; 0: BM). A memory-bound router whose
    // T / BM tiles would leave SMs idle takes shorter tiles, one per SM: the
    // MMAs still run 128 rows, the copies and stores cover router_tm
    int router_tm;
    RouterSel rs;
    unsigned long long wait_ns;  // limit of each pipeline mbarrier wait
    // 1: the MMA warp withholds the "accumulator ready" signal of its CTA's
    // first tile, so the epilogue's first wait can only end by running out
    // (moe_set_wait_limits; tests of the failure path)
    int hold_first_acc;
};

template <int BN>
struct Cfg {
    static constexpr int A_HALF = BM * BKH * 2;  // one 64-wide K half of the A tile
    static constexpr int B_HALF = BN * BKH * 2;
    static constexpr int A_BYTES = A_HALF * KH;
    static constexpr int B_BYTES = B_HALF * KH;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_FIT = MOE_TC_SMEM / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > MOE_TC_MAX_STAGES ? MOE_TC_MAX_STAGES : STAGES_FIT;
    static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;  // power of two for BN in {32..256}
    static constexpr int B_BOX_ROWS = BN < 128 ? BN : 128;
    static constexpr int B_LOADS = BN / B_BOX_ROWS;
    // M=128, N=BN, D=f32, A=B=bf16, both K-major
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                                      ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
    // the same with M=64, for tiles of at most 64 rows
    static constexpr uint32_t IDESC64 = (1u << 4) | (1u << 7) | (1u << 10) |
                                        ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(64 >> 4) << 24);
    // epilogue staging per epilogue warp: the router's 32x32 fp32 block
    // (padded rows), or 32 rows x 80 bytes of bf16 (store_rows32_bf16)
    static constexpr int STAGING_BYTES = 4 * 32 * 33 * 4;
    // layout after the stages: barriers (256 B), tile table [G+1], group rows
    // [G], then the staging area
    static constexpr size_t smem_bytes(int G) {
        return 1024 + (size_t)STAGES * STAGE_BYTES + 256 + sizeof(int) * (size_t)(2 * G + 1) +
               16 + STAGING_BYTES;
    }
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete. Returns false if the
// CTA is aborting or the wait exceeded limit_ns (which starts the abort).
__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                       int* status, unsigned long long limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            flag_status(status, DEV_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}
// As mbar_wait, for a barrier whose phase is completed by a remote arrive
// with release at cluster scope: the completed wait acquires at cluster
// scope, so the releasing CTA's shared::cluster stores are visible.
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ bool mbar_wait_acq_cluster(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort_flag, int* status,
                                                   unsigned long long limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_acq_cluster(a, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_acq_cluster(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            flag_status(status, DEV_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
// As tma_load_2d, with an L2 eviction policy (createpolicy) for the lines read.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_global_hint(void* dst, uint4 v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// ---- CTA-pair (cluster of two) forms, used by grouped_gemm_pair_kernel
// TMEM allocation shared by the CTA pair: one warp of each CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D (both CTAs' TMEM, 128 rows each) (+)= A (128 rows in each CTA's shared
// memory) * B^T (N/2 rows in each CTA's shared memory), issued by one thread
// of the even CTA
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier at this shared-memory offset in every CTA of mask
// once the pair MMAs issued so far by this thread are done.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}
// TMA 2-D tile load into this CTA's shared memory whose completion is
// counted on the mbarrier at `bar_cluster` (shared::cluster address), which
// may be in the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_to_pair_bar(void* dst, const CUtensorMap* map,
                                                        uint32_t bar_cluster, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared-memory address of the same object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on a barrier of another CTA of the cluster. Default semantics
// (release at CTA scope): no cluster-wide fence, which would cost about a
// microsecond per call. The arrival passes on a hardware-completed event (the
// tcgen05.ld of an accumulator finished), not data written by this thread.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Remote arrive that releases this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote_release(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// barrier among the 128 epilogue threads (warps 2..5) only
struct EpilogueBar {
    __device__ void operator()() const { asm volatile("bar.sync 1, 128;" ::: "memory"); }
};
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once all tcgen05 operations issued so far by this thread are done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset
    d |= (uint64_t)1 << 46;                    // descriptor version
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 columns at taddr_a and 16 at taddr_b, one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,"
        "%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}

// ------------------------------------------------------------ epilogue math
__device__ __forceinline__ float act_apply(int act, float u) {
    if (act == MOE_RELU) return fmaxf(u, 0.f);
    if (act == MOE_GELU) return 0.5f * u * erfcf(-u * 0.70710678118654752f);
    return u;
}
__device__ __forceinline__ float silu(float u) { return u / (1.f + expf(-u)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// Stores columns n0 .. n0+31 of the 32 rows of this warp's TMEM lanes; thread
// `lane` holds its row in v[] and gives its output row index in dst_row (-1:
// not stored). The values go through shared memory (stg: 32 rows x 80 bytes,
// the 16 spare bytes spread the rows over the banks) so that each store
// instruction writes 8 rows x 64 contiguous bytes rather than 32 rows x 16.
// N is a multiple of 8, so a 16-byte piece lies wholly inside or outside.
// keep_l2: store with the evict-last policy `pol` (the output is read back
// soon, by the next GEMM).
__device__ __forceinline__ void store_rows32_bf16(__nv_bfloat16* out, int N, int n0, int dst_row,
                                                  const float (&v)[32], uint32_t* stg,
                                                  bool keep_l2, uint64_t pol) {
    const int lane = threadIdx.x & 31;
    uint32_t* mine = stg + lane * 20;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(mine + 4 * q) =
            make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                       pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    __syncwarp();
    const int piece = lane & 3;
    const int col = n0 + 8 * piece;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = (lane >> 2) + 8 * j;
        const int drow = __shfl_sync(0xffffffffu, dst_row, r);
        const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 20 + 4 * piece);
        if (drow >= 0 && col < N) {
            uint4* dst = reinterpret_cast<uint4*>(out + (size_t)drow * N + col);
            if (keep_l2)
                st_global_hint(dst, val, pol);
            else
                *dst = val;
        }
    }
    __syncwarp();
}

// --------------------------------------------------------- folded combine
static_assert(MOE_TC_BN_ACT == kDownTileN, "the folded combine counts 256-column tiles");

// Combine folded into the down projection (GroupedGemm::fold_cnt), run by an
// epilogue warp once its rows of the tile are stored. Every valid row counts
// itself for its token and this column tile. For each token whose count the
// warp completed, the warp then adds up the token's rows over the tile's 256
// columns (lane = 8 consecutive columns) exactly as the combine kernel does:
// acc = fmaf(gate_j, row_j, acc) over the kept choices j = 0, 1, ..., then
// acc += shared row s for s = 0, 1, ..., all on the bf16 values as stored,
// and the sum rounded to bf16 into y. The result does not depend on which
// row arrived last.
__device__ __noinline__ void fold_tile(const GroupedGemm& p, const GroupTile& gt, bool routed,
                                       int trow, bool rv) {
    const int lane = threadIdx.x & 31;
    const int nt = (p.N + kDownTileN - 1) / kDownTileN;
    bool bad = false, nonfinite = false;
    int t = -1;
    if (rv) {
        t = routed ? __ldcg(p.fold_rows + gt.out_row + trow) : gt.m0 + trow;
        if (t < 0 || t >= p.T) {
            bad = true;
            t = -1;
        }
    }
    __threadfence();  // this lane's stores of the tile's rows ...
    __syncwarp();     // ... come before any row of the warp is counted
    bool last = false;
    if (t >= 0) {
        int* cnt = p.fold_cnt + (size_t)t * nt + gt.n_tile;
        const int need = __ldcg(p.fold_need + t) + p.S;
        last = atomicAdd(cnt, 1) == need - 1;
        if (last) *cnt = 0;  // every row of (t, tile) is in: ready for the next call
    }
    unsigned todo = __ballot_sync(0xffffffffu, last);
    if (todo) __threadfence();  // the other rows' stores are visible to the loads below
    const __nv_bfloat16* yp = reinterpret_cast<const __nv_bfloat16*>(p.out0);
    const __nv_bfloat16* ys = reinterpret_cast<const __nv_bfloat16*>(p.out1);
    __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.fold_y);
    const int n0 = gt.n_tile * kDownTileN + 8 * lane;
    const bool cv = n0 < p.N;  // N is a multiple of 8
    // lane j holds choice j's row and gate of token tt (-1: dropped or none)
    auto load_choices = [&](int tt, int& r, float& g) {
        r = -1;
        g = 0.f;
        if (tt >= 0 && lane < p.fold_nc) {
            r = __ldcg(p.fold_slot + (size_t)tt * p.fold_nc + lane);
            g = __ldcg(p.fold_w + (size_t)tt * p.fold_nc + lane);
            if (r >= p.max_rows0) {
                bad = true;
                r = -1;
            }
        }
    };
    int tt = todo ? __shfl_sync(0xffffffffu, t, __ffs(todo) - 1) : -1;
    int my_r, nx_r;
    float my_g, nx_g;
    load_choices(tt, my_r, my_g);
    while (todo) {
        todo &= todo - 1;
        // the next token's choices load while this one's rows are summed
        const int nx = todo ? __shfl_sync(0xffffffffu, t, __ffs(todo) - 1) : -1;
        load_choices(nx, nx_r, nx_g);
        // the token's rows in the combine's order: kept choices, then shared
        // experts; loaded kChunk at a time, added in order
        constexpr int kChunk = 12;
        unsigned live = __ballot_sync(0xffffffffu, my_r >= 0);
        const int nlive = __popc(live);
        const int nrow = nlive + p.S;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        unsigned rem = live;  // kept choices not yet loaded, in order
        for (int c0 = 0; c0 < nrow; c0 += kChunk) {
            uint4 raw[kChunk];
            float g[kChunk];
#pragma unroll
            for (int q = 0; q < kChunk; ++q) {
                const int i = c0 + q;
                g[q] = 0.f;
                if (i < nlive) {  // warp-uniform
                    const int j = __ffs(rem) - 1;  // the i-th kept choice
                    rem &= rem - 1;
                    const int r = __shfl_sync(0xffffffffu, my_r, j);
                    g[q] = __shfl_sync(0xffffffffu, my_g, j);
                    if (cv) raw[q] = __ldcg(reinterpret_cast<const uint4*>(yp + (size_t)r * p.N + n0));
                } else if (i < nrow && cv) {
                    raw[q] = __ldcg(reinterpret_cast<const uint4*>(
                        ys + ((size_t)(i - nlive) * p.T + tt) * p.N + n0));
                }
            }
#pragma unroll
            for (int q = 0; q < kChunk; ++q) {
                const int i = c0 + q;
                if (i < nrow && cv) {
                    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[q]);
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        const float2 v = __bfloat1622float2(h[k2]);
                        if (i < nlive) {
                            acc[2 * k2] = fmaf(g[q], v.x, acc[2 * k2]);
                            acc[2 * k2 + 1] = fmaf(g[q], v.y, acc[2 * k2 + 1]);
                        } else {
                            acc[2 * k2] += v.x;
                            acc[2 * k2 + 1] += v.y;
                        }
                    }
                }
            }
        }
        if (cv) {
            uint4 out;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                nonfinite |= !isfinite(acc[2 * i]) || !isfinite(acc[2 * i + 1]);
                h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            }
            *reinterpret_cast<uint4*>(y + (size_t)tt * p.N + n0) = out;
        }
        tt = nx;
        my_r = nx_r;
        my_g = nx_g;
    }
    if (bad) flag_status(p.status, DEV_BAD_ARG);
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0) flag_status(p.status, DEV_NONFINITE);
}

// ------------------------------------------------------------------ kernel
// First B row of each B box of tile gt: SwiGLU tiles take 128 gate rows and
// the matching 128 up rows; other tiles take BN consecutive rows.
template <int BN, int EPI>
__device__ __forceinline__ void b_tile_rows(const GroupedGemm& p, const GroupTile& gt,
                                            int (&brow)[Cfg<BN>::B_LOADS]) {
#pragma unroll
    for (int h = 0; h < Cfg<BN>::B_LOADS; ++h) {
        if (EPI == EPI_GLU)
            brow[h] = gt.b_row + h * p.N + gt.n_tile * 128;
        else
            brow[h] = gt.b_row + gt.n_tile * BN + h * Cfg<BN>::B_BOX_ROWS;
    }
}
// The B tile of k block kb into one ring stage.
// WEF: the weights are read with the evict-first policy pol
// (GroupedGemm::b_evict_first); otherwise with no cache hint at all.
template <int BN, bool WEF>
__device__ __forceinline__ void load_b_stage(uint8_t* sB_stage, const CUtensorMap* mb,
                                             uint64_t* bar, int kb,
                                             const int (&brow)[Cfg<BN>::B_LOADS], uint64_t pol) {
#pragma unroll
    for (int hk = 0; hk < KH; ++hk)
#pragma unroll
        for (int h = 0; h < Cfg<BN>::B_LOADS; ++h) {
            uint8_t* dst = sB_stage + hk * Cfg<BN>::B_HALF + h * Cfg<BN>::B_BOX_ROWS * 128;
            if (WEF)
                tma_load_2d_hint(dst, mb, bar, kb * BK + hk * BKH, brow[h], pol);
            else
                tma_load_2d(dst, mb, bar, kb * BK + hk * BKH, brow[h]);
        }
}

// Bytes a ring stage receives for a tile whose group has `rows` rows from the
// tile's first row on: tiles of at most 64 rows (M=64 MMAs) load a 64-row A
// box, half the A bytes; the rest of the A slot stays unused.
template <int BN, int EPI>
__device__ __forceinline__ uint32_t stage_bytes(int rows) {
    const bool short_a = EPI != EPI_ROUTER && rows <= 64;
    return (uint32_t)((short_a ? Cfg<BN>::A_BYTES / 2 : Cfg<BN>::A_BYTES) + Cfg<BN>::B_BYTES);
}

#ifndef MOE_TC_ROUTER_ROT
#define MOE_TC_ROUTER_ROT 1
#endif
#ifndef MOE_ROUTER_PAIR
#define MOE_ROUTER_PAIR 1  // 256-wide router GEMMs on CTA pairs
#endif
#ifndef MOE_ROUTER_SEL_IN_GEMM
#define MOE_ROUTER_SEL_IN_GEMM 1  // selection in the epilogue of narrow unsplit routers
#endif
#ifndef MOE_ROUTER_SHORT_TILES
#define MOE_ROUTER_SHORT_TILES 1  // memory-bound routers: one tile per SM
#endif

// The K block loaded at step j of a work item whose K range is [lo, hi). The
// router's CTAs all start together, one tile each, and would otherwise read
// the same K offset of every row at the same time; with MOE_TC_ROUTER_ROT
// each starts its K range at a tile-dependent block and wraps around, so the
// CTAs' concurrent loads spread over the rows' K extent (Mixtral-shaped
// router: 37.8 -> 35.8 us a route call). Only the order of the K blocks in a
// tile's sum changes with it, not the result beyond rounding.
template <int EPI>
__device__ __forceinline__ int k_block(int j, int lo, int hi, int tile) {
    if (MOE_TC_ROUTER_ROT && EPI == EPI_ROUTER) {
        const int n = hi - lo;
        int x = j - lo + (tile * 5) % n;
        if (x >= n) x -= n;
        return lo + x;
    }
    return j;
}

// The selection of token t from its row of raw router sums v[0..E) (E <= EMAX
// <= 32), as router_select_kernel does it for a token: logits z = v + offset,
// the max-subtracted fp32 softmax, keys ordered by (score desc, index asc) with
// score H (or p + bias), the first nc candidates, and gates p_j over the sum of
// the first k candidates' p (renorm) or p_j. Only the summation order of the
// softmax denominator and of the gates' sum differs (a pairwise tree and a
// sequential sum here). With aux statistics, each warp adds its tokens'
// probabilities (fp32, butterfly order, then fixed point), gates (fixed point)
// and counts per expert into the accumulators, and every choice into the
// capacity histogram. One warp per SM sub-partition runs this, so the chains
// are kept short: EMAX = 8 sorts 64-bit keys (score key, complemented index)
// with a register network and reduces all experts' statistics together.
__device__ __forceinline__ unsigned sel_key(float v) {
    const unsigned b = __float_as_uint(__fadd_rn(v, 0.f));
    return b ^ ((b >> 31) ? 0xFFFFFFFFu : 0x80000000u);
}
// Row t of a [T, E] fp32 output from a thread's registers: two 16-byte
// stores when E = 8 and the base is 16-byte aligned, else E scalar stores.
template <int EMAX>
__device__ __forceinline__ void store_row(float* base, int E, int t, const float (&x)[EMAX]) {
    float* dst = base + (size_t)t * E;
    if (EMAX == 8 && E == 8 && (reinterpret_cast<uintptr_t>(base) & 15) == 0) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
#pragma unroll
        for (int i = 0; i < EMAX; ++i)
            if (i < E) dst[i] = x[i];
    }
}

// logits: NULL when the caller has written them, else the [T, E] output.
template <int EMAX>
__device__ __forceinline__ void router_select_rows(const RouterSel rs, const float* offset,
                                                   int E, int t, bool valid,
                                                   const float (&v)[32], float* logits,
                                                   float* stg, int* status) {
    const int lane = threadIdx.x & 31;
    float h[EMAX], pr[EMAX];
    bool nonfinite = false;
#pragma unroll
    for (int i = 0; i < EMAX; ++i) {
        h[i] = -FLT_MAX;
        if (i < E) {
            h[i] = v[i] + (offset ? offset[i] : 0.f);
            if (!isfinite(h[i])) nonfinite = true;
        }
    }
    // pairwise maximum and sum (log-depth chains)
    float red[EMAX];
#pragma unroll
    for (int i = 0; i < EMAX; ++i) red[i] = h[i];
#pragma unroll
    for (int w = EMAX / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) red[i] = fmaxf(red[i], red[i + w]);
    const float m = red[0];
#pragma unroll
    for (int i = 0; i < EMAX; ++i) {
        pr[i] = i < E ? __expf(h[i] - m) : 0.f;
        red[i] = pr[i];
    }
#pragma unroll
    for (int w = EMAX / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) red[i] += red[i + w];
    const float inv = __frcp_rn(red[0]);
    unsigned key[EMAX];
    float sc[EMAX];
#pragma unroll
    for (int i = 0; i < EMAX; ++i) {
        key[i] = 0u;
        sc[i] = 0.f;
        if (i < E) {
            pr[i] = pr[i] * inv;
            sc[i] = rs.bias ? pr[i] + rs.bias[i] : h[i];
            key[i] = sel_key(sc[i]);
        }
    }
    if (valid) {
        if (logits) store_row<EMAX>(logits, E, t, h);
        store_row<EMAX>(rs.probs, E, t, pr);
        if (rs.sel) store_row<EMAX>(rs.sel, E, t, sc);
    }
    if (__any_sync(0xffffffffu, valid && nonfinite) && lane == 0) flag_status(status, DEV_NONFINITE);
    int id[8];
    float pj[8];
    if constexpr (EMAX == 8) {
        // one sort of (score key, complemented index): keys are distinct and
        // the unsigned order is (score desc, index asc); 0 marks no expert
        unsigned long long k64[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            k64[i] = i < E ? ((unsigned long long)key[i] << 32) | (unsigned)~i : 0ull;
        sort_desc64<8>(k64);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            id[j] = (int)(~(unsigned)k64[j]) & 7;
            pj[j] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i == id[j]) pj[j] = pr[i];
        }
    } else {
        // repeated arg-max; a strict > keeps the lower index among equal keys
        unsigned taken = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            id[j] = 0;
            pj[j] = 0.f;
            if (j < rs.nc) {
                int be = -1;
                unsigned bk = 0u;
                float bp = 0.f;
#pragma unroll
                for (int i = 0; i < EMAX; ++i)
                    if (i < E && !((taken >> i) & 1u) && (be < 0 || key[i] > bk)) {
                        be = i;
                        bk = key[i];
                        bp = pr[i];
                    }
                if (be >= 0) taken |= 1u << be;  // nc <= E: always
                id[j] = be < 0 ? 0 : be;
                pj[j] = bp;
            }
        }
    }
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < rs.k) psum += pj[j];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < rs.nc) {
            const float wj = rs.renorm ? pj[j] / psum : pj[j];
            pj[j] = wj;
            if (valid && rs.ids) {
                rs.ids[(size_t)t * rs.nc + j] = id[j];
                rs.w[(size_t)t * rs.nc + j] = wj;
                if (j < rs.k && rs.blk_hist)
                    atomicAdd(&rs.blk_hist[(size_t)id[j] * rs.nblk_cap + t / kCapBlockTokens], 1);
            }
        }
    }
    if (rs.acc_mem == nullptr) return;
    const AuxAcc acc = aux_acc_at(rs.acc_mem, E, kAuxGroups);
    const size_t g = (size_t)(blockIdx.x % acc.groups) * E;
    if constexpr (EMAX == 8) {
        // the warp's 32 x 8 probabilities and its gate and count sums per
        // expert in its staging area (free once the logits are out); lane e
        // then adds expert e's column in row order
        float* cs = stg;                                                // [8][33]
        unsigned long long* si = reinterpret_cast<unsigned long long*>(stg + 264);  // [8]
        unsigned* sc = reinterpret_cast<unsigned*>(stg + 280);          // [8]
        if (lane < 8) {
            si[lane] = 0ull;
            sc[lane] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) cs[e * 33 + lane] = valid ? pr[e] : 0.f;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (valid && j < rs.k) {
                atomicAdd(&si[id[j]], to_fix(pj[j]));
                atomicAdd(&sc[id[j]], 1u);
            }
        __syncwarp();
        if (lane < E) {
            float pe = 0.f;
#pragma unroll 8
            for (int r = 0; r < 32; ++r) pe += cs[lane * 33 + r];
            const unsigned long long pf = to_fix(pe);
            if (pf) atomicAdd(&acc.P[g + lane], pf);
            if (si[lane]) atomicAdd(&acc.I[g + lane], si[lane]);
            if (sc[lane]) atomicAdd(&acc.cnt[g + lane], sc[lane]);
        }
        __syncwarp();
    } else {
        for (int e = 0; e < E; ++e) {
            float pe = 0.f;
            unsigned long long ie = 0ull;
            unsigned ce = 0u;
#pragma unroll
            for (int i = 0; i < EMAX; ++i)
                if (i == e) pe = valid ? pr[i] : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (valid && j < rs.k && id[j] == e) {
                    ie += to_fix(pj[j]);
                    ++ce;
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                pe += __shfl_xor_sync(0xffffffffu, pe, o);
                ie += __shfl_xor_sync(0xffffffffu, ie, o);
            }
            ce = __reduce_add_sync(0xffffffffu, ce);
            if (lane == 0) {
                const unsigned long long pf = to_fix(pe);
                if (pf) atomicAdd(&acc.P[g + e], pf);
                if (ie) atomicAdd(&acc.I[g + e], ie);
                if (ce) atomicAdd(&acc.cnt[g + e], ce);
            }
        }
    }
}

// WEF: weights evict-first in L2 (a separate instantiation: the hinted copy
// form, even with the normal policy, slowed the launches with weight reuse).
template <int BN, int EPI, bool WEF>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0,
                           const __grid_constant__ CUtensorMap tmA1,
                           const __grid_constant__ CUtensorMap tmA0s,
                           const __grid_constant__ CUtensorMap tmA1s,
                           const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const TcArgs args) {
    using C = Cfg<BN>;
    const GroupedGemm& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    static_assert((2 * C::STAGES + 5) * 8 + 8 <= 256, "barrier area");
    int* mt_start = reinterpret_cast<int*>(smem + C::STAGES * C::STAGE_BYTES + 256);
    int* grows = mt_start + p.E + p.S + 1;  // [G] rows of each group
    float* staging = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(grows + p.E + p.S) + 15) & ~(uintptr_t)15);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.E + p.S;
    const int ncol_tile = EPI == EPI_GLU ? 128 : BN;
    const int nt = (p.N + ncol_tile - 1) / ncol_tile;
    const int nkb = (p.K + BK - 1) / BK;
    // rows of a tile: BM, or the router's shorter tiles
    const int TM = EPI == EPI_ROUTER && args.router_tm > 0 ? args.router_tm : BM;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA0);
        prefetch_tmap(&tmA1);
        prefetch_tmap(&tmA0s);
        prefetch_tmap(&tmA1s);
        prefetch_tmap(&tmB0);
        prefetch_tmap(&tmB1);
    }
    // early launch: the offsets are final and B is never written by the
    // preceding kernels, so the tile table and the first B tiles do not wait
    // for the preceding kernel (A, the outputs and TMEM do)
    const bool early = p.early != 0;
    if (!early) pdl_wait();
    if (early)
        build_tile_table<true>(p, TM, mt_start, grows);
    else
        build_tile_table<false>(p, TM, mt_start, grows);
    __syncthreads();
    // work items: output tiles, times the K parts of a split router GEMM
    const int ks = EPI == EPI_ROUTER ? args.ksplit : 1;
    const int total = mt_start[G] * nt * ks;
    // no work: leave before any allocation (CTA 0 stays when it owes the
    // statistics finalisation); every CTA passes the wait before it exits, so
    // this kernel completes only after the preceding one has
    if ((int)blockIdx.x >= total && !(p.fin_acc_mem && blockIdx.x == 0)) {
        if (early) pdl_wait();
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // first ring stages: expected bytes and B tiles (A follows after the wait)
    const uint64_t pol_w = WEF ? l2_evict_first_policy() : 0ull;
    int prefilled = 0;
    if (early && threadIdx.x == 0) {
        for (int w = blockIdx.x; w < total && prefilled < C::STAGES; w += gridDim.x) {
            const int tile = w / ks, sp = w - tile * ks;
            const GroupTile gt = decode_tile<true>(p, mt_start, nt, TM, tile);
            const CUtensorMap* mb = gt.g < p.E ? &tmB0 : &tmB1;
            int brow[C::B_LOADS];
            b_tile_rows<BN, EPI>(p, gt, brow);
            const int kb_lo = sp * nkb / ks, kb_hi = (sp + 1) * nkb / ks;
            const uint32_t bytes = EPI == EPI_ROUTER
                                       ? (uint32_t)(TM * BK * 2 + C::B_BYTES)
                                       : stage_bytes<BN, EPI>(gt.rows);
            for (int kb = kb_lo; kb < kb_hi && prefilled < C::STAGES; ++kb) {
                mbar_arrive_expect_tx(&full[prefilled], bytes);
                load_b_stage<BN, WEF>(sB + prefilled * C::B_BYTES, mb, &full[prefilled],
                                      k_block<EPI>(kb, kb_lo, kb_hi, tile), brow, pol_w);
                ++prefilled;
            }
        }
    }
    if (early) pdl_wait();
    // dependents may launch once every CTA is past the wait: a kernel that
    // follows this one can rely on the kernel before this one being complete
    if (!(EPI == EPI_ROUTER && args.rs.late_trigger)) pdl_trigger();
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;
            bool ok = true;
            int item = 0;  // (tile, k block) pairs issued so far
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
                const int tile = w / ks, sp = w - tile * ks;
                const GroupTile gt = decode_tile(p, mt_start, nt, TM, tile);
                const bool routed = gt.g < p.E;
                // tiles of at most 64 rows (M=64 MMAs) load 64-row A boxes
                const bool short_a = EPI != EPI_ROUTER && gt.rows <= 64;
                const CUtensorMap* ma = short_a ? (routed ? &tmA0s : &tmA1s)
                                                : (routed ? &tmA0 : &tmA1);
                const CUtensorMap* mb = routed ? &tmB0 : &tmB1;
                const uint32_t bytes = EPI == EPI_ROUTER
                                           ? (uint32_t)(TM * BK * 2 + C::B_BYTES)
                                           : stage_bytes<BN, EPI>(gt.rows);
                int brow[C::B_LOADS];
                b_tile_rows<BN, EPI>(p, gt, brow);
                const int kb_lo = sp * nkb / ks, kb_hi = (sp + 1) * nkb / ks;
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++item) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // prefilled stages already expect their bytes and hold B
                    const bool fresh = item >= prefilled;
                    if (fresh) mbar_arrive_expect_tx(&full[stage], bytes);
                    const int kbe = k_block<EPI>(kb, kb_lo, kb_hi, tile);
#pragma unroll
                    for (int hk = 0; hk < KH; ++hk)
                        tma_load_2d(sA + stage * C::A_BYTES + hk * C::A_HALF, ma, &full[stage],
                                    kbe * BK + hk * BKH, gt.a_row);
                    if (fresh)
                        load_b_stage<BN, WEF>(sB + stage * C::B_BYTES, mb, &full[stage], kbe,
                                              brow, pol_w);
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                // aborting: let the copies already issued land before smem is released
                for (int s = 0; s < C::STAGES; ++s)
                    if ((filled >> s) & 1u) {
                        volatile int never = 0;
                        mbar_wait(&full[s], (fill_parity >> s) & 1u, &never, p.status, kDrainNs);
                    }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++local) {
                const int tile = w / ks, sp = w - tile * ks;
                const int b = local & 1;
                const uint32_t tph = (local >> 1) & 1;
                if (!mbar_wait(&tempty[b], tph ^ 1, abort_flag, p.status, args.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
                // expert tiles of at most 64 rows (few-token experts) run M=64 MMAs
                const bool m64 =
                    EPI != EPI_ROUTER && tile_rows(mt_start, grows, G, nt, BM, tile, p.row_block) <= 64;
                const uint32_t idesc = m64 ? C::IDESC64 : C::IDESC;
                const int kb_lo = sp * nkb / ks, kb_hi = (sp + 1) * nkb / ks;
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int hk = 0; hk < KH; ++hk) {
                        const uint64_t ad =
                            sdesc_sw128(smem_u32(sA + stage * C::A_BYTES + hk * C::A_HALF));
                        const uint64_t bd =
                            sdesc_sw128(smem_u32(sB + stage * C::B_BYTES + hk * C::B_HALF));
#pragma unroll
                        for (int kk = 0; kk < BKH / 16; ++kk)
                            umma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                                      (kb != kb_lo || hk | kk) ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok && !(args.hold_first_acc && local == 0)) umma_commit(&tfull[b]);
            }
            if (!ok || args.hold_first_acc) {
                // every MMA this thread issued completes before TMEM is freed
                umma_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, &never, p.status, kDrainNs);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        if (p.fin_acc_mem && blockIdx.x == 0) {
            // the statistics sums are complete (previous kernels); finalise them
            // while the first accumulator is still being computed
            const AuxAcc acc = aux_acc_at(p.fin_acc_mem, p.E, kAuxGroups);
            const AuxOut out{p.fin_f, p.fin_P, p.fin_I, p.fin_out3, p.fin_w_imp};
            aux_finalize(p.T, p.E, p.fin_k, acc, out, threadIdx.x - 64, 128, EpilogueBar{});
        }
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint64_t pol_o = l2_evict_last_policy();
        int local = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x, ++local) {
            const int tile = w / ks, sp = w - tile * ks;
            const GroupTile gt = decode_tile(p, mt_start, nt, TM, tile);
            const int b = local & 1;
            const uint32_t tph = (local >> 1) & 1;
            if (!mbar_wait(&tfull[b], tph, abort_flag, p.status, args.wait_ns)) break;
            tc_fence_after();
            if (EPI == EPI_ROUTER && args.rs.late_trigger && w + (int)gridDim.x >= total &&
                threadIdx.x == 64)
                pdl_trigger();  // this CTA's last accumulator: its reads are all done
            const uint32_t taddr = tmem_base + (uint32_t)(b * BN) + ((uint32_t)(32 * q) << 16);
            // M=64 tiles: accumulator row r is in TMEM lane 32 (r / 16) + r % 16,
            // so lanes 0..15 of each lane quadrant hold 16 rows and 16..31 none
            const bool m64 = EPI != EPI_ROUTER && gt.rows <= 64;
            const int trow = m64 ? (lane < 16 ? 16 * q + lane : BM) : row;
            const bool rv = trow < gt.rows;
            const bool routed = gt.g < p.E;
            if (EPI == EPI_ROUTER) {
                // thread = row; stage 32 rows x 32 columns, then each warp writes
                // whole 128-byte row segments (lane = column)
                float* stg = staging + q * 32 * 33;
                const int rows_here = min(32, min(gt.rows, TM) - 32 * q);
                const int E_r = args.E_router;
                // at most 8 experts selected here: the selection writes the logits
                const int c_end = (BN == 32 && args.rs.on && E_r <= 8) ? 0 : BN;
#pragma unroll 1
                for (int c = 0; c < c_end; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) stg[lane * 33 + i] = v[i];
                    __syncwarp();
                    const int n = gt.n_tile * BN + c + lane;
                    if (n < p.N && args.part) {
                        float* dst = args.part + (size_t)sp * p.T * p.N + n;
                        for (int r = 0; r < rows_here; ++r)
                            dst[(size_t)(gt.out_row + 32 * q + r) * p.N] = stg[r * 33 + lane];
                    } else if (n < p.N) {
                        const bool is_logit = n < E_r;
                        const float off = (is_logit && args.offset) ? args.offset[n] : 0.f;
                        float* dst = is_logit ? args.logits + n : args.zn + (n - E_r);
                        for (int r = 0; r < rows_here; ++r) {
                            const size_t t = (size_t)(gt.out_row + 32 * q + r);
                            dst[t * E_r] = stg[r * 33 + lane] + off;
                        }
                    }
                    __syncwarp();
                }
                if constexpr (BN == 32) {
                    if (args.rs.on) {
                        float v[32];
                        tmem_ld32(taddr, v);
                        const bool tv = row < rows_here + 32 * q;
                        if (E_r <= 8)
                            router_select_rows<8>(args.rs, args.offset, E_r, gt.out_row + row, tv,
                                                  v, args.logits, stg, p.status);
                        else
                            router_select_rows<32>(args.rs, args.offset, E_r, gt.out_row + row,
                                                   tv, v, nullptr, stg, p.status);
                    }
                }
            } else {
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(routed ? p.out0 : p.out1);
                uint32_t* stg = reinterpret_cast<uint32_t*>(staging) + q * 32 * 20;
                const bool keep_l2 = MOE_TC_L2_HINTS && p.out_l2_keep;
                int dst_row = rv ? gt.out_row + trow : -1;
                if (EPI == EPI_GLU) {
#pragma unroll 1
                    for (int c = 0; c < 128; c += 32) {
                        float g[16], u[16], v[32];
                        tmem_ld16x2(taddr + c, taddr + 128 + c, g, u);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = silu(g[i]) * u[i];
                        tmem_ld16x2(taddr + c + 16, taddr + 128 + c + 16, g, u);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[16 + i] = silu(g[i]) * u[i];
                        const int n0 = gt.n_tile * 128 + c;
                        if (n0 < p.N)
                            store_rows32_bf16(out, p.N, n0, dst_row, v, stg, keep_l2, pol_o);
                    }
                } else {
                    const int act = p.glu ? -1 : p.act;
                    float scale = 1.f;
                    if (routed && p.scatter_rows) {
                        // top-1 combine: this row is token t's output, times its gate
                        const int t = rv ? p.scatter_rows[gt.out_row + trow] : 0;
                        out = reinterpret_cast<__nv_bfloat16*>(p.scatter_out);
                        dst_row = rv ? t : -1;
                        scale = rv ? p.scatter_scale[t] : 0.f;
                    }
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        float v[32];
                        tmem_ld32(taddr + c, v);
                        const int n0 = gt.n_tile * BN + c;
                        if (n0 < p.N) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = act_apply(act, v[i]) * scale;
                            store_rows32_bf16(out, p.N, n0, dst_row, v, stg, keep_l2, pol_o);
                        }
                    }
                    if (EPI == EPI_ACT && p.fold_cnt) fold_tile(p, gt, routed, trow, rv);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[b]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);

}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix; box [box_rows, 64].
static bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BKH, (cuuint32_t)box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride,
                    box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    MOE_TC_PROMO == 0   ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                    : MOE_TC_PROMO == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                        : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, int EPI, bool WEF>
static cudaError_t launch(const TcArgs& a, cudaStream_t st) {
    using C = Cfg<BN>;
    const GroupedGemm& p = a.p;
    CUtensorMap mA0, mA1, mA0s, mA1s, mB0, mB1;
    const int G = p.E + p.S;
    const int tm = EPI == EPI_ROUTER && a.router_tm > 0 ? a.router_tm : BM;  // rows of a tile
    // A maps with tile-high boxes, and with 64-row boxes for tiles of <= 64 rows
    for (int i = 0; i < 2; ++i) {
        const int box = i == 0 ? tm : 64;
        CUtensorMap* m0 = i == 0 ? &mA0 : &mA0s;
        CUtensorMap* m1 = i == 0 ? &mA1 : &mA1s;
        if (!make_map(m0, p.A0 ? p.A0 : p.A1, p.A0 ? p.rows_a0 : p.rows_a1, p.K, box) ||
            !make_map(m1, p.A1 ? p.A1 : p.A0, p.A1 ? p.rows_a1 : p.rows_a0, p.K, box))
            return cudaErrorInvalidValue;
    }
    const int brows0 = p.E * p.b_rows_group, brows1 = p.S * p.b_rows_group;
    if (!make_map(&mB0, p.B0 ? p.B0 : p.B1, p.B0 ? brows0 : brows1, p.K, C::B_BOX_ROWS) ||
        !make_map(&mB1, p.B1 ? p.B1 : p.B0, p.B1 ? brows1 : brows0, p.K, C::B_BOX_ROWS))
        return cudaErrorInvalidValue;
    const size_t smem = C::smem_bytes(G);
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_tc_kernel<BN, EPI, WEF>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    // upper bound of the tile count, from host-known sizes
    const int ncol_tile = EPI == EPI_GLU ? 128 : BN;
    const long long nt = (p.N + ncol_tile - 1) / ncol_tile;
    long long mt = (long long)p.max_rows0 / tm + p.E + (long long)p.S * ((p.T + tm - 1) / tm);
    if (p.E == 0) mt = (long long)p.S * ((p.T + tm - 1) / tm);
    const long long bound = std::max<long long>(1, mt * nt * (EPI == EPI_ROUTER ? a.ksplit : 1));
    const int grid = (int)std::min<long long>(bound, num_sms());
    return launch_k(grouped_gemm_tc_kernel<BN, EPI, WEF>, dim3(grid), dim3(kThreads), smem, st, mA0,
                    mA1, mA0s, mA1s, mB0, mB1, a);
}

// ------------------------------------------------------------ CTA-pair kernel
// The expert GEMM on 256-row tiles computed by a cluster of two CTAs with the
// pair MMA (tcgen05.mma.cta_group::2, M = 256, N = 256): each CTA holds its
// own 128 A rows and one half of the 256-wide weight tile in shared memory
// and receives its 128 rows x 256 columns of the accumulator in its own TMEM.
// Per SM a K block is 16 KB of A plus 16 KB of B for 128 x 256 x 64 of MMA
// work, a third fewer operand bytes than the single-CTA tile (16 + 32 KB), so
// the same 192 KB holds 6 ring stages instead of 4; both TMEM buffers stay,
// so the epilogue of one tile overlaps the next tile's MMAs.
//
// Signals. Both CTAs' TMA copies of a stage complete on the even CTA's
// `full` barrier (the odd CTA's copies through the pair form of the TMA
// load), which the even CTA's producer arms with both CTAs' bytes. The even
// CTA's warp 1 issues the MMAs once a stage is in, and its commits arrive on
// `empty` (stage free) and `tfull` (accumulator ready) in both CTAs at once
// (multicast). Each CTA's epilogue warps release an accumulator on the even
// CTA's `tempty` (remote arrive from the odd CTA). Every wait is bounded in
// time as in the single-CTA kernel; neither CTA frees TMEM or leaves before a
// cluster barrier that both reach once every MMA of the pair is done. An
// aborting odd CTA cannot see its own copies complete (they count on the
// other CTA's barrier), so it waits 200 us, far longer than a copy takes,
// before that barrier.
//
// Tile order. With GroupedGemm::tile_ctr the pairs take their tiles in order
// from a launch-wide counter, so the tiles in flight stay a window of
// consecutive tiles (sharing weight panels and token blocks through L2);
// pairs that each took every nclusters-th tile drifted apart over a launch
// and tripled the DRAM reads of the Mixtral-shaped GEMMs.

// Work-item ring of the pair kernel's dynamic tile order: slots, and the
// consumers of each item (the even CTA's MMA issuer, 4 epilogue warps in each
// CTA, the odd CTA's producer).
constexpr int kItemRing = 4;
constexpr int kItemConsumers = 10;
// tile_ctr[0] is the launch's tile counter, tile_ctr[1] counts the pairs that
// are done with it; the last pair to finish puts both back to zero for the
// next launch (which touches them only after its wait for this one).
__device__ __forceinline__ void release_tile_counter(int* tile_ctr, int nclusters) {
    __threadfence();
    if (atomicAdd(tile_ctr + 1, 1) == nclusters - 1) {
        atomicExch(tile_ctr, 0);
        atomicExch(tile_ctr + 1, 0);
    }
}

struct PairCfg {
    static constexpr int BN = 256;
    static constexpr int A_BYTES = BM * BKH * 2;    // own 128 rows x 64
    static constexpr int B_BYTES = 128 * BKH * 2;   // own half of the weight tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_FIT = MOE_TC_SMEM / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > MOE_TC_MAX_STAGES ? MOE_TC_MAX_STAGES : STAGES_FIT;
    static constexpr int TMEM_COLS = 2 * BN;        // two accumulators
    // M=256 (128 rows in each CTA), N=256, D=f32, A=B=bf16, both K-major
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                                      ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
    static constexpr int STAGING_BYTES = 4 * 32 * 33 * 4;
    static constexpr size_t smem_bytes(int G) {
        return 1024 + (size_t)STAGES * STAGE_BYTES + 256 + sizeof(int) * (size_t)(2 * G + 1) +
               16 + STAGING_BYTES;
    }
};
static_assert(KH == 1, "the pair kernel loads one 64-wide K block per stage");
// barriers, TMEM slot, abort flag and the work-item ring fit the 256 bytes
// before the tile table
static_assert((2 * PairCfg::STAGES + 7 + 2 * kItemRing) * 8 + 4 * kItemRing <= 256,
              "pair kernel barrier area");

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                             const __grid_constant__ CUtensorMap tmA1,
                             const __grid_constant__ CUtensorMap tmB0,
                             const __grid_constant__ CUtensorMap tmB1, const TcArgs args) {
    using C = PairCfg;
    constexpr int BN = C::BN;
    const GroupedGemm& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // work-item ring of the dynamic tile order (GroupedGemm::tile_ctr)
    uint64_t* item_full = drain + 2;
    uint64_t* item_empty = item_full + kItemRing;
    volatile int* s_item = reinterpret_cast<volatile int*>(item_empty + kItemRing);
    int* mt_start = reinterpret_cast<int*>(smem + C::STAGES * C::STAGE_BYTES + 256);
    int* grows = mt_start + p.E + p.S + 1;
    float* staging = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(grows + p.E + p.S) + 15) & ~(uintptr_t)15);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = (int)cluster_id_x(), nclusters = (int)cluster_count_x();
    const int G = p.E + p.S;
    const int ncol_tile = EPI == EPI_GLU ? 128 : BN;
    const int nt = (p.N + ncol_tile - 1) / ncol_tile;
    const int nkb = (p.K + BK - 1) / BK;
    const bool dyn = EPI != EPI_ROUTER && p.tile_ctr != nullptr;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA0);
        prefetch_tmap(&tmA1);
        prefetch_tmap(&tmB0);
        prefetch_tmap(&tmB1);
    }
    const bool early = p.early != 0;
    if (!early) pdl_wait();
    if (early)
        build_tile_table<true>(p, 2 * BM, mt_start, grows);
    else
        build_tile_table<false>(p, 2 * BM, mt_start, grows);
    __syncthreads();
    // work items: output tiles, times the K parts of a split router GEMM
    const int ks = EPI == EPI_ROUTER ? args.ksplit : 1;
    const int total = mt_start[G] * nt * ks;
    // no work for this pair: both CTAs leave together, before any allocation
    // or cluster-wide step (pair 0 stays when it owes the statistics)
    if (cluster >= total && !(p.fin_acc_mem && cluster == 0)) {
        if (early) pdl_wait();
        if (dyn && leader && threadIdx.x == 0) release_tile_counter(p.tile_ctr, nclusters);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);  // lane 0 of the 4 epilogue warps of each CTA
        }
        mbar_init(drain, 1);
        for (int s = 0; s < kItemRing; ++s) {
            mbar_init(&item_full[s], 1);
            mbar_init(&item_empty[s], kItemConsumers);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // both CTAs' barriers are initialised before any remote arrive or
    // multicast commit can reach them
    cluster_sync_all();
    const uint64_t pol_w = 0ull;
    int prefilled = 0;
    if (early && threadIdx.x == 0) {
        // (dynamic order: only item 0, the one tile known before the wait)
        for (int w = cluster; w < total && prefilled < C::STAGES && !(dyn && w != cluster);
             w += nclusters) {
            const int tile = w / ks, sp = w - tile * ks;
            const GroupTile gt = decode_tile<true>(p, mt_start, nt, 2 * BM, tile);
            const CUtensorMap* mb = gt.g < p.E ? &tmB0 : &tmB1;
            int brow[Cfg<BN>::B_LOADS];
            b_tile_rows<BN, EPI>(p, gt, brow);
            const int kb_hi = (sp + 1) * nkb / ks;
            for (int kb = sp * nkb / ks; kb < kb_hi && prefilled < C::STAGES; ++kb) {
                if (leader) {
                    mbar_arrive_expect_tx(&full[prefilled], 2 * C::STAGE_BYTES);
                    tma_load_2d(sB + prefilled * C::B_BYTES, mb, &full[prefilled], kb * BK,
                                brow[rank]);
                } else {
                    tma_load_2d_to_pair_bar(sB + prefilled * C::B_BYTES, mb,
                                            mapa_shared(smem_u32(&full[prefilled]), 0), kb * BK,
                                            brow[rank]);
                }
                ++prefilled;
            }
        }
    }
    (void)pol_w;
    if (early) pdl_wait();
    pdl_trigger();
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Work items of the pair, in order i = 0, 1, ...: item 0 is tile `cluster`;
    // after it, every nclusters-th tile (static order), or (dynamic order) the
    // next tile of the launch-wide counter, which the even CTA's producer
    // takes two items ahead and hands to the 10 consumers (its MMA issuer,
    // both CTAs' 4 epilogue warps, the odd CTA's producer) one item ahead
    // through the ring, the odd CTA's copy by a remote store released with the
    // remote arrive. Values >= total end the sequence.
    auto item_put = [&](int i, int v) -> bool {
        const int s = i % kItemRing;
        const uint32_t ph = (uint32_t)(i / kItemRing) & 1u;
        if (!mbar_wait(&item_empty[s], ph ^ 1u, abort_flag, p.status, args.wait_ns)) return false;
        s_item[s] = v;
        st_shared_cluster(mapa_shared(smem_u32((const void*)&s_item[s]), 1), v);
        mbar_arrive(&item_full[s]);
        mbar_arrive_remote_release(mapa_shared(smem_u32(&item_full[s]), 1));
        return true;
    };
    // -1: the wait gave up (timeout or abort)
    auto item_get = [&](int i) -> int {
        const int s = i % kItemRing;
        const uint32_t ph = (uint32_t)(i / kItemRing) & 1u;
        const bool okw =
            leader ? mbar_wait(&item_full[s], ph, abort_flag, p.status, args.wait_ns)
                   : mbar_wait_acq_cluster(&item_full[s], ph, abort_flag, p.status, args.wait_ns);
        return okw ? s_item[s] : -1;
    };
    auto item_release = [&](int i) {
        const int s = i % kItemRing;
        if (leader)
            mbar_arrive(&item_empty[s]);
        else
            mbar_arrive_remote_release(mapa_shared(smem_u32(&item_empty[s]), 0));
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;
            bool ok = true;
            int item = 0;
            // dynamic order, even CTA: item it+1 is handed out before item it
            // is loaded (so the odd CTA's producer never waits for it at a
            // tile boundary), and its tile comes from a counter read one item
            // earlier still (so the atomic's latency is hidden)
            int w_cur = cluster, w_nxt = 0;
            if (dyn && leader) {
                ok = item_put(0, w_cur < total ? w_cur : total);
                w_nxt = nclusters + atomicAdd(p.tile_ctr, 1);
            }
            for (int it = 0; ok; ++it) {
                int w = cluster + it * nclusters;
                if (dyn && leader) {
                    w = w_cur;
                    if (w >= total) break;  // the end mark went out as item it
                    const int w_after = nclusters + atomicAdd(p.tile_ctr, 1);  // item it+2
                    if (!item_put(it + 1, w_nxt < total ? w_nxt : total)) {
                        ok = false;
                        break;
                    }
                    w_cur = w_nxt;
                    w_nxt = w_after;
                } else if (dyn) {
                    w = item_get(it);
                    if (w < 0) {
                        ok = false;
                        break;
                    }
                    item_release(it);
                }
                if (w >= total) break;
                const int tile = w / ks, sp = w - tile * ks;
                const GroupTile gt = decode_tile(p, mt_start, nt, 2 * BM, tile);
                const bool routed = gt.g < p.E;
                const CUtensorMap* ma = routed ? &tmA0 : &tmA1;
                const CUtensorMap* mb = routed ? &tmB0 : &tmB1;
                int brow[Cfg<BN>::B_LOADS];
                b_tile_rows<BN, EPI>(p, gt, brow);
                const int a_row = gt.a_row + BM * (int)rank;  // this CTA's 128 rows
                const int kb_lo = sp * nkb / ks, kb_hi = (sp + 1) * nkb / ks;
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++item) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const bool fresh = item >= prefilled;
                    if (leader) {
                        // arms the stage for both CTAs' bytes
                        if (fresh) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                        tma_load_2d(sA + stage * C::A_BYTES, ma, &full[stage], kb * BK, a_row);
                        if (fresh)
                            tma_load_2d(sB + stage * C::B_BYTES, mb, &full[stage], kb * BK,
                                        brow[rank]);
                    } else {
                        const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
                        tma_load_2d_to_pair_bar(sA + stage * C::A_BYTES, ma, bar, kb * BK, a_row);
                        if (fresh)
                            tma_load_2d_to_pair_bar(sB + stage * C::B_BYTES, mb, bar, kb * BK,
                                                    brow[rank]);
                    }
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok && leader) {
                // aborting: let the copies of the armed stages land (both CTAs' bytes)
                for (int s = 0; s < C::STAGES; ++s)
                    if ((filled >> s) & 1u) {
                        volatile int never = 0;
                        mbar_wait(&full[s], (fill_parity >> s) & 1u, &never, p.status, kDrainNs);
                    }
            } else if (!ok) {
                // the odd CTA's copies count on the even CTA's barriers: give
                // any still in flight time to land in this CTA's shared memory
                const unsigned long long t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // -------------------------------------------- MMA issuer (even CTA)
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int it = 0; ok; ++it, ++local) {
                int w = cluster + it * nclusters;
                if (dyn) {
                    w = item_get(it);
                    if (w < 0) {
                        ok = false;
                        break;
                    }
                    item_release(it);
                }
                if (w >= total) break;
                const int sp = w % ks;
                const int b = local & 1;
                const uint32_t tph = (local >> 1) & 1;
                if (!mbar_wait(&tempty[b], tph ^ 1, abort_flag, p.status, args.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
                const int kb_lo = sp * nkb / ks, kb_hi = (sp + 1) * nkb / ks;
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_sw128(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bd = sdesc_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BKH / 16; ++kk)
                        umma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, C::IDESC,
                                       (kb != kb_lo || kk != 0) ? 1u : 0u);
                    umma_commit_pair_mc(&empty[stage], 0x3);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok && !(args.hold_first_acc && local == 0)) umma_commit_pair_mc(&tfull[b], 0x3);
            }
            // every pair MMA completes before the pair's TMEM and shared memory are released
            umma_commit_pair_mc(drain, 0x1);
            volatile int never = 0;
            mbar_wait(drain, 0, &never, p.status, kDrainNs);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, both CTAs)
        if (p.fin_acc_mem && blockIdx.x == 0) {
            const AuxAcc acc = aux_acc_at(p.fin_acc_mem, p.E, kAuxGroups);
            const AuxOut out{p.fin_f, p.fin_P, p.fin_I, p.fin_out3, p.fin_w_imp};
            aux_finalize(p.T, p.E, p.fin_k, acc, out, threadIdx.x - 64, 128, EpilogueBar{});
        }
        const int q = warp & 3;
        const int trow = BM * (int)rank + 32 * q + lane;  // this thread's row of the 256-row tile
        const uint64_t pol_o = l2_evict_last_policy();
        const uint32_t tempty_remote0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t tempty_remote1 = mapa_shared(smem_u32(&tempty[1]), 0);
        int local = 0;
        for (int it = 0;; ++it, ++local) {
            int w = cluster + it * nclusters;
            if (dyn) {
                // lane 0 takes the item for the warp, so the warp stays converged
                int v = 0;
                if (lane == 0) {
                    v = item_get(it);
                    if (v >= 0) item_release(it);
                }
                w = __shfl_sync(0xffffffffu, v, 0);
                if (w < 0) break;
            }
            if (w >= total) break;
            const int tile = w / ks, sp = w - tile * ks;
            const GroupTile gt = decode_tile(p, mt_start, nt, 2 * BM, tile);
            const int b = local & 1;
            const uint32_t tph = (local >> 1) & 1;
            if (!mbar_wait(&tfull[b], tph, abort_flag, p.status, args.wait_ns)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(b * BN) + ((uint32_t)(32 * q) << 16);
            const bool rv = trow < gt.rows;
            const bool routed = gt.g < p.E;
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(routed ? p.out0 : p.out1);
            uint32_t* stg = reinterpret_cast<uint32_t*>(staging) + q * 32 * 20;
            const bool keep_l2 = MOE_TC_L2_HINTS && p.out_l2_keep;
            int dst_row = rv ? gt.out_row + trow : -1;
            if (EPI == EPI_ROUTER) {
                // as in the single-CTA kernel: 32 rows x 32 columns staged per
                // warp, then whole 128-byte row segments (lane = column)
                (void)out;
                (void)dst_row;
                float* rstg = staging + q * 32 * 33;
                const int row0 = BM * (int)rank + 32 * q;  // the warp's first tile row
                const int rows_here = min(32, gt.rows - row0);
                const int E_r = args.E_router;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) rstg[lane * 33 + i] = v[i];
                    __syncwarp();
                    const int n = gt.n_tile * BN + c + lane;
                    if (n < p.N && args.part) {
                        float* dst = args.part + (size_t)sp * p.T * p.N + n;
                        for (int r = 0; r < rows_here; ++r)
                            dst[(size_t)(gt.out_row + row0 + r) * p.N] = rstg[r * 33 + lane];
                    } else if (n < p.N) {
                        const bool is_logit = n < E_r;
                        const float off = (is_logit && args.offset) ? args.offset[n] : 0.f;
                        float* dst = is_logit ? args.logits + n : args.zn + (n - E_r);
                        for (int r = 0; r < rows_here; ++r) {
                            const size_t t = (size_t)(gt.out_row + row0 + r);
                            dst[t * E_r] = rstg[r * 33 + lane] + off;
                        }
                    }
                    __syncwarp();
                }
            } else if (EPI == EPI_GLU) {
                // columns 0..127 hold the gate half (from the even CTA's
                // weight rows), 128..255 the up half (the odd CTA's)
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    float g[16], u[16], v[32];
                    tmem_ld16x2(taddr + c, taddr + 128 + c, g, u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = silu(g[i]) * u[i];
                    tmem_ld16x2(taddr + c + 16, taddr + 128 + c + 16, g, u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[16 + i] = silu(g[i]) * u[i];
                    const int n0 = gt.n_tile * 128 + c;
                    if (n0 < p.N) store_rows32_bf16(out, p.N, n0, dst_row, v, stg, keep_l2, pol_o);
                }
            } else {
                const int act = p.glu ? -1 : p.act;
                float scale = 1.f;
                if (routed && p.scatter_rows) {
                    const int t = rv ? p.scatter_rows[gt.out_row + trow] : 0;
                    out = reinterpret_cast<__nv_bfloat16*>(p.scatter_out);
                    dst_row = rv ? t : -1;
                    scale = rv ? p.scatter_scale[t] : 0.f;
                }
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
                    const int n0 = gt.n_tile * BN + c;
                    if (n0 < p.N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = act_apply(act, v[i]) * scale;
                        store_rows32_bf16(out, p.N, n0, dst_row, v, stg, keep_l2, pol_o);
                    }
                }
                if (p.fold_cnt) fold_tile(p, gt, routed, trow, rv);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&tempty[b]);
                else
                    mbar_arrive_remote(b ? tempty_remote1 : tempty_remote0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // no CTA of the pair frees its TMEM or shared memory, or exits, while
    // the pair's MMAs (drained above), copies or remote arrives may use them
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    if (dyn && leader && threadIdx.x == 0) release_tile_counter(p.tile_ctr, nclusters);
}

// Launches the pair kernel: clusters of two CTAs on SM pairs, at most one
// cluster per two SMs.
template <int EPI>
static cudaError_t launch_pair(const TcArgs& a, cudaStream_t st) {
    using C = PairCfg;
    const GroupedGemm& p = a.p;
    CUtensorMap mA0, mA1, mB0, mB1;
    const int G = p.E + p.S;
    if (!make_map(&mA0, p.A0 ? p.A0 : p.A1, p.A0 ? p.rows_a0 : p.rows_a1, p.K, BM) ||
        !make_map(&mA1, p.A1 ? p.A1 : p.A0, p.A1 ? p.rows_a1 : p.rows_a0, p.K, BM))
        return cudaErrorInvalidValue;
    const int brows0 = p.E * p.b_rows_group, brows1 = p.S * p.b_rows_group;
    if (!make_map(&mB0, p.B0 ? p.B0 : p.B1, p.B0 ? brows0 : brows1, p.K, 128) ||
        !make_map(&mB1, p.B1 ? p.B1 : p.B0, p.B1 ? brows1 : brows0, p.K, 128))
        return cudaErrorInvalidValue;
    const size_t smem = C::smem_bytes(G);
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<EPI>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int ncol_tile = EPI == EPI_GLU ? 128 : C::BN;
    const long long nt = (p.N + ncol_tile - 1) / ncol_tile;
    const int MT = 2 * BM;
    long long mt = (long long)p.max_rows0 / MT + p.E + (long long)p.S * ((p.T + MT - 1) / MT);
    if (p.E == 0) mt = (long long)p.S * ((p.T + MT - 1) / MT);
    const long long bound = std::max<long long>(1, mt * nt * (EPI == EPI_ROUTER ? a.ksplit : 1));
    const int nclusters = (int)std::min<long long>(bound, std::max(1, num_sms() / 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * nclusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<EPI>, mA0, mA1, mB0, mB1, a);
}

}  // namespace tc

cudaError_t launch_grouped_gemm_tc(const Shape& s, const GroupedGemm& g, cudaStream_t st) {
    tc::TcArgs a{};
    a.p = g;
    a.ksplit = 1;
    a.wait_ns = wait_limit_ns();
    a.hold_first_acc = hold_first_accumulator();
    const bool wef = MOE_TC_L2_HINTS && g.b_evict_first;
    if (g.pair && !wef)
        return g.glu ? tc::launch_pair<tc::EPI_GLU>(a, st) : tc::launch_pair<tc::EPI_ACT>(a, st);
    if (g.glu)
        return wef ? tc::launch<256, tc::EPI_GLU, true>(a, st)
                   : tc::launch<256, tc::EPI_GLU, false>(a, st);
    return wef ? tc::launch<MOE_TC_BN_ACT, tc::EPI_ACT, true>(a, st)
               : tc::launch<MOE_TC_BN_ACT, tc::EPI_ACT, false>(a, st);
}

// Plan of the router GEMM (T x Nr outputs, K = d). The column tile is the
// narrowest of 32/64/128/256 that covers Nr, so x is read once per row tile.
// A 256-wide router runs on CTA pairs (256-row tiles, each SM loading its own
// 128 rows of x and half of the 256 router columns: a third fewer operand
// bytes per MMA than a 128-row tile on one SM). When the output tiles would
// leave SMs idle, the K range of each tile is split over 2, 4, ... CTAs (each
// keeping at least 4 blocks of K) while the work items fit one wave. The plan
// assumes a 148-SM part whatever the device, so the split, and with it every
// rounding of the logits, is the same on any GPU.
void router_plan(int T, int d, int Nr, int* bn, int* ksplit, int* pair, int* tile_rows) {
    constexpr int kPlanSms = 148;
    const int b = Nr <= 32 ? 32 : Nr <= 64 ? 64 : Nr <= 128 ? 128 : 256;
    const int pr = MOE_ROUTER_PAIR && b == 256 ? 1 : 0;
    const int nkb = (d + tc::BK - 1) / tc::BK;
    const long long ncol = (Nr + b - 1) / b;
    // a memory-bound router (at most 128 columns) that would leave SMs idle
    // with 128-row tiles and no split takes tiles of ceil(T / 148) rows
    // (at least 64), one per SM
    int tm = pr ? 2 * tc::BM : tc::BM;  // rows of a tile
    if (MOE_ROUTER_SHORT_TILES && !pr && ncol == 1) {
        const long long t128 = (T + tc::BM - 1) / tc::BM;
        if (t128 < kPlanSms && !(t128 * 2 <= kPlanSms && nkb / 2 >= 4)) {
            const int want = (int)((T + kPlanSms - 1) / kPlanSms);
            if (want >= 64 && want < tc::BM) tm = want;
        }
    }
    const long long tiles = (long long)((T + tm - 1) / tm) * ncol;
    const long long ctas = tiles * (pr ? 2 : 1);  // CTAs per K part
    int s = 1;
    while (ctas * s * 2 <= kPlanSms && nkb / (s * 2) >= 4) s *= 2;
    *bn = b;
    *ksplit = s;
    if (pair) *pair = pr;
    if (tile_rows) *tile_rows = pr ? 0 : tm;
}

bool router_sel_in_gemm(const Shape& s, bool noisy) {
    if (!MOE_ROUTER_SEL_IN_GEMM || s.dtype != MOE_BF16 || noisy || s.E > 32 || s.nc > 8)
        return false;
    int bn, ks, pair;
    router_plan(s.T, s.d, s.E, &bn, &ks, &pair);
    return bn == 32 && ks == 1 && !pair;
}

cudaError_t launch_router_gemm_bf16(const Shape& s, int Nr, const void* x, const void* wgT,
                                    const float* offset, float* logits, float* zn, float* part,
                                    int* status, cudaStream_t st, const RouterSelOut* so) {
    tc::TcArgs a{};
    GroupedGemm& p = a.p;
    p.offsets = nullptr;
    p.E = 0;
    p.S = 1;
    p.T = s.T;
    p.a1_row0 = 0;
    p.a1_stride = 0;
    p.rows_a0 = 0;
    p.max_rows0 = 0;
    p.rows_a1 = s.T;
    p.N = Nr;
    p.K = s.d;
    p.b_rows_group = Nr;
    p.glu = 0;
    p.act = -1;
    p.A0 = nullptr;
    p.A1 = x;
    p.B0 = nullptr;
    p.B1 = wgT;
    p.out0 = nullptr;
    p.out1 = nullptr;
    p.status = status;
    a.offset = offset;
    a.logits = logits;
    a.zn = zn;
    a.E_router = s.E;
    a.wait_ns = wait_limit_ns();
    a.hold_first_acc = hold_first_accumulator();
    int bn, ks, pair, tm;
    router_plan(s.T, s.d, Nr, &bn, &ks, &pair, &tm);
    a.ksplit = ks;
    a.router_tm = tm;
    if (so) {
        if (!router_sel_in_gemm(s, zn != nullptr) || Nr != s.E) return cudaErrorInvalidValue;
        a.rs.on = 1;
        a.rs.k = s.k;
        a.rs.nc = s.nc;
        a.rs.renorm = s.renorm;
        a.rs.bias = so->bias;
        a.rs.probs = so->probs;
        a.rs.sel = so->sel;
        a.rs.ids = so->ids;
        a.rs.w = so->w;
        a.rs.blk_hist = so->blk_hist;
        a.rs.nblk_cap = (s.T + kCapBlockTokens - 1) / kCapBlockTokens;
        a.rs.acc_mem = so->acc_mem;
        a.rs.late_trigger = so->late_trigger;
    }
    a.part = ks > 1 ? part : nullptr;
    if (ks > 1 && !part) return cudaErrorInvalidValue;
    if (pair) return tc::launch_pair<tc::EPI_ROUTER>(a, st);
    if (bn == 32) return tc::launch<32, tc::EPI_ROUTER, false>(a, st);
    if (bn == 64) return tc::launch<64, tc::EPI_ROUTER, false>(a, st);
    if (bn == 128) return tc::launch<128, tc::EPI_ROUTER, false>(a, st);
    return tc::launch<256, tc::EPI_ROUTER, false>(a, st);
}

}  // namespace moe
