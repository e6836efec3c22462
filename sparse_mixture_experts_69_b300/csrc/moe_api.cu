// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace carving and the order of launches on the caller's stream.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "aux_common.cuh"

// Token rows (A operand) of one block of the expert GEMMs' tile order, in MB
// (group_table.cuh); 0: no blocks (each weight tile sweeps all of a group's
// rows before the next).
#ifndef MOE_ROW_BLOCK_MB
#define MOE_ROW_BLOCK_MB 32
#endif

// 1: the expert GEMMs of layers whose experts hold many rows run 256-row
// tiles on CTA pairs (gemm_tc.cu, grouped_gemm_pair_kernel); 0: never.
#ifndef MOE_PAIR_TILES
#define MOE_PAIR_TILES 1
#endif
// ... when the experts hold at least this many rows on average (R_max / E)
#ifndef MOE_PAIR_MIN_ROWS
#define MOE_PAIR_MIN_ROWS 1024
#endif
// 1: layers of mixed expert sizes run each expert projection as two launches
// (few-row experts on single CTAs, many-row experts on CTA pairs); 0: one.
#ifndef MOE_SPLIT_LAUNCH
#define MOE_SPLIT_LAUNCH 1
#endif
// 1: the CTA-pair expert GEMMs take their tiles from a launch-wide counter
// (in order), so the tiles in flight stay a window of consecutive tiles
#ifndef MOE_PAIR_DYNAMIC
#define MOE_PAIR_DYNAMIC 1
#endif

namespace moe {

cudaError_t launch_grouped_gemm_tc(const Shape& s, const GroupedGemm& g, cudaStream_t st);
cudaError_t launch_grouped_gemm_simt(const Shape& s, const GroupedGemm& g, cudaStream_t st);

cudaError_t launch_grouped_gemm(const Shape& s, const GroupedGemm& g, cudaStream_t st) {
    return s.dtype == MOE_BF16 ? launch_grouped_gemm_tc(s, g, st)
                               : launch_grouped_gemm_simt(s, g, st);
}

int num_sms() {
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_policy_passes{kDefaultPolicyPasses};
std::atomic<int> g_hold_first_acc{0};
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int policy_max_passes() { return g_policy_passes.load(std::memory_order_relaxed); }
int hold_first_accumulator() { return g_hold_first_acc.load(std::memory_order_relaxed); }

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

WsLayout ws_layout(const Shape& s) {
    WsLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align256(off + std::max<size_t>(bytes, 1));
        return o;
    };
    const size_t T = s.T, E = s.E, d = s.d, F = s.F, S = s.S, R = s.R_max;
    const size_t es = s.esize;
    const size_t nblk = (T + kCapBlockTokens - 1) / kCapBlockTokens;
    L.status = take(256);
    L.aux_acc = take(aux_acc_bytes((int)E, kAuxGroups));
    L.blk_hist = take(nblk * E * 4);
    L.cap_ticket = take(16);
    L.seq_ticket = take(16);
    L.tile_ctr = take(16);
    L.fold_cnt = take(s.dtype == MOE_BF16 ? T * ((d + kDownTileN - 1) / kDownTileN) * 4 : 0);
    L.zero_end = off;
    L.zn = take(T * E * 4);
    size_t part = 0;  // K parts of the router GEMM, for Nr = E or 2E (noisy)
    if (s.dtype == MOE_BF16)
        for (int nr = (int)E; nr <= 2 * (int)E; nr += (int)E) {
            int bn, ks;
            router_plan(s.T, s.d, nr, &bn, &ks);
            if (ks > 1) part = std::max(part, (size_t)ks * T * nr * 4);
        }
    L.rpart = take(part);
    L.wgT = take(2 * E * d * es);
    L.logits = take(T * E * 4);
    L.probs = take(T * E * 4);
    const size_t nc = s.nc;
    const bool ec = s.routing == MOE_EXPERT_CHOICE;
    L.ids = take(T * nc * 4);
    L.w = take(T * nc * 4);
    L.slot = take(T * nc * 4);
    L.tok_row = take(ec ? T * E * 4 : 0);
    L.row_w = take(ec ? R * 4 : 0);
    L.seq_acc = take(seq_aux_scratch_bytes((int)E, (int)T + 1));
    L.counts = take(E * 4);
    L.kept = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.row_token = take(R * 4);
    L.tok_need = take(T * 4);
    L.blk_base = take(nblk * E * 4);
    L.xp = take(R * d * es);
    L.h = take((R + S * T) * F * es);
    L.yp = take(R * d * es);
    L.ys = take(S * T * d * es);
    L.aux_vecs = take(3 * E * 4);
    L.out3 = take(16);
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status make_shape(const moe_config* c, Shape* s) {
    if (!c || !s) return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->d_model < 1 || c->n_experts < 1 || c->top_k < 1 || c->d_ff < 1 ||
        c->n_shared < 0 || c->top_k > c->n_experts)
        return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->act < MOE_RELU || c->act > MOE_SWIGLU) return MOE_ERR_INVALID_ARG;
    if (c->renorm_topk != 0 && c->renorm_topk != 1) return MOE_ERR_INVALID_ARG;
    if (!isfinite(c->capacity_factor) || !isfinite(c->importance_weight))
        return MOE_ERR_INVALID_ARG;
    if (c->reroute < 0 || c->priority < MOE_PRIORITY_TOKEN || c->priority > MOE_PRIORITY_RANK ||
        (c->pad_to_capacity != 0 && c->pad_to_capacity != 1) || c->routing < MOE_TOKEN_CHOICE ||
        c->routing > MOE_EXPERT_CHOICE)
        return MOE_ERR_INVALID_ARG;
    const bool ec = c->routing == MOE_EXPERT_CHOICE;
    if (ec && (c->reroute != 0 || c->priority != MOE_PRIORITY_TOKEN)) return MOE_ERR_INVALID_ARG;
    if ((long long)c->top_k + c->reroute > c->n_experts) return MOE_ERR_INVALID_ARG;
    if (c->n_experts > 1024 || c->top_k + c->reroute > 32 || c->n_shared > 64)
        return MOE_ERR_UNSUPPORTED;
    if (c->d_model % 8 != 0 || c->d_ff % 8 != 0) return MOE_ERR_UNSUPPORTED;
    // capacity with re-routing or rank priority runs in one thread-block cluster
    const bool policy = !ec && (c->reroute > 0 || c->priority == MOE_PRIORITY_RANK);
    if (policy && (c->n_experts > 512 || c->T > 131072)) return MOE_ERR_UNSUPPORTED;
    // expert choice keeps one expert's column of probabilities in shared memory
    if (ec && c->T > 32768) return MOE_ERR_UNSUPPORTED;
    const long long T = c->T, E = c->n_experts, k = c->top_k, S = c->n_shared;
    const long long nc = k + c->reroute;
    long long C = T;
    if (c->capacity_factor > 0.f) {
        C = (long long)ceil((double)T * (double)c->capacity_factor / (double)E);
        if (C > T) C = T;  // no expert can receive more than T tokens
    }
    const long long R = (ec || c->pad_to_capacity) ? E * C : std::min(T * k, E * C);
    const long long F1 = c->act == MOE_SWIGLU ? 2LL * c->d_ff : c->d_ff;
    // row indices and TMA coordinates are 32-bit
    if (T * nc >= (1LL << 31) || T * E >= (1LL << 31) || R + S * T >= (1LL << 31) ||
        E * F1 >= (1LL << 31) ||
        E * (long long)c->d_model >= (1LL << 31))
        return MOE_ERR_UNSUPPORTED;
    s->T = c->T;
    s->d = c->d_model;
    s->E = c->n_experts;
    s->k = c->top_k;
    s->F = c->d_ff;
    s->S = c->n_shared;
    s->F1 = (int)F1;
    s->C = (int)C;
    s->R_max = (int)R;
    s->dtype = c->dtype;
    s->act = c->act;
    s->renorm = c->renorm_topk;
    s->nc = (int)nc;
    s->priority = c->priority;
    s->pad = ec ? 0 : c->pad_to_capacity;
    s->routing = c->routing;
    s->w_imp = c->importance_weight;
    s->esize = c->dtype == MOE_BF16 ? 2 : 4;
    if (c->noise_draw != 0 && c->noise_draw != 1) return MOE_ERR_INVALID_ARG;
    s->noise_draw = c->noise_draw;
    s->noise_seed = c->noise_seed;
    s->noise_counter = c->noise_counter;
    if (c->combine_mode < MOE_COMBINE_AUTO || c->combine_mode > MOE_COMBINE_KERNEL)
        return MOE_ERR_INVALID_ARG;
    s->combine_mode = c->combine_mode;
    return MOE_OK;
}

// Noise arguments of the router: with Wnoise, the draws are either passed in
// (noise) or drawn (noise_draw = 1, noise NULL); without Wnoise neither.
bool noise_args_ok(const Shape& s, const void* Wnoise, const float* noise) {
    if (!Wnoise) return noise == nullptr;
    return s.noise_draw ? noise == nullptr : noise != nullptr;
}

moe_status check_ws(const Shape& s, void* ws, size_t ws_bytes, WsLayout* L) {
    *L = ws_layout(s);
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

#define MOE_TRY(expr)                          \
    do {                                       \
        moe_status _st = (expr);               \
        if (_st != MOE_OK) return _st;         \
    } while (0)
#define MOE_CUDA(expr)                               \
    do {                                             \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

// Re-routing or rank priority: the cluster capacity kernel (policy.cu);
// otherwise the plain token-order dropping kernels (capacity.cu).
bool uses_policy(const Shape& s) { return s.nc > s.k || s.priority != MOE_PRIORITY_TOKEN; }

// -------------------------------------------------------------- stage bodies
// aux: if non-NULL ([3E] f, P, importance followed by out3 at aux_out3), the
// selection kernel also counts the capacity histogram and the statistics.
moe_status route_impl(const Shape& s, const WsLayout& L, void* ws, const void* x, const void* Wg,
                      const void* Wnoise, const float* noise, const float* offset,
                      const float* bias, float* logits, float* probs, float* sel, int32_t* ids,
                      float* w, float* aux_vecs, float* aux_out3, cudaStream_t st) {
    int* status = at<int>(ws, L.status);
    const bool noisy = Wnoise != nullptr;
    const int Nr = noisy ? 2 * s.E : s.E;
    float* zn = noisy ? at<float>(ws, L.zn) : nullptr;
    RouterLogits rl{logits, zn, nullptr, 1, Nr, offset};
    if (s.dtype == MOE_BF16) {
        void* wgT = at<void>(ws, L.wgT);
        int bn, ks;
        router_plan(s.T, s.d, Nr, &bn, &ks);
        if (ks > 1) {
            rl.part = at<float>(ws, L.rpart);
            rl.nsplit = ks;
        }
        MOE_CUDA(launch_transpose_router_w(s, Wg, Wnoise, wgT, st));
        if (router_sel_in_gemm(s, noisy)) {
            // the GEMM's epilogue selects: no selection kernel
            RouterSelOut so{bias, probs, sel, ids, w, nullptr, nullptr, 1};
            if (aux_out3) {
                so.blk_hist = uses_policy(s) ? nullptr : at<int32_t>(ws, L.blk_hist);
                so.acc_mem = at<void>(ws, L.aux_acc);
                so.late_trigger = 0;  // the capacity kernel follows (statistics: the up GEMM)
            }
            MOE_CUDA(launch_router_gemm_bf16(s, Nr, x, wgT, offset, logits, zn,
                                             at<float>(ws, L.rpart), status, st, &so));
            return MOE_OK;
        }
        MOE_CUDA(launch_router_gemm_bf16(s, Nr, x, wgT, offset, logits, zn,
                                         at<float>(ws, L.rpart), status, st));
    } else {
        MOE_CUDA(launch_router_gemm_f32(s, Nr, static_cast<const float*>(x),
                                        static_cast<const float*>(Wg),
                                        static_cast<const float*>(Wnoise), offset, logits, zn,
                                        st));
    }
    if (aux_out3) {
        // bf16: the up GEMM (tcgen05) finalises the statistics later in the layer
        MOE_CUDA(launch_router_select_fused(s, rl, noisy ? noise : nullptr, bias, probs, ids, w,
                                            status,
                                            uses_policy(s) ? nullptr : at<int32_t>(ws, L.blk_hist),
                                            at<void>(ws, L.aux_acc), aux_vecs, aux_vecs + s.E,
                                            aux_vecs + 2 * s.E, aux_out3,
                                            s.dtype == MOE_BF16, st));
    } else {
        // moe_route's logits are an output: formed here when the GEMM was split
        MOE_CUDA(launch_router_select(s, rl, rl.nsplit > 1 ? logits : nullptr,
                                      noisy ? noise : nullptr, bias, probs, sel, ids, w, 0,
                                      nullptr, nullptr, status, st));
    }
    return MOE_OK;
}

moe_status dispatch_impl(const Shape& s, const WsLayout& L, void* ws, const void* x,
                         const int32_t* ids, int32_t* counts, int32_t* kept, int32_t* offsets,
                         int32_t* slot, void* xp, int32_t* row_token, bool hist_ready,
                         void* y_zero, int32_t* tok_need, cudaStream_t st) {
    int* status = at<int>(ws, L.status);
    // padded blocks: rows no token takes must read zero, so clear the block
    // buffer first (the permute then fills the taken rows)
    if (s.pad)
        MOE_CUDA(cudaMemsetAsync(xp, 0, (size_t)s.R_max * s.d * s.esize, st));
    if (uses_policy(s)) {
        MOE_CUDA(launch_capacity_policy(s, ids, counts, kept, offsets, slot, row_token, status,
                                        st));
    } else {
        MOE_CUDA(launch_capacity(s, ids, at<int32_t>(ws, L.blk_hist),
                                 at<unsigned int>(ws, L.cap_ticket), at<int32_t>(ws, L.blk_base),
                                 counts, kept, offsets, slot, row_token, status, hist_ready, st));
    }
    MOE_CUDA(launch_permute(s, x, slot, xp, y_zero, tok_need, status, st));
    return MOE_OK;
}

// Expert choice: select per expert, gather the chosen rows.
moe_status ec_dispatch_impl(const Shape& s, const WsLayout& L, void* ws, const void* x,
                            const float* probs, int32_t* offsets, int32_t* row_token,
                            float* row_w, int32_t* tok_row, void* xp, cudaStream_t st) {
    MOE_CUDA(launch_expert_choice_select(s, probs, offsets, row_token, row_w, tok_row,
                                         at<int>(ws, L.status), st));
    MOE_CUDA(launch_gather_rows(s, s.E * s.C, x, row_token, xp, st));
    return MOE_OK;
}

// scatter (top-1, no shared experts, bf16): the down GEMM writes y[token] =
// gate * output directly through row_token instead of yp (no combine pass).
// fold (bf16, otherwise): the down GEMM writes yp and ys and also sums each
// token's rows into y once the last of them is stored (no combine launch).
// fin_aux_vecs / fin_out3 (layer path, bf16): the up GEMM finalises the
// statistics the selection kernel accumulated.
// The combine of the layer path, done by the down projection (ffn_impl).
struct Fold {
    const int32_t* row_token;  // [R_max]
    const int32_t* slot;       // [T,nc]
    const float* w;            // [T,nc]
    void* y;                   // [T,d]
};

moe_status ffn_impl(const Shape& s, const WsLayout& L, void* ws, const void* xp,
                    const int32_t* offsets, const void* W1, const void* W2, const void* x,
                    const void* W1s, const void* W2s, void* yp, void* ys,
                    const int32_t* scatter_rows, const float* scatter_gate, void* y,
                    float* fin_aux_vecs, float* fin_out3, bool up_early, const Fold* fold,
                    cudaStream_t st) {
    int* status = at<int>(ws, L.status);
    void* h = at<void>(ws, L.h);
    void* h_shared = static_cast<char*>(h) + (size_t)s.R_max * s.F * s.esize;
    GroupedGemm up{};
    up.offsets = offsets;
    up.E = s.E;
    up.S = s.S;
    up.T = s.T;
    up.a1_row0 = 0;
    up.a1_stride = 0;
    up.rows_a0 = s.R_max;
    up.max_rows0 = s.R_max;
    up.rows_a1 = s.T;
    up.N = s.F;
    up.K = s.d;
    up.b_rows_group = s.F1;
    up.glu = s.act == MOE_SWIGLU;
    up.act = s.act;
    up.A0 = xp;
    up.A1 = s.S ? x : nullptr;
    up.B0 = W1;
    up.B1 = s.S ? W1s : nullptr;
    up.out0 = h;
    up.out1 = h_shared;
    if (fin_out3) {
        up.fin_acc_mem = at<void>(ws, L.aux_acc);
        up.fin_f = fin_aux_vecs;
        up.fin_P = fin_aux_vecs + s.E;
        up.fin_I = fin_aux_vecs + 2 * s.E;
        up.fin_out3 = fin_out3;
        up.fin_k = s.k;
        up.fin_w_imp = s.w_imp;
    }
    up.status = status;
    up.tile_ctr = MOE_PAIR_DYNAMIC ? at<int32_t>(ws, L.tile_ctr) : nullptr;
    // T <= 128 (decode): every expert, routed or shared, gets at most one
    // 128-row tile, so every weight tile is read once and the weights may leave
    // L2 first. Measured: decode layer 467 -> 455 us; on the Switch layer,
    // whose experts also have one tile each, the standalone FFN was 2% slower.
    const int one_tile = s.T <= 128 ? 1 : 0;
    up.b_evict_first = one_tile;
    up.early = up_early ? 1 : 0;
    // h is read back by the down projection: keep it in L2 when it fits with
    // room to spare (126 MB of L2), else let it stream
    up.out_l2_keep = (double)(s.R_max + (double)s.S * s.T) * s.F * s.esize <= 80e6 ? 1 : 0;
    // experts of at least 1024 rows on average (the Mixtral-shaped layer):
    // 256-row tiles on CTA pairs, which halve each SM's weight bytes per MMA
    const int pair = MOE_PAIR_TILES && (long long)s.R_max >= (long long)MOE_PAIR_MIN_ROWS * s.E ? 1 : 0;
    // experts of mixed sizes (at least 256 rows per expert on average, but
    // not all large: the DeepSeek-shaped layer): each projection runs as two
    // launches, the experts of fewer than kSplitRows rows on single CTAs,
    // then the others (and the shared experts) on CTA pairs
    constexpr int kSplitRows = 512;
    const bool split = MOE_PAIR_TILES && MOE_SPLIT_LAUNCH && !pair && !one_tile &&
                       s.dtype == MOE_BF16 && (long long)s.T * s.k >= 256LL * s.E;
    auto row_block = [&](int K, int tile_rows) {
        const double tile_mb = (double)tile_rows * K * s.esize / 1e6;
        return MOE_ROW_BLOCK_MB > 0 ? std::max(1, (int)(MOE_ROW_BLOCK_MB / tile_mb)) : 0;
    };
    // one projection, as one launch or as the two launches described above
    auto launch_parts = [&](GroupedGemm g, int K) -> cudaError_t {
        g.pair = pair;
        g.row_block = row_block(K, pair ? 256 : 128);
        if (!split) return launch_grouped_gemm(s, g, st);
        GroupedGemm light = g;
        light.rows_hi = kSplitRows - 1;
        cudaError_t err = launch_grouped_gemm(s, light, st);
        if (err != cudaSuccess) return err;
        GroupedGemm heavy = g;
        heavy.rows_lo = kSplitRows;
        heavy.pair = 1;
        heavy.row_block = row_block(K, 256);
        heavy.fin_acc_mem = nullptr;  // the first launch finalises the statistics
        heavy.early = 1;              // the launch before it signals after its wait
        return launch_grouped_gemm(s, heavy, st);
    };
    MOE_CUDA(launch_parts(up, s.d));
    GroupedGemm dn{};
    dn.offsets = offsets;
    dn.E = s.E;
    dn.S = s.S;
    dn.T = s.T;
    dn.a1_row0 = s.R_max;
    dn.a1_stride = s.T;
    dn.rows_a0 = s.R_max;
    dn.max_rows0 = s.R_max;
    dn.rows_a1 = s.R_max + s.S * s.T;
    dn.N = s.d;
    dn.K = s.F;
    dn.b_rows_group = s.d;
    dn.glu = 0;
    dn.act = -1;
    dn.A0 = h;
    dn.A1 = s.S ? h : nullptr;
    dn.B0 = W2;
    dn.B1 = s.S ? W2s : nullptr;
    dn.out0 = yp;
    dn.out1 = s.S ? ys : nullptr;
    dn.scatter_rows = scatter_rows;
    dn.scatter_scale = scatter_gate;
    dn.scatter_out = y;
    if (fold) {
        dn.fold_cnt = at<int32_t>(ws, L.fold_cnt);
        dn.fold_need = at<int32_t>(ws, L.tok_need);
        dn.fold_rows = fold->row_token;
        dn.fold_slot = fold->slot;
        dn.fold_w = fold->w;
        dn.fold_nc = s.nc;
        dn.fold_y = fold->y;
    }
    dn.status = status;
    dn.tile_ctr = MOE_PAIR_DYNAMIC ? at<int32_t>(ws, L.tile_ctr) + 2 : nullptr;
    dn.b_evict_first = one_tile;
    // the up projection just launched signals only after its wait: when this
    // launch starts, whatever wrote the offsets before it is complete
    dn.early = 1;
    MOE_CUDA(launch_parts(dn, s.F));
    return MOE_OK;
}

}  // namespace

extern "C" {

MOE_API const char* moe_status_string(moe_status status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: unsupported size or alignment";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA call or launch failed";
        case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE: NaN or Inf found on the device";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a device pipeline wait ran out";
        case MOE_ERR_DEVICE_ARG: return "MOE_ERR_DEVICE_ARG: expert id or offsets out of range";
    }
    return "unknown moe_status";
}

MOE_API moe_status moe_capacity(const moe_config* cfg, int32_t* capacity, int32_t* rows_max) {
    Shape s;
    MOE_TRY(make_shape(cfg, &s));
    if (capacity) *capacity = s.C;
    if (rows_max) *rows_max = s.R_max;
    return MOE_OK;
}

MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
    Shape s;
    MOE_TRY(make_shape(cfg, &s));
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(s).total;
    return MOE_OK;
}

MOE_API moe_status moe_workspace_reset(const moe_config* cfg, void* ws, size_t ws_bytes,
                                       moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    MOE_CUDA(cudaMemsetAsync(ws, 0, L.zero_end, (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const void* Wg,
                             const void* Wnoise, const float* noise, const float* logit_offset,
                             const float* sel_bias, float* logits, float* probs,
                             float* sel_scores, int32_t* topk_ids, float* topk_w,
                             int32_t from_scores, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    cudaStream_t st = (cudaStream_t)stream;
    if (!probs) return MOE_ERR_INVALID_ARG;
    if ((!topk_ids || !topk_w) && !(s.routing == MOE_EXPERT_CHOICE && !topk_ids && !topk_w))
        return MOE_ERR_INVALID_ARG;
    if (from_scores) {
        if (!sel_scores) return MOE_ERR_INVALID_ARG;
        const RouterLogits none{nullptr, nullptr, nullptr, 1, s.E, nullptr};
        MOE_CUDA(launch_router_select(s, none, nullptr, nullptr, nullptr, nullptr, nullptr,
                                      topk_ids, topk_w, 1, sel_scores, probs,
                                      at<int>(ws, L.status), st));
        return MOE_OK;
    }
    if (!x || !Wg || !logits) return MOE_ERR_INVALID_ARG;
    if (!noise_args_ok(s, Wnoise, noise)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg) || (Wnoise && !aligned16(Wnoise)))
        return MOE_ERR_UNSUPPORTED;
    return route_impl(s, L, ws, x, Wg, Wnoise, noise, logit_offset, sel_bias, logits, probs,
                      sel_scores, topk_ids, topk_w, nullptr, nullptr, st);
}

MOE_API moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                                int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* slot,
                                void* xp, int32_t* row_token, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (!x || !topk_ids || !counts || !kept || !offsets || !slot || !xp || !row_token)
        return MOE_ERR_INVALID_ARG;
    if (s.routing == MOE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_UNSUPPORTED;
    return dispatch_impl(s, L, ws, x, topk_ids, counts, kept, offsets, slot, xp, row_token,
                         false, nullptr, nullptr, (cudaStream_t)stream);
}

MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* offsets,
                                  const void* W1, const void* W2, const void* x,
                                  const void* W1s, const void* W2s, void* yp, void* ys,
                                  void* ws, size_t ws_bytes, moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (!xp || !offsets || !W1 || !W2 || !yp) return MOE_ERR_INVALID_ARG;
    if (s.S > 0 && (!x || !W1s || !W2s || !ys)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(xp) || !aligned16(W1) || !aligned16(W2) || !aligned16(yp)) return MOE_ERR_UNSUPPORTED;
    if (s.S > 0 && (!aligned16(x) || !aligned16(W1s) || !aligned16(W2s) || !aligned16(ys)))
        return MOE_ERR_UNSUPPORTED;
    // the preceding kernel is the caller's: the up projection waits for it
    // before it reads the offsets
    return ffn_impl(s, L, ws, xp, offsets, W1, W2, x, W1s, W2s, yp, ys, nullptr, nullptr, nullptr,
                    nullptr, nullptr, false, nullptr, (cudaStream_t)stream);
}

MOE_API moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot,
                               const float* topk_w, const void* ys, void* y, void* ws,
                               size_t ws_bytes, moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (!yp || !slot || !topk_w || !y) return MOE_ERR_INVALID_ARG;
    if (s.routing == MOE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (s.S > 0 && !ys) return MOE_ERR_INVALID_ARG;
    if (!aligned16(yp) || !aligned16(y) || (ys && !aligned16(ys))) return MOE_ERR_UNSUPPORTED;
    MOE_CUDA(launch_combine(s, yp, slot, topk_w, s.S ? ys : nullptr, y, at<int>(ws, L.status),
                            (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_aux_stats(const moe_config* cfg, const float* probs,
                                 const int32_t* topk_ids, const float* topk_w, float* f,
                                 float* P, float* importance, float* out3, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (!probs || !topk_ids || !topk_w || !out3) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_aux(s, probs, topk_ids, topk_w, at<void>(ws, L.aux_acc), kAuxGroups, f, P,
                        importance,
                        out3, (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_bias_update(const moe_config* cfg, const int32_t* counts, float* bias,
                                   float rate, moe_stream_t stream) {
    Shape s;
    MOE_TRY(make_shape(cfg, &s));
    if (!counts || !bias || !isfinite(rate)) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_bias_update(s, counts, bias, rate, (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_layer_fwd(const moe_config* cfg, const void* x, const void* Wg,
                                 const void* Wnoise, const float* noise,
                                 const float* logit_offset, const float* sel_bias,
                                 const void* W1, const void* W2, const void* W1s,
                                 const void* W2s, void* y, int32_t* topk_ids, float* topk_w,
                                 int32_t* counts, float* aux_vecs, float* out3, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    cudaStream_t st = (cudaStream_t)stream;
    if (!x || !Wg || !W1 || !W2 || !y) return MOE_ERR_INVALID_ARG;
    if (!noise_args_ok(s, Wnoise, noise)) return MOE_ERR_INVALID_ARG;
    if (s.S > 0 && (!W1s || !W2s)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg) || (Wnoise && !aligned16(Wnoise)) || !aligned16(W1) ||
        !aligned16(W2) || !aligned16(y) || (s.S > 0 && (!aligned16(W1s) || !aligned16(W2s))))
        return MOE_ERR_UNSUPPORTED;
    float* logits = at<float>(ws, L.logits);
    float* probs = at<float>(ws, L.probs);
    int32_t* ids = topk_ids ? topk_ids : at<int32_t>(ws, L.ids);
    float* w = topk_w ? topk_w : at<float>(ws, L.w);
    int32_t* cnt = counts ? counts : at<int32_t>(ws, L.counts);
    int32_t* kept = at<int32_t>(ws, L.kept);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* slot = at<int32_t>(ws, L.slot);
    int32_t* row_token = at<int32_t>(ws, L.row_token);
    void* xp = at<void>(ws, L.xp);
    void* yp = at<void>(ws, L.yp);
    void* ys = at<void>(ws, L.ys);
    float* av = aux_vecs ? aux_vecs : at<float>(ws, L.aux_vecs);
    float* o3 = out3 ? out3 : at<float>(ws, L.out3);
    if (s.routing == MOE_EXPERT_CHOICE) {
        if (topk_ids || topk_w || counts || aux_vecs || out3) return MOE_ERR_INVALID_ARG;
        int32_t* tok_row = at<int32_t>(ws, L.tok_row);
        float* row_w = at<float>(ws, L.row_w);
        MOE_TRY(route_impl(s, L, ws, x, Wg, Wnoise, noise, logit_offset, sel_bias, logits, probs,
                           nullptr, nullptr, nullptr, nullptr, nullptr, st));
        MOE_TRY(ec_dispatch_impl(s, L, ws, x, probs, offsets, row_token, row_w, tok_row, xp, st));
        // the gather signals its dependents after its wait: the offsets the
        // selection wrote are final when the up projection launches
        MOE_TRY(ffn_impl(s, L, ws, xp, offsets, W1, W2, x, W1s, W2s, yp, ys, nullptr, nullptr,
                         nullptr, nullptr, nullptr, true, nullptr, st));
        MOE_CUDA(launch_expert_choice_combine(s, yp, tok_row, probs, s.S ? ys : nullptr, y, st));
        return MOE_OK;
    }
    // route + capacity histogram + statistics, then scan/slots, permute,
    // expert GEMMs, combine
    MOE_TRY(route_impl(s, L, ws, x, Wg, Wnoise, noise, logit_offset, sel_bias, logits, probs,
                       nullptr, ids, w, av, o3, st));
    // top-1 without shared experts: each token has at most one expert row, so the
    // down GEMM writes y itself (dropped tokens are zeroed by the permute kernel).
    // Not with re-route candidates (a token's gate depends on which candidate
    // is kept) or padding (padding rows belong to no token).
    const bool scatter = s.k == 1 && s.nc == 1 && !s.pad && s.S == 0 && s.dtype == MOE_BF16;
    // otherwise (bf16, packed rows) the down GEMM can also combine, on request:
    // each token's rows are summed in the fixed combine order once the last
    // one is stored. It re-reads every row it adds, like the combine kernel,
    // and on the workloads measured it was no faster (the Mixtral-shaped layer
    // within noise, the DeepSeek-shaped one slower), so the automatic choice
    // is the separate kernel.
    const bool fold = !scatter && !s.pad && s.dtype == MOE_BF16 &&
                      s.combine_mode == MOE_COMBINE_IN_GEMM;
    const Fold fold_args{row_token, slot, w, y};
    MOE_TRY(dispatch_impl(s, L, ws, x, ids, cnt, kept, offsets, slot, xp, row_token,
                          !uses_policy(s), (scatter || (fold && s.S == 0)) ? y : nullptr,
                          fold ? at<int32_t>(ws, L.tok_need) : nullptr, st));
    // the permute signals its dependents after its wait: the offsets the
    // capacity kernel wrote are final when the up projection launches
    MOE_TRY(ffn_impl(s, L, ws, xp, offsets, W1, W2, x, W1s, W2s, yp, ys,
                     scatter ? row_token : nullptr, scatter ? w : nullptr,
                     scatter ? y : nullptr, s.dtype == MOE_BF16 ? av : nullptr,
                     s.dtype == MOE_BF16 ? o3 : nullptr, true, fold ? &fold_args : nullptr, st));
    if (!scatter && !fold)
        MOE_CUDA(launch_combine(s, yp, slot, w, s.S ? ys : nullptr, y, at<int>(ws, L.status), st));
    return MOE_OK;
}

MOE_API moe_status moe_expert_choice_dispatch(const moe_config* cfg, const void* x,
                                              const float* probs, int32_t* offsets,
                                              int32_t* row_token, float* row_w,
                                              int32_t* tok_row, void* xp, void* ws,
                                              size_t ws_bytes, moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (s.routing != MOE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (!x || !probs || !offsets || !row_token || !row_w || !tok_row || !xp)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_UNSUPPORTED;
    return ec_dispatch_impl(s, L, ws, x, probs, offsets, row_token, row_w, tok_row, xp,
                            (cudaStream_t)stream);
}

MOE_API moe_status moe_expert_choice_combine(const moe_config* cfg, const void* yp,
                                             const int32_t* tok_row, const float* probs,
                                             const void* ys, void* y, void* ws, size_t ws_bytes,
                                             moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (s.routing != MOE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (!yp || !tok_row || !probs || !y) return MOE_ERR_INVALID_ARG;
    if (s.S > 0 && !ys) return MOE_ERR_INVALID_ARG;
    if (!aligned16(yp) || !aligned16(y) || (ys && !aligned16(ys))) return MOE_ERR_UNSUPPORTED;
    MOE_CUDA(launch_expert_choice_combine(s, yp, tok_row, probs, s.S ? ys : nullptr, y,
                                          (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_draw_noise(const moe_config* cfg, float* noise, moe_stream_t stream) {
    Shape s;
    MOE_TRY(make_shape(cfg, &s));
    if (!noise) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_draw_noise(s, noise, (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_seq_aux_stats(const moe_config* cfg, const float* probs,
                                     const int32_t* topk_ids, const int32_t* seq_offsets,
                                     int32_t n_seq, float* f_seq, float* P_seq, float* aux_seq,
                                     float* aux_mean, void* ws, size_t ws_bytes,
                                     moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    if (!probs || !topk_ids || !seq_offsets || !aux_seq || !aux_mean || n_seq < 1)
        return MOE_ERR_INVALID_ARG;
    if (n_seq > s.T + 1) return MOE_ERR_UNSUPPORTED;  // the workspace holds T + 1 sequences
    MOE_CUDA(launch_seq_aux(s, probs, topk_ids, seq_offsets, n_seq, f_seq, P_seq, aux_seq,
                            aux_mean, at<void>(ws, L.seq_acc), at<unsigned int>(ws, L.seq_ticket),
                            at<int>(ws, L.status), (cudaStream_t)stream));
    return MOE_OK;
}

MOE_API moe_status moe_set_wait_limits(uint64_t wait_ns, int32_t policy_passes,
                                       int32_t hold_first_accumulator) {
    if (policy_passes < 0 || (hold_first_accumulator != 0 && hold_first_accumulator != 1))
        return MOE_ERR_INVALID_ARG;
    g_wait_ns.store(wait_ns ? (unsigned long long)wait_ns : kDefaultWaitNs);
    g_policy_passes.store(policy_passes ? policy_passes : kDefaultPolicyPasses);
    g_hold_first_acc.store(hold_first_accumulator);
    return MOE_OK;
}

MOE_API moe_status moe_read_device_error(const moe_config* cfg, void* ws, size_t ws_bytes,
                                         moe_stream_t stream) {
    Shape s;
    WsLayout L;
    MOE_TRY(make_shape(cfg, &s));
    MOE_TRY(check_ws(s, ws, ws_bytes, &L));
    cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    MOE_CUDA(cudaMemcpyAsync(&word, at<int>(ws, L.status), sizeof(int), cudaMemcpyDeviceToHost, st));
    MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.status), 0, sizeof(int), st));
    MOE_CUDA(cudaStreamSynchronize(st));
    if (word & DEV_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (word & DEV_BAD_ARG) return MOE_ERR_DEVICE_ARG;
    if (word & DEV_NONFINITE) return MOE_ERR_NONFINITE;
    return MOE_OK;
}

}  // extern "C"

// ------------------------------------------------ statistics without a workspace
// moe_aux_stats_noalloc keeps its accumulators in this file-scope device array
// instead of a caller-provided workspace. Every GPU that loads the library
// holds one copy until the process exits. It fits up to
// MOE_AUX_NOALLOC_MAX_EXPERTS experts: two u64 sums and one u32 count per
// expert, plus the ticket counter of the statistics kernel.
#define MOE_AUX_NOALLOC_MAX_EXPERTS 512
static __device__ __align__(256) unsigned char g_aux_noalloc_scratch[MOE_AUX_NOALLOC_MAX_EXPERTS * 20 + 16];

namespace {

// Host code may not hand g_aux_noalloc_scratch itself to a kernel: on the host
// that name is a stand-in, not a device address. Its device address is
// looked up once per device, with that device current, and cached together
// with the CUDA context it belongs to. A call from another context on that
// device (the primary context was destroyed by cudaDeviceReset and made
// again, which loads the library's device code again) looks the address up
// afresh.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
CUcontext g_noalloc_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

CUcontext current_context() {
    CUcontext ctx = nullptr;
    CtxGetCurrentFn fn = ctx_get_current_fn();
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

moe_status noalloc_scratch_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const CUcontext ctx = current_context();
    if (!g_noalloc_ptr[dev] || !ctx || ctx != g_noalloc_ctx[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_aux_noalloc_scratch) != cudaSuccess || !ptr)
            return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
        // the lookup makes the device's primary context current if no context was
        g_noalloc_ctx[dev] = current_context();
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status moe_aux_stats_noalloc(const moe_config* cfg, const float* probs,
                                                    const int32_t* topk_ids,
                                                    const float* topk_w, float* f, float* P,
                                                    float* importance, float* out3,
                                                    moe_stream_t stream) {
    Shape s;
    MOE_TRY(make_shape(cfg, &s));
    if (!probs || !topk_ids || !topk_w || !out3) return MOE_ERR_INVALID_ARG;
    if (s.E > MOE_AUX_NOALLOC_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    MOE_TRY(noalloc_scratch_current_device(&scratch));
    cudaStream_t st = (cudaStream_t)stream;
    // the array keeps whatever the previous call left: start this call from zero
    MOE_CUDA(cudaMemsetAsync(scratch, 0, (size_t)s.E * 20 + 16, st));
    MOE_CUDA(launch_aux(s, probs, topk_ids, topk_w, scratch, 1, f, P, importance, out3, st));
    return MOE_OK;
}
