// The C ABI declared in include/moetree.h: argument checks, workspace layout and
// the launch sequence of the layer (router -> selection -> permute -> grouped
// SwiGLU experts -> combine), plus the host-side expert-residency table and the
// host-to-device expert upload used when experts are offloaded.
#include <algorithm>
#include <chrono>
#include <new>
#include <thread>
#include <vector>

#include "common.cuh"

namespace moe {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Workspace workspace_layout(const moe_layer_desc &L, int B, int N) {
    const size_t R = (size_t)B * N, A = R * L.k, E = L.E;
    Workspace w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    w.flags = take(64 * sizeof(int));
    w.logits = take(R * E * 4);
    w.idx = take(A * 4);
    w.gates = take(A * 4);
    w.elig = take((size_t)B * E);
    w.info = take((size_t)B * MOE_INFO_FIELDS * 4);
    w.counts = take(E * 4);
    w.offsets = take((E + 1) * 4);
    w.perm = take(A * 4);
    w.pos = take(A * 4);
    w.rbmask = take((size_t)2 * E * ((R + 31) / 32) * 4);
    w.active = take((E + 1) * 4);
    w.slotmap = take(E * 4);
    w.resident = take(E);
    w.pass = take(E);
    w.rowtiles = take((size_t)(kRowTileHeader + 4 * max_rowtiles(L.E, (int)A)) * 4);
    w.sched = take((size_t)(1 + max_rowtiles(L.E, (int)A)) * 4);
    w.xp = take(A * L.d * elem_size(L.dtype));
    w.h = take(A * L.f * 4);
    w.o = take(A * L.d * 4);
    w.xn = take(R * L.d * elem_size(L.dtype));
    w.total = off;
    return w;
}

bool desc_ok(const moe_layer_desc *L) {
    return L && L->k >= 1 && L->k <= kMaxK && L->E >= L->k && L->E <= kMaxE && L->d >= 8 &&
           L->d % 8 == 0 && L->d <= kMaxD && L->f >= 8 && L->f % 8 == 0 && L->f <= kMaxD &&
           (L->dtype == MOE_DTYPE_F32 || L->dtype == MOE_DTYPE_BF16) && L->slots >= 0 &&
           L->slots <= 65535;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }


bool select_args(const moe_select_params *P, int k, SelectArgs *a) {
    if (!P) return false;
    if (P->mode < MOE_ROUTE_NATURAL || P->mode > MOE_ROUTE_FIXED_B) return false;
    if (P->mode != MOE_ROUTE_NATURAL && (P->n_c < 1 || P->n_c > MOE_MAX_DEPTHS)) return false;
    if (P->prune && (P->reroute_budget < 0 || P->min_set < 0)) return false;
    if (P->mode == MOE_ROUTE_FIXED_B && P->fixed_B < 1) return false;
    a->mode = P->mode;
    a->n_c = P->mode == MOE_ROUTE_NATURAL ? 1 : P->n_c;
    a->pool_all = P->pool_all ? 1 : 0;
    a->anchor = P->anchor ? 1 : 0;
    a->prune = P->prune ? 1 : 0;
    a->budget = P->reroute_budget;
    a->min_set = P->min_set;
    a->fixed_B = P->fixed_B;
    a->cmax = 0.f;
    for (int t = 0; t < MOE_MAX_DEPTHS; ++t) {
        a->c64[t] = (P->mode != MOE_ROUTE_NATURAL && t < P->n_c) ? P->c_by_depth[t] : 0.0;
        a->c[t] = (float)a->c64[t];
        a->cmax = std::max(a->cmax, a->c[t]);
    }
    (void)k;
    return true;
}


moe_status run_permute(const moe_layer_desc &L, const int *idx, int R, void *ws,
                       const Workspace &w, int *counts, int *offsets, int *perm,
                       bool after_router, cudaStream_t s) {
    return cuda_status(launch_permute(L, idx, R, counts, offsets, perm, at<int>(ws, w.pos),
                                      at<int>(ws, w.active), at<int>(ws, w.rowtiles),
                                      at<int>(ws, w.flags), at<uint32_t>(ws, w.rbmask),
                                      after_router, s));
}

moe_status run_ffn(const moe_layer_desc &L, const void *x, const void *Wg, const void *Wu,
                   const void *Wd, const int *slot, const uint8_t *pass, int R, void *ws,
                   const Workspace &w, const int *counts, const int *offsets, const int *perm,
                   const moe_run_opts *opts, cudaStream_t s) {
    FfnArgs fa{};
    fa.x = x;
    fa.Wg = Wg;
    fa.Wu = Wu;
    fa.Wd = Wd;
    fa.slot = slot;
    fa.pass = pass;
    fa.counts = counts;
    fa.offsets = offsets;
    fa.perm = perm;
    fa.pos = at<int>(ws, w.pos);
    fa.active = at<int>(ws, w.active);
    fa.rowtiles = at<int>(ws, w.rowtiles);
    fa.R = R;
    fa.d = L.d;
    fa.f = L.f;
    fa.E = L.E;
    fa.k = L.k;
    fa.dtype = L.dtype;
    fa.slots = L.slots > 0 ? L.slots : L.E;
    fa.flags = at<int>(ws, w.flags);
    fa.sched = at<int>(ws, w.sched);
    fa.xp = at<void>(ws, w.xp);
    fa.h = at<void>(ws, w.h);
    fa.o = at<void>(ws, w.o);
    fa.max_ctas = opts ? opts->ffn_max_ctas : 0;

    const int path = resolve_ffn_path(L, opts);
    if (path < 0) return MOE_ERR_UNSUPPORTED;
    const bool timed = opts && opts->ffn_begin && opts->ffn_end;
    if (timed && cudaEventRecord((cudaEvent_t)opts->ffn_begin, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const cudaError_t err = path == MOE_FFN_TCGEN05 ? launch_ffn_tc(fa, s) : launch_ffn_simt(fa, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    if (timed && cudaEventRecord((cudaEvent_t)opts->ffn_end, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int resolve_ffn_path(const moe_layer_desc &L, const moe_run_opts *opts) {
    int path = opts ? opts->ffn_path : MOE_FFN_AUTO;
    if (path == MOE_FFN_AUTO) path = ffn_tc_supported(L) ? MOE_FFN_TCGEN05 : MOE_FFN_SIMT;
    if (path == MOE_FFN_TCGEN05 && !ffn_tc_supported(L)) return -1;
    return path;
}

moe_status run_combine(const moe_layer_desc &L, const void *residual, const float *gates, int R,
                       void *y, void *ws, const Workspace &w, cudaStream_t s) {
    return cuda_status(launch_combine(L, at<void>(ws, w.o), at<int>(ws, w.pos), gates, residual,
                                      R, y, s));
}

// permute (unless the selection did it) -> experts -> combine, shared by
// moe_expert_forward and moe_tree_forward. The experts read x; the combine adds `residual`
// (may be null).
static moe_status run_experts(const moe_layer_desc &L, const void *x, const void *Wg,
                              const void *Wu, const void *Wd, const int *slot, const int *idx,
                              const float *gates, int R, void *y, void *ws, const Workspace &w,
                              int *counts, int *offsets, int *perm, const moe_run_opts *opts,
                              bool after_router, bool permuted, const void *residual,
                              cudaStream_t s) {
    moe_status st = MOE_OK;
    if (!permuted) st = run_permute(L, idx, R, ws, w, counts, offsets, perm, after_router, s);
    if (st != MOE_OK) return st;
    st = run_ffn(L, x, Wg, Wu, Wd, slot, nullptr, R, ws, w, counts, offsets, perm, opts, s);
    if (st != MOE_OK) return st;
    return run_combine(L, residual, gates, R, y, ws, w, s);
}

// The input the router and experts read: x, or its pre-norm written into the workspace.
const void *layer_input(const moe_layer_desc &L, const void *x, int R, void *ws,
                        const Workspace &w, const moe_run_opts *opts, cudaStream_t s,
                        moe_status *st) {
    *st = MOE_OK;
    if (!opts || !opts->norm_input) return x;
    void *xn = at<void>(ws, w.xn);
    if (launch_rmsnorm(L, x, R, xn, s) != cudaSuccess) *st = MOE_ERR_CUDA;
    return xn;
}

}  // namespace moe

using namespace moe;

// Every argument check of moe_tree_forward except the workspace's.
moe_status moe::tree_forward_check(const moe_layer_desc *L, const moe_select_params *P,
                                   const void *x, const void *W_r, const void *W_gate,
                                   const void *W_up, const void *W_down, const int *depth,
                                   int B, int N, const uint8_t *resident, const void *y) {
    SelectArgs a;
    if (!desc_ok(L) || !select_args(P, L->k, &a) || B < 1 || N < 1) return MOE_ERR_ARG;
    if (!x || !W_r || !W_gate || !W_up || !W_down || !depth || !y) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(W_r) || !aligned16(W_gate) || !aligned16(W_up) ||
        !aligned16(W_down) || !aligned16(y))
        return MOE_ERR_ARG;
    if (a.prune && !resident) return MOE_ERR_ARG;
    if ((long long)B * N > (1 << 30)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

struct moe_residency {
    int n_layers = 0, E = 0, slots = 0;
    std::vector<int> slot_of;     // [layer][E], -1 = not resident
    std::vector<int> expert_in;   // [layer][slots], -1 = free
    std::vector<long long> used;  // [layer][slots], last-use tick
    long long tick = 0;
    // Timing events of the offloaded layer, per layer: pairs recorded on the compute
    // stream just before and just after each wait for an upload, and how many pairs the
    // last call on that layer used (created on first use, reused by later calls).
    std::vector<std::vector<cudaEvent_t>> wait_ev;
    std::vector<int> n_wait;
    ~moe_residency() {
        for (auto &v : wait_ev)
            for (cudaEvent_t e : v)
                if (e) cudaEventDestroy(e);
    }
};

// Event `which` (0: before the wait, 1: after it) of the i-th upload wait of `layer`.
cudaEvent_t moe::residency_wait_event(moe_residency *t, int layer, int i, int which) {
    auto &v = t->wait_ev[layer];
    while ((int)v.size() < 2 * (i + 1)) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        v.push_back(e);
    }
    return v[2 * i + which];
}

void moe::residency_set_waits(moe_residency *t, int layer, int n) { t->n_wait[layer] = n; }

extern "C" {

const char *moe_status_str(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_ARG: return "invalid argument";
        case MOE_ERR_CUDA: return "CUDA call failed";
        case MOE_ERR_NOSLOT: return "more experts needed at once than the layer has slots";
        case MOE_ERR_TIMEOUT: return "bounded wait timed out";
        case MOE_ERR_DEVICE_CHECK: return "kernel-side check failed";
        case MOE_ERR_UNSUPPORTED: return "shape or dtype not supported by this kernel";
        default: return "unknown status";
    }
}

int moe_abi_version(void) { return 202; }

size_t moe_workspace_bytes(const moe_layer_desc *L, int B, int N) {
    if (!desc_ok(L) || B < 1 || N < 1) return 0;
    return workspace_layout(*L, B, N).total;
}

moe_status moe_router_logits(const moe_layer_desc *L, const void *x, const void *W_r, int R,
                             float *logits, moe_stream_t stream) {
    if (!desc_ok(L) || R < 0 || (R > 0 && (!x || !W_r || !logits))) return MOE_ERR_ARG;
    if (R > 0 && (!aligned16(x) || !aligned16(W_r))) return MOE_ERR_ARG;
    return cuda_status(launch_router(*L, x, W_r, R, logits, nullptr, (cudaStream_t)stream));
}

moe_status moe_rms_norm(const moe_layer_desc *L, const void *x, int R, void *xn,
                        moe_stream_t stream) {
    if (!desc_ok(L) || R < 0 || (R > 0 && (!x || !xn))) return MOE_ERR_ARG;
    if (R > 0 && (!aligned16(x) || !aligned16(xn))) return MOE_ERR_ARG;
    return cuda_status(launch_rmsnorm(*L, x, R, xn, (cudaStream_t)stream));
}

moe_status moe_tree_select(const moe_layer_desc *L, const moe_select_params *P,
                           const float *logits, const int *depth, int B, int N,
                           const uint8_t *resident, int *topk_idx, float *gates,
                           uint8_t *eligible, int *info, moe_stream_t stream) {
    SelectArgs a;
    if (!desc_ok(L) || !select_args(P, L->k, &a) || B < 0 || N < 0) return MOE_ERR_ARG;
    if (B * N > 0 && (!logits || !depth || !topk_idx || !gates)) return MOE_ERR_ARG;
    if (a.prune && !resident) return MOE_ERR_ARG;
    return cuda_status(launch_select(*L, a, logits, depth, B, N, resident, topk_idx, gates,
                                     eligible, info, WeightPrefetch{}, PermuteOut{}, nullptr,
                                     (cudaStream_t)stream));
}

moe_status moe_tree_route(const moe_layer_desc *L, const moe_select_params *P, const void *x,
                          const void *W_r, const int *depth, int B, int N,
                          const uint8_t *resident, float *logits, int *topk_idx, float *gates,
                          uint8_t *eligible, int *info, moe_stream_t stream) {
    SelectArgs a;
    if (!desc_ok(L) || !select_args(P, L->k, &a) || B < 0 || N < 0) return MOE_ERR_ARG;
    if (B * N > 0 && (!x || !W_r || !logits || !depth || !topk_idx || !gates))
        return MOE_ERR_ARG;
    if (B * N > 0 && (!aligned16(x) || !aligned16(W_r))) return MOE_ERR_ARG;
    if (a.prune && !resident) return MOE_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_router(*L, x, W_r, B * N, logits, nullptr, s) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_select(*L, a, logits, depth, B, N, resident, topk_idx, gates,
                                     eligible, info, WeightPrefetch{}, PermuteOut{}, nullptr, s));
}

moe_status moe_tree_block_stats(const moe_layer_desc *L, int B, int N, const int *info,
                                const int *counts, const void *workspace, moe_tree_stats *stats,
                                moe_stream_t stream) {
    if (!desc_ok(L) || B < 1 || N < 1 || !stats) return MOE_ERR_ARG;
    if ((!info || !counts) && !workspace) return MOE_ERR_ARG;
    const Workspace w = workspace_layout(*L, B, N);
    void *ws = const_cast<void *>(workspace);
    const int *inf = info ? info : at<int>(ws, w.info);
    const int *cnt = counts ? counts : at<int>(ws, w.counts);
    cudaStream_t s = (cudaStream_t)stream;
    int c[kMaxE];
    if (cudaMemcpyAsync(c, cnt, sizeof(int) * L->E, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    double sums[4] = {0, 0, 0, 0};
    int exact = 0;
    constexpr int kChunk = 128;  // trees per copy: the host buffer stays on the stack
    int buf[kChunk * MOE_INFO_FIELDS];
    for (int b0 = 0; b0 < B; b0 += kChunk) {
        const int nb = std::min(kChunk, B - b0);
        if (cudaMemcpyAsync(buf, inf + (size_t)b0 * MOE_INFO_FIELDS,
                            sizeof(int) * nb * MOE_INFO_FIELDS, cudaMemcpyDeviceToHost,
                            s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return MOE_ERR_CUDA;
        for (int b = 0; b < nb; ++b) {
            for (int f = 0; f < 4; ++f) sums[f] += buf[b * MOE_INFO_FIELDS + f];
            exact += buf[b * MOE_INFO_FIELDS + 4] != 0;
        }
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    moe_tree_stats st{};
    st.trees = B;
    for (int e = 0; e < L->E; ++e) {
        st.assignments += c[e];
        st.union_experts += c[e] > 0;
        st.max_per_expert = std::max(st.max_per_expert, c[e]);
    }
    st.reuse = st.assignments > 0 ? 1.0 - (double)st.union_experts / st.assignments : 0.0;
    st.union_nat_mean = sums[0] / B;
    st.union_sel_mean = sums[1] / B;
    st.m_mean = sums[2] / B;
    st.pruned_mean = sums[3] / B;
    st.exact_trees = exact;
    *stats = st;
    return MOE_OK;
}

moe_status moe_expert_permute(const moe_layer_desc *L, const int *topk_idx, int R, int *counts,
                              int *offsets, int *perm, void *workspace, moe_stream_t stream) {
    if (!desc_ok(L) || R < 1 || !topk_idx || !counts || !offsets || !perm || !workspace)
        return MOE_ERR_ARG;
    const Workspace w = workspace_layout(*L, 1, R);
    return cuda_status(launch_permute(*L, topk_idx, R, counts, offsets, perm,
                                      at<int>(workspace, w.pos), at<int>(workspace, w.active),
                                      at<int>(workspace, w.rowtiles),
                                      at<int>(workspace, w.flags),
                                      at<uint32_t>(workspace, w.rbmask), false,
                                      (cudaStream_t)stream));
}

moe_status moe_expert_forward(const moe_layer_desc *L, const void *x, const void *W_gate,
                              const void *W_up, const void *W_down, const int *slot_of_expert,
                              const int *topk_idx, const float *gates, int R, void *y,
                              void *workspace, const moe_run_opts *opts, moe_stream_t stream) {
    if (!desc_ok(L) || R < 1 || !x || !W_gate || !W_up || !W_down || !topk_idx || !gates ||
        !y || !workspace)
        return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) ||
        !aligned16(y) || ((uintptr_t)workspace & 255u))
        return MOE_ERR_ARG;
    const Workspace w = workspace_layout(*L, 1, R);
    cudaStream_t s = (cudaStream_t)stream;
    moe_status st;
    const void *xin = layer_input(*L, x, R, workspace, w, opts, s, &st);
    if (st != MOE_OK) return st;
    return run_experts(*L, xin, W_gate, W_up, W_down, slot_of_expert, topk_idx, gates, R, y,
                       workspace, w, at<int>(workspace, w.counts), at<int>(workspace, w.offsets),
                       at<int>(workspace, w.perm), opts, false, false,
                       (opts && opts->residual) ? x : nullptr, s);
}

moe_status moe_tree_forward(const moe_layer_desc *L, const moe_select_params *P, const void *x,
                            const void *W_r, const void *W_gate, const void *W_up,
                            const void *W_down, const int *slot_of_expert, const int *depth,
                            int B, int N, const uint8_t *resident, void *y,
                            const moe_tree_outputs *out, void *workspace,
                            const moe_run_opts *opts, moe_stream_t stream) {
    const moe_status st =
        tree_forward_check(L, P, x, W_r, W_gate, W_up, W_down, depth, B, N, resident, y);
    if (st != MOE_OK) return st;
    if (!workspace || ((uintptr_t)workspace & 255u)) return MOE_ERR_ARG;
    SelectArgs a;
    select_args(P, L->k, &a);
    const int R = B * N;
    cudaStream_t s = (cudaStream_t)stream;
    const Workspace w = workspace_layout(*L, B, N);
    moe_tree_outputs o{};
    if (out) o = *out;
    float *logits = o.logits ? o.logits : at<float>(workspace, w.logits);
    int *idx = o.topk_idx ? o.topk_idx : at<int>(workspace, w.idx);
    float *gates = o.gates ? o.gates : at<float>(workspace, w.gates);
    uint8_t *elig = o.eligible ? o.eligible : at<uint8_t>(workspace, w.elig);
    int *info = o.info ? o.info : at<int>(workspace, w.info);
    int *counts = o.counts ? o.counts : at<int>(workspace, w.counts);
    int *offsets = o.offsets ? o.offsets : at<int>(workspace, w.offsets);
    int *perm = o.perm ? o.perm : at<int>(workspace, w.perm);

    moe_status sn;
    const void *xin = layer_input(*L, x, R, workspace, w, opts, s, &sn);
    if (sn != MOE_OK) return sn;
    if (launch_router(*L, xin, W_r, R, logits, at<int>(workspace, w.flags) + kRouterCheckWord,
                      s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const WeightPrefetch pf = weight_prefetch(*L, B, W_gate, W_up, W_down, slot_of_expert);
    const PermuteOut po{counts, offsets, perm, at<int>(workspace, w.pos),
                        at<int>(workspace, w.active), at<int>(workspace, w.rowtiles),
                        at<int>(workspace, w.flags), 1};
    bool permuted = false;
    if (opts && opts->select_begin &&
        cudaEventRecord((cudaEvent_t)opts->select_begin, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_select(*L, a, logits, depth, B, N, resident, idx, gates, elig, info, pf, po,
                      &permuted, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return run_experts(*L, xin, W_gate, W_up, W_down, slot_of_expert, idx, gates, R, y,
                       workspace, w, counts, offsets, perm, opts, true, permuted,
                       (opts && opts->residual) ? x : nullptr, s);
}

moe_status moe_workspace_check(void *workspace, int *flags, moe_stream_t stream) {
    if (!workspace || !flags) return MOE_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    *flags = v;
    return v ? MOE_ERR_DEVICE_CHECK : MOE_OK;
}

// ------------------------------------------------------------------- offload

moe_status moe_residency_create(int n_layers, int E, int slots, moe_residency **table) {
    if (!table || n_layers < 1 || E < 1 || E > kMaxE || slots < 1 || slots > E) return MOE_ERR_ARG;
    moe_residency *t = new (std::nothrow) moe_residency();
    if (!t) return MOE_ERR_ARG;
    t->n_layers = n_layers;
    t->E = E;
    t->slots = slots;
    t->slot_of.assign((size_t)n_layers * E, -1);
    t->expert_in.assign((size_t)n_layers * slots, -1);
    t->used.assign((size_t)n_layers * slots, 0);
    t->wait_ev.resize(n_layers);
    t->n_wait.assign(n_layers, 0);
    *table = t;
    return MOE_OK;
}

moe_status moe_residency_destroy(moe_residency *table) {
    delete table;
    return MOE_OK;
}

moe_status moe_residency_query(const moe_residency *t, int layer, int *slot_of_expert,
                               uint8_t *resident) {
    if (!t || layer < 0 || layer >= t->n_layers) return MOE_ERR_ARG;
    for (int e = 0; e < t->E; ++e) {
        const int s = t->slot_of[(size_t)layer * t->E + e];
        if (slot_of_expert) slot_of_expert[e] = s;
        if (resident) resident[e] = s >= 0;
    }
    return MOE_OK;
}

moe_status moe_residency_plan(moe_residency *t, int layer, const int *needed, int n_needed,
                              int *up_expert, int *up_slot, int *n_up, int *hits) {
    if (!t || layer < 0 || layer >= t->n_layers || n_needed < 0 || (n_needed && !needed) ||
        !n_up || (n_needed && (!up_expert || !up_slot)))
        return MOE_ERR_ARG;
    if (n_needed > t->slots) return MOE_ERR_NOSLOT;
    std::vector<char> need(t->E, 0);
    for (int i = 0; i < n_needed; ++i) {
        const int e = needed[i];
        if (e < 0 || e >= t->E || need[e]) return MOE_ERR_ARG;
        need[e] = 1;
    }
    int *slot_of = &t->slot_of[(size_t)layer * t->E];
    int *expert_in = &t->expert_in[(size_t)layer * t->slots];
    long long *used = &t->used[(size_t)layer * t->slots];
    int h = 0, nu = 0;
    for (int i = 0; i < n_needed; ++i) {
        const int s = slot_of[needed[i]];
        if (s >= 0) {
            used[s] = ++t->tick;
            ++h;
        }
    }
    for (int i = 0; i < n_needed; ++i) {
        const int e = needed[i];
        if (slot_of[e] >= 0) continue;
        int victim = -1;
        for (int s = 0; s < t->slots && victim < 0; ++s)
            if (expert_in[s] < 0) victim = s;
        if (victim < 0)
            for (int s = 0; s < t->slots; ++s) {
                if (need[expert_in[s]]) continue;
                if (victim < 0 || used[s] < used[victim]) victim = s;
            }
        if (victim < 0) return MOE_ERR_NOSLOT;  // unreachable: n_needed <= slots
        if (expert_in[victim] >= 0) slot_of[expert_in[victim]] = -1;
        expert_in[victim] = e;
        slot_of[e] = victim;
        used[victim] = ++t->tick;
        up_expert[nu] = e;
        up_slot[nu] = victim;
        ++nu;
    }
    *n_up = nu;
    if (hits) *hits = h;
    return MOE_OK;
}

moe_status moe_residency_publish(const moe_residency *t, int layer, int *slot_of_expert,
                                 uint8_t *resident, moe_stream_t stream) {
    if (!t || layer < 0 || layer >= t->n_layers) return MOE_ERR_ARG;
    if (!slot_of_expert && !resident) return MOE_OK;
    std::vector<uint8_t> res(t->E);
    const int *so = &t->slot_of[(size_t)layer * t->E];
    for (int e = 0; e < t->E; ++e) res[e] = so[e] >= 0;
    return cuda_status(launch_publish(t->E, so, res.data(), slot_of_expert, resident,
                                      (cudaStream_t)stream));
}

moe_status moe_expert_upload(const moe_layer_desc *L, const void *host_gate, const void *host_up,
                             const void *host_down, void *slot_gate, void *slot_up,
                             void *slot_down, const int *up_expert, const int *up_slot, int n,
                             moe_stream_t side, moe_event_t done) {
    if (!desc_ok(L) || n < 0 || (n && (!up_expert || !up_slot)) || !host_gate || !host_up ||
        !host_down || !slot_gate || !slot_up || !slot_down)
        return MOE_ERR_ARG;
    const size_t bytes = (size_t)L->d * L->f * elem_size(L->dtype);
    cudaStream_t s = (cudaStream_t)side;
    for (int i = 0; i < n; ++i) {
        if (up_expert[i] < 0 || up_expert[i] >= L->E || up_slot[i] < 0) return MOE_ERR_ARG;
        const size_t src = (size_t)up_expert[i] * bytes, dst = (size_t)up_slot[i] * bytes;
        const void *hs[3] = {host_gate, host_up, host_down};
        void *ds[3] = {slot_gate, slot_up, slot_down};
        for (int m = 0; m < 3; ++m)
            if (cudaMemcpyAsync((char *)ds[m] + dst, (const char *)hs[m] + src, bytes,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
                return MOE_ERR_CUDA;
    }
    if (done && cudaEventRecord((cudaEvent_t)done, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_offload_upload_wait(moe_residency *t, int layer, double timeout_s,
                                   double *wait_ms, int *waits) {
    if (!t || layer < 0 || layer >= t->n_layers || !wait_ms || timeout_s < 0)
        return MOE_ERR_ARG;
    double sum = 0.0;
    const int n = t->n_wait[layer];
    for (int i = 0; i < n; ++i) {
        cudaEvent_t a = t->wait_ev[layer][2 * i], b = t->wait_ev[layer][2 * i + 1];
        const moe_status st = moe_event_wait((moe_event_t)b, timeout_s);
        if (st != MOE_OK) return st;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return MOE_ERR_CUDA;
        sum += ms;
    }
    *wait_ms = sum;
    if (waits) *waits = n;
    return MOE_OK;
}

moe_status moe_event_wait(moe_event_t ev, double timeout_s) {
    if (!ev || timeout_s < 0) return MOE_ERR_ARG;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery((cudaEvent_t)ev);
        if (e == cudaSuccess) return MOE_OK;
        if (e != cudaErrorNotReady) return MOE_ERR_CUDA;
        const double el =
            std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        if (el >= timeout_s) return MOE_ERR_TIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

}  // extern "C"
