// moe_offload_forward: the layer with its experts offloaded to host memory ("AcceptMoE"
// news article, section 03: expert slots per layer on the GPU, the other experts in CPU
// memory, uploaded on demand; section 02: residency-aware pruning decides eligibility
// from what is resident now instead of predicting and prefetching).
//
// Per call (one verification block, one layer):
//   1. publish the layer's residency (slot map, resident mask) as it stands before any
//      upload, then router + selection (pruning sees that mask) + permute on `stream`;
//   2. one host wait for the per-expert counts: the needed set is every expert with an
//      assignment;
//   3. the resident needed experts are computed at once (first expert pass) while the
//      missing ones are copied host -> device on `side` (one cudaMemcpyAsync per
//      matrix); each later pass waits for its uploads with an event. When the missing
//      experts do not fit next to the experts of the pass before, they go in chunks,
//      and a chunk that must evict the previous pass's experts waits for that pass;
//   4. the gated combine once all passes are enqueued.
// Slots are replaced least-recently-used (moe_residency_plan). An upload never evicts
// an expert that an enqueued pass may still be reading: the host wait in step 2 orders
// everything enqueued before this call, and inside the call every upload waits for all
// passes except the one just before it, whose experts it keeps.
#include <algorithm>
#include <chrono>
#include <thread>
#include <vector>

#include "common.cuh"

namespace {

using namespace moe;

// Bounded host wait for an event (polls cudaEventQuery).
moe_status wait_event(cudaEvent_t ev, double timeout_s) {
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return MOE_OK;
        if (e != cudaErrorNotReady) return MOE_ERR_CUDA;
        if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() >
            timeout_s)
            return MOE_ERR_TIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
}

struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
    cudaEvent_t make() {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        ev.push_back(e);
        return e;
    }
};

}  // namespace

extern "C" moe_status moe_offload_forward(
    const moe_layer_desc *L, const moe_select_params *P, const void *x, const void *W_r,
    const void *host_gate, const void *host_up, const void *host_down, void *slot_gate,
    void *slot_up, void *slot_down, moe_residency *table, int layer, const int *depth, int B,
    int N, void *y, const moe_tree_outputs *out, moe_offload_stats *stats, void *workspace,
    const moe_run_opts *opts, moe_stream_t stream, moe_stream_t side) {
    SelectArgs a;
    if (!desc_ok(L) || !select_args(P, L->k, &a) || B < 1 || N < 1 || !table) return MOE_ERR_ARG;
    if (!x || !W_r || !host_gate || !host_up || !host_down || !slot_gate || !slot_up ||
        !slot_down || !depth || !y || !workspace || L->slots < 1)
        return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(W_r) || !aligned16(slot_gate) || !aligned16(slot_up) ||
        !aligned16(slot_down) || !aligned16(y) || ((uintptr_t)workspace & 255u))
        return MOE_ERR_ARG;
    const int E = L->E, R = B * N;
    std::vector<int> slot_host(E);
    std::vector<uint8_t> res_host(E);
    if (moe_residency_query(table, layer, slot_host.data(), res_host.data()) != MOE_OK)
        return MOE_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream, sd = (cudaStream_t)side;
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
    int *slot_dev = at<int>(workspace, w.slotmap);
    uint8_t *res_dev = at<uint8_t>(workspace, w.resident);
    uint8_t *pass_dev = at<uint8_t>(workspace, w.pass);
    Events events;

    // 1. residency before uploads, routing, selection, permutation
    if (launch_publish(E, slot_host.data(), res_host.data(), slot_dev, res_dev, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    moe_status sn;
    const void *xin = layer_input(*L, x, R, workspace, w, opts, s, &sn);
    if (sn != MOE_OK) return sn;
    if (launch_router(*L, xin, W_r, R, logits, at<int>(workspace, w.flags) + kRouterCheckWord,
                      s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_select(*L, a, logits, depth, B, N, a.prune ? res_dev : nullptr, idx, gates, elig,
                      info, WeightPrefetch{}, PermuteOut{}, nullptr, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    moe_status st = run_permute(*L, idx, R, workspace, w, counts, offsets, perm, true, s);
    if (st != MOE_OK) return st;

    // 2. the needed set
    std::vector<int> cnt(E);
    cudaEvent_t ev_counts = events.make();
    if (!ev_counts ||
        cudaMemcpyAsync(cnt.data(), counts, E * sizeof(int), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaEventRecord(ev_counts, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if ((st = wait_event(ev_counts, 10.0)) != MOE_OK) return st;
    std::vector<int> resident_needed, missing;
    for (int e = 0; e < E; ++e)
        if (cnt[e] > 0) (slot_host[e] >= 0 ? resident_needed : missing).push_back(e);
    const int slots = L->slots;
    const size_t mat_bytes = (size_t)L->d * L->f * elem_size(L->dtype);
    long long h2d = 0;
    int uploads = 0, passes = 0;

    auto pass_run = [&](const std::vector<int> &experts) -> moe_status {
        std::vector<uint8_t> mask(E, 0);
        for (int e : experts) mask[e] = 1;
        int sl[kMaxE];
        if (moe_residency_query(table, layer, sl, nullptr) != MOE_OK) return MOE_ERR_ARG;
        if (launch_publish(E, sl, mask.data(), slot_dev, pass_dev, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        ++passes;
        return run_ffn(*L, xin, slot_gate, slot_up, slot_down, slot_dev, pass_dev, R, workspace, w,
                       counts, offsets, perm, opts, s);
    };

    // 3a. resident experts: refresh their LRU age and compute them now
    std::vector<int> ue(E), us(E);
    int n_up = 0;
    std::vector<int> prev = resident_needed;  // experts of the pass just enqueued
    cudaEvent_t ev_prev = nullptr, ev_prev2 = nullptr;  // ends of the last two passes
    if (!resident_needed.empty()) {
        if (moe_residency_plan(table, layer, resident_needed.data(), (int)resident_needed.size(),
                               ue.data(), us.data(), &n_up, nullptr) != MOE_OK)
            return MOE_ERR_ARG;
        if ((st = pass_run(resident_needed)) != MOE_OK) return st;
        ev_prev = events.make();
        if (!ev_prev || cudaEventRecord(ev_prev, s) != cudaSuccess) return MOE_ERR_CUDA;
    }

    // 3b. missing experts in chunks, uploads on the side stream
    size_t next = 0;
    int n_wait = 0;
    residency_set_waits(table, layer, 0);
    while (next < missing.size()) {
        const size_t left = missing.size() - next;
        const size_t room = slots > (int)prev.size() ? slots - prev.size() : 0;
        const bool keep_prev = room >= std::min<size_t>(left, std::max(1, slots / 2));
        const size_t take = keep_prev ? std::min(left, room) : std::min<size_t>(left, slots);
        std::vector<int> chunk(missing.begin() + next, missing.begin() + next + take);
        next += take;
        // passes before `prev` must be done before their slots may be reused; without
        // room next to `prev`, `prev` itself too
        if (ev_prev2 && cudaStreamWaitEvent(sd, ev_prev2, 0) != cudaSuccess) return MOE_ERR_CUDA;
        std::vector<int> plan_set = chunk;
        if (keep_prev) {
            plan_set.insert(plan_set.end(), prev.begin(), prev.end());
        } else if (ev_prev && cudaStreamWaitEvent(sd, ev_prev, 0) != cudaSuccess) {
            return MOE_ERR_CUDA;
        }
        if (moe_residency_plan(table, layer, plan_set.data(), (int)plan_set.size(), ue.data(),
                               us.data(), &n_up, nullptr) != MOE_OK)
            return MOE_ERR_NOSLOT;
        cudaEvent_t ev_up = events.make();
        if (!ev_up) return MOE_ERR_CUDA;
        if ((st = moe_expert_upload(L, host_gate, host_up, host_down, slot_gate, slot_up,
                                    slot_down, ue.data(), us.data(), n_up, side,
                                    (moe_event_t)ev_up)) != MOE_OK)
            return st;
        uploads += n_up;
        h2d += (long long)n_up * 3 * (long long)mat_bytes;
        // the compute stream's wait for this upload, bracketed by timing events: the
        // second completes when both the work before it and the upload are done
        cudaEvent_t w0 = residency_wait_event(table, layer, n_wait, 0);
        cudaEvent_t w1 = residency_wait_event(table, layer, n_wait, 1);
        if (!w0 || !w1 || cudaEventRecord(w0, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamWaitEvent(s, ev_up, 0) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaEventRecord(w1, s) != cudaSuccess) return MOE_ERR_CUDA;
        residency_set_waits(table, layer, ++n_wait);
        if ((st = pass_run(chunk)) != MOE_OK) return st;
        ev_prev2 = ev_prev;
        ev_prev = events.make();
        if (!ev_prev || cudaEventRecord(ev_prev, s) != cudaSuccess) return MOE_ERR_CUDA;
        prev = chunk;
    }

    // 4. combine
    st = run_combine(*L, (opts && opts->residual) ? x : nullptr, gates, R, y, workspace, w, s);
    if (st != MOE_OK) return st;
    if (stats) {
        stats->needed = (int)(resident_needed.size() + missing.size());
        stats->hits = (int)resident_needed.size();
        stats->uploads = uploads;
        stats->passes = passes;
        stats->h2d_bytes = h2d;
    }
    return MOE_OK;
}
