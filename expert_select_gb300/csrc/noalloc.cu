// moe_tree_forward_noalloc: the whole MoE tree-verification layer without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they run the layer: a
// serving engine that has already handed all free HBM to its KV-cache pool (one more
// cudaMalloc would fail or fragment that pool), a plug-in that only receives device
// pointers for its inputs and outputs from a host runtime with no allocator binding,
// or a latency-critical loop where cudaMalloc/cudaFree would synchronise the device.
// For them the scratch that moe_tree_forward takes as `workspace` lives here, in one
// file-scope device array of fixed size. The kernels and their launch order are
// exactly those of moe_tree_forward; only the source of the scratch differs.
#include <mutex>

#include "common.cuh"

namespace {

// Holds one 65-node tree of a Qwen3-30B-A3B- or GPT-OSS-120B-shaped layer with room
// to spare. Requests whose moe_workspace_bytes() exceed it are rejected.
constexpr size_t kScratchBytes = (size_t)16 << 20;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device addresses of g_scratch, one per device, looked up on the first call made
// with that device current. (In host code `g_scratch` names a host-side shadow, not
// device memory, so it must never be handed to a kernel directly.)
constexpr int kMaxDevices = 64;
void *g_scratch_dev[kMaxDevices];
std::mutex g_scratch_mu;

// The built-in scratch's device address on the current device (set up on first use).
moe_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_tree_forward_noalloc(
    const moe_layer_desc *L, const moe_select_params *P, const void *x, const void *W_r,
    const void *W_gate, const void *W_up, const void *W_down, const int *slot_of_expert,
    const int *depth, int B, int N, const uint8_t *resident, void *y,
    const moe_tree_outputs *out, const moe_run_opts *opts, moe_stream_t stream) {
    // bad arguments are reported as such before any CUDA call
    const moe_status st = moe::tree_forward_check(L, P, x, W_r, W_gate, W_up, W_down, depth, B,
                                                  N, resident, y);
    if (st != MOE_OK) return st;
    const size_t need = moe_workspace_bytes(L, B, N);
    if (need == 0) return MOE_ERR_ARG;
    if (need > kScratchBytes) return MOE_ERR_UNSUPPORTED;
    void *ws = nullptr;
    const moe_status sa = scratch_address(&ws);
    if (sa != MOE_OK) return sa;
    // The check word and scheduler counters that must start at zero are cleared by
    // the first kernel that uses them (the permute kernel), as for any workspace.
    return moe_tree_forward(L, P, x, W_r, W_gate, W_up, W_down, slot_of_expert, depth, B, N,
                            resident, y, out, ws, opts, stream);
}

extern "C" moe_status moe_noalloc_check(int *flags, moe_stream_t stream) {
    if (!flags) return MOE_ERR_ARG;
    void *ws = nullptr;
    const moe_status sa = scratch_address(&ws);
    if (sa != MOE_OK) return sa;
    // the check word is the first int of the workspace layout, as in any workspace
    return moe_workspace_check(ws, flags, stream);
}
