// Internal declarations shared by the libmoetree translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <utility>

#include "moetree.h"

namespace moe {

// Bits of the kernel-side check word (first int of the workspace).
enum : int { FLAG_BAD_EXPERT = 1, FLAG_WAIT_TIMEOUT = 2 };
// Workspace flag words: [0] the check word moe_workspace_check reads; [kRouterCheckWord]
// the router's, which runs before the permute kernel clears the words and is carried into
// [0] by it.
constexpr int kRouterCheckWord = 1;

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxD = 6144;  // SIMT experts stage 8 rows of d (or f) fp32 in shared memory

// Byte offsets of the scratch arrays inside one workspace.
struct Workspace {
    size_t flags;     // int32[64]: [0] check word, the rest scheduler counters
    size_t logits;    // f32 [R, E]
    size_t idx;       // i32 [R, k]
    size_t gates;     // f32 [R, k]
    size_t elig;      // u8  [B, E]
    size_t info;      // i32 [B, 4]
    size_t counts;    // i32 [E]
    size_t offsets;   // i32 [E + 1]
    size_t perm;      // i32 [A]  permuted position -> assignment id
    size_t pos;       // i32 [A]  assignment id -> permuted position (-1 = skipped)
    size_t rbmask;    // u32 [2][E][ceil(R/32)]  row-block masks and prefixes of the permute
    size_t active;    // i32 [E + 1]  [0] = n_active, then active experts ascending
    size_t slotmap;   // i32 [E]  expert -> slot (offload)
    size_t resident;  // u8  [E]  residency before this call's uploads (offload)
    size_t pass;      // u8  [E]  experts computed by the current expert pass (offload)
    size_t rowtiles;  // i32 [4 + 4 * max_rowtiles]: count, tile height, 0, 0, then
                      // (expert, first permuted row, tokens, 0) per tile
    size_t sched;     // i32 [1 + max_rowtiles]: ticket counter, finished phase-1 units per row tile
    size_t xp;        // layer dtype [A, d]  x rows gathered in permuted order
    size_t h;         // f32 [A, f]  SwiGLU activations (bf16 [A, f] on the tensor-core path)
    size_t o;         // f32 [A, d]  expert outputs in permuted order
    size_t xn;        // layer dtype [R, d]  the normalised input (moe_run_opts.norm_input)
    size_t total;
};

Workspace workspace_layout(const moe_layer_desc &L, int B, int N);

inline size_t elem_size(int dtype) { return dtype == MOE_DTYPE_F32 ? 4 : 2; }

// ---- launchers (each returns the launch's cudaError_t) ----
cudaError_t launch_router(const moe_layer_desc &L, const void *x, const void *Wr, int R,
                          float *logits, int *flags, cudaStream_t s);  // flags may be null

struct SelectArgs {
    int mode, n_c, pool_all, anchor, prune, budget, min_set, fixed_B;
    float c[MOE_MAX_DEPTHS];     // the commitment table rounded to fp32 (the fast pass)
    double c64[MOE_MAX_DEPTHS];  // as given (the exact pass)
    float cmax;                  // the largest entry
};
// L2 prefetch of expert weights during routing (AcceptMoE and fixed-size selection). The
// root's natural top-k is the anchor that AcceptMoE keeps in every eligible set, and with
// it the root's own routing, so those experts are in the block's union whatever the
// selection decides. Extra CTAs of the selection launch take tree 0's root top-k from the
// logits and ask L2 for the three weight matrices of each of those experts: the expert
// kernel then finds part of them in L2, read from HBM while the routing kernels left it
// idle.
struct WeightPrefetch {
    const char *wg, *wu, *wd;   // W_gate, W_up, W_down slot pools
    const int *slot_of_expert;  // null: slot = expert id
    int slots;                  // slots in each pool
    int ctas;                   // extra CTAs doing the prefetch (a multiple of 8); 0 = none
    unsigned long long bytes;   // bytes of one slot of one matrix (a multiple of 16)
};
// The prefetch for a layer's weight pools, sized for a launch of B trees (ctas = 0 when
// the weights cannot be prefetched or the SMs are taken by the selection itself).
WeightPrefetch weight_prefetch(const moe_layer_desc &L, int B, const void *W_gate,
                               const void *W_up, const void *W_down, const int *slot_of_expert);
// The arrays of the permute step (see launch_permute), for a selection launch that also
// performs it: one tree per block on the cluster path. counts == nullptr: it does not.
struct PermuteOut {
    int *counts, *offsets, *perm, *pos, *active, *rowtiles, *flags;
    int after_router;
};
// *permuted (may be null) tells whether the launch also performed the permute step.
cudaError_t launch_select(const moe_layer_desc &L, const SelectArgs &a, const float *logits,
                          const int *depth, int B, int N, const uint8_t *resident, int *idx,
                          float *gates, uint8_t *elig, int *info, const WeightPrefetch &pf,
                          const PermuteOut &po, bool *permuted, cudaStream_t s);

// Row tiles of the tensor-core expert kernel: at most kMaxRowTile tokens of one expert
// (its MMA N is at most 256), or at most kPairRowTile when no expert has more than
// 2 * kPairRowTile tokens: then every tile has 128 tokens or fewer and the expert kernel
// can run two weight tiles over one tile of token rows. An expert with c tokens takes
// ceil(c / limit) tiles of near-equal size (at most E + A / kPairRowTile tiles in all); the
// height is the largest tile rounded up to 16, and the expert kernel sizes its per-stage
// token buffer to it: small blocks leave shared memory for more stages of weight bytes in
// flight. Each tile entry is (expert, first permuted row, tokens, group) with group =
// rowtile_group(j, g): the tile is the j-th of the expert's g tiles (the expert kernel hands
// the g tiles of one weight tile out together, so they read the weights from HBM once).
constexpr int kMaxRowTile = 256;
constexpr int kPairRowTile = 128;
constexpr int kRowTileHeader = 4;  // count, height, two unused ints
inline int max_rowtiles(int E, int A) { return E + (A + kPairRowTile - 1) / kPairRowTile + 1; }
// The tile limit of a block whose largest expert has cmax tokens.
__host__ __device__ inline int rowtile_limit(int cmax) {
    return cmax <= 2 * kPairRowTile ? kPairRowTile : kMaxRowTile;
}
__host__ __device__ inline int rowtile_group(int j, int g) { return (j << 16) | g; }

// The kernel starts the call's check word: the router's word is carried into it when the
// router ran earlier in the same call (after_router).
cudaError_t launch_permute(const moe_layer_desc &L, const int *idx, int R, int *counts,
                           int *offsets, int *perm, int *pos, int *active, int *rowtiles,
                           int *flags, uint32_t *rbmask, bool after_router, cudaStream_t s);
size_t permute_smem_bytes(int R, int E);

struct FfnArgs {
    const void *x;       // [R, d]
    const void *Wg, *Wu; // [S, f, d]
    const void *Wd;      // [S, d, f]
    const int *slot;     // [E] or nullptr
    const uint8_t *pass; // [E] or nullptr: experts with 0 are skipped (not an error)
    const int *counts, *offsets, *perm, *active, *rowtiles;
    const int *pos;      // [R*k] permuted position of each assignment (-1: skipped)
    int R, d, f, E, k, dtype;
    int slots;           // expert slots in the weight pools
    int *flags;
    int max_ctas;        // tensor-core path: CTAs at most (0: one per SM)
    int *sched;          // tensor-core path: ticket + row-tile counters
    void *xp;            // gathered x (tensor-core path)
    void *h;             // activations
    void *o;             // expert outputs, permuted order, in the layer dtype
};
cudaError_t launch_ffn_simt(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_ffn_tc(const FfnArgs &a, cudaStream_t s);
bool ffn_tc_supported(const moe_layer_desc &L);

cudaError_t launch_combine(const moe_layer_desc &L, const void *o, const int *pos,
                           const float *gates, const void *residual, int R, void *y,
                           cudaStream_t s);

cudaError_t launch_publish(int E, const int *slot_host, const uint8_t *res_host, int *slot_dev,
                           uint8_t *res_dev, cudaStream_t s);

// Pre-norm (moe_run_opts.norm_input): xn[r] = x[r] / sqrt(mean_i x[r, i]^2 + kNormEps).
constexpr double kNormEps = 1e-6;
cudaError_t launch_rmsnorm(const moe_layer_desc &L, const void *x, int R, void *xn,
                           cudaStream_t s);

// ---- host helpers shared by the entry points (api.cu, offload.cu) ----
// Timing events of the offloaded layer's upload waits, kept in the residency table.
cudaEvent_t residency_wait_event(moe_residency *t, int layer, int i, int which);
void residency_set_waits(moe_residency *t, int layer, int n);
inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T>
inline T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(reinterpret_cast<char *>(ws) + off);
}

bool desc_ok(const moe_layer_desc *L);
bool select_args(const moe_select_params *P, int k, SelectArgs *a);
bool aligned16(const void *p);
// The argument checks of moe_tree_forward other than those of the workspace.
moe_status tree_forward_check(const moe_layer_desc *L, const moe_select_params *P,
                              const void *x, const void *W_r, const void *W_gate,
                              const void *W_up, const void *W_down, const int *depth, int B,
                              int N, const uint8_t *resident, const void *y);
moe_status run_permute(const moe_layer_desc &L, const int *idx, int R, void *ws,
                       const Workspace &w, int *counts, int *offsets, int *perm,
                       bool after_router, cudaStream_t s);
moe_status run_ffn(const moe_layer_desc &L, const void *x, const void *Wg, const void *Wu,
                   const void *Wd, const int *slot, const uint8_t *pass, int R, void *ws,
                   const Workspace &w, const int *counts, const int *offsets, const int *perm,
                   const moe_run_opts *opts, cudaStream_t s);
int resolve_ffn_path(const moe_layer_desc &L, const moe_run_opts *opts);  // -1: unsupported
// x, or (opts->norm_input) its pre-norm written into the workspace by a launch on s.
const void *layer_input(const moe_layer_desc &L, const void *x, int R, void *ws,
                        const Workspace &w, const moe_run_opts *opts, cudaStream_t s,
                        moe_status *st);
moe_status run_combine(const moe_layer_desc &L, const void *residual, const float *gates, int R,
                       void *y, void *ws, const Workspace &w, cudaStream_t s);

// ---- launches ----
// Every kernel of the library is launched with programmatic stream serialization, so a
// kernel may be scheduled while its predecessor in the stream drains, and every kernel
// calls pdl_wait() before it touches memory: the wait returns once the predecessor grid
// has completed and its writes are visible. (Because every kernel waits, completion stays
// ordered along the whole chain.) No kernel releases its successor early
// (griddepcontrol.launch_dependents): measured on GB300, placing the successor's CTAs on
// the SMs while this kernel runs made the layer 0.6-1.2% slower, and the gap between two
// kernels (~1.5-3 us from the last CTA's exit to the successor's wait returning) stayed
// the same, so it is the grid's completion, not the successor's launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- device helpers ----
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Loads 8 consecutive elements starting at element `i` of a row as fp32.
// bf16: one 16-byte load; fp32: two 16-byte loads. `p` must be 16-byte aligned at i.
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float v[8]) {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
    }
};
template <> struct Vec8<float> {
    __device__ __forceinline__ static void load(const float *p, float v[8]) {
        float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// Sums 32 per-lane values across a warp; afterwards lane L holds the total of
// value index L (a transpose-reduction: 31 shuffles for 32 sums).
__device__ __forceinline__ float warp_transpose_sum32(float v[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            float send = up ? v[i] : v[i + s];
            float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

}  // namespace moe
