/*
 * moetree.h -- C ABI of libmoetree: a GB300 (sm_103a) MoE layer run over one
 * speculative-decoding verification block (a draft tree verified in one pass),
 * with AcceptMoE-style verifier-side expert selection.
 *
 * What the operations compute (page title + section):
 *   - "MoE and speculative decoding" blog, section "starting from one MoE layer":
 *     the layer E(x) = TopR(softmax(W_r x)), y = sum_{e in E(x)} g_e(x) E_e(x), run
 *     as router -> permute/group by expert -> grouped GEMM over the active experts
 *     -> unpermute + weighted combine.
 *   - "AcceptMoE" news article, section 02, and the AcceptMoE abstract (arXiv
 *     2608.02989): commitment-weighted demand, root anchor, self-sizing by the
 *     effective rank of the demand, residency-aware pruning, and re-routing every
 *     node inside the eligible set.
 *   - same article, section 03 and the abstract: expert offload with 48 expert
 *     slots per layer and host-to-device uploads of non-resident experts.
 *   - "Fewer experts, faster decoding: cost-aware speculative decoding for MoE"
 *     (EcoSpec), section 1 and Fig. 2-3, with the scoring rule of the blog above:
 *     a cost-aware choice of which drafted nodes to verify (moe_draft_select).
 *
 * Conventions shared by every entry point:
 *   - All tensors are plain pointers, row-major, densely packed. "device" means
 *     CUDA device memory of the current device; "host" means CPU memory. The
 *     caller owns every buffer and every stream; the library allocates nothing
 *     except the residency table's host metadata.
 *   - Work is enqueued on the caller's stream and returns without waiting, unless
 *     an entry point says otherwise. Arguments are checked on the host before any
 *     launch; a bad argument returns MOE_ERR_ARG and enqueues nothing.
 *   - x, W_r and expert weights share the layer dtype (fp32 or bf16). Router
 *     logits and gates are fp32. Expert ids and indices are int32.
 *   - `workspace` is device memory of at least moe_workspace_bytes() bytes, 256-byte
 *     aligned. It is scratch: its contents on entry are ignored and on return are
 *     unspecified. Two calls that overlap in time must use different workspaces.
 *   - No C++ exception crosses this ABI; every failure is a moe_status.
 */
#ifndef MOETREE_H
#define MOETREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* a cudaStream_t (NULL = legacy default) */
typedef struct CUevent_st *moe_event_t;   /* a cudaEvent_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = -1,          /* bad argument; nothing was enqueued */
    MOE_ERR_CUDA = -2,         /* a CUDA runtime/driver call failed */
    MOE_ERR_NOSLOT = -3,       /* more experts needed at once than the layer has slots */
    MOE_ERR_TIMEOUT = -4,      /* a bounded wait gave up */
    MOE_ERR_DEVICE_CHECK = -5, /* a kernel-side check failed (see moe_workspace_check) */
    MOE_ERR_UNSUPPORTED = -6   /* shape or dtype outside what the kernels support */
} moe_status;

typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

/* Routing modes. NATURAL is plain top-k routing (the pages' "Standard SD");
 * ACCEPT is AcceptMoE selection; FIXED_B keeps the demand ranking but takes the
 * set size from `fixed_B` instead of the effective rank (AcceptMoE-B; with a
 * uniform commitment table and no anchor it is the MoE-Spec budget rule). */
typedef enum { MOE_ROUTE_NATURAL = 0, MOE_ROUTE_ACCEPT = 1, MOE_ROUTE_FIXED_B = 2 } moe_route_mode;

/* Which grouped-expert kernel runs. AUTO picks by dtype and shape. */
typedef enum { MOE_FFN_AUTO = 0, MOE_FFN_SIMT = 1, MOE_FFN_TCGEN05 = 2 } moe_ffn_path;

/* One MoE layer: hidden size d, E routed experts, top-k, SwiGLU width f.
 * `slots` is the number of expert slots in the weight pools the expert entry points
 * read (0 means E: one slot per expert). Limits: 1 <= k <= 16, k <= E <= 256, d and f
 * multiples of 8 and at most 6144 (multiples of 64 for the tcgen05 expert kernel),
 * 0 <= slots <= 65535. */
typedef struct {
    int d, E, k, f;
    int dtype; /* moe_dtype */
    int slots;
} moe_layer_desc;

#define MOE_MAX_DEPTHS 16

/* Expert-selection parameters ("AcceptMoE" news article, section 02).
 *   c_by_depth[t]  commitment probability of a node at draft depth t (root = 0);
 *                  depths >= n_c use c_by_depth[n_c-1].
 *   pool_all       0: fill candidates come from the natural union of the tree
 *                  (default); 1: from all E experts.
 *   anchor         1: the root's natural top-k is always eligible (default).
 *   prune          1: residency-aware pruning against `resident` (needs resident).
 *   reroute_budget most experts pruning may remove from a tree's eligible set.
 *   min_set        pruning stops when the set has max(min_set, k) experts.
 *   fixed_B        set size for MOE_ROUTE_FIXED_B. */
typedef struct {
    int mode; /* moe_route_mode */
    int n_c;
    double c_by_depth[MOE_MAX_DEPTHS];
    int pool_all;
    int anchor;
    int prune;
    int reroute_budget;
    int min_set;
    int fixed_B;
} moe_select_params;

/* Per-tree counters written by selection, int32 [B][MOE_INFO_FIELDS] in device memory:
 * natural union, selected union, eligible-set size m before pruning, pruned count, and
 * 1 if the tree's decisions needed the fp64 pass (see moe_tree_select), else 0. */
#define MOE_INFO_FIELDS 5

/* Optional device outputs of moe_tree_forward; any member may be NULL. */
typedef struct {
    float *logits;    /* [R, E] router logits */
    int *topk_idx;    /* [R, k] routed experts (after selection) */
    float *gates;     /* [R, k] renormalised gate weights */
    uint8_t *eligible;/* [B, E] eligible set per tree */
    int *info;        /* [B, MOE_INFO_FIELDS] */
    int *counts;      /* [E] assignments per expert */
    int *offsets;     /* [E+1] exclusive prefix of counts */
    int *perm;        /* [R*k] permuted order of assignment ids r*k+j */
} moe_tree_outputs;

/* Run options; pass NULL for defaults. If both events are non-NULL they are
 * recorded on the stream immediately before and after the grouped-expert kernel
 * (for timing the dominant kernel with CUDA events). `select_begin`, if non-NULL, is
 * recorded just before the selection launch of moe_tree_forward (whose extra CTAs
 * start streaming the root's experts into L2), so that select_begin .. ffn_end times
 * the whole expert stage. An event between two launches keeps the second from
 * starting early, so timed calls run slightly slower than untimed ones. With `residual`
 * set the layer returns y = x + MoE(x) instead of MoE(x), for a residual stack of
 * layers; y may then be the same buffer as x. With `norm_input` set the router and the
 * experts read the pre-norm x_n[r] = x[r] / sqrt(mean_i x[r, i]^2 + 1e-6) (no learned
 * weight; mean and scale in fp64, each element rounded once to the layer dtype, written
 * into the workspace) instead of x, as the pre-norm blocks of the target models do; the
 * residual still adds x itself: y = x + MoE(x_n). Used by moe_tree_forward,
 * moe_expert_forward and moe_offload_forward. */
typedef struct {
    int ffn_path; /* moe_ffn_path */
    moe_event_t ffn_begin;
    moe_event_t ffn_end;
    int residual;
    moe_event_t select_begin;
    int norm_input;
    int ffn_max_ctas; /* tensor-core expert kernel: CTAs at most (0: one per SM). Fewer
                         leave SMs free for another stream's routing kernels, so that two
                         independent blocks can be in flight at once */
} moe_run_opts;

/* Text for a status code. Never NULL. */
const char *moe_status_str(int status);

/* ABI version of this header (major*100 + minor). */
int moe_abi_version(void);

/* Bytes of workspace needed for blocks of up to B trees of N nodes (R = B*N rows). */
size_t moe_workspace_bytes(const moe_layer_desc *L, int B, int N);

/* Router scores ("MoE and speculative decoding" blog, "starting from one MoE layer",
 * the W_r x inside E(x) = TopR(softmax(W_r x))): logits[r, e] = sum_i x[r, i] W_r[e, i],
 * fp32 accumulation, no bias. From 192 rows on (bf16, d a multiple of 64, sm_100 or
 * later) the product runs on the tensor cores; the accumulation order then differs
 * from the CUDA-core kernel's at the level of fp32 rounding.
 *   x [R, d] and W_r [E, d] device, layer dtype; logits [R, E] device fp32. */
moe_status moe_router_logits(const moe_layer_desc *L, const void *x, const void *W_r, int R,
                             float *logits, moe_stream_t stream);

/* Pre-norm of the layer input, the RMS normalisation the target models (Qwen3, GPT-OSS)
 * apply before the MoE layer, without a learned weight: per row
 * xn[r, i] = x[r, i] / sqrt(mean_i x[r, i]^2 + 1e-6); the mean and scale are computed in
 * fp64, each element is rounded once (nearest, ties to even) to the layer dtype. The
 * layer calls apply it themselves when moe_run_opts.norm_input is set; this call exposes
 * it on its own.
 *   x, xn [R, d] device, layer dtype, 16-byte aligned, must not overlap. */
moe_status moe_rms_norm(const moe_layer_desc *L, const void *x, int R, void *xn,
                        moe_stream_t stream);

/* Expert selection for B trees of N nodes from router logits ("AcceptMoE" news
 * article, section 02; AcceptMoE abstract). Per tree: natural top-k of every node,
 * demand D_e = sum_n c(depth_n) softmax(logits_n)_e (nodes in order), set size
 * m = max(k, ceil(exp(H(D / sum D)))) capped at the pool, an exp(H) within 1e-9
 * (relative) of an integer counting as that integer (FIXED_B: m = fixed_B), root anchor
 * + fill by (D desc, id asc), optional residency-aware pruning, then each node's top-k
 * restricted to the eligible set, gates = softmax over the k chosen logits. NATURAL
 * mode: plain top-k with the same renormalised gates.
 * The demand, entropy and exp(H) are defined in fp64. The kernels compute them in fp32
 * with a bound on their own rounding error and keep the fp32 decisions only where that
 * bound proves them equal to the fp64 ones; any other tree is recomputed in fp64
 * (info[b][4] = 1). Given the same logits, the results are those of the fp64 definition
 * up to ties closer than fp64 rounding.
 *   logits   [B*N, E] device fp32, node n of tree b at row b*N + n, node 0 = root.
 *   depth    [B*N] device int32, draft depth of each node (root 0).
 *   resident [E] device uint8 (1 = expert resident) or NULL; required if P->prune.
 *   topk_idx [B*N, k] device int32, descending logit order, ties to the lower id.
 *   gates    [B*N, k] device fp32.
 *   eligible [B, E] device uint8 or NULL; info [B, MOE_INFO_FIELDS] device int32 or
 *   NULL. */
moe_status moe_tree_select(const moe_layer_desc *L, const moe_select_params *P,
                           const float *logits, const int *depth, int B, int N,
                           const uint8_t *resident, int *topk_idx, float *gates,
                           uint8_t *eligible, int *info, moe_stream_t stream);

/* Permute / group by expert ("MoE and speculative decoding" blog, pipeline step
 * "permute / group by expert"): stable counting sort of the assignments (r, j) by
 * (expert, row, slot).
 *   topk_idx [R, k] device int32; counts [E], offsets [E+1], perm [R*k] device int32
 *   (perm[p] = r*k + j of the assignment at permuted position p). Expert ids out of
 *   range are counted as a device-check failure and skipped. */
moe_status moe_expert_permute(const moe_layer_desc *L, const int *topk_idx, int R, int *counts,
                              int *offsets, int *perm, void *workspace, moe_stream_t stream);

/* Grouped SwiGLU experts + gated combine for a given routing ("MoE and speculative
 * decoding" blog, "grouped GEMM for active experts" and "unpermute + weighted
 * combine"): y[r] = sum_j gates[r, j] W_down[e] (silu(W_gate[e] x_r) * (W_up[e] x_r)),
 * e = topk_idx[r, j], slots summed in ascending j. Each expert with at least one
 * assignment streams its weights from HBM once per launch; an expert with more tokens
 * than one row tile holds (128 when no expert of the call has more than 256, else 256)
 * takes several row tiles, which read each weight tile at the same time, so their repeat
 * reads mostly hit L2.
 *   x [R, d] device; y [R, d] device, layer dtype.
 *   W_gate, W_up [S, f, d] and W_down [S, d, f] device: a pool of S = L->slots (or E)
 *   expert slots.
 *   slot_of_expert [E] device int32 maps expert -> slot, or NULL for slot = expert. An
 *   expert routed to a slot outside [0, S) is skipped and flagged (moe_workspace_check).
 *   topk_idx [R, k] device int32, gates [R, k] device fp32. */
moe_status moe_expert_forward(const moe_layer_desc *L, const void *x, const void *W_gate,
                              const void *W_up, const void *W_down, const int *slot_of_expert,
                              const int *topk_idx, const float *gates, int R, void *y,
                              void *workspace, const moe_run_opts *opts, moe_stream_t stream);

/* The whole layer over one verification block: router, selection (or natural
 * routing), permute, grouped SwiGLU experts, combine. Arguments as in the calls
 * above; `out` (may be NULL) receives intermediate results. */
moe_status moe_tree_forward(const moe_layer_desc *L, const moe_select_params *P, const void *x,
                            const void *W_r, const void *W_gate, const void *W_up,
                            const void *W_down, const int *slot_of_expert, const int *depth,
                            int B, int N, const uint8_t *resident, void *y,
                            const moe_tree_outputs *out, void *workspace,
                            const moe_run_opts *opts, moe_stream_t stream);

/* Router and selection from hidden states: moe_router_logits followed by
 * moe_tree_select on the same stream, for callers that hold x and W_r rather than
 * logits. `logits` [B*N, E] device fp32 is written (the selection reads it); the other
 * arguments are those of the two calls. */
moe_status moe_tree_route(const moe_layer_desc *L, const moe_select_params *P, const void *x,
                          const void *W_r, const int *depth, int B, int N,
                          const uint8_t *resident, float *logits, int *topk_idx, float *gates,
                          uint8_t *eligible, int *info, moe_stream_t stream);

/* Counters of one verification block ("MoE and speculative decoding" blog, measurement
 * section: unique experts, assignments per expert, and the reuse of the union
 * 1 - |union of E(x_i)| / sum |E(x_i)|; "AcceptMoE" news article, section 02: the set
 * size and what pruning removed). */
typedef struct {
    int trees;               /* B */
    int assignments;         /* R * k routed (row, expert) pairs */
    int union_experts;       /* experts with at least one assignment in the block */
    int max_per_expert;      /* the largest per-expert count */
    double reuse;            /* 1 - union_experts / assignments */
    double union_nat_mean;   /* per tree: natural union (the pages' Standard SD) */
    double union_sel_mean;   /* per tree: union after selection */
    double m_mean;           /* per tree: eligible-set size before pruning */
    double pruned_mean;      /* per tree: experts removed by residency-aware pruning */
    int exact_trees;         /* trees whose decisions took the fp64 pass */
} moe_tree_stats;

/* Reads the counters of the last block routed with these arrays: info [B,
 * MOE_INFO_FIELDS] and counts [E] (device), as written by moe_tree_forward /
 * moe_tree_select + moe_expert_permute. NULL info or counts: the copies inside
 * `workspace` (the one the forward call used; info/counts must not have been redirected
 * by moe_tree_outputs then). Waits for `stream`; allocates nothing. */
moe_status moe_tree_block_stats(const moe_layer_desc *L, int B, int N, const int *info,
                                const int *counts, const void *workspace, moe_tree_stats *stats,
                                moe_stream_t stream);

/* moe_tree_forward without a `workspace` argument, for callers that cannot allocate
 * device memory when they run the layer: an engine whose free HBM is already reserved
 * for its KV cache, a plug-in that is handed only input/output device pointers, or a
 * loop that must not let cudaMalloc/cudaFree synchronise the device. The pages have no
 * counterpart to this entry point; it is a deployment convenience of this library.
 *   - Scratch is one built-in 16 MiB device array (a file-scope __device__ buffer).
 *     Every device that has loaded it keeps those 16 MiB until the process exits.
 *     Requests whose moe_workspace_bytes(L, B, N) exceed 16 MiB return
 *     MOE_ERR_UNSUPPORTED (one 65-node tree of the Qwen3-30B-A3B- or GPT-OSS-120B-shaped
 *     layer needs about 8 MiB); nothing is enqueued then.
 *   - The first call on a device looks up that array's device address (with that
 *     device current); make that first call before any stream capture begins.
 *   - All calls in the process share the one array, and it keeps the last call's
 *     contents; what must start at zero is cleared by the call itself. Calls whose work
 *     overlaps on the GPU (different streams, or different host threads without
 *     ordering) race on the array: order them on one stream.
 *   - Calls no allocating routine. Other arguments and results are those of
 *     moe_tree_forward. Kernel-side checks (a skipped expert id or slot, a bounded wait
 *     that gave up) land in the built-in array's check word: read and clear it with
 *     moe_noalloc_check. */
moe_status moe_tree_forward_noalloc(const moe_layer_desc *L, const moe_select_params *P,
                                    const void *x, const void *W_r, const void *W_gate,
                                    const void *W_up, const void *W_down,
                                    const int *slot_of_expert, const int *depth, int B, int N,
                                    const uint8_t *resident, void *y,
                                    const moe_tree_outputs *out, const moe_run_opts *opts,
                                    moe_stream_t stream);

/* The check word of moe_tree_forward_noalloc's built-in scratch on the current device,
 * read and cleared like moe_workspace_check (waits for `stream`; no allocation). Each
 * call of the layer starts the word afresh, so it reports the kernels of the last call:
 * *flags = 0 when they reported no problem (also when the entry point has not run on
 * this device or the word was read since); bits as in moe_workspace_check. Returns
 * MOE_ERR_DEVICE_CHECK when *flags != 0. */
moe_status moe_noalloc_check(int *flags, moe_stream_t stream);

/* Cost-aware choice of the draft tree to verify ("Fewer experts, faster decoding:
 * cost-aware speculative decoding for MoE" (EcoSpec, arXiv 2607.12696), section 1 and
 * Fig. 2-3; Score(v) = log P_q(v) - lambda * dC_expert(v) in the "MoE and speculative
 * decoding" blog). From C drafted candidates (node 0 the root, parent[v] < v) take
 * gamma nodes: the root, then repeatedly the candidate whose parent is already taken with
 * the largest logp[v] - lambda * (number of its predicted experts not yet covered), fp32,
 * ties to the lower index; the covered set grows by each chosen node's footprint.
 * Verification of the chosen tree is unchanged (plain moe_tree_forward).
 *   parent, depth [C] int32, logp [C] fp32 (cumulative draft log-probability),
 *   footprint [C, L->k] int32 predicted experts per candidate (e.g. the natural top-k of
 *   the target router). The cost counts experts: an id listed twice counts once, ids
 *   outside [0, L->E) are ignored, and a candidate whose parent is outside [0, C) is
 *   never taken -- all device. logp must be finite.
 *   selected [gamma]: candidate ids in selection order (parents first; -1 past the end
 *   when fewer than gamma can be taken); sel_parent [gamma]: parent as a position in
 *   `selected` (root -1); sel_depth [gamma]; x [C, d] / x_sel [gamma, d] (layer dtype,
 *   both or neither): the chosen rows gathered in selection order; n_union (may be NULL):
 *   covered experts. All device. 1 <= C <= 4097, gamma >= 1, lambda >= 0, else
 *   MOE_ERR_ARG (nothing enqueued). One CTA; the gamma - 1 greedy steps are sequential. */
moe_status moe_draft_select(const moe_layer_desc *L, int C, const int *parent, const int *depth,
                            const float *logp, const int *footprint, float lambda, int gamma,
                            const void *x, int *selected, int *sel_parent, int *sel_depth,
                            void *x_sel, int *n_union, moe_stream_t stream);

/* Reads and clears the kernel-side check word of a workspace. Waits for `stream`.
 * *flags = 0 when no kernel reported a problem since the last call; bit 0 = an
 * expert id outside [0, E) was skipped; bit 1 = a bounded device wait gave up. */
moe_status moe_workspace_check(void *workspace, int *flags, moe_stream_t stream);

/* ---------------------------------------------------------------- offload ----
 * Expert residency for offloaded layers ("AcceptMoE" news article, section 03:
 * 48 expert slots per layer on the GPU, the other experts in CPU memory and
 * uploaded on demand). The table lives in host memory; each layer has `slots`
 * device slots and an LRU order over them. */
typedef struct moe_residency moe_residency;

moe_status moe_residency_create(int n_layers, int E, int slots, moe_residency **table);
moe_status moe_residency_destroy(moe_residency *table);

/* Host copy of one layer's state: slot_of_expert [E] (-1 = not resident) and
 * resident [E] (0/1); either may be NULL. */
moe_status moe_residency_query(const moe_residency *table, int layer, int *slot_of_expert,
                               uint8_t *resident);

/* Makes the `n_needed` experts of `needed` (host) resident in `layer`: experts
 * already in a slot are hits and move to the front of the LRU order; each miss
 * takes a free slot or evicts the least recently used slot not needed now. Writes
 * the uploads to perform to up_expert/up_slot (host, room for n_needed) and their
 * number to *n_up; *hits may be NULL. MOE_ERR_NOSLOT if n_needed > slots (split the
 * set and call once per part). Host only; enqueues nothing. */
moe_status moe_residency_plan(moe_residency *table, int layer, const int *needed, int n_needed,
                              int *up_expert, int *up_slot, int *n_up, int *hits);

/* Writes the layer's slot map and resident mask to device arrays (int32 [E] and
 * uint8 [E]; either may be NULL) with a kernel on `stream`. */
moe_status moe_residency_publish(const moe_residency *table, int layer, int *slot_of_expert,
                                 uint8_t *resident, moe_stream_t stream);

/* Copies whole experts host -> device slot: for each i, expert up_expert[i]'s
 * W_gate, W_up, W_down from the host stores (pinned, [E, f, d], [E, f, d], [E, d, f])
 * into slot up_slot[i] of the device pools ([S, ...]) with one cudaMemcpyAsync per
 * matrix on `side`, then records `done` (may be NULL) on `side`. Arrays are host. */
moe_status moe_expert_upload(const moe_layer_desc *L, const void *host_gate, const void *host_up,
                             const void *host_down, void *slot_gate, void *slot_up,
                             void *slot_down, const int *up_expert, const int *up_slot, int n,
                             moe_stream_t side, moe_event_t done);

/* Counters of one moe_offload_forward call. */
typedef struct {
    int needed;          /* experts with at least one assignment in the block */
    int hits;            /* of those, already resident when the call began */
    int uploads;         /* experts copied host -> device by the call */
    int passes;          /* grouped-expert launches (resident experts, then upload chunks) */
    long long h2d_bytes; /* bytes copied host -> device */
} moe_offload_stats;

/* The whole layer with offloaded experts ("AcceptMoE" news article, section 03: a fixed
 * number of expert slots per layer on the GPU, the rest in CPU memory uploaded on
 * demand; section 02 and the abstract: residency-aware pruning conditions eligibility
 * on what is resident now). Router, selection (pruning, if P->prune, sees the residency
 * as it was before this call), permute; then ONE host wait for the per-expert counts;
 * the resident needed experts are computed at once while missing experts are copied on
 * `side` (one cudaMemcpyAsync per matrix, least-recently-used slots replaced, in chunks
 * when they do not fit next to the experts being computed); finally the gated combine.
 *   L->slots        device slots of this layer (the table's `slots`).
 *   host_gate/up/down  pinned host stores [E, f, d], [E, f, d], [E, d, f].
 *   slot_gate/up/down  device pools [slots, f, d], [slots, f, d], [slots, d, f].
 *   table, layer    the residency table and this layer's index in it; updated.
 *   stats           host, optional.
 * Other arguments as moe_tree_forward. Returns after enqueueing the last kernel; the
 * call itself waits (bounded, 10 s -> MOE_ERR_TIMEOUT) only for the routing of this
 * block. Uploads never overwrite a slot that an enqueued kernel may still read. */
moe_status moe_offload_forward(const moe_layer_desc *L, const moe_select_params *P,
                               const void *x, const void *W_r, const void *host_gate,
                               const void *host_up, const void *host_down, void *slot_gate,
                               void *slot_up, void *slot_down, moe_residency *table, int layer,
                               const int *depth, int B, int N, void *y,
                               const moe_tree_outputs *out, moe_offload_stats *stats,
                               void *workspace, const moe_run_opts *opts, moe_stream_t stream,
                               moe_stream_t side);

/* Time the compute stream of the last moe_offload_forward call on `layer` spent waiting
 * for expert uploads ("AcceptMoE" news article, section 03: the share of runtime spent
 * waiting on expert loads): the sum over that call's upload waits of the time between
 * the stream reaching the wait and the upload completing (0 for a wait the upload had
 * already met). Waits (bounded by timeout_s per event -> MOE_ERR_TIMEOUT) for those
 * events; *waits (may be NULL) = the number of upload waits. Host only. */
moe_status moe_offload_upload_wait(moe_residency *table, int layer, double timeout_s,
                                   double *wait_ms, int *waits);

/* Host poll of cudaEventQuery(ev) for at most timeout_s seconds. MOE_ERR_TIMEOUT if
 * the event has not completed by then. */
moe_status moe_event_wait(moe_event_t ev, double timeout_s);

#ifdef __cplusplus
}
#endif
#endif /* MOETREE_H */
