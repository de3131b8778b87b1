// Cost-aware selection of the draft tree to verify ("Fewer experts, faster decoding:
// cost-aware speculative decoding for MoE" (EcoSpec, arXiv 2607.12696), section 1 and
// Fig. 2-3; the scoring rule Score(v) = log P_q(v) - lambda * dC_expert(v) as written in
// the "MoE and speculative decoding" blog).
//
// One CTA. S starts as {root}, the expert buffer B as the root's predicted footprint.
// Each of the gamma - 1 steps scores every candidate whose parent is in S,
// logp[v] - lambda * |footprint(v) \ B| (fp32: one product, one difference), takes the
// best (ties to the lower index) with a block-wide argmax, and adds it to S and its
// footprint to B (a bitmask of E <= 256 bits; footprint ids outside [0, E) are ignored,
// and so are candidates whose parent index is outside [0, C)). The selection order is a
// valid node order for the verified tree (parents first), so the kernel also writes that
// tree's parent indices and depths and gathers its token rows for moe_tree_forward.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ bool better(float s, int i, float bs, int bi) {
    return bi < 0 || s > bs || (s == bs && i < bi);
}

__global__ void __launch_bounds__(kThreads)
draft_select_kernel(int C, int k, int E, const int *__restrict__ parent,
                    const int *__restrict__ depth,
                    const float *__restrict__ logp, const int *__restrict__ fp, float lambda,
                    int gamma, int *__restrict__ selected, int *__restrict__ sel_parent,
                    int *__restrict__ sel_depth, int *__restrict__ n_union,
                    const uint4 *__restrict__ x, uint4 *__restrict__ x_sel, int row_vec) {
    pdl_wait();
    extern __shared__ int dsm[];
    int *inS = dsm;      // [C]
    int *pos = dsm + C;  // [C] position in the selection order, -1 if not selected
    __shared__ uint32_t buf[kMaxE / 32];
    __shared__ float wbs[kWarps];
    __shared__ int wbi[kWarps];
    __shared__ int s_best;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int c = tid; c < C; c += kThreads) {
        inS[c] = 0;
        pos[c] = -1;
    }
    if (tid < kMaxE / 32) buf[tid] = 0u;
    __syncthreads();
    if (tid == 0) {
        inS[0] = 1;
        pos[0] = 0;
        selected[0] = 0;
        sel_parent[0] = -1;
        sel_depth[0] = depth[0];
        for (int j = 0; j < k; ++j) {
            const int e = fp[j];
            if (e >= 0 && e < E) buf[e >> 5] |= 1u << (e & 31);
        }
    }
    __syncthreads();
    int n = 1;
    for (; n < gamma; ++n) {
        float bs = 0.f;
        int bi = -1;
        for (int c = 1 + tid; c < C; c += kThreads) {
            const int pc = parent[c];
            if (inS[c] || pc < 0 || pc >= C || !inS[pc]) continue;
            int dc = 0;
            for (int j = 0; j < k; ++j) {
                const int e = fp[(size_t)c * k + j];
                if (e >= 0 && e < E) dc += (buf[e >> 5] >> (e & 31)) & 1u ? 0 : 1;
            }
            const float sc = __fsub_rn(logp[c], __fmul_rn(lambda, (float)dc));
            if (better(sc, c, bs, bi)) {
                bs = sc;
                bi = c;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, bs, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi >= 0 && better(os, oi, bs, bi)) {
                bs = os;
                bi = oi;
            }
        }
        if (lane == 0) {
            wbs[warp] = bs;
            wbi[warp] = bi;
        }
        __syncthreads();
        if (warp == 0) {
            bs = wbs[lane];
            bi = wbi[lane];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (oi >= 0 && better(os, oi, bs, bi)) {
                    bs = os;
                    bi = oi;
                }
            }
            if (lane == 0) {
                s_best = bi;
                if (bi >= 0) {
                    inS[bi] = 1;
                    pos[bi] = n;
                    selected[n] = bi;
                    sel_parent[n] = pos[parent[bi]];
                    sel_depth[n] = depth[bi];
                    for (int j = 0; j < k; ++j) {
                        const int e = fp[(size_t)bi * k + j];
                        if (e >= 0 && e < E) buf[e >> 5] |= 1u << (e & 31);
                    }
                }
            }
        }
        __syncthreads();
        if (s_best < 0) break;
    }
    for (int i = n + tid; i < gamma; i += kThreads) {  // fewer candidates than gamma
        selected[i] = -1;
        sel_parent[i] = -1;
        sel_depth[i] = -1;
    }
    if (tid == 0 && n_union) {
        int u = 0;
        for (int w = 0; w < kMaxE / 32; ++w) u += __popc(buf[w]);
        *n_union = u;
    }
    if (x && x_sel) {
        for (int i = warp; i < n; i += kWarps) {
            const uint4 *src = x + (size_t)selected[i] * row_vec;
            uint4 *dst = x_sel + (size_t)i * row_vec;
            for (int v = lane; v < row_vec; v += 32) dst[v] = __ldg(src + v);
        }
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_draft_select(const moe_layer_desc *L, int C, const int *parent,
                                       const int *depth, const float *logp,
                                       const int *footprint, float lambda, int gamma,
                                       const void *x, int *selected, int *sel_parent,
                                       int *sel_depth, void *x_sel, int *n_union,
                                       moe_stream_t stream) {
    if (!desc_ok(L) || C < 1 || C > 8192 || gamma < 1 || !parent || !depth || !logp ||
        !footprint || !selected || !sel_parent || !sel_depth || !(lambda >= 0.f))
        return MOE_ERR_ARG;
    if ((x == nullptr) != (x_sel == nullptr)) return MOE_ERR_ARG;
    if (x && (!aligned16(x) || !aligned16(x_sel))) return MOE_ERR_ARG;
    const int row_vec = (int)((size_t)L->d * elem_size(L->dtype) / 16);
    const size_t smem = (size_t)2 * C * sizeof(int);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(draft_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return cuda_status(launch_pdl(draft_select_kernel, dim3(1), dim3(kThreads), smem,
                                  (cudaStream_t)stream, C, L->k, L->E, parent, depth, logp,
                                  footprint, lambda, gamma, selected, sel_parent, sel_depth,
                                  n_union, (const uint4 *)x, (uint4 *)x_sel, row_vec));
}
