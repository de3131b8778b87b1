// Cost-aware selection of the draft tree to verify ("Fewer experts, faster decoding:
// cost-aware speculative decoding for MoE" (EcoSpec, arXiv 2607.12696), section 1 and
// Fig. 2-3; the scoring rule Score(v) = log P_q(v) - lambda * dC_expert(v) as written in
// the "MoE and speculative decoding" blog).
//
// One CTA. S starts as {root}, the expert buffer B as the root's predicted footprint.
// Each of the gamma - 1 steps scores every candidate whose parent is in S,
// logp[v] - lambda * |footprint(v) \ B| (fp32: one product, one difference), takes the
// best (ties to the lower index), and adds it to S and its footprint to B.
//
// The steps are sequential, so the kernel is built for the latency of one step:
//   - every footprint is turned once into a bit set of E <= 256 bits in shared memory;
//     |footprint(v) \ B| is then a popcount of (footprint(v) & ~B) over E / 32 words
//     (duplicate ids count once, ids outside [0, E) are ignored);
//   - each thread owns up to kMaxCpt candidates and keeps their log-probability,
//     parent and state (waiting / eligible / taken) in registers, and every thread keeps
//     its own copy of B; nothing is written to shared memory inside a step except the
//     per-warp best;
//   - the best is an order-preserving 32-bit key of the score (max) and the lowest
//     index among equal keys (min), two warp reductions per level; the per-warp results
//     are double-buffered by step parity, so one barrier per step suffices: every warp
//     then reduces the warp results itself and learns the winner.
// The parent positions, depths, covered count and gathered rows are written after the
// last step from the list of winners.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxThreads = 1024;
constexpr int kMaxCpt = 4;  // candidates per thread: C <= 1 + 4 * 1024
constexpr int kMaxWords = kMaxE / 32;
constexpr uint32_t kNone = 0u;

// Order-preserving key of a float score (larger score, larger key); 0 is "no candidate".
// -0 is folded into +0 first, so equal scores give equal keys.
__device__ __forceinline__ uint32_t score_key(float s) {
    const uint32_t u = __float_as_uint(s + 0.f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int CPT>
__global__ void __launch_bounds__(kMaxThreads)
draft_select_kernel(int C, int k, int E, const int *__restrict__ parent,
                    const int *__restrict__ depth, const float *__restrict__ logp,
                    const int *__restrict__ fp, float lambda, int gamma,
                    int *__restrict__ selected, int *__restrict__ sel_parent,
                    int *__restrict__ sel_depth, int *__restrict__ n_union,
                    const uint4 *__restrict__ x, uint4 *__restrict__ x_sel, int row_vec) {
    pdl_wait();
    const int nw = (E + 31) >> 5;  // words of a bit set
    extern __shared__ uint32_t dsm[];
    uint32_t *fpm = dsm;                       // [C][nw] footprint bit sets
    int *win = (int *)(dsm + (size_t)C * nw);  // [C] winners in selection order
    int *pos = win + C;                        // [C] position of a winner
    __shared__ uint32_t wkey[2][32];
    __shared__ int widx[2][32];
    const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = T >> 5;

    // footprint bit sets
    for (int i = tid; i < C * nw; i += T) fpm[i] = 0u;
    __syncthreads();
    for (int i0 = tid; i0 < C * k; i0 += 8 * T) {  // eight loads in flight, then the ORs
        int ev[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) ev[u] = i0 + u * T < C * k ? fp[i0 + u * T] : -1;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = ev[u], i = i0 + u * T;
            if (e >= 0 && e < E) atomicOr(&fpm[(size_t)(i / k) * nw + (e >> 5)], 1u << (e & 31));
        }
    }
    // owned candidates: c = 1 + tid + s * T
    float lp[CPT];
    int par[CPT];
    int st[CPT];  // 0 waiting for its parent, 1 eligible, 2 taken or not a candidate
#pragma unroll
    for (int s = 0; s < CPT; ++s) {
        const int c = 1 + tid + s * T;
        if (c < C) {
            lp[s] = logp[c];
            par[s] = parent[c];
            st[s] = par[s] == 0 ? 1 : 0;
        } else {
            lp[s] = 0.f;
            par[s] = -1;
            st[s] = 2;
        }
    }
    if (tid == 0) win[0] = 0;
    __syncthreads();
    uint32_t B[kMaxWords];
#pragma unroll
    for (int q = 0; q < kMaxWords; ++q) B[q] = q < nw ? fpm[q] : 0u;

    int n = 1;
    const int steps = min(gamma, C);
    for (; n < steps; ++n) {
        uint32_t key = kNone;
        int bi = 0x7fffffff;
#pragma unroll
        for (int s = 0; s < CPT; ++s) {
            if (st[s] != 1) continue;
            const int c = 1 + tid + s * T;
            int dc = 0;
#pragma unroll
            for (int q = 0; q < kMaxWords; ++q)
                if (q < nw) dc += __popc(fpm[(size_t)c * nw + q] & ~B[q]);
            const uint32_t kc = score_key(__fsub_rn(lp[s], __fmul_rn(lambda, (float)dc)));
            if (kc > key) {  // owned candidates ascend with s: ties keep the lower index
                key = kc;
                bi = c;
            }
        }
        uint32_t km = __reduce_max_sync(0xffffffffu, key);
        int wi = (int)__reduce_min_sync(0xffffffffu, key == km ? (uint32_t)bi : 0x7fffffffu);
        const int b = n & 1;
        if (lane == 0) {
            wkey[b][warp] = km;
            widx[b][warp] = wi;
        }
        __syncthreads();
        key = lane < nwarps ? wkey[b][lane] : kNone;
        bi = lane < nwarps ? widx[b][lane] : 0x7fffffff;
        km = __reduce_max_sync(0xffffffffu, key);
        if (km == kNone) break;  // no candidate left
        const int w = (int)__reduce_min_sync(0xffffffffu, key == km ? (uint32_t)bi : 0x7fffffffu);
#pragma unroll
        for (int q = 0; q < kMaxWords; ++q)
            if (q < nw) B[q] |= fpm[(size_t)w * nw + q];
#pragma unroll
        for (int s = 0; s < CPT; ++s) {
            if (1 + tid + s * T == w) st[s] = 2;
            else if (st[s] == 0 && par[s] == w) st[s] = 1;
        }
        if (tid == 0) win[n] = w;
    }
    __syncthreads();
    for (int i = tid; i < n; i += T) pos[win[i]] = i;
    __syncthreads();
    for (int i = tid; i < gamma; i += T) {
        if (i < n) {
            const int v = win[i];
            selected[i] = v;
            sel_parent[i] = i == 0 ? -1 : pos[parent[v]];
            sel_depth[i] = depth[v];
        } else {  // fewer candidates than gamma
            selected[i] = -1;
            sel_parent[i] = -1;
            sel_depth[i] = -1;
        }
    }
    if (tid == 0 && n_union) {
        int u = 0;
#pragma unroll
        for (int q = 0; q < kMaxWords; ++q) u += __popc(B[q]);
        *n_union = u;
    }
    if (x && x_sel) {
        for (int i = warp; i < n; i += nwarps) {
            const uint4 *src = x + (size_t)win[i] * row_vec;
            uint4 *dst = x_sel + (size_t)i * row_vec;
            for (int v = lane; v < row_vec; v += 32) dst[v] = __ldg(src + v);
        }
    }
}

template <int CPT>
cudaError_t launch_draft(int T, size_t smem, cudaStream_t s, int C, int k, int E,
                         const int *parent, const int *depth, const float *logp, const int *fp,
                         float lambda, int gamma, int *selected, int *sel_parent, int *sel_depth,
                         int *n_union, const void *x, void *x_sel, int row_vec) {
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(
            draft_select_kernel<CPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(draft_select_kernel<CPT>, dim3(1), dim3(T), smem, s, C, k, E, parent,
                      depth, logp, fp, lambda, gamma, selected, sel_parent, sel_depth, n_union,
                      (const uint4 *)x, (uint4 *)x_sel, row_vec);
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
    if (!desc_ok(L) || C < 1 || C > 1 + kMaxCpt * kMaxThreads || gamma < 1 || !parent ||
        !depth || !logp || !footprint || !selected || !sel_parent || !sel_depth ||
        !(lambda >= 0.f))
        return MOE_ERR_ARG;
    if ((x == nullptr) != (x_sel == nullptr)) return MOE_ERR_ARG;
    if (x && (!aligned16(x) || !aligned16(x_sel))) return MOE_ERR_ARG;
    const int row_vec = (int)((size_t)L->d * elem_size(L->dtype) / 16);
    const int nw = (L->E + 31) / 32;
    const size_t smem = (size_t)C * (nw + 2) * sizeof(uint32_t);
    const int cand = C > 1 ? C - 1 : 1;
    // two candidates per thread from 257 candidates on (fewer warps in each step's
    // reduction; measured faster than one per thread at 411 candidates), four past 2048
    const int cpt = cand <= 256 ? 1 : (cand <= 2 * kMaxThreads ? 2 : 4);
    const int T = std::min(kMaxThreads, ((cand + cpt - 1) / cpt + 31) / 32 * 32);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (cpt == 1)
        e = launch_draft<1>(T, smem, s, C, L->k, L->E, parent, depth, logp, footprint, lambda,
                            gamma, selected, sel_parent, sel_depth, n_union, x, x_sel, row_vec);
    else if (cpt == 2)
        e = launch_draft<2>(T, smem, s, C, L->k, L->E, parent, depth, logp, footprint, lambda,
                            gamma, selected, sel_parent, sel_depth, n_union, x, x_sel, row_vec);
    else
        e = launch_draft<4>(T, smem, s, C, L->k, L->E, parent, depth, logp, footprint, lambda,
                            gamma, selected, sel_parent, sel_depth, n_union, x, x_sel, row_vec);
    return cuda_status(e);
}
