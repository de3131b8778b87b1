// Verifier-side expert selection for a block of draft trees ("AcceptMoE" news
// article, section 02; AcceptMoE abstract, arXiv 2608.02989).
//
// One CTA per tree. Phase A: a warp per node takes the node's natural top-k (the
// natural routing and the natural union U) and, unless routing is natural, its
// softmax weighted by the commitment probability of the node's depth; the CTA
// then adds those rows into the demand D in node order. Phase B (one CTA, O(E^2)
// rank counting, E <= 256): set size from the effective rank exp(H(D / sum D)),
// root anchor + fill in (D desc, id asc) order, residency-aware pruning in
// (D asc, id asc) order. Phase C: a warp per node re-runs top-k inside the
// eligible set and writes renormalised gates.
//
// Demand, entropy and gates are computed in fp32 (GB300's fp64 rate is a small
// fraction of its fp32 rate): the softmax row sum in a warp tree, the demand per
// expert in ascending node order, sum D and H in ascending expert order in one
// thread, each product and sum rounded on its own (no FMA contraction).
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kVPL = kMaxE / 32;  // logits held per lane

// Relative distance to an integer under which exp(H) counts as that integer.
constexpr float kSnap = 1e-5f;

struct Top {
    int idx;    // valid in lanes j < k: the j-th choice
    float val;
};

// Warp-wide top-k of v (lane holds experts lane + 32 i) among experts whose bit is set
// in `allowed` (bit i of lane's mask). Descending value, ties to the lower id.
// Lane j < k receives the j-th choice.
__device__ __forceinline__ Top warp_topk(const float v[kVPL], unsigned allowed, int E, int k) {
    const int lane = threadIdx.x & 31;
    unsigned taken = 0;
    Top mine{-1, -INFINITY};
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kVPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && ((allowed >> i) & 1u) && !((taken >> i) & 1u)) {
                if (v[i] > bv || (v[i] == bv && e < bi)) {
                    bv = v[i];
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) mine = Top{bi == 0x7fffffff ? -1 : bi, bv};
    }
    return mine;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Gates: softmax over the k chosen logits (lane j holds choice j), written with idx.
__device__ __forceinline__ void write_choice(const Top &t, int k, int *idx, float *gates) {
    const int lane = threadIdx.x & 31;
    const float top = __shfl_sync(0xffffffffu, t.val, 0);
    const float ex = lane < k ? expf(t.val - top) : 0.f;
    const float s = warp_sum(ex);
    if (lane < k) {
        idx[lane] = t.idx;
        gates[lane] = ex / s;
    }
}

__global__ void __launch_bounds__(kThreads)
select_kernel(SelectArgs a, const float *__restrict__ logits, const int *__restrict__ depth,
              int N, int E, int k, const uint8_t *__restrict__ resident, int *__restrict__ idx_out,
              float *__restrict__ gates_out, uint8_t *__restrict__ elig_out,
              int *__restrict__ info_out) {
    __shared__ float D[kMaxE];
    __shared__ float wbuf[kWarps][kMaxE];
    __shared__ float term[kMaxE];
    __shared__ int inU[kMaxE], inS[kMaxE], inA[kMaxE], inSel[kMaxE], rem[kMaxE];
    __shared__ int natRoot[kMaxK];
    __shared__ int s_m, s_removed;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const float *L = logits + (size_t)b * N * E;
    const int *dep = depth + (size_t)b * N;
    int *idxb = idx_out + (size_t)b * N * k;
    float *gb = gates_out + (size_t)b * N * k;
    const bool natural = a.mode == MOE_ROUTE_NATURAL;

    for (int e = tid; e < kMaxE; e += kThreads) {
        D[e] = 0.f;
        inU[e] = 0;
        inSel[e] = 0;
    }
    __syncthreads();

    // ---- phase A: natural top-k, natural union, demand rows ----
    for (int base = 0; base < N; base += kWarps) {
        const int n = base + warp;
        if (n < N) {
            float v[kVPL];
#pragma unroll
            for (int i = 0; i < kVPL; ++i) {
                const int e = lane + 32 * i;
                v[i] = e < E ? L[(size_t)n * E + e] : -INFINITY;
            }
            const Top t = warp_topk(v, 0xffffffffu, E, k);
            if (lane < k && t.idx >= 0) inU[t.idx] = 1;
            if (n == 0 && lane < k) natRoot[lane] = t.idx;
            if (natural) {
                write_choice(t, k, idxb + (size_t)n * k, gb + (size_t)n * k);
            } else {
                const float mx = __shfl_sync(0xffffffffu, t.val, 0);
                float ex[kVPL], s = 0.f;
#pragma unroll
                for (int i = 0; i < kVPL; ++i) {
                    const int e = lane + 32 * i;
                    ex[i] = e < E ? expf(v[i] - mx) : 0.f;
                    s += ex[i];
                }
                s = warp_sum(s);
                const int dd = dep[n] < a.n_c ? dep[n] : a.n_c - 1;
                const float c = a.c[dd < 0 ? 0 : dd];
#pragma unroll
                for (int i = 0; i < kVPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E) wbuf[warp][e] = __fmul_rn(c, __fdiv_rn(ex[i], s));
                }
            }
        }
        __syncthreads();
        if (!natural) {
            for (int e = tid; e < E; e += kThreads) {
                float acc = D[e];
                for (int w = 0; w < kWarps && base + w < N; ++w) acc = __fadd_rn(acc, wbuf[w][e]);
                D[e] = acc;
            }
        }
        __syncthreads();
    }

    if (natural) {
        if (tid == 0) {
            int u = 0;
            for (int e = 0; e < E; ++e) u += inU[e];
            if (info_out) {
                info_out[b * MOE_INFO_FIELDS + 0] = u;
                info_out[b * MOE_INFO_FIELDS + 1] = u;
                info_out[b * MOE_INFO_FIELDS + 2] = E;
                info_out[b * MOE_INFO_FIELDS + 3] = 0;
            }
        }
        if (elig_out)
            for (int e = tid; e < E; e += kThreads) elig_out[(size_t)b * E + e] = 1;
        return;
    }

    // ---- phase B: size, anchor + fill, prune ----
    if (tid == 0) {
        float sum = 0.f;
        for (int e = 0; e < E; ++e) sum = __fadd_rn(sum, D[e]);
        term[0] = sum;  // borrowed as a broadcast slot until the terms are written
    }
    __syncthreads();
    const float sumD = term[0];
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        const float q = __fdiv_rn(D[e], sumD);
        term[e] = q > 0.f ? __fmul_rn(q, logf(q)) : 0.f;
        inA[e] = 0;
    }
    __syncthreads();
    if (tid == 0) {
        int pool = 0;
        for (int e = 0; e < E; ++e) pool += (a.pool_all || inU[e]) ? 1 : 0;
        int m;
        if (a.mode == MOE_ROUTE_ACCEPT) {
            float H = 0.f;
            for (int e = 0; e < E; ++e) H = __fsub_rn(H, term[e]);
            const float r = expf(H);
            const float rn = rintf(r);
            m = (fabsf(r - rn) <= kSnap * r) ? (int)rn : (int)ceilf(r);
        } else {
            m = a.fixed_B;
        }
        if (m < k) m = k;
        if (m > pool) m = pool;
        s_m = m;
        if (a.anchor)
            for (int j = 0; j < k; ++j) inA[natRoot[j]] = 1;
    }
    __syncthreads();
    int nA = 0;
    if (a.anchor) nA = k;
    const int m = s_m;
    for (int e = tid; e < E; e += kThreads) {
        int in = inA[e];
        const bool cand = !inA[e] && (a.pool_all || inU[e]);
        if (cand) {
            const float De = D[e];
            int rank = 0;
            for (int q = 0; q < E; ++q) {
                const bool cq = !inA[q] && (a.pool_all || inU[q]);
                rank += (cq && (D[q] > De || (D[q] == De && q < e))) ? 1 : 0;
            }
            in = rank < m - nA;
        }
        inS[e] = in;
    }
    __syncthreads();
    if (a.prune && resident) {
        for (int e = tid; e < E; e += kThreads) rem[e] = inS[e] && !inA[e] && !resident[e];
        __syncthreads();
        if (tid == 0) {
            int nrem = 0;
            for (int e = 0; e < E; ++e) nrem += rem[e];
            const int fl = a.min_set > k ? a.min_set : k;
            int can = m - fl;
            if (can < 0) can = 0;
            if (can > a.budget) can = a.budget;
            if (can > nrem) can = nrem;
            s_removed = can;
        }
        __syncthreads();
        const int nr = s_removed;
        for (int e = tid; e < E; e += kThreads) {
            if (!rem[e]) continue;
            const float De = D[e];
            int rank = 0;
            for (int q = 0; q < E; ++q)
                rank += (rem[q] && (D[q] < De || (D[q] == De && q < e))) ? 1 : 0;
            if (rank < nr) inS[e] = 0;
        }
    } else if (tid == 0) {
        s_removed = 0;
    }
    __syncthreads();

    // ---- phase C: restricted top-k and gates ----
    unsigned allowed = 0;
#pragma unroll
    for (int i = 0; i < kVPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && inS[e]) allowed |= 1u << i;
    }
    for (int n = warp; n < N; n += kWarps) {
        float v[kVPL];
#pragma unroll
        for (int i = 0; i < kVPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? L[(size_t)n * E + e] : -INFINITY;
        }
        const Top t = warp_topk(v, allowed, E, k);
        if (lane < k && t.idx >= 0) inSel[t.idx] = 1;
        write_choice(t, k, idxb + (size_t)n * k, gb + (size_t)n * k);
    }
    __syncthreads();
    if (tid == 0 && info_out) {
        int u = 0, us = 0;
        for (int e = 0; e < E; ++e) {
            u += inU[e];
            us += inSel[e];
        }
        info_out[b * MOE_INFO_FIELDS + 0] = u;
        info_out[b * MOE_INFO_FIELDS + 1] = us;
        info_out[b * MOE_INFO_FIELDS + 2] = m;
        info_out[b * MOE_INFO_FIELDS + 3] = s_removed;
    }
    if (elig_out)
        for (int e = tid; e < E; e += kThreads) elig_out[(size_t)b * E + e] = (uint8_t)inS[e];
}

}  // namespace

cudaError_t launch_select(const moe_layer_desc &L, const SelectArgs &a, const float *logits,
                          const int *depth, int B, int N, const uint8_t *resident, int *idx,
                          float *gates, uint8_t *elig, int *info, cudaStream_t s) {
    if (B <= 0 || N <= 0) return cudaSuccess;
    select_kernel<<<B, kThreads, 0, s>>>(a, logits, depth, N, L.E, L.k, resident, idx, gates, elig,
                                         info);
    return cudaGetLastError();
}

}  // namespace moe
