// Verifier-side expert selection for a block of draft trees ("AcceptMoE" news
// article, section 02; AcceptMoE abstract, arXiv 2608.02989).
//
// Natural routing needs none of the per-tree steps and has its own kernel (the last one
// in this file). For AcceptMoE and fixed-size routing, trees of up to 256 nodes run as
// one cluster of 8 CTAs per tree (see the cluster variant below); larger trees run on
// one CTA of 32 warps per tree, described here. The
// tree's logits are staged in shared memory once (when they fit) and every later pass
// reads them from there.
//   Phase A  a warp per node: natural top-k (the natural routing and the natural
//            union U), and the node's softmax maximum and normaliser.
//   Demand   every term c(depth_n) * exp(l_ne - max_n) / sum_n in parallel, then a
//            thread per expert adds its terms in ascending node order.
//   Phase B  set size from the effective rank exp(H(D / sum D)), root anchor + fill in
//            (D desc, id asc) order, residency-aware pruning in (D asc, id asc) order
//            (ranks by counting, E <= 256).
//   Phase C  a warp per node: top-k restricted to the eligible set S, renormalised
//            gates. A node whose natural top-k lies inside S keeps it (it is then the
//            restricted top-k by definition).
//
// Top-k: each lane holds experts lane + 32 i; a round takes every lane's best
// candidate as an order-preserving 32-bit key of its logit (-0 folded onto +0) and
// finds the winner with two warp reductions (max key, then min expert id among the
// lanes holding that key): descending logits, ties to the lower id, as exact as a
// comparison of the fp32 values.
//
// Precision of the decisions. The demand, its entropy and the effective rank are defined in
// fp64 (softmax of each node's logits, D_e summed over the nodes, H and exp(H)). A first
// pass computes them in fp32, every operation rounded on its own, and bounds its own
// rounding error (see phase_b): when every decision that depends on them (the set size
// from exp(H), the fill cut, the prune cut) is farther from its decision point than that
// bound, the fp32 pass has decided exactly as the fp64 definition does. Otherwise the
// tree's demand is recomputed in fp64 and phase B runs again in fp64 (GB300's fp64 rate is
// a small fraction of its fp32 rate, so that pass is kept for the trees that need it).
// info[4] reports which trees took it.
//
// Two more jobs ride on the selection launches of the whole layer (moe_tree_forward):
// for a block of one tree of up to 256 nodes the cluster (AcceptMoE or natural) also
// performs the permute step (permute_tree), and the AcceptMoE / fixed-size launches carry
// extra CTAs that prefetch the root's experts into L2 (prefetch_root_experts).
#include <cooperative_groups.h>
#include <math.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 32;
constexpr int kThreads = kWarps * 32;
constexpr int kVPL = kMaxE / 32;     // logits held per lane
constexpr int kStageFloats = 16384;  // logits staged in shared memory up to 64 KB
static_assert(kThreads >= kMaxE, "block-wide counts take one expert per thread");

// Relative distance to an integer under which exp(H) counts as that integer: an effective
// rank that is mathematically an integer (demand uniform over j experts) still counts as
// j after fp64 rounding.
constexpr double kSnap = 1e-9;
constexpr float kU = 5.9604645e-8f;  // 2^-24, the unit roundoff of fp32
// Terms whose exponent lies below about -87 underflow in fp32 (denormal or zero): their
// error is not relative but below 2^-126 in absolute value. The certificate adds
// kUnderflow * N * max(c) to every demand's error.
constexpr float kUnderflow = 2.4e-38f;  // 2^-125, twice the smallest normal fp32

__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.f);  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp top-k of v (lane holds experts lane + 32 i, i < VPL) among the experts whose bit i is
// set in `allowed`, in k rounds: every lane offers its best remaining candidate, two warp
// reductions (max key, then the lowest id holding it) pick the round's winner. Returns,
// in lane j < k, the expert id of the j-th choice (-1 if fewer than k experts are
// allowed).
template <int VPL>
__device__ __forceinline__ int warp_topk(const float (&v)[VPL], unsigned allowed, int E, int k) {
    const int lane = threadIdx.x & 31;
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        key[i] = (lane + 32 * i < E && ((allowed >> i) & 1u)) ? order_key(v[i]) : 0u;
    int mine = -1;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (key[i] > bk) {
                bk = key[i];
                bi = lane + 32 * i;
            }
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t w = __reduce_min_sync(0xffffffffu, (bk == m && m != 0u) ? (uint32_t)bi
                                                                               : 0xffffffffu);
        if (w != 0xffffffffu && (int)(w & 31u) == lane) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if ((int)(w >> 5) == i) key[i] = 0u;
        }
        if (lane == j) mine = w == 0xffffffffu ? -1 : (int)w;
    }
    return mine;
}


// c(depth) of the commitment table (the last entry repeats past the table). The table is
// a kernel parameter: selecting the entry with unrolled compares keeps it in the
// parameter bank (an indexed access would copy the whole argument block to local memory).
__device__ __forceinline__ float commitment(const SelectArgs &a, int depth) {
    const int dd = max(0, min(depth, a.n_c - 1));
    float c = a.c[0];
#pragma unroll
    for (int i = 1; i < MOE_MAX_DEPTHS; ++i)
        if (i == dd) c = a.c[i];
    return c;
}

__device__ __forceinline__ double commitment64(const SelectArgs &a, int depth) {
    const int dd = max(0, min(depth, a.n_c - 1));
    double c = a.c64[0];
#pragma unroll
    for (int i = 1; i < MOE_MAX_DEPTHS; ++i)
        if (i == dd) c = a.c64[i];
    return c;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ double warp_sum64(double v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// The logit range of a node (its largest minus its smallest logit), >= 0; lanes hold
// experts lane + 32 i (entries past E are -inf and ignored); `top` is the largest.
template <int VPL>
__device__ __forceinline__ float node_range(const float (&v)[VPL], int E, float top) {
    const int lane = threadIdx.x & 31;
    float lo = INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) lo = fminf(lo, v[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    return fmaxf(top - lo, 0.f);
}

// fp32 / fp64 arithmetic of phase B, every operation rounded on its own.
template <typename T> struct Num;
template <> struct Num<float> {
    __device__ static float add(float a, float b) { return __fadd_rn(a, b); }
    __device__ static float mul(float a, float b) { return __fmul_rn(a, b); }
    __device__ static float div(float a, float b) { return __fdiv_rn(a, b); }
    __device__ static float ln(float a) { return logf(a); }
    __device__ static float wsum(float v) { return warp_sum(v); }
};
template <> struct Num<double> {
    __device__ static double add(double a, double b) { return __dadd_rn(a, b); }
    __device__ static double mul(double a, double b) { return __dmul_rn(a, b); }
    __device__ static double div(double a, double b) { return __ddiv_rn(a, b); }
    __device__ static double ln(double a) { return log(a); }
    __device__ static double wsum(double v) { return warp_sum64(v); }
};

// Sum of v over the block's NW warps, identical in every thread: a butterfly per warp,
// then the warps' sums in warp order (red holds one value per warp; the call ends with a
// barrier, and `red` may be reused after the next barrier).
template <typename T, int NW>
__device__ __forceinline__ T block_sum(T v, T *red) {
    v = Num<T>::wsum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    T s = T(0);
#pragma unroll
    for (int w = 0; w < NW; ++w) s = Num<T>::add(s, red[w]);
    return s;
}

// Rank of expert e under the order of the keys rk (desc: larger first, else smaller
// first; equal keys: lower id first), i.e. the number of experts before it. `per`
// consecutive threads (a power of two dividing 32) share e: thread `part` counts the
// experts q = part (mod per), so that at each step a warp reads `per` consecutive words,
// and the counts are added with shuffles.
template <typename T>
__device__ __forceinline__ int rank_of(const T *rk, int e, int E, int per, int part, bool desc) {
    const T me = rk[e];
    int r = 0;
#pragma unroll 8
    for (int q = part; q < E; q += per) {
        const T o = rk[q];
        r += ((desc ? o > me : o < me) || (o == me && q < e)) ? 1 : 0;
    }
    for (int off = 1; off < per; off <<= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

struct PhaseB {
    int m, removed;
    bool sure;  // fp32 pass: every decision is certain to equal the fp64 definition's
};

// Phase B of one tree in precision T, on a whole block of NW warps: the set size from the
// effective rank exp(H(D / sum D)) (or fixed_B), the root anchor + fill in (D desc, id asc)
// order among the pool, residency-aware pruning in (D asc, id asc) order. D[E] holds the
// demand; inU / inA the natural union and the anchor; writes inS. rk, red, cut are
// scratch. Returns the size, the number pruned and, for T = float, whether the decisions
// are certain.
//
// The fp32 certificate. dD bounds the relative error of every fp32 D_e against the exact
// demand (computed by the caller from the logit range and the number of roundings). Then
//  - q_e = D_e / sum D is within dq = 2 dD + 21 u (sum: 20 roundings of positive terms);
//  - each term q ln q is within q (dq |ln q| + dq) + 3u q |ln q| (logf: 1 ulp; the
//    product: 1 rounding), so H (a block sum of same-sign terms, 20 roundings) is within
//    dH = (dq + 23 u) H + dq, and r = expf(H) (2 ulp) within dr = dH + 4u, taken with 5%
//    and 8u of slack for second-order terms and the rounding of the bounds themselves;
//  - the size rule is m = clamp(ceil(r (1 - 1e-9))): it is certain when the rule gives the
//    same m over [r (1 - dr), r (1 + dr)];
//  - a cut (fill: last taken vs first left; prune: last removed vs next) is certain when
//    the two demands stay ordered after moving each by dD + 2u (relative) and dA
//    (absolute: terms that underflowed in fp32) towards the other.
template <typename T, int NW>
__device__ PhaseB phase_b(const SelectArgs &a, int E, int k, const T *D, const int *inU,
                          const int *inA, int *inS, const uint8_t *resident, T *rk,
                          T (*red)[NW], T *cut, float dD, float dA) {
    using F = Num<T>;
    constexpr bool exact = sizeof(T) == sizeof(double);
    constexpr int NT = NW * 32;
    const int tid = threadIdx.x;
    const T De = tid < E ? D[tid] : T(0);
    if (tid < 4) cut[tid] = T(-1);
    const T sumD = block_sum<T, NW>(De, red[0]);
    const int pool = __syncthreads_count(tid < E && (a.pool_all || inU[tid]));
    T term = T(0);
    if (tid < E) {
        const T q = F::div(De, sumD);
        term = q > T(0) ? F::mul(q, F::ln(q)) : T(0);
    }
    const T H = -block_sum<T, NW>(term, red[1]);
    bool sure = true;
    int m;
    if (a.mode == MOE_ROUTE_ACCEPT) {
        if constexpr (exact) {
            const double r = exp(H);
            const double rn = rint(r);
            m = (fabs(r - rn) <= kSnap * r) ? (int)rn : (int)ceil(r);
            m = min(max(m, k), pool);
        } else {
            const float r = expf(H);
            const float dq = 2.f * dD + 21.f * kU;
            // + the underflowed terms: each q moves by at most dA / sum D, and |ln q| < 100
            const float dH = (dq + 23.f * kU) * fmaxf(H, 0.f) + dq +
                             (float)E * 100.f * dA / fmaxf((float)sumD, 1e-30f);
            const float dr = (dH + 4.f * kU) * 1.05f + 8.f * kU;
            const int lo = min(max((int)ceilf(r * (1.f - dr)), k), pool);
            const int hi = min(max((int)ceilf(r * (1.f + dr)), k), pool);
            sure = lo == hi && isfinite(r);
            m = hi;
        }
    } else {
        m = min(max(a.fixed_B, k), pool);
    }
    const int nA = a.anchor ? k : 0;
    // fill: candidates (pool minus anchor) ranked by (D desc, id asc); demand is >= 0, so
    // -1 marks a non-candidate. `per` threads share an expert.
    if (tid < E) rk[tid] = (!inA[tid] && (a.pool_all || inU[tid])) ? De : T(-1);
    __syncthreads();
    const int per = NT >= 4 * E ? 4 : 2;
    const int e = tid / per, pe = tid % per;
    const int ec = min(e, E - 1);
    const int F_ = m - nA;
    int in = 0;
    {
        const bool cand = e < E && rk[ec] >= T(0);
        const int ncand = __syncthreads_count(cand && pe == 0);
        if (F_ > 0 && F_ < ncand) {  // uniform: rank the candidates, keep the first F_
            const int rnk = rank_of<T>(rk, ec, E, per, pe, true);  // every thread
            if (e < E) in = inA[e] || (cand && rnk < F_);
            if (!exact && cand && pe == 0) {
                if (rnk == F_ - 1) cut[0] = rk[ec];
                if (rnk == F_) cut[1] = rk[ec];
            }
            __syncthreads();  // rk is rewritten below
            if (!exact)
                sure = sure && (float)cut[0] * (1.f - dD - 2.f * kU) - dA >
                                   (float)cut[1] * (1.f + dD + 2.f * kU) + dA;
        } else if (e < E) {  // every candidate fits (or none does): no ranking needed
            in = inA[e] || (cand && F_ > 0);
        }
    }
    if (e < E && pe == 0) inS[e] = in;
    int removed = 0;
    if (a.prune && resident) {
        // removable members (non-resident, not anchor) ranked by (D asc, id asc); +inf
        // marks the others
        int is_rem = 0;
        if (e < E) {
            is_rem = in && !inA[e] && !resident[e];
            if (pe == 0) rk[e] = is_rem ? D[e] : T(INFINITY);
        }
        const int nrem = __syncthreads_count(is_rem && pe == 0);
        const int fl = a.min_set > k ? a.min_set : k;
        removed = min(min(max(m - fl, 0), a.budget), nrem);
        const int rnk = rank_of<T>(rk, ec, E, per, pe, false);  // every thread
        if (is_rem && pe == 0) {
            if (rnk < removed) inS[e] = 0;
            if (!exact) {
                if (rnk == removed - 1) cut[2] = D[e];
                if (rnk == removed) cut[3] = D[e];
            }
        }
        __syncthreads();
        if (!exact && removed > 0 && removed < nrem)
            sure = sure && (float)cut[3] * (1.f - dD - 2.f * kU) - dA >
                               (float)cut[2] * (1.f + dD + 2.f * kU) + dA;
    }
    __syncthreads();  // inS complete
    return PhaseB{m, removed, sure};
}

// The fp64 phase B, kept out of line: it runs for few trees, and the selection kernels
// are short enough that the instruction fetch of their common path shows.
template <int NW>
__device__ __noinline__ PhaseB phase_b_exact(const SelectArgs &a, int E, int k, const double *D,
                                             const int *inU, const int *inA, int *inS,
                                             const uint8_t *resident, double *rk,
                                             double (*red)[NW], double *cut) {
    return phase_b<double, NW>(a, E, k, D, inU, inA, inS, resident, rk, red, cut, 0.f, 0.f);
}

// Relative error bound of the fp32 demand of a tree of N nodes whose logit ranges are at
// most A, VPL logits per lane: per term, the commitment (1 rounding), the argument
// l - max (|l - max| u), expf (2 ulp = 4u), the node's normaliser (its VPL - 1 + 5
// additions and its terms' errors), the quotient and the product (1 rounding each); then
// at most N + 8 additions of positive terms into D_e. 5% slack for second-order terms.
__device__ __forceinline__ float demand_bound(float A, int N, int VPL) {
    return kU * (2.f * A + (float)VPL + 15.f + (float)N + 8.f) * 1.05f;
}

// Absolute error bound of the fp32 demand from terms that underflow: at most one
// kUnderflow per node, times the largest commitment (computed on the host: indexing the
// table here would copy the whole argument block to local memory).
__device__ __forceinline__ float demand_floor(const SelectArgs &a, int N) {
    return kUnderflow * (float)N * a.cmax;
}

// Loads the E logits of one node into v[] (lane holds experts lane + 32 i).
template <int VPL>
__device__ __forceinline__ void load_row(const float *Ln, int E, float (&v)[VPL]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? Ln[e] : -INFINITY;
    }
}

// The logit of expert `idx` (idx < 0: -inf), fetched from the lane that holds it.
template <int VPL>
__device__ __forceinline__ float chosen_value(const float (&v)[VPL], int idx) {
    const int lane = threadIdx.x & 31;
    float out = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const float got = __shfl_sync(0xffffffffu, v[i], idx < 0 ? lane : (idx & 31));
        if (idx >= 0 && (idx >> 5) == i) out = got;
    }
    return out;
}

// Gates: softmax over the k chosen logits (lane j holds choice j), written with idx.
__device__ __forceinline__ void write_choice(int idx, float val, int k, int *out_idx,
                                             float *out_gates) {
    const int lane = threadIdx.x & 31;
    const float top = __shfl_sync(0xffffffffu, val, 0);
    const float ex = lane < k ? expf(val - top) : 0.f;
    const float s = warp_sum(ex);
    if (lane < k) {
        out_idx[lane] = idx;
        out_gates[lane] = ex / s;
    }
}

// L2 prefetch of the weights of tree 0's root experts (see WeightPrefetch): a CTA that
// is one of pf.ctas prefetch CTAs (part = its index among them) takes the root's natural
// top-k from `row0` and issues its share of bulk L2 prefetches over the three weight
// matrices of those experts. Chunks are dealt round-robin over all prefetch threads, so
// every CTA (and its SM's copy engine) covers part of every expert. Nothing waits for the
// prefetches; a slot outside [0, pf.slots) is skipped.
constexpr unsigned kPfChunk = 32768;  // bytes per bulk prefetch

__device__ void prefetch_root_experts(const WeightPrefetch &pf, const float *row0, int E, int k,
                                      int part) {
    __shared__ int s_slot[kMaxK];
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 32) {
        float v[kVPL];
        load_row(row0, E, v);
        const int c = warp_topk(v, 0xffffffffu, E, k);
        if (lane < k) {
            int sl = c;
            if (c >= 0 && pf.slot_of_expert) sl = pf.slot_of_expert[c];
            s_slot[lane] = (sl >= 0 && sl < pf.slots) ? sl : -1;
        }
    }
    __syncthreads();
    const unsigned long long per = (pf.bytes + kPfChunk - 1) / kPfChunk;  // chunks per matrix
    const unsigned long long total = per * 3ull * (unsigned long long)k;
    const unsigned long long stride = (unsigned long long)pf.ctas * blockDim.x;
    for (unsigned long long c = part + (unsigned long long)pf.ctas * tid; c < total; c += stride) {
        const unsigned long long q = c / per;  // expert rank * 3 + matrix
        const int sl = s_slot[q / 3];
        if (sl < 0) continue;
        const int mtx = (int)(q - (q / 3) * 3);
        const unsigned long long off = (c - q * per) * kPfChunk;
        const char *base = mtx == 0 ? pf.wg : (mtx == 1 ? pf.wu : pf.wd);
        const char *ptr = base + (size_t)sl * pf.bytes + off;
        const unsigned long long left = pf.bytes - off;
        const uint32_t sz = (uint32_t)(left < kPfChunk ? left : kPfChunk);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(sz) : "memory");
    }
}

__global__ void __launch_bounds__(kThreads)
select_kernel(SelectArgs a, const float *__restrict__ logits, const int *__restrict__ depth,
              int N, int E, int k, const uint8_t *__restrict__ resident, int *__restrict__ idx_out,
              float *__restrict__ gates_out, uint8_t *__restrict__ elig_out,
              int *__restrict__ info_out, WeightPrefetch pf) {
    // the last pf.ctas CTAs only prefetch
    if ((int)blockIdx.x >= (int)gridDim.x - pf.ctas) {
        prefetch_root_experts(pf, logits, E, k, (int)blockIdx.x - ((int)gridDim.x - pf.ctas));
        return;
    }
    // nz64 [N] (fp64 normalisers, the fp64 pass), staged logits, mx, nz, cN, nat, demand terms
    extern __shared__ double dyn64[];
    __shared__ float D[kMaxE];
    __shared__ double D64[kMaxE], rkb[kMaxE], redb[2][kWarps], cutb[4];
    __shared__ int inU[kMaxE], inS[kMaxE], inA[kMaxE], inSel[kMaxE];
    __shared__ int natRoot[kMaxK];
    __shared__ int s_range;  // largest node logit range (a non-negative float's bits)

    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const float *Lg = logits + (size_t)b * N * E;
    const int *dep = depth + (size_t)b * N;
    int *idxb = idx_out + (size_t)b * N * k;
    float *gb = gates_out + (size_t)b * N * k;
    const bool staged = N * E <= kStageFloats;
    double *nz64 = dyn64;
    float *stage = reinterpret_cast<float *>(dyn64 + N);
    float *mx = stage + (staged ? N * E : 0);  // [N] softmax maxima
    float *nz = mx + N;                        // [N] softmax normalisers
    float *cN = nz + N;                        // [N] commitment of each node
    int *nat = reinterpret_cast<int *>(cN + N);  // [N][k] natural choices

    if (staged) {
        if ((reinterpret_cast<uintptr_t>(Lg) & 15u) == 0 &&
            (reinterpret_cast<uintptr_t>(stage) & 15u) == 0) {
            const int n4 = (N * E) / 4;
            const float4 *src = reinterpret_cast<const float4 *>(Lg);
            float4 *dst = reinterpret_cast<float4 *>(stage);
            for (int i = tid; i < n4; i += kThreads) dst[i] = __ldg(src + i);
            for (int i = n4 * 4 + tid; i < N * E; i += kThreads) stage[i] = __ldg(Lg + i);
        } else {
            for (int i = tid; i < N * E; i += kThreads) stage[i] = __ldg(Lg + i);
        }
    }
    for (int e = tid; e < kMaxE; e += kThreads) {
        inU[e] = 0;
        inSel[e] = 0;
        inA[e] = 0;
    }
    if (tid == 0) s_range = 0;
    __syncthreads();
    const float *L = staged ? stage : Lg;

    // ---- phase A: natural top-k, natural union, softmax max / normaliser, logit range ----
    for (int n = warp; n < N; n += kWarps) {
        float v[kVPL];
        load_row(L + (size_t)n * E, E, v);
        const int t = warp_topk(v, 0xffffffffu, E, k);
        const float val = chosen_value(v, t);
        if (lane < k && t >= 0) inU[t] = 1;
        if (n == 0 && lane < k) natRoot[lane] = t;
        if (lane < k) nat[n * k + lane] = t;
        const float m = __shfl_sync(0xffffffffu, val, 0);  // the top-1 logit
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kVPL; ++i)
            if (lane + 32 * i < E) s += expf(v[i] - m);
        s = warp_sum(s);
        const float range = node_range(v, E, m);
        if (lane == 0) {
            mx[n] = m;
            nz[n] = s;
            cN[n] = commitment(a, dep[n]);
            atomicMax(&s_range, __float_as_int(range));
        }
    }
    __syncthreads();

    // ---- demand: D_e = sum over nodes (ascending) of c_n * exp(l_ne - max_n) / sum_n ----
    if (staged) {
        // all N*E terms in parallel, then a thread per expert adds its column in order
        float *wt = reinterpret_cast<float *>(nat + N * k);  // [N][E]
        for (int i = tid; i < N * E; i += kThreads) {
            const int n = i / E;
            wt[i] = __fmul_rn(cN[n], __fdiv_rn(expf(L[i] - mx[n]), nz[n]));
        }
        __syncthreads();
        for (int e = tid; e < E; e += kThreads) {
            float acc = 0.f;
#pragma unroll 8
            for (int n = 0; n < N; ++n) acc = __fadd_rn(acc, wt[(size_t)n * E + e]);
            D[e] = acc;
        }
    } else {
        for (int e = tid; e < E; e += kThreads) {
            float acc = 0.f;
#pragma unroll 4
            for (int n = 0; n < N; ++n) {
                const float ex = expf(L[(size_t)n * E + e] - mx[n]);
                acc = __fadd_rn(acc, __fmul_rn(cN[n], __fdiv_rn(ex, nz[n])));
            }
            D[e] = acc;
        }
    }
    if (a.anchor && tid < k) inA[natRoot[tid]] = 1;
    __syncthreads();

    // ---- phase B: size, anchor + fill, prune; fp32 with its certificate, else fp64 ----
    const float A = __int_as_float(s_range);
    PhaseB pb = phase_b<float, kWarps>(a, E, k, D, inU, inA, inS, resident,
                                       reinterpret_cast<float *>(rkb),
                                       reinterpret_cast<float(*)[kWarps]>(&redb[0][0]),
                                       reinterpret_cast<float *>(cutb),
                                       demand_bound(A, N, kVPL), demand_floor(a, N));
    const bool exact_pass = !pb.sure || !isfinite(A);
    if (exact_pass) {
        // fp64 normaliser of every node, then a thread per expert adds its terms in order
        for (int n = warp; n < N; n += kWarps) {
            double s = 0.0;
#pragma unroll
            for (int i = 0; i < kVPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E) s = __dadd_rn(s, exp((double)L[(size_t)n * E + e] - (double)mx[n]));
            }
            s = warp_sum64(s);
            if (lane == 0) nz64[n] = s;
        }
        __syncthreads();
        for (int n = warp; n < N; n += kWarps)  // c_n / sum_n once per node
            if (lane == 0) nz64[n] = __ddiv_rn(commitment64(a, dep[n]), nz64[n]);
        __syncthreads();
        for (int e = tid; e < E; e += kThreads) {
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                const double ex = exp((double)L[(size_t)n * E + e] - (double)mx[n]);
                acc = __dadd_rn(acc, __dmul_rn(nz64[n], ex));
            }
            D64[e] = acc;
        }
        __syncthreads();
        pb = phase_b_exact<kWarps>(a, E, k, D64, inU, inA, inS, resident, rkb, redb, cutb);
    }
    const int m = pb.m, removed = pb.removed;

    // ---- phase C: restricted top-k and gates ----
    unsigned allowed = 0;
#pragma unroll
    for (int i = 0; i < kVPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && inS[e]) allowed |= 1u << i;
    }
    for (int n = warp; n < N; n += kWarps) {
        float v[kVPL];
        load_row(L + (size_t)n * E, E, v);
        const int nt = lane < k ? nat[n * k + lane] : -1;
        const bool keep = __all_sync(0xffffffffu, lane >= k || (nt >= 0 && inS[nt]));
        const int t = keep ? nt : warp_topk(v, allowed, E, k);
        const float val = chosen_value(v, t);
        if (lane < k && t >= 0) inSel[t] = 1;
        write_choice(t, val, k, idxb + (size_t)n * k, gb + (size_t)n * k);
    }
    const int u_nat = __syncthreads_count(tid < E && inU[tid]);
    const int u_sel = __syncthreads_count(tid < E && inSel[tid]);
    if (tid == 0 && info_out) {
        info_out[b * MOE_INFO_FIELDS + 0] = u_nat;
        info_out[b * MOE_INFO_FIELDS + 1] = u_sel;
        info_out[b * MOE_INFO_FIELDS + 2] = m;
        info_out[b * MOE_INFO_FIELDS + 3] = removed;
        info_out[b * MOE_INFO_FIELDS + 4] = exact_pass ? 1 : 0;
    }
    if (elig_out)
        for (int e = tid; e < E; e += kThreads) elig_out[(size_t)b * E + e] = (uint8_t)inS[e];
}

// ---------------------------------------------------------------------------
// Cluster variant: one cluster of kCC CTAs (kCW warps each) per tree, for trees of up to
// kClusterMaxN nodes. Node n belongs to global warp g = n mod (kCC*kCW), i.e. CTA
// g / kCW, warp g mod kCW, local slot (n / (kCC*kCW)) * kCW + warp. Each CTA takes its
// nodes' natural top-k and softmax terms, adds the terms of its nodes per expert in node
// order, and stores the partial demand and the natural choices into CTA 0's shared memory
// (distributed shared memory). CTA 0 adds the partials in CTA order and runs the size /
// anchor / fill / prune phase, with sum D and H as block reductions and the ranks counted
// by two or four threads per expert; meanwhile the other CTAs write their nodes' natural
// routing, which stands for every node whose natural top-k lies in the eligible set. Every
// CTA then reads the eligible set back and re-routes the nodes that need it. When CTA 0's
// fp32 phase B cannot certify its decisions, every CTA adds its nodes' fp64 demand terms
// (from the logit rows it holds in shared memory), CTA 0 adds the partials in CTA order
// and runs phase B again in fp64, before the re-routing.
namespace cg = cooperative_groups;
constexpr int kCC = 8;                  // CTAs per tree
constexpr int kCW = 16;                 // warps per CTA
constexpr int kCThreads = kCW * 32;
constexpr int kClusterMaxN = 256;
static_assert(kCThreads >= 2 * kMaxE, "phase B takes at least two threads per expert");

// Cluster barrier whose arrival releases this thread's earlier writes to the cluster only
// when `release` (uniform over the CTA); the wait always acquires. A CTA whose writes no
// other CTA reads next need not wait for them (global stores in flight) before arriving.
__device__ __forceinline__ void cluster_barrier(bool release) {
    if (release)
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    else
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The permute step for a block of one tree, on CTA 0 of the selection cluster ("MoE and
// speculative decoding" blog, pipeline step "permute / group by expert"), with the same
// results as the permute kernel: a stable counting sort of the assignments (n, j) by
// (expert, node, slot). rmask[e] holds the nodes that chose e (a node chooses an expert
// at most once, so within an expert the order is node order) and fin_all[n][j] the choices.
// Writes counts, offsets, the active-expert list, the row tiles (split and sized as the
// permute kernel splits and sizes them), perm and pos, and starts the
// call's check word (keeping router_word, the router's, read by thread 0 long before).
__device__ void permute_tree(const PermuteOut &po, const int *fin_all,
                             const uint32_t (*rmask)[kClusterMaxN / 32], int *soff,
                             int (*wsc)[kCW], int N, int E, int k, int router_word) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nbw = (N + 31) >> 5;
    const int A = N * k;
    if (tid == 0) {
        po.flags[0] = po.after_router ? router_word : 0;
        po.flags[kRouterCheckWord] = 0;
    } else if (tid < 64 && tid != kRouterCheckWord) {
        po.flags[tid] = 0;
    }
    int c = 0;
    if (tid < E)
        for (int q = 0; q < nbw; ++q) c += __popc(rmask[tid][q]);
    const int nw = (E + 31) >> 5;
    if (warp < nw) {
        const int wm = __reduce_max_sync(0xffffffffu, c);
        if (lane == 0) wsc[3][warp] = wm;
    }
    __syncthreads();
    int cmax = 0;
    for (int w = 0; w < nw; ++w) cmax = max(cmax, wsc[3][w]);
    // as in the permute kernel: ceil(c / limit) tiles of near-equal size, the height the
    // largest tile of any expert rounded up to 16 (an expert of limit tokens can have a
    // larger tile than one of more)
    const int lim = rowtile_limit(cmax);
    const int act = c > 0, nt = (c + lim - 1) / lim;
    const int tmax = nt > 0 ? (c + nt - 1) / nt : 0;
    if (warp < nw) {
        const int wm = __reduce_max_sync(0xffffffffu, tmax);
        if (lane == 0) wsc[2][warp] = wm;
    }
    __syncthreads();
    int hmax = 0;
    for (int w = 0; w < nw; ++w) hmax = max(hmax, wsc[2][w]);
    const int rt_size = min(lim, max(16, (hmax + 15) & ~15));
    int ci = c, ai = act, ti = nt;  // inclusive scans within the warp
    if (warp < nw) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int c2 = __shfl_up_sync(0xffffffffu, ci, o);
            const int a2 = __shfl_up_sync(0xffffffffu, ai, o);
            const int t2 = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) {
                ci += c2;
                ai += a2;
                ti += t2;
            }
        }
        if (lane == 31) {  // wsc[2] may still be read above: the tile totals go to wsc[3]
            wsc[0][warp] = ci;
            wsc[1][warp] = ai;
            wsc[3][warp] = ti;
        }
    }
    __syncthreads();
    if (tid < E) {
        for (int w = 0; w < warp; ++w) {
            ci += wsc[0][w];
            ai += wsc[1][w];
            ti += wsc[3][w];
        }
        const int c_ex = ci - c;
        int t_ex = ti - nt;
        soff[tid] = c_ex;
        po.counts[tid] = c;
        po.offsets[tid] = c_ex;
        if (act) po.active[1 + ai - act] = tid;
        for (int j = 0, n0 = 0; j < nt; ++j) {
            const int sz = c / nt + (j < c % nt ? 1 : 0);
            int *t = po.rowtiles + kRowTileHeader + 4 * t_ex++;
            t[0] = tid;
            t[1] = c_ex + n0;  // first permuted row of the tile
            t[2] = sz;
            t[3] = rowtile_group(j, nt);
            n0 += sz;
        }
        if (tid == E - 1) {
            soff[E] = ci;
            po.offsets[E] = ci;
            po.active[0] = ai;
            po.rowtiles[0] = ti;
            po.rowtiles[1] = rt_size;
        }
    }
    __syncthreads();
    for (int a = tid; a < A; a += kCThreads) {
        const int e = fin_all[a];
        if (e < 0 || e >= E) {  // cannot happen for a selection of k distinct experts
            po.pos[a] = -1;
            atomicOr(po.flags, FLAG_BAD_EXPERT);
            continue;
        }
        const int n = a / k, q1 = n >> 5;
        int pre = __popc(rmask[e][q1] & ((1u << (n & 31)) - 1u));
        for (int q = 0; q < q1; ++q) pre += __popc(rmask[e][q]);
        const int p = soff[e] + pre;
        po.perm[p] = a;
        po.pos[a] = p;
    }
    for (int p = soff[E] + tid; p < A; p += kCThreads) po.perm[p] = -1;
}

// The fp64 demand terms of one CTA's nodes in the cluster kernel (the fp64 pass, out of
// line): a warp per node takes exp(l - max) in fp64 from the logit rows the CTA holds, the
// node's sum, and c_n / sum_n once per node (one fp64 divide instead of one per expert;
// the product differs from c_n * (ex / sum_n) by an fp64 rounding); then a thread per
// expert adds the CTA's nodes in node order and stores the partial into part0[rank][e]
// (CTA 0's shared memory).
template <int VPL>
__device__ __noinline__ void cluster_exact_terms(const SelectArgs &a, const int *dep, int N,
                                                 int E, int k, int rank, const float *lrow,
                                                 const float *nat_val, double *w64,
                                                 double *part0) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int n = rank * kCW + warp, t = 0; n < N; n += kCC * kCW, ++t) {
        const int slot = t * kCW + warp;
        const double top = (double)nat_val[slot * k];  // the node's largest logit
        const double cn = commitment64(a, dep[n]);
        double ex[VPL], s = 0.0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            ex[i] = e < E ? exp((double)lrow[slot * E + e] - top) : 0.0;
            s = __dadd_rn(s, ex[i]);
        }
        s = warp_sum64(s);
        const double scale = __ddiv_rn(cn, s);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) w64[slot * E + e] = __dmul_rn(scale, ex[i]);
        }
    }
    __syncthreads();
    if (tid < E) {
        double acc = 0.0;
        for (int t = 0; t * kCC * kCW < N; ++t) {
            const int cnt = min(kCW, max(0, N - t * kCC * kCW - rank * kCW));
            for (int w = 0; w < cnt; ++w) acc = __dadd_rn(acc, w64[(size_t)(t * kCW + w) * E + tid]);
        }
        part0[rank * kMaxE + tid] = acc;
    }
}

template <int VPL>
__global__ void __cluster_dims__(kCC, 1, 1) __launch_bounds__(kCThreads, 1)
select_cluster_kernel(SelectArgs a, const float *__restrict__ logits,
                      const int *__restrict__ depth, int N, int E, int k,
                      const uint8_t *__restrict__ resident, int *__restrict__ idx_out,
                      float *__restrict__ gates_out, uint8_t *__restrict__ elig_out,
                      int *__restrict__ info_out, WeightPrefetch pf, PermuteOut po) {
    // the last pf.ctas CTAs (whole clusters of their own) only prefetch
    if ((int)blockIdx.x >= (int)gridDim.x - pf.ctas) {
        prefetch_root_experts(pf, logits, E, k, (int)blockIdx.x - ((int)gridDim.x - pf.ctas));
        return;
    }
    // w64 [slots][E] (fp64 demand terms, the fp64 pass), wt [slots][E], lrow [slots][E]
    // (this CTA's logit rows), nat_all [N][k] (CTA 0), nat_loc [slots][k], nat_val
    // [slots][k] (their logits), fin_all [N][k] (CTA 0: the final choices, for the permute
    // step)
    extern __shared__ double cdyn64[];
    __shared__ float part[kCC][kMaxE];    // CTA 0: partial demand of every CTA
    __shared__ double part64[kCC][kMaxE]; // CTA 0: the same in fp64 (the fp64 pass)
    __shared__ float rangeAll[kCC];       // CTA 0: largest node logit range of every CTA
    __shared__ int selAll[kCC][kMaxE];    // CTA 0: experts chosen by every CTA's nodes
    __shared__ float D[kMaxE];
    __shared__ double D64[kMaxE], rkb[kMaxE], redb[2][kCW], cutb[4];
    __shared__ int inU[kMaxE], inS[kMaxE], inA[kMaxE], inSel[kMaxE];
    __shared__ int s_m, s_removed, s_exact;
    __shared__ float wrange[kCW];  // largest node logit range of each warp
    // CTA 0, permute step: bit n of rmask[e][n / 32] = node n chose e; offsets per expert
    __shared__ uint32_t rmask[kMaxE][kClusterMaxN / 32];
    __shared__ int soff[kMaxE + 1];
    __shared__ int wsc[4][kCW];

    // every CTA of the cluster must be running before any touches another's shared
    // memory: arrive now, wait just before the first remote store
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / kCC;
    const int slots = ((N + kCC * kCW - 1) / (kCC * kCW)) * kCW;
    double *w64 = cdyn64;
    float *wt = reinterpret_cast<float *>(w64 + (size_t)slots * E);
    float *lrow = wt + (size_t)slots * E;
    int *nat_all = reinterpret_cast<int *>(lrow + (size_t)slots * E);
    int *nat_loc = nat_all + (size_t)N * k;
    float *nat_val = reinterpret_cast<float *>(nat_loc + (size_t)slots * k);
    int *fin_all = reinterpret_cast<int *>(nat_val + (size_t)slots * k);
    int *nat0 = cl.map_shared_rank(nat_all, 0);
    const bool fuse = po.counts != nullptr;
    // the router's check word, used at the very end (its load latency is hidden)
    const int router_word = (fuse && rank == 0 && tid == 0) ? po.flags[kRouterCheckWord] : 0;
    const float *Lg = logits + (size_t)b * N * E;
    const int *dep = depth + (size_t)b * N;
    int *idxb = idx_out + (size_t)b * N * k;
    float *gb = gates_out + (size_t)b * N * k;

    for (int e = tid; e < kMaxE; e += kCThreads) {
        inU[e] = 0;
        inSel[e] = 0;
        inA[e] = 0;
    }
    if (fuse)
        for (int i = tid; i < kMaxE * (kClusterMaxN / 32); i += kCThreads) (&rmask[0][0])[i] = 0u;
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    // ---- phase A: this CTA's nodes ----
    float my_range = 0.f;  // uniform over the warp
    for (int n = rank * kCW + warp, t = 0; n < N; n += kCC * kCW, ++t) {
        const int slot = t * kCW + warp;
        const int dn = dep[n];  // in flight with the logits
        float v[VPL];
        load_row(Lg + (size_t)n * E, E, v);
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (lane + 32 * i < E) lrow[slot * E + lane + 32 * i] = v[i];
        const int c = warp_topk(v, 0xffffffffu, E, k);
        const float val = chosen_value(v, c);
        if (lane < k) {
            nat_loc[slot * k + lane] = c;
            nat_val[slot * k + lane] = val;
            nat0[n * k + lane] = c;
        }
        const float m = __shfl_sync(0xffffffffu, val, 0);
        float ex[VPL], s = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            ex[i] = lane + 32 * i < E ? expf(v[i] - m) : 0.f;
            s += ex[i];
        }
        s = warp_sum(s);
        const float cn = commitment(a, dn);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) wt[slot * E + e] = __fmul_rn(cn, __fdiv_rn(ex[i], s));
        }
        my_range = fmaxf(my_range, node_range(v, E, m));
    }
    if (lane == 0) wrange[warp] = my_range;
    __syncthreads();
    if (tid == 0) {
        float A = 0.f;
        for (int w = 0; w < kCW; ++w) A = fmaxf(A, wrange[w]);
        cl.map_shared_rank(rangeAll, 0)[rank] = A;
    }
    if (tid < E) {  // partial demand of this CTA's nodes, node order
        float acc = 0.f;
        for (int t = 0; t * kCC * kCW < N; ++t) {
            const int cnt = min(kCW, max(0, N - t * kCC * kCW - rank * kCW));
            const float *w0 = wt + (size_t)t * kCW * E + tid;
            if (cnt == kCW) {
#pragma unroll
                for (int w = 0; w < kCW; ++w) acc = __fadd_rn(acc, w0[(size_t)w * E]);
            } else {
                for (int w = 0; w < cnt; ++w) acc = __fadd_rn(acc, w0[(size_t)w * E]);
            }
        }
        cl.map_shared_rank(&part[0][0], 0)[rank * kMaxE + tid] = acc;
    }
    cl.sync();

    // ---- phase B on CTA 0; the other CTAs write their nodes' natural routing, which
    // stands unless phase C re-routes the node ----
    if (rank == 0) {
        for (int i = tid; i < N * k; i += kCThreads) inU[nat_all[i]] = 1;
        if (tid < E) {
            float De = 0.f;
            for (int r = 0; r < kCC; ++r) De = __fadd_rn(De, part[r][tid]);
            D[tid] = De;
        }
        if (a.anchor && tid < k) inA[nat_all[tid]] = 1;
        float A = 0.f;
        for (int r = 0; r < kCC; ++r) A = fmaxf(A, rangeAll[r]);
        __syncthreads();
        const PhaseB pb = phase_b<float, kCW>(a, E, k, D, inU, inA, inS, resident,
                                              reinterpret_cast<float *>(rkb),
                                              reinterpret_cast<float(*)[kCW]>(&redb[0][0]),
                                              reinterpret_cast<float *>(cutb),
                                              demand_bound(A, N, VPL), demand_floor(a, N));
        if (tid == 0) {
            s_m = pb.m;
            s_removed = pb.removed;
            s_exact = (!pb.sure || !isfinite(A)) ? 1 : 0;
        }
    } else {
        for (int n = rank * kCW + warp, t = 0; n < N; n += kCC * kCW, ++t) {
            const int slot = t * kCW + warp;
            write_choice(lane < k ? nat_loc[slot * k + lane] : -1,
                         lane < k ? nat_val[slot * k + lane] : -INFINITY, k,
                         idxb + (size_t)n * k, gb + (size_t)n * k);
        }
    }
    // only CTA 0's writes (the eligible set, the verdict) must be visible past this
    // barrier: the other CTAs arrive without waiting for their global stores
    cluster_barrier(rank == 0);

    // ---- the fp64 pass, when CTA 0 could not certify the fp32 decisions (uniform over
    // the cluster). The other CTAs read CTA 0's verdict and eligible set together (one
    // round trip); after an fp64 pass they read the set again. ----
    int exact_pass = s_exact;
    if (rank != 0) {
        const int *inS0 = cl.map_shared_rank(inS, 0);
        if (tid < E) inS[tid] = inS0[tid];
        exact_pass = *cl.map_shared_rank(&s_exact, 0);
    }
    if (exact_pass) {
        cluster_exact_terms<VPL>(a, dep, N, E, k, rank, lrow, nat_val, w64,
                                 cl.map_shared_rank(&part64[0][0], 0));
        cluster_barrier(true);
        if (rank == 0) {
            if (tid < E) {
                double De = 0.0;
                for (int r = 0; r < kCC; ++r) De = __dadd_rn(De, part64[r][tid]);
                D64[tid] = De;
            }
            __syncthreads();
            const PhaseB pb =
                phase_b_exact<kCW>(a, E, k, D64, inU, inA, inS, resident, rkb, redb, cutb);
            if (tid == 0) {
                s_m = pb.m;
                s_removed = pb.removed;
            }
        }
        cluster_barrier(rank == 0);
        if (rank != 0 && tid < E) inS[tid] = cl.map_shared_rank(inS, 0)[tid];
    }

    // ---- phase C: this CTA's nodes, restricted to the eligible set ----
    if (rank == 0) {  // the set's size and the block's eligibility mask
        if (tid == 0 && info_out) {
            info_out[b * MOE_INFO_FIELDS + 2] = s_m;
            info_out[b * MOE_INFO_FIELDS + 3] = s_removed;
            info_out[b * MOE_INFO_FIELDS + 4] = exact_pass;
        }
        if (elig_out && tid < E) elig_out[(size_t)b * E + tid] = (uint8_t)inS[tid];
    }
    __syncthreads();
    unsigned allowed = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && inS[e]) allowed |= 1u << i;
    }
    int *fin0 = cl.map_shared_rank(fin_all, 0);
    uint32_t *rm0 = cl.map_shared_rank(&rmask[0][0], 0);
    for (int n = rank * kCW + warp, t = 0; n < N; n += kCC * kCW, ++t) {
        const int slot = t * kCW + warp;
        const int nt = lane < k ? nat_loc[slot * k + lane] : -1;
        const bool keep = __all_sync(0xffffffffu, lane >= k || (nt >= 0 && inS[nt]));
        int c = nt;
        if (keep) {  // the natural routing stands (CTAs other than 0 wrote it already)
            if (rank == 0)
                write_choice(nt, lane < k ? nat_val[slot * k + lane] : -INFINITY, k,
                             idxb + (size_t)n * k, gb + (size_t)n * k);
        } else {
            float v[VPL];
            load_row(lrow + (size_t)slot * E, E, v);
            c = warp_topk(v, allowed, E, k);
            write_choice(c, chosen_value(v, c), k, idxb + (size_t)n * k, gb + (size_t)n * k);
        }
        if (lane < k) {
            if (c >= 0) inSel[c] = 1;
            if (fuse) {  // into CTA 0's shared memory, for the permute step
                fin0[n * k + lane] = c;
                if (c >= 0) atomicOr(rm0 + c * (kClusterMaxN / 32) + (n >> 5), 1u << (n & 31));
            }
        }
    }
    __syncthreads();
    if (!fuse && tid < E) cl.map_shared_rank(&selAll[0][0], 0)[rank * kMaxE + tid] = inSel[tid];
    // the other CTAs' writes into CTA 0's shared memory must be visible to CTA 0 past this
    // barrier; CTA 0 arrives without waiting for its global stores. After it CTA 0 reads
    // only its own shared memory.
    cluster_barrier(rank != 0);
    if (rank == 0) {
        int sel = 0;
        if (tid < E) {
            if (fuse)  // the node masks of the permute step hold the union too
                for (int q = 0; q < kClusterMaxN / 32; ++q) sel |= rmask[tid][q] != 0u;
            else
                for (int r = 0; r < kCC; ++r) sel |= selAll[r][tid];
        }
        const int u_sel = __syncthreads_count(sel);
        const int u_nat = __syncthreads_count(tid < E && inU[tid]);
        if (tid == 0 && info_out) {
            info_out[b * MOE_INFO_FIELDS + 0] = u_nat;
            info_out[b * MOE_INFO_FIELDS + 1] = u_sel;
        }
        if (fuse) permute_tree(po, fin_all, rmask, soff, wsc, N, E, k, router_word);
    }
}

// Raises a kernel's dynamic shared-memory limit to `bytes` when it is above the largest
// limit set so far (static + dynamic shared memory may not exceed 48 KB without it).
template <typename K>
cudaError_t allow_smem(K kernel, std::atomic<size_t> &set, size_t bytes) {
    size_t cur = set.load();
    if (bytes <= cur) return cudaSuccess;
    const cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess)
        while (cur < bytes && !set.compare_exchange_weak(cur, bytes)) {
        }
    return err;
}
std::atomic<size_t> cluster4_smem_set{0}, cluster8_smem_set{0}, single_smem_set{0};

}  // namespace

// ---------------------------------------------------------------------------
// Natural routing (every expert eligible): each node's top-k and renormalised gates are
// independent of the other nodes, so a tree of any size runs on one cluster of kNC CTAs
// of kNW warps, a warp per node (node n on global warp n mod (kNC*kNW)). The only
// per-tree quantity is the natural union |U|: each CTA marks its nodes' experts in a bit
// set, ORs it into CTA 0's bit set through distributed shared memory, and CTA 0 counts
// the bits after the cluster barrier.
constexpr int kNC = 8;    // CTAs per tree
constexpr int kNW = 16;   // warps per CTA
constexpr int kNWords = kMaxE / 32;

__global__ void __cluster_dims__(kNC, 1, 1) __launch_bounds__(kNW * 32, 1)
select_natural_kernel(const float *__restrict__ logits, int N, int E, int k,
                      int *__restrict__ idx_out, float *__restrict__ gates_out,
                      uint8_t *__restrict__ elig_out, int *__restrict__ info_out,
                      PermuteOut po) {
    static_assert(kNW == kCW, "the permute step assumes the selection kernels' block size");
    extern __shared__ int nfin[];  // CTA 0, permute step: the choices [N][k]
    __shared__ uint32_t mask[kNWords];
    // CTA 0, permute step: bit n of rmask[e][n / 32] = node n chose e; offsets per expert
    __shared__ uint32_t rmask[kMaxE][kClusterMaxN / 32];
    __shared__ int soff[kMaxE + 1];
    __shared__ int wsc[4][kCW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool fuse = po.counts != nullptr;
    if (tid < kNWords) mask[tid] = 0u;
    if (fuse)
        for (int i = tid; i < kMaxE * (kClusterMaxN / 32); i += kNW * 32) (&rmask[0][0])[i] = 0u;
    // CTA 0's bit sets must be cleared before any CTA ORs into them: the arrive releases
    // the clearing stores, the wait before the first remote update acquires them
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    pdl_wait();
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int b = blockIdx.x / kNC;
    const float *Lg = logits + (size_t)b * N * E;
    int *idxb = idx_out + (size_t)b * N * k;
    float *gb = gates_out + (size_t)b * N * k;
    int *fin0 = cl.map_shared_rank(nfin, 0);
    uint32_t *rm0 = cl.map_shared_rank(&rmask[0][0], 0);
    // the router's check word, used at the very end (its load latency is hidden)
    const int router_word = (fuse && rank == 0 && tid == 0) ? po.flags[kRouterCheckWord] : 0;
    __syncthreads();  // the local bit set is clear
    if (fuse) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    for (int n = rank * kNW + warp; n < N; n += kNC * kNW) {
        float v[kVPL];
        load_row(Lg + (size_t)n * E, E, v);
        const int c = warp_topk(v, 0xffffffffu, E, k);
        const float val = chosen_value(v, c);
        write_choice(c, val, k, idxb + (size_t)n * k, gb + (size_t)n * k);
        if (lane < k && c >= 0) atomicOr(&mask[c >> 5], 1u << (c & 31));
        if (fuse && lane < k) {  // into CTA 0's shared memory, for the permute step
            fin0[n * k + lane] = c;
            if (c >= 0) atomicOr(rm0 + c * (kClusterMaxN / 32) + (n >> 5), 1u << (n & 31));
        }
    }
    __syncthreads();
    if (!fuse) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (tid < kNWords && mask[tid]) atomicOr(cl.map_shared_rank(&mask[tid], 0), mask[tid]);
    cl.sync();
    if (rank == 0) {
        if (tid == 0 && info_out) {
            int u = 0;
            for (int w = 0; w < kNWords; ++w) u += __popc(mask[w]);
            info_out[b * MOE_INFO_FIELDS + 0] = u;
            info_out[b * MOE_INFO_FIELDS + 1] = u;
            info_out[b * MOE_INFO_FIELDS + 2] = E;
            info_out[b * MOE_INFO_FIELDS + 3] = 0;
            info_out[b * MOE_INFO_FIELDS + 4] = 0;
        }
        if (elig_out)
            for (int e = tid; e < E; e += kNW * 32) elig_out[(size_t)b * E + e] = 1;
        if (fuse) permute_tree(po, nfin, rmask, soff, wsc, N, E, k, router_word);
    }
}

namespace {

// Clusters of 8 CTAs of `kernel` (with `smem` bytes of dynamic shared memory) that the
// device runs at once; 0 if the query fails. Cached per (kernel, shared memory, device).
template <typename K>
int active_clusters(K kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, size_t, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(reinterpret_cast<const void *>(kernel), smem, dev);
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(8);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 8;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[key] = n;
    return n;
}

// Prefetch CTAs for a launch whose selection takes `used` of the `avail` concurrent
// slots (clusters, or CTAs of the one-CTA kernel): at most kPfMaxCtas, whole clusters of 8,
// and only in slots the selection leaves free, so the prefetch never waits for a second
// wave. Measured on GB300 (65-node trees, Qwen3-30B-A3B-shaped layer): 64 CTAs made the
// layer 0.9% (router std 0.02) and 1.3% (std 0.1) faster; 128 CTAs, or 4 experts instead
// of the root's 8, gained less: the prefetch traffic also lengthens the memory latency
// of the routing kernels it overlaps.
constexpr int kPfMaxCtas = 64;
WeightPrefetch sized(WeightPrefetch pf, int used, int avail, int per_slot) {
    const int free_ctas = (avail - used) * per_slot;
    pf.ctas = std::max(0, std::min(kPfMaxCtas, free_ctas) / 8 * 8);
    return pf;
}

// Dynamic shared memory of the cluster kernel for N-node trees: w64 [slots][E] doubles; wt
// and lrow [slots][E]; nat_all and fin_all [N][k]; nat_loc and nat_val [slots][k].
size_t cluster_smem(const moe_layer_desc &L, int N) {
    const int slots = ((N + kCC * kCW - 1) / (kCC * kCW)) * kCW;
    return (size_t)slots * L.E * sizeof(double) +
        ((size_t)2 * slots * L.E + (size_t)2 * N * L.k + (size_t)2 * slots * L.k) * sizeof(float);
}

// Whether B clusters of the kernel for this layer run in at most three waves. The kernel's
// shared-memory limit is raised first, so the occupancy query sees the launch as it will be.
bool clusters_in_three_waves(const moe_layer_desc &L, int B, int N) {
    const size_t smem = cluster_smem(L, N);
    if (L.E <= 128)
        return allow_smem(select_cluster_kernel<4>, cluster4_smem_set, smem) == cudaSuccess &&
               B <= 3 * active_clusters(select_cluster_kernel<4>, kCThreads, smem);
    return allow_smem(select_cluster_kernel<8>, cluster8_smem_set, smem) == cudaSuccess &&
           B <= 3 * active_clusters(select_cluster_kernel<8>, kCThreads, smem);
}

// One 8-CTA cluster per tree (+ the prefetch CTAs), VPL logits per lane (E <= 32 VPL).
template <int VPL>
cudaError_t launch_cluster(const moe_layer_desc &L, const SelectArgs &a, const float *logits,
                           const int *depth, int B, int N, const uint8_t *resident, int *idx,
                           float *gates, uint8_t *elig, int *info, WeightPrefetch pf,
                           PermuteOut po, std::atomic<size_t> &smem_set, cudaStream_t s) {
    const size_t smem = cluster_smem(L, N);
    cudaError_t err = allow_smem(select_cluster_kernel<VPL>, smem_set, smem);
    if (err != cudaSuccess) return err;
    if (pf.ctas > 0)
        pf = sized(pf, B, active_clusters(select_cluster_kernel<VPL>, kCThreads, smem), 8);
    return launch_pdl(select_cluster_kernel<VPL>, dim3(B * kCC + pf.ctas), dim3(kCThreads), smem,
                      s, a, logits, depth, N, L.E, L.k, resident, idx, gates, elig, info, pf, po);
}

}  // namespace

WeightPrefetch weight_prefetch(const moe_layer_desc &L, int B, const void *W_gate,
                               const void *W_up, const void *W_down, const int *slot_of_expert) {
    WeightPrefetch pf{};
    const unsigned long long esz = L.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    const unsigned long long bytes = (unsigned long long)L.f * L.d * esz;
    if (!W_gate || !W_up || !W_down || bytes % 16 != 0 || B < 1) return pf;
    pf.wg = static_cast<const char *>(W_gate);
    pf.wu = static_cast<const char *>(W_up);
    pf.wd = static_cast<const char *>(W_down);
    pf.slot_of_expert = slot_of_expert;
    pf.slots = L.slots > 0 ? L.slots : L.E;
    pf.bytes = bytes;
    pf.ctas = kPfMaxCtas;  // launch_select trims it to the SMs the selection leaves free
    return pf;
}

cudaError_t launch_select(const moe_layer_desc &L, const SelectArgs &a, const float *logits,
                          const int *depth, int B, int N, const uint8_t *resident, int *idx,
                          float *gates, uint8_t *elig, int *info, const WeightPrefetch &pf_in,
                          const PermuteOut &po_in, bool *permuted, cudaStream_t s) {
    if (permuted) *permuted = false;
    if (B <= 0 || N <= 0) return cudaSuccess;
    WeightPrefetch pf = pf_in;
    // Natural routing: no prefetch. Its selection is short (a few microseconds), so the
    // prefetch CTAs would outlast it and delay the chain; measured on GB300 the layer was
    // 1% slower with them.
    if (a.mode == MOE_ROUTE_NATURAL) {
        // a block of one tree of up to kClusterMaxN nodes: the cluster also permutes
        const PermuteOut po =
            (B == 1 && N <= kClusterMaxN && po_in.counts) ? po_in : PermuteOut{};
        const size_t smem = po.counts ? (size_t)N * L.k * sizeof(int) : 0;
        const cudaError_t err = launch_pdl(select_natural_kernel, dim3(B * kNC), dim3(kNW * 32),
                                           smem, s, logits, N, L.E, L.k, idx, gates, elig, info,
                                           po);
        if (err == cudaSuccess && permuted) *permuted = po.counts != nullptr;
        return err;
    }
    // trees of up to kClusterMaxN nodes take a cluster each while the clusters run in at
    // most three waves; more trees than that take the one-CTA kernel, one CTA per tree in
    // one wave. Measured on GB300 (65-node trees, Qwen3-30B-A3B-shaped layer): at 48 and 64
    // trees per block (more than three waves of clusters) the one-CTA kernel made the block
    // 1.2% and 2.5% faster, at 16-32 trees (one to three waves) up to 2.4% slower.
    if (N <= kClusterMaxN && (B == 1 || clusters_in_three_waves(L, B, N))) {
        // a block of one tree: the cluster also performs the permute step
        const PermuteOut po = (B == 1 && po_in.counts) ? po_in : PermuteOut{};
        const cudaError_t err =
            L.E <= 128 ? launch_cluster<4>(L, a, logits, depth, B, N, resident, idx, gates, elig,
                                           info, pf, po, cluster4_smem_set, s)
                       : launch_cluster<8>(L, a, logits, depth, B, N, resident, idx, gates, elig,
                                           info, pf, po, cluster8_smem_set, s);
        if (err == cudaSuccess && permuted) *permuted = po.counts != nullptr;
        return err;
    }
    const bool staged = N * L.E <= kStageFloats;
    // nz64 [N] doubles; staged: logits and demand terms [N][E] each; always: mx, nz, cN [N]
    // and nat [N][k]
    const size_t smem = (size_t)N * sizeof(double) +
        ((staged ? 2 * (size_t)N * L.E : 0) + 3 * (size_t)N + (size_t)N * L.k) * sizeof(float);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    cudaError_t err = allow_smem(select_kernel, single_smem_set, smem);
    if (err != cudaSuccess) return err;
    if (pf.ctas > 0) {  // one CTA of this kernel per SM
        int dev = 0, nsm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            nsm = 0;
        pf = sized(pf, B, nsm, 1);
    }
    return launch_pdl(select_kernel, dim3(B + pf.ctas), dim3(kThreads), smem, s, a, logits, depth,
                      N, L.E, L.k, resident, idx, gates, elig, info, pf);
}

}  // namespace moe
