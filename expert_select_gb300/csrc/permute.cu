// Permute / group by expert ("MoE and speculative decoding" blog, pipeline step
// "permute / group by expert"): a stable counting sort of the assignments (r, j)
// by the key (expert, row, slot).
//
// A row picks each expert at most once, so inside one expert the key order is row
// order. One CTA builds, per block of 32 rows and per expert, the bitmask of rows
// that chose the expert; a scan over row blocks gives each (block, expert) its
// prefix; an assignment's position is then
//   offsets[e] + prefix[e][block] + popc(mask[e][block] & lanes_below(row)).
// The masks and prefixes live in shared memory: (R/32) x E x 8 bytes (133 KB at 4160
// rows and 128 experts). The same kernel also writes the active-expert list and the list
// of row tiles that the tensor-core expert kernel walks: an expert with c tokens takes
// ceil(c / 128) tiles of near-equal size (sizes differ by at most one) when no expert has
// more than 256 tokens, else ceil(c / 256), and the tile height is the largest tile
// rounded up to 16. Up to 2048 assignments it keeps the expert ids in shared memory and places the
// assignments itself; past that it leaves the masks and prefixes in the workspace and a
// second, many-CTA kernel places the assignments. Past 8192 assignments a many-CTA kernel
// also builds the masks beforehand (a CTA per row block), and the one CTA only loads them.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;

// The masks of a large block: CTA b takes row block b (32 rows, their 32 k assignments)
// and writes mask[e][b] for every expert e into gmask ([E][nb]).
constexpr int kMaskThreads = 256;

__global__ void __launch_bounds__(kMaskThreads)
permute_masks_kernel(const int *__restrict__ idx, int R, int k, int E,
                     uint32_t *__restrict__ gmask) {
    pdl_wait();
    __shared__ uint32_t m[kMaxE];
    const int nb = (R + 31) >> 5, b = blockIdx.x, tid = threadIdx.x;
    for (int e = tid; e < E; e += kMaskThreads) m[e] = 0u;
    __syncthreads();
    const int a0 = b * 32 * k, a1 = min(R, (b + 1) * 32) * k;
    for (int a = a0 + tid; a < a1; a += kMaskThreads) {
        const int e = idx[a];
        if (e < 0 || e >= E) continue;  // flagged where the assignments are placed
        atomicOr(&m[e], 1u << ((a / k) & 31));
    }
    __syncthreads();
    for (int e = tid; e < E; e += kMaskThreads) gmask[(size_t)e * nb + b] = m[e];
}

// kMode 0: the CTA builds the masks in shared memory. 1: permute_masks_kernel has built
// them in gmask and the CTA loads them into shared memory. 2: the same, but the [E][nb]
// masks and prefixes would not fit in shared memory: the CTA scans the masks in place and
// writes the prefixes beside them, keeping only the per-expert counts and offsets.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
permute_kernel(const int *__restrict__ idx, int R, int k, int E, int *__restrict__ counts,
               int *__restrict__ offsets, int *__restrict__ perm, int *__restrict__ pos,
               int *__restrict__ active, int *__restrict__ rowtiles, int *__restrict__ flags,
               uint32_t *__restrict__ gmask, int after_router) {
    pdl_wait();
    extern __shared__ uint32_t sm[];
    const int nb = (R + 31) >> 5;
    constexpr bool kMasksReady = kMode != 0, kInPlace = kMode == 2;
    uint32_t *mask = kInPlace ? gmask : sm;                              // [E][nb]
    uint32_t *pre = kInPlace ? gmask + (size_t)nb * E : sm + (size_t)nb * E;  // [E][nb]
    int *cnt = (int *)(kInPlace ? sm : pre + (size_t)nb * E);
    int *off = cnt + E;                   // [E + 1]
    int *sidx = off + E + 1;              // [A] the expert ids, when this CTA places them
    const int tid = threadIdx.x;
    const int A = R * k;

    // the first four expert ids of each thread are in flight while the masks are cleared
    // (or, when permute_masks_kernel built them in gmask, loaded)
    int ev0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        ev0[u] = !kMasksReady && tid + u * kThreads < A ? idx[tid + u * kThreads] : -1;
    if (!kInPlace)
        for (int i = tid; i < nb * E; i += kThreads) mask[i] = kMasksReady ? gmask[i] : 0u;
    if (tid == 0) {  // a fresh check word for this call, keeping what the router reported
        flags[0] = after_router ? flags[kRouterCheckWord] : 0;
        flags[kRouterCheckWord] = 0;
    } else if (tid < 64 && tid != kRouterCheckWord) {
        flags[tid] = 0;
    }
    __syncthreads();
    // four loads in flight per thread before their atomics
    for (int a0 = tid; !kMasksReady && a0 < A; a0 += 4 * kThreads) {
        int ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            ev[u] = a0 == tid ? ev0[u] : (a0 + u * kThreads < A ? idx[a0 + u * kThreads] : -1);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = ev[u];
            if (!gmask && a0 + u * kThreads < A) sidx[a0 + u * kThreads] = e;
            if (e < 0 || e >= E) continue;
            const int r = (a0 + u * kThreads) / k;
            atomicOr(&mask[e * nb + (r >> 5)], 1u << (r & 31));
        }
    }
    __syncthreads();
    if (nb <= 8) {  // few row blocks: a thread per expert
        for (int e = tid; e < E; e += kThreads) {
            int run = 0;
            for (int b = 0; b < nb; ++b) {
                pre[e * nb + b] = run;
                run += __popc(mask[e * nb + b]);
            }
            cnt[e] = run;
        }
    } else {  // per expert, a warp scans the row blocks' counts (exclusive prefix over blocks)
        const int lane = tid & 31;
        for (int e = tid >> 5; e < E; e += kThreads / 32) {
            int run = 0;
            for (int b0 = 0; b0 < nb; b0 += 32) {
                const int b = b0 + lane;
                const int c = b < nb ? __popc(mask[e * nb + b]) : 0;
                int incl = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                if (b < nb) pre[e * nb + b] = run + incl - c;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) cnt[e] = run;
        }
    }
    __syncthreads();
    {
        // exclusive scans over experts (ascending) of the assignment counts, of the active
        // flags and of the row-tile counts: a thread per expert, scans within each warp,
        // then the totals of the lower warps
        __shared__ int wred[4][kMaxE / 32];
        const int lane = tid & 31, warp = tid >> 5;
        const int nw = (E + 31) >> 5;
        const int c = tid < E ? cnt[tid] : 0;
        // the tile limit from the largest count, then an expert's tiles: ceil(c / limit)
        // of near-equal size
        if (warp < nw) {
            const int wm = __reduce_max_sync(0xffffffffu, c);
            if (lane == 0) wred[2][warp] = wm;
        }
        __syncthreads();
        int cbig = 0;
        for (int w = 0; w < nw; ++w) cbig = max(cbig, wred[2][w]);
        const int lim = rowtile_limit(cbig);
        const int nt = (c + lim - 1) / lim;
        const int tmax = nt > 0 ? (c + nt - 1) / nt : 0;  // its largest tile
        if (warp < nw) {
            const int wm = __reduce_max_sync(0xffffffffu, tmax);
            if (lane == 0) wred[3][warp] = wm;
        }
        __syncthreads();
        // row-tile height: the largest tile rounded up to 16
        int cmax = 0;
        for (int w = 0; w < nw; ++w) cmax = max(cmax, wred[3][w]);
        const int rt_size = min(lim, max(16, (cmax + 15) & ~15));
        const int a = c > 0;
        int ci = c, ai = a, ti = nt;  // inclusive scans within the warp
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
            if (lane == 31) {
                wred[0][warp] = ci;
                wred[1][warp] = ai;
                wred[2][warp] = ti;
            }
        }
        __syncthreads();
        if (tid < E) {
            for (int w = 0; w < warp; ++w) {
                ci += wred[0][w];
                ai += wred[1][w];
                ti += wred[2][w];
            }
            const int c_ex = ci - c, a_ex = ai - a;
            int t_ex = ti - nt;
            off[tid] = c_ex;
            if (a) active[1 + a_ex] = tid;
            // the expert's row tiles for the tensor-core kernel: nt near-equal tiles, each
            // knowing its index in the expert's group and the group's size
            for (int j = 0, n0 = 0; j < nt; ++j) {
                const int sz = c / nt + (j < c % nt ? 1 : 0);
                int *t = rowtiles + kRowTileHeader + 4 * t_ex++;
                t[0] = tid;
                t[1] = c_ex + n0;  // first permuted row of the tile
                t[2] = sz;
                t[3] = rowtile_group(j, nt);
                n0 += sz;
            }
            if (tid == E - 1) {
                off[E] = ci;
                active[0] = ai;
                rowtiles[0] = ti;
                rowtiles[1] = rt_size;
            }
        }
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kThreads) {
        offsets[e] = off[e];
        if (e < E) counts[e] = cnt[e];
    }
    if (gmask) {  // large blocks: permute_scatter_kernel places the assignments
        if (!kInPlace)
            for (int i = tid; i < 2 * nb * E; i += kThreads)
                if (!kMasksReady || i >= nb * E) gmask[i] = sm[i];
        return;
    }
    // a thread per assignment; a repeated expert keeps its first slot
    for (int a = tid; a < A; a += kThreads) {
        const int e = sidx[a];
        const int r = a / k, j = a - r * k;
        bool ok = e >= 0 && e < E;
#pragma unroll
        for (int q = 0; q < kMaxK; ++q)
            if (q < j && sidx[r * k + q] == e) ok = false;
        if (!ok) {
            pos[a] = -1;
            atomicOr(flags, FLAG_BAD_EXPERT);
            continue;
        }
        const int b = r >> 5;
        const int p = off[e] + (int)pre[e * nb + b] +
                      __popc(mask[e * nb + b] & ((1u << (r & 31)) - 1u));
        perm[p] = a;
        pos[a] = p;
    }
    for (int p = off[E] + tid; p < A; p += kThreads) perm[p] = -1;
}

// Places the assignments of a large block from the row-block masks and prefixes the
// permute kernel left in `gmask` ([E][nb] masks, then [E][nb] prefixes): a thread per
// assignment, spread over many CTAs (one CTA's stores would bound the whole step).
__global__ void __launch_bounds__(256)
permute_scatter_kernel(const int *__restrict__ idx, int R, int k, int E,
                       const int *__restrict__ offsets, const uint32_t *__restrict__ gmask,
                       int *__restrict__ perm, int *__restrict__ pos, int *__restrict__ flags) {
    pdl_wait();
    const int nb = (R + 31) >> 5;
    const int A = R * k;
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= A) return;
    const int total = offsets[E];
    if (a >= total) perm[a] = -1;  // positions past the placed assignments
    const int e = idx[a];
    const int r = a / k, j = a - r * k;
    bool ok = e >= 0 && e < E;
#pragma unroll
    for (int q = 0; q < kMaxK; ++q)  // first slot wins; the loads are independent
        if (q < j && idx[r * k + q] == e) ok = false;
    if (!ok) {
        pos[a] = -1;
        atomicOr(flags, FLAG_BAD_EXPERT);
        return;
    }
    const int b = r >> 5;
    const int p = offsets[e] + (int)gmask[(size_t)nb * E + e * nb + b] +
                  __popc(gmask[e * nb + b] & ((1u << (r & 31)) - 1u));
    perm[p] = a;
    pos[a] = p;
}

// Up to this many assignments one CTA also places them.
constexpr int kOneCtaAssignments = 2048;
// Past this many, permute_masks_kernel builds the masks first. Measured on GB300
// (Qwen3-30B-A3B-shaped layer): at 2080 assignments the extra launch cost 0.3%, at 33280
// it saved 1.5-1.8% of the block.
constexpr int kManyCtaMasks = 8192;

}  // namespace

size_t permute_smem_bytes(int R, int E) {
    const size_t nb = (size_t)(R + 31) / 32;
    return nb * E * 8 + (size_t)(2 * E + 1) * 4;
}

namespace {
// Shared memory of the one-CTA scan of masks left in place: counts, offsets.
size_t masks_ready_smem_bytes(int E) { return (size_t)(2 * E + 1) * 4; }
constexpr size_t kPermuteSmemLimit = 227 * 1024;
}  // namespace

cudaError_t launch_permute(const moe_layer_desc &L, const int *idx, int R, int *counts,
                           int *offsets, int *perm, int *pos, int *active, int *rowtiles,
                           int *flags, uint32_t *rbmask, bool after_router, cudaStream_t s) {
    const int A = R * L.k;
    uint32_t *gm = A > kOneCtaAssignments ? rbmask : nullptr;
    // past kManyCtaMasks assignments, or when the masks and prefixes would not fit in shared
    // memory, a many-CTA kernel builds the masks and the one CTA scans them in place; else
    // they live in shared memory, with the staged expert ids when this CTA places the
    // assignments (A <= 2048, so R <= 2048 and the masks take at most 64 row blocks: the
    // total stays far below the limit)
    const bool in_place = gm && permute_smem_bytes(R, L.E) > kPermuteSmemLimit;
    const bool masks_ready = A > kManyCtaMasks || in_place;
    const size_t smem = in_place ? masks_ready_smem_bytes(L.E)
                                 : permute_smem_bytes(R, L.E) + (gm ? 0 : (size_t)A * 4);
    auto kernel = in_place      ? permute_kernel<2>
                  : masks_ready ? permute_kernel<1>
                                : permute_kernel<0>;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if (masks_ready) {
        err = launch_pdl(permute_masks_kernel, dim3((R + 31) / 32), dim3(kMaskThreads), 0, s, idx,
                         R, L.k, L.E, gm);
        if (err != cudaSuccess) return err;
    }
    err = launch_pdl(kernel, dim3(1), dim3(kThreads), smem, s, idx, R, L.k, L.E, counts, offsets,
                     perm, pos, active, rowtiles, flags, gm, after_router ? 1 : 0);
    if (err != cudaSuccess || !gm) return err;
    return launch_pdl(permute_scatter_kernel, dim3((A + 255) / 256), dim3(256), 0, s, idx, R,
                      L.k, L.E, (const int *)offsets, (const uint32_t *)gm, perm, pos, flags);
}

}  // namespace moe
