// Permute / group by expert ("MoE and speculative decoding" blog, pipeline step
// "permute / group by expert"): a stable counting sort of the assignments (r, j)
// by the key (expert, row, slot).
//
// A row picks each expert at most once, so inside one expert the key order is row
// order. One CTA builds, per block of 32 rows and per expert, the bitmask of rows
// that chose the expert; a scan over row blocks gives each (block, expert) its
// prefix; an assignment's position is then
//   offsets[e] + prefix[block][e] + popc(mask[block][e] & lanes_below(row)).
// Everything stays in shared memory: (R/32) x E x 8 bytes (133 KB at 4160 rows and
// 128 experts). The same kernel also writes the active-expert list and the list of
// row tiles (at most 64 or 256 tokens of one expert) that the grouped expert kernels walk.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads)
permute_kernel(const int *__restrict__ idx, int R, int k, int E, int *__restrict__ counts,
               int *__restrict__ offsets, int *__restrict__ perm, int *__restrict__ pos,
               int *__restrict__ active, int *__restrict__ rowtiles, int *__restrict__ flags,
               int rt_size, int after_router) {
    pdl_wait();
    extern __shared__ uint32_t sm[];
    const int nb = (R + 31) >> 5;
    uint32_t *mask = sm;                  // [nb][E]
    uint32_t *pre = sm + (size_t)nb * E;  // [nb][E]
    int *cnt = (int *)(pre + (size_t)nb * E);
    int *off = cnt + E;                   // [E + 1]
    const int tid = threadIdx.x;
    const int A = R * k;

    for (int i = tid; i < nb * E; i += kThreads) mask[i] = 0u;
    if (tid == 0) {  // a fresh check word for this call, keeping what the router reported
        flags[0] = after_router ? flags[kRouterCheckWord] : 0;
        flags[kRouterCheckWord] = 0;
    } else if (tid < 64 && tid != kRouterCheckWord) {
        flags[tid] = 0;
    }
    __syncthreads();
    for (int a = tid; a < A; a += kThreads) {
        const int e = idx[a];
        if (e < 0 || e >= E) continue;
        const int r = a / k;
        atomicOr(&mask[(r >> 5) * E + e], 1u << (r & 31));
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        int run = 0;
        for (int b = 0; b < nb; ++b) {
            pre[b * E + e] = run;
            run += __popc(mask[b * E + e]);
        }
        cnt[e] = run;
    }
    __syncthreads();
    if (tid < 32) {
        // warp 0: exclusive scans over experts (ascending) of the assignment counts, of
        // the active flags and of the row-tile counts; lane owns experts [lane*per, +per)
        const int per = (E + 31) / 32;
        int c_tot = 0, a_tot = 0, t_tot = 0;
        for (int i = 0; i < per; ++i) {
            const int e = tid * per + i;
            const int c = e < E ? cnt[e] : 0;
            c_tot += c;
            a_tot += c > 0;
            t_tot += (c + rt_size - 1) / rt_size;
        }
        int c_ex = c_tot, a_ex = a_tot, t_ex = t_tot;  // inclusive scans across lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int c2 = __shfl_up_sync(0xffffffffu, c_ex, o);
            const int a2 = __shfl_up_sync(0xffffffffu, a_ex, o);
            const int t2 = __shfl_up_sync(0xffffffffu, t_ex, o);
            if (tid >= o) {
                c_ex += c2;
                a_ex += a2;
                t_ex += t2;
            }
        }
        c_ex -= c_tot;
        a_ex -= a_tot;
        t_ex -= t_tot;
        for (int i = 0; i < per; ++i) {
            const int e = tid * per + i;
            if (e >= E) break;
            const int c = cnt[e];
            off[e] = c_ex;
            c_ex += c;
            if (c > 0) active[1 + a_ex++] = e;
            // row tiles of at most rt_size tokens of one expert, for the tensor-core kernel
            for (int n0 = 0; n0 < c; n0 += rt_size) {
                int *t = rowtiles + 1 + 4 * t_ex++;
                t[0] = e;
                t[1] = n0;
                t[2] = min(rt_size, c - n0);
                t[3] = 0;
            }
        }
        if (tid == 31) {
            off[E] = c_ex;
            active[0] = a_ex;
            rowtiles[0] = t_ex;
        }
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kThreads) {
        offsets[e] = off[e];
        if (e < E) counts[e] = cnt[e];
    }
    for (int a = tid; a < A; a += kThreads) {
        const int e = idx[a];
        const int r = a / k, j = a - r * k;
        bool ok = e >= 0 && e < E;
        for (int q = 0; ok && q < j; ++q) ok = idx[r * k + q] != e;  // first slot wins
        if (!ok) {
            pos[a] = -1;
            atomicOr(flags, FLAG_BAD_EXPERT);
            continue;
        }
        const int b = r >> 5;
        const int p = off[e] + (int)pre[b * E + e] +
                      __popc(mask[b * E + e] & ((1u << (r & 31)) - 1u));
        perm[p] = a;
        pos[a] = p;
    }
    for (int p = off[E] + tid; p < A; p += kThreads) perm[p] = -1;
}

}  // namespace

size_t permute_smem_bytes(int R, int E) {
    const size_t nb = (size_t)(R + 31) / 32;
    return nb * E * 8 + (size_t)(2 * E + 1) * 4;
}

cudaError_t launch_permute(const moe_layer_desc &L, const int *idx, int R, int *counts,
                           int *offsets, int *perm, int *pos, int *active, int *rowtiles,
                           int *flags, bool after_router, cudaStream_t s) {
    const size_t smem = permute_smem_bytes(R, L.E);
    cudaError_t err = cudaFuncSetAttribute(permute_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(permute_kernel, dim3(1), dim3(kThreads), smem, s, idx, R, L.k, L.E, counts,
                      offsets, perm, pos, active, rowtiles, flags, rowtile_size(R),
                      after_router ? 1 : 0);
}

}  // namespace moe
