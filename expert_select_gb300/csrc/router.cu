// Router scores l = W_r x ("MoE and speculative decoding" blog, section "starting from
// one MoE layer": the W_r x inside E(x) = TopR(softmax(W_r x))).
//
// A warp computes a 4-row x 8-expert block of logits: lanes split the hidden
// dimension in 8-element (16-byte for bf16) slices, so every load is coalesced and
// each x/W fragment feeds 8 (resp. 4) FMAs, and a transpose-reduction leaves one
// finished logit per lane. Two launch shapes:
//   * small blocks (a few trees): the 8 warps of a CTA split the hidden dimension of
//     one 4 x 8 block, so each lane issues all of its loads at once, and the CTA adds
//     the 8 partial sums in shared memory (latency-bound regime);
//   * large blocks: the 8 warps share their 8 experts and take consecutive row
//     blocks, so a W_r slice is fetched from L2 once per CTA and served from L1.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRows = 4;     // rows per warp
constexpr int kExp = 8;      // experts per warp
constexpr int kWarps = 8;    // warps per CTA (consecutive row blocks)

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
router_kernel(const T *__restrict__ x, const T *__restrict__ Wr, int R, int d, int E,
              float *__restrict__ logits) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int e0 = blockIdx.y * kExp;
    const int r0 = (blockIdx.x * kWarps + warp) * kRows;
    if (r0 >= R) return;

    const T *xr[kRows];
    const T *wr[kExp];
#pragma unroll
    for (int i = 0; i < kRows; ++i) xr[i] = x + (size_t)min(r0 + i, R - 1) * d;
#pragma unroll
    for (int j = 0; j < kExp; ++j) wr[j] = Wr + (size_t)min(e0 + j, E - 1) * d;

    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;

    for (int c = lane * 8; c < d; c += 32 * 8) {
        float xv[kRows][8];
#pragma unroll
        for (int i = 0; i < kRows; ++i) Vec8<T>::load(xr[i] + c, xv[i]);
#pragma unroll
        for (int j = 0; j < kExp; ++j) {
            float wv[8];
            Vec8<T>::load(wr[j] + c, wv);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                float s = acc[i * kExp + j];
#pragma unroll
                for (int t = 0; t < 8; ++t) s = fmaf(xv[i][t], wv[t], s);
                acc[i * kExp + j] = s;
            }
        }
    }
    const float v = warp_transpose_sum32(acc);
    const int r = r0 + lane / kExp, e = e0 + lane % kExp;
    if (r < R && e < E) logits[(size_t)r * E + e] = v;
}

// Small-R shape: one 4-row x 8-expert block per CTA, hidden dimension split over warps.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
router_splitd_kernel(const T *__restrict__ x, const T *__restrict__ Wr, int R, int d, int E,
                     float *__restrict__ logits) {
    pdl_wait();
    __shared__ float part[kWarps][32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int r0 = blockIdx.x * kRows, e0 = blockIdx.y * kExp;
    const T *xr[kRows];
    const T *wr[kExp];
#pragma unroll
    for (int i = 0; i < kRows; ++i) xr[i] = x + (size_t)min(r0 + i, R - 1) * d;
#pragma unroll
    for (int j = 0; j < kExp; ++j) wr[j] = Wr + (size_t)min(e0 + j, E - 1) * d;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    for (int c = (warp * 32 + lane) * 8; c < d; c += kWarps * 32 * 8) {
        float xv[kRows][8];
#pragma unroll
        for (int i = 0; i < kRows; ++i) Vec8<T>::load(xr[i] + c, xv[i]);
#pragma unroll
        for (int j = 0; j < kExp; ++j) {
            float wv[8];
            Vec8<T>::load(wr[j] + c, wv);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                float s = acc[i * kExp + j];
#pragma unroll
                for (int t = 0; t < 8; ++t) s = fmaf(xv[i][t], wv[t], s);
                acc[i * kExp + j] = s;
            }
        }
    }
    part[warp][lane] = warp_transpose_sum32(acc);
    __syncthreads();
    if (warp == 0) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += part[w][lane];
        const int r = r0 + lane / kExp, e = e0 + lane % kExp;
        if (r < R && e < E) logits[(size_t)r * E + e] = v;
    }
}

// Up to this many rows the split-hidden shape is used.
constexpr int kSplitRows = 1024;

}  // namespace

cudaError_t launch_router(const moe_layer_desc &L, const void *x, const void *Wr, int R,
                          float *logits, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (R <= kSplitRows) {
        dim3 g((R + kRows - 1) / kRows, (L.E + kExp - 1) / kExp);
        if (L.dtype == MOE_DTYPE_BF16)
            return launch_pdl(router_splitd_kernel<__nv_bfloat16>, g, dim3(kWarps * 32), 0, s,
                              (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wr, R, L.d, L.E,
                              logits);
        return launch_pdl(router_splitd_kernel<float>, g, dim3(kWarps * 32), 0, s,
                          (const float *)x, (const float *)Wr, R, L.d, L.E, logits);
    }
    dim3 grid((R + kWarps * kRows - 1) / (kWarps * kRows), (L.E + kExp - 1) / kExp);
    if (L.dtype == MOE_DTYPE_BF16)
        return launch_pdl(router_kernel<__nv_bfloat16>, grid, dim3(kWarps * 32), 0, s,
                          (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wr, R, L.d, L.E,
                          logits);
    return launch_pdl(router_kernel<float>, grid, dim3(kWarps * 32), 0, s, (const float *)x,
                      (const float *)Wr, R, L.d, L.E, logits);
}

}  // namespace moe
