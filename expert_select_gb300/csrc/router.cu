// Router scores l = W_r x ("MoE and speculative decoding" blog, section "starting from
// one MoE layer": the W_r x inside E(x) = TopR(softmax(W_r x))).
//
// One warp computes a 4-row x 8-expert block of logits. Lanes split the hidden
// dimension in 8-element (16-byte for bf16) slices, so every load is coalesced and
// each x/W fragment feeds 8 (resp. 4) FMAs. A transpose-reduction then leaves one
// finished logit per lane. The 8 warps of a CTA share their experts and take
// consecutive row blocks, so a W_r slice is fetched from L2 once per CTA and served
// to the other warps from L1.
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

}  // namespace

cudaError_t launch_router(const moe_layer_desc &L, const void *x, const void *Wr, int R,
                          float *logits, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    dim3 grid((R + kWarps * kRows - 1) / (kWarps * kRows), (L.E + kExp - 1) / kExp);
    if (L.dtype == MOE_DTYPE_BF16)
        router_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, s>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wr, R, L.d, L.E, logits);
    else
        router_kernel<float><<<grid, kWarps * 32, 0, s>>>((const float *)x, (const float *)Wr,
                                                          R, L.d, L.E, logits);
    return cudaGetLastError();
}

}  // namespace moe
