// Pre-norm of the layer input: every row scaled to unit root-mean-square,
//   xn[r] = x[r] / sqrt(mean_i x[r, i]^2 + eps),
// as the blocks of the target models put a normalisation in front of the MoE layer (a
// stack of layers without one lets the residual stream grow until it overflows). No
// learned weight. The mean of squares and the scale are computed in fp64 (the squares of
// fp32 / bf16 values are exact in fp64), and each element x * scale is rounded once to the
// layer dtype (bf16: through an fp32 product where that provably rounds the same).
//
// GB300's fp64 rate is a small fraction of its fp32 rate (~2 fp64 operations per clock per
// SM), so the fp64 work is spread over as many SMs as there are rows: a CTA of 256 threads
// per row. (A warp per row put a 65-row block on 9 SMs and took ~31 us; measured on GB300.)
#include "common.cuh"

namespace moe {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormWarps = kNormThreads / 32;

__device__ __forceinline__ double norm_warp_sum(double v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Adds v[q]^2, q < 8, to s (v^2 is exact in fp64: one rounding per fused add).
__device__ __forceinline__ double norm_add_squares(double s, const float v[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) s = __fma_rn((double)v[q], (double)v[q], s);
    return s;
}

// The row's scale from each thread's partial sum; every thread of the CTA calls it (two
// block barriers). Thread 0 alone adds the warps' partials and forms the scale (an fp64
// square root and divide are dozens of fp64 operations), then shares it. part: kNormWarps
// doubles of shared memory.
__device__ __forceinline__ double norm_scale(double s, int d, double eps, double *part) {
    s = norm_warp_sum(s);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
#pragma unroll
        for (int w = 0; w < kNormWarps; ++w) tot = __dadd_rn(tot, part[w]);
        part[0] = 1.0 / sqrt(tot / (double)d + eps);
    }
    __syncthreads();
    return part[0];
}

// bf16(fp64(v * scale)), rounded to nearest even, for v an fp32 value. The fp32 product
// p = v * (float)scale lies within 2^-22.8 |p| of the fp64 product (one rounding of the
// scale to fp32 and one of the product, 2^-24 relative each); bf16 rounding midpoints are
// at least 2^-9 |p| apart, so when p is farther than 2^-21 |p| from the midpoint between
// its two bf16 neighbours, both products round to the same bf16 value and p's rounding is
// the answer. Otherwise (about one element in 4000, for zero, tiny or non-finite p, and for
// a scale whose fp32 rounding is not a normal number far from the range ends) the product
// is formed and rounded in fp64.
__device__ __forceinline__ uint32_t scaled_bf16(float v, double scale, float scale_f) {
    const float p = v * scale_f;
    const float ap = fabsf(p);
    if (scale_f >= 0x1p-100f && scale_f <= 0x1p+100f && ap >= 0x1p-100f && ap <= 0x1p+100f) {
        const __nv_bfloat16 lo = __float2bfloat16_rd(p), hi = __float2bfloat16_ru(p);
        const float flo = __bfloat162float(lo), fhi = __bfloat162float(hi);
        if (flo == fhi) return __bfloat16_as_ushort(lo);  // p is a bf16 value
        const float mid = 0.5f * (flo + fhi);              // exact: a 9-bit value
        const float dist = fabsf(p - mid);                 // exact (Sterbenz)
        if (dist > ap * 0x1p-21f) return __bfloat16_as_ushort(p < mid ? lo : hi);
    }
    return __bfloat16_as_ushort(__double2bfloat16((double)v * scale));
}

// Stores v[q] * scale, q < 8, rounded once (nearest, ties to even) to T, as 16-byte stores.
template <typename T> __device__ __forceinline__ void store_scaled(T *p, const float v[8],
                                                                  double scale);
template <>
__device__ __forceinline__ void store_scaled<__nv_bfloat16>(__nv_bfloat16 *p, const float v[8],
                                                            double scale) {
    const float scale_f = __double2float_rn(scale);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = scaled_bf16(v[2 * q], scale, scale_f) |
               (scaled_bf16(v[2 * q + 1], scale, scale_f) << 16);
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ void store_scaled<float>(float *p, const float v[8], double scale) {
    float o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = __double2float_rn((double)v[q] * scale);
    reinterpret_cast<float4 *>(p)[0] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(o[4], o[5], o[6], o[7]);
}

// A CTA per row: the 8-element groups at columns 8 t + 8 kNormThreads j to thread t, its
// fp64 sum of squares over them, then over the warp, then the warps' partials in order.
template <typename T>
__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(const T *__restrict__ x, int R, int d, double eps, T *__restrict__ xn) {
    pdl_wait();
    __shared__ double part[kNormWarps];
    const int row = blockIdx.x, tid = threadIdx.x;
    const T *xr = x + (size_t)row * d;
    double s = 0.0;
    for (int c = tid * 8; c < d; c += kNormThreads * 8) {
        float v[8];
        Vec8<T>::load(xr + c, v);
        s = norm_add_squares(s, v);
    }
    const double scale = norm_scale(s, d, eps, part);
    T *out = xn + (size_t)row * d;
    for (int c = tid * 8; c < d; c += kNormThreads * 8) {
        float v[8];
        Vec8<T>::load(xr + c, v);
        store_scaled<T>(out + c, v, scale);
    }
}

}  // namespace

cudaError_t launch_rmsnorm(const moe_layer_desc &L, const void *x, int R, void *xn,
                           cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const dim3 grid(R);
    if (L.dtype == MOE_DTYPE_BF16)
        return launch_pdl(rmsnorm_kernel<__nv_bfloat16>, grid, dim3(kNormThreads), 0, s,
                          (const __nv_bfloat16 *)x, R, L.d, kNormEps, (__nv_bfloat16 *)xn);
    return launch_pdl(rmsnorm_kernel<float>, grid, dim3(kNormThreads), 0, s, (const float *)x,
                      R, L.d, kNormEps, (float *)xn);
}

}  // namespace moe
