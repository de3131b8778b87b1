// Unpermute + weighted combine ("MoE and speculative decoding" blog, pipeline step
// "unpermute + weighted combine"): y[r] = sum_j gates[r, j] O[pos(r, j)], slots in
// ascending j, fp32 accumulation, rounded once to the layer dtype. The expert outputs O
// arrive in the layer dtype (bf16 layers: rounded once from the experts' fp32 sums). With a residual
// input the sum starts from it (y = x + MoE(x), as in a stack of layers).
//
// Also holds the small kernel that publishes a residency table to the device.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <typename TO>
__device__ __forceinline__ void store4(TO *y, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float *y, float4 v) {
    *reinterpret_cast<float4 *>(y) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *y, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(y) = u;
}

template <typename TO>
__device__ __forceinline__ float4 load4(const TO *p);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

// The same through the read-only cache (for the expert outputs, never written here).
template <typename TO>
__device__ __forceinline__ float4 ldg4(const TO *p);
template <>
__device__ __forceinline__ float4 ldg4<float>(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
template <>
__device__ __forceinline__ float4 ldg4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

// `res` (may be null, may alias y) is added first: y = res + sum_j g_j O_j, over the slots
// in ascending j. A thread per 4 columns of a row.
template <typename TO>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const TO *__restrict__ o, const int *__restrict__ pos,
               const float *__restrict__ gates, const TO *res, int d, int k, TO *y) {
    pdl_wait();
    const int r = blockIdx.x;
    const int c = (blockIdx.y * kThreads + threadIdx.x) * 4;
    if (c >= d) return;
    float4 acc = res ? load4<TO>(res + (size_t)r * d + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int p = pos[r * k + j];
        if (p < 0) continue;
        const float g = gates[r * k + j];
        const float4 v = ldg4<TO>(o + (size_t)p * d + c);
        acc.x = fmaf(g, v.x, acc.x);
        acc.y = fmaf(g, v.y, acc.y);
        acc.z = fmaf(g, v.z, acc.z);
        acc.w = fmaf(g, v.w, acc.w);
    }
    store4<TO>(y + (size_t)r * d + c, acc);
}

// The same for small blocks, where the kernel is bound by load latency: every slot's
// position and gate are loaded first, then every slot's output piece (up to KMAX slots in
// flight per thread), and the sum runs over the slots in ascending j as above. Large
// blocks keep the kernel above: its fewer registers let more threads stream.
template <typename TO, int KMAX>
__global__ void __launch_bounds__(kThreads)
combine_small_kernel(const TO *__restrict__ o, const int *__restrict__ pos,
                     const float *__restrict__ gates, const TO *res, int d, int k, TO *y) {
    pdl_wait();
    const int r = blockIdx.x;
    const int c = (blockIdx.y * kThreads + threadIdx.x) * 4;
    if (c >= d) return;
    int p[KMAX];
    float g[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        p[j] = j < k ? pos[r * k + j] : -1;
        g[j] = j < k ? gates[r * k + j] : 0.f;
    }
    float4 acc = res ? load4<TO>(res + (size_t)r * d + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
        if (p[j] >= 0) v[j] = ldg4<TO>(o + (size_t)p[j] * d + c);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (p[j] < 0) continue;
        acc.x = fmaf(g[j], v[j].x, acc.x);
        acc.y = fmaf(g[j], v[j].y, acc.y);
        acc.z = fmaf(g[j], v[j].z, acc.z);
        acc.w = fmaf(g[j], v[j].w, acc.w);
    }
    store4<TO>(y + (size_t)r * d + c, acc);
}

// Assignments up to which the combine takes the small-block kernel.
constexpr int kSmallCombine = 2048;

template <typename TO>
cudaError_t launch_combine_t(const TO *o, const int *pos, const float *gates,
                             const TO *res, int R, int d, int k, TO *y, cudaStream_t s) {
    const dim3 grid(R, (d / 4 + kThreads - 1) / kThreads);
    if (R * k <= kSmallCombine) {
        if (k <= 8)
            return launch_pdl(combine_small_kernel<TO, 8>, grid, dim3(kThreads), 0, s, o, pos,
                              gates, res, d, k, y);
        return launch_pdl(combine_small_kernel<TO, kMaxK>, grid, dim3(kThreads), 0, s, o, pos,
                          gates, res, d, k, y);
    }
    return launch_pdl(combine_kernel<TO>, grid, dim3(kThreads), 0, s, o, pos, gates, res, d, k,
                      y);
}

struct PublishArgs {
    int slot[kMaxE];
    uint8_t res[kMaxE];
};

__global__ void publish_kernel(PublishArgs p, int E, int *slot, uint8_t *res) {
    pdl_wait();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (slot) slot[e] = p.slot[e];
        if (res) res[e] = p.res[e];
    }
}

}  // namespace

cudaError_t launch_combine(const moe_layer_desc &L, const void *o, const int *pos,
                           const float *gates, const void *residual, int R, void *y,
                           cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (L.dtype == MOE_DTYPE_BF16)
        return launch_combine_t((const __nv_bfloat16 *)o, pos, gates,
                                (const __nv_bfloat16 *)residual, R, L.d, L.k, (__nv_bfloat16 *)y, s);
    return launch_combine_t((const float *)o, pos, gates, (const float *)residual, R, L.d, L.k,
                            (float *)y, s);
}

cudaError_t launch_publish(int E, const int *slot_host, const uint8_t *res_host, int *slot_dev,
                           uint8_t *res_dev, cudaStream_t s) {
    PublishArgs p;
    for (int e = 0; e < E; ++e) {
        p.slot[e] = slot_host[e];
        p.res[e] = res_host[e];
    }
    return launch_pdl(publish_kernel, dim3(1), dim3(256), 0, s, p, E, slot_dev, res_dev);
}

}  // namespace moe
