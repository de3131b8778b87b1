// Grouped SwiGLU experts on CUDA cores ("MoE and speculative decoding" blog,
// "grouped GEMM for active experts"): for every expert with assignments,
//   h = silu(X_e W_gate[e]^T) * (X_e W_up[e]^T),   O_e = h W_down[e]^T,
// X_e being the expert's token rows in permuted order.
//
// This is the general path (fp32 or bf16 layers, any d, f multiple of 8). Two
// launches: gate/up then down. A CTA owns one expert and a 32-row slice of the
// weight matrix; its 8 warps each take 4 weight rows, lanes split the reduction
// dimension in 8-element (16-byte) slices, and up to 8 token rows are staged in
// shared memory as fp32 so each weight fragment feeds 8 tokens. Weight bytes are
// read once per 8 tokens of an expert. A transpose-reduction finishes 32 dot
// products per warp at a time. The weight loads are software-pipelined: a lane issues
// the next slice's four 16-byte loads (kept raw) before it computes on the current
// slice, so twice as many bytes are in flight per warp; registers stay within the
// 128 that two CTAs per SM allow. (Measured on GB300: 0.43 of the copy bandwidth at one
// to two rows per expert against 0.39 without; passes compiled per live token count, or
// one CTA per SM without the register cap, were slower.)
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 32
constexpr int kTok = 8;                              // token rows per pass

template <typename T>
__device__ __forceinline__ const T *expert_base(const void *W, const int *slot, int slots, int e,
                                                size_t per_expert, int *flags, bool &ok) {
    const int s = slot ? slot[e] : e;
    ok = s >= 0 && s < slots;
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(flags, FLAG_BAD_EXPERT);
        return nullptr;
    }
    return reinterpret_cast<const T *>(W) + (size_t)s * per_expert;
}

// Stages rows src[row(t)] (t < nt) of length n as fp32 into xs[t][n]; rows nt..kTok-1
// are zero.
template <typename T, typename RowOf>
__device__ __forceinline__ void stage_rows(float *xs, int n, int nt, RowOf row_of, const T *src) {
    const int per = n / 8;
    for (int i = threadIdx.x; i < kTok * per; i += kThreads) {
        const int t = i / per, c = (i - t * per) * 8;
        float v[8];
        if (t < nt) {
            Vec8<T>::load(src + (size_t)row_of(t) * n + c, v);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0.f;
        }
        float4 *d = reinterpret_cast<float4 *>(xs + (size_t)t * n + c);
        d[0] = make_float4(v[0], v[1], v[2], v[3]);
        d[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// Eight consecutive weights kept as loaded (one 16-byte load for bf16, two for fp32) and
// widened to fp32 when used, so that loads can be issued a slice ahead of their use.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        u = __ldg(reinterpret_cast<const uint4 *>(p));
    }
    __device__ __forceinline__ void widen(float v[8]) const {
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p) {
        a = __ldg(reinterpret_cast<const float4 *>(p));
        b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void widen(float v[8]) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// Stores an fp32 result in the layer dtype (bf16: rounded to nearest even).
__device__ __forceinline__ void store_as(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_as(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float dot8(const float w[8], const float *x) {
    const float4 a = reinterpret_cast<const float4 *>(x)[0];
    const float4 b = reinterpret_cast<const float4 *>(x)[1];
    float s = w[0] * a.x;
    s = fmaf(w[1], a.y, s); s = fmaf(w[2], a.z, s); s = fmaf(w[3], a.w, s);
    s = fmaf(w[4], b.x, s); s = fmaf(w[5], b.y, s); s = fmaf(w[6], b.z, s);
    return fmaf(w[7], b.w, s);
}

// h[p, i] = silu(Wg[i] . x_p) * (Wu[i] . x_p) for the expert's permuted rows p.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) ffn_gateup_simt(FfnArgs a) {
    pdl_wait();
    const int e = blockIdx.x;
    const int cnt = a.counts[e];
    if (cnt == 0 || (a.pass && !a.pass[e])) return;
    bool ok;
    const T *Wg = expert_base<T>(a.Wg, a.slot, a.slots, e, (size_t)a.f * a.d, a.flags, ok);
    if (!ok) return;
    const T *Wu = reinterpret_cast<const T *>(a.Wu) + (Wg - reinterpret_cast<const T *>(a.Wg));
    extern __shared__ float xs[];  // [kTok][d]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int off = a.offsets[e];
    const int d = a.d, f = a.f;
    const T *x = reinterpret_cast<const T *>(a.x);
    float *h = reinterpret_cast<float *>(a.h);

    for (int t0 = 0; t0 < cnt; t0 += kTok) {
        const int nt = min(kTok, cnt - t0);
        __syncthreads();
        stage_rows<T>(xs, d, nt, [&](int t) { return a.perm[off + t0 + t] / a.k; }, x);
        __syncthreads();
        for (int pr = 0; pr < kRowsPerWarp; pr += 2) {
            const int i0 = blockIdx.y * kRowsPerCta + warp * kRowsPerWarp + pr;
            if (i0 >= f) break;
            const int i1 = min(i0 + 1, f - 1);
            // acc[q*16 + g*8 + t]: row i0+q, g = 0 gate / 1 up, token t
            float acc[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = 0.f;
            const T *rows[4] = {Wg + (size_t)i0 * d, Wu + (size_t)i0 * d, Wg + (size_t)i1 * d,
                                Wu + (size_t)i1 * d};
            Raw8<T> nxt[4];
            if (lane * 8 < d) {
#pragma unroll
                for (int q = 0; q < 4; ++q) nxt[q].load(rows[q] + lane * 8);
            }
            for (int c = lane * 8; c < d; c += 256) {
                float w[4][8];
#pragma unroll
                for (int q = 0; q < 4; ++q) nxt[q].widen(w[q]);
                if (c + 256 < d) {  // the next slice's loads go out before this slice's math
#pragma unroll
                    for (int q = 0; q < 4; ++q) nxt[q].load(rows[q] + c + 256);
                }
#pragma unroll
                for (int t = 0; t < kTok; ++t) {
                    const float *xr = xs + (size_t)t * d + c;
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[q * 8 + t] += dot8(w[q], xr);
                }
            }
            const float v = warp_transpose_sum32(acc);
            const float u = __shfl_xor_sync(0xffffffffu, v, 8);
            const int q = lane >> 4, gate = ((lane >> 3) & 1) == 0, t = lane & 7;
            const int i = i0 + q;
            if (gate && t < nt && i < f && (q == 0 || i0 + 1 < f)) {
                const float s = v / (1.f + expf(-v));
                h[(size_t)(off + t0 + t) * f + i] = s * u;
            }
        }
    }
}

// O[p, i] = Wd[i] . h_p for the expert's permuted rows p.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) ffn_down_simt(FfnArgs a) {
    pdl_wait();
    const int e = blockIdx.x;
    const int cnt = a.counts[e];
    if (cnt == 0 || (a.pass && !a.pass[e])) return;
    bool ok;
    const T *Wd = expert_base<T>(a.Wd, a.slot, a.slots, e, (size_t)a.f * a.d, a.flags, ok);
    if (!ok) return;
    extern __shared__ float hs[];  // [kTok][f]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int off = a.offsets[e];
    const int d = a.d, f = a.f;
    const float *h = reinterpret_cast<const float *>(a.h);
    const int i0 = blockIdx.y * kRowsPerCta + warp * kRowsPerWarp;

    for (int t0 = 0; t0 < cnt; t0 += kTok) {
        const int nt = min(kTok, cnt - t0);
        __syncthreads();
        stage_rows<float>(hs, f, nt, [&](int t) { return off + t0 + t; }, h);
        __syncthreads();
        if (i0 >= d) continue;
        float acc[32];  // acc[r*8 + t]: row i0+r, token t
#pragma unroll
        for (int q = 0; q < 32; ++q) acc[q] = 0.f;
        const T *rows[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) rows[r] = Wd + (size_t)min(i0 + r, d - 1) * f;
        Raw8<T> nxt[4];
        if (lane * 8 < f) {
#pragma unroll
            for (int r = 0; r < 4; ++r) nxt[r].load(rows[r] + lane * 8);
        }
        for (int c = lane * 8; c < f; c += 256) {
            float w[4][8];
#pragma unroll
            for (int r = 0; r < 4; ++r) nxt[r].widen(w[r]);
            if (c + 256 < f) {  // the next slice's loads go out before this slice's math
#pragma unroll
                for (int r = 0; r < 4; ++r) nxt[r].load(rows[r] + c + 256);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int t = 0; t < kTok; ++t)
                    acc[r * 8 + t] += dot8(w[r], hs + (size_t)t * f + c);
            }
        }
        const float v = warp_transpose_sum32(acc);
        const int r = lane >> 3, t = lane & 7;
        if (t < nt && i0 + r < d) store_as(static_cast<T *>(a.o) + (size_t)(off + t0 + t) * d + i0 + r, v);
    }
}

}  // namespace

cudaError_t launch_ffn_simt(const FfnArgs &a, cudaStream_t s) {
    const size_t smem_gu = (size_t)kTok * a.d * sizeof(float);
    const size_t smem_dn = (size_t)kTok * a.f * sizeof(float);
    dim3 g1(a.E, (a.f + kRowsPerCta - 1) / kRowsPerCta);
    dim3 g2(a.E, (a.d + kRowsPerCta - 1) / kRowsPerCta);
    cudaError_t err;
    if (a.dtype == MOE_DTYPE_BF16) {
        err = cudaFuncSetAttribute(ffn_gateup_simt<__nv_bfloat16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(ffn_down_simt<__nv_bfloat16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
        if (err != cudaSuccess) return err;
        err = launch_pdl(ffn_gateup_simt<__nv_bfloat16>, g1, dim3(kThreads), smem_gu, s, a);
        if (err != cudaSuccess) return err;
        err = launch_pdl(ffn_down_simt<__nv_bfloat16>, g2, dim3(kThreads), smem_dn, s, a);
    } else {
        err = cudaFuncSetAttribute(ffn_gateup_simt<float>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(ffn_down_simt<float>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
        if (err != cudaSuccess) return err;
        err = launch_pdl(ffn_gateup_simt<float>, g1, dim3(kThreads), smem_gu, s, a);
        if (err != cudaSuccess) return err;
        err = launch_pdl(ffn_down_simt<float>, g2, dim3(kThreads), smem_dn, s, a);
    }
    return err;
}

}  // namespace moe
