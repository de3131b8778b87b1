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
// From a few hundred rows on (bf16), the scores are a dense [R x d] x [d x E] product and
// run on the tensor cores instead (router_tc_kernel below).
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace moe {
namespace {

// The router's check word starts every call at zero: the first thread of the grid
// clears it before anything else (only the tensor-core kernel ever sets it, and only
// after a wait of two seconds).
__device__ __forceinline__ void clear_check_word(int *flags) {
    if (flags && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *flags = 0;
}

constexpr int kRows = 4;     // rows per warp
constexpr int kExp = 8;      // experts per warp
constexpr int kWarps = 8;    // warps per CTA (consecutive row blocks)

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
router_kernel(const T *__restrict__ x, const T *__restrict__ Wr, int R, int d, int E,
              float *__restrict__ logits, int *flags) {
    clear_check_word(flags);
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
                     float *__restrict__ logits, int *flags) {
    clear_check_word(flags);
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

// ------------------------------------------------------------------ tensor cores
// One CTA per (nt-row tile of x, 128 experts, 1/KS of the hidden dimension): the 128 router
// rows W_r[e0 .. e0+127] are the MMA's A operand (M = 128; experts past E are zero-filled by
// TMA), the token rows the B operand (N = nt, 32 to 256), the fp32 accumulator [128 experts
// x nt tokens] lives in tensor memory. The CTA's share of the hidden dimension streams
// through a ring of stages of 64 elements (one 128-byte swizzle atom) loaded by TMA. Warp 0
// loads, warp 1 allocates tensor memory and issues the MMAs, then all four warps read the
// accumulator back (warp q owns experts e0 + 32q .. +31, one per lane).
//
// Every CTA reads its whole W_r slice, so a CTA per row tile over the full hidden dimension
// moves 512 KB of W_r per 32 rows; the KS CTAs of a cluster (KS = 1, 2, 4 or 8) instead split
// the hidden dimension, each adding over its slice, and the cluster sums the KS partial
// logits: each CTA writes its partial into its own (drained) stage ring, and after a
// cluster barrier CTA c adds rows [c nt / KS, (c + 1) nt / KS) of every CTA's partial in
// rank order through distributed shared memory (a fixed order: the logits are the same on
// every run). The host picks the tile height and KS that put the fewest bytes through one
// CTA while the launch stays within one wave.
// Every wait is bounded; a wait that gives up leaves NaN in the CTA's logits and sets
// FLAG_WAIT_TIMEOUT in the router's check word `flags` when one is given.
namespace rtc {

using namespace tc;

constexpr int kThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kBK = 64;
constexpr int kM = 128;
constexpr uint32_t kABytes = kM * kBK * 2;  // 16 KB of W_r per stage
constexpr size_t kSmemBudget = 227 * 1024;
constexpr size_t kCtlBytes = 256;

struct Maps {
    CUtensorMap w;  // W_r [E][d], box 64 x 128
    CUtensorMap x;  // x [R][d], box 64 x nt
};

// Stages of the ring for tile height nt: as many as fit, at most kMaxStages.
__host__ __device__ constexpr int stages_for(int nt) {
    return (int)((kSmemBudget - 1024 - kCtlBytes) / (kABytes + (size_t)nt * 128)) < kMaxStages
               ? (int)((kSmemBudget - 1024 - kCtlBytes) / (kABytes + (size_t)nt * 128))
               : kMaxStages;
}

__host__ __device__ constexpr size_t smem_bytes(int nt) {
    return 1024 + (size_t)stages_for(nt) * (kABytes + (size_t)nt * 128) + kCtlBytes;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Four consecutive floats at the shared-memory address `local` of cluster CTA `rank`.
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t local, uint32_t rank) {
    uint32_t remote;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

template <int KS>
__global__ void __cluster_dims__(KS, 1, 1) __launch_bounds__(kThreads, 1)
router_tc_kernel(const __grid_constant__ Maps maps, int R, int E, int d, int nt,
                 float *__restrict__ logits, int *flags) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int S = stages_for(nt);
    const uint32_t b_bytes = (uint32_t)nt * 128u;
    const uint32_t sA = base, sB = base + (uint32_t)S * kABytes;
    const uint32_t ctl = sB + (uint32_t)S * b_bytes;
    // control block: full[kMaxStages], empty[kMaxStages], tfull, done, tmem slot, abort, ok
    const uint32_t full = ctl, empty = ctl + 8 * kMaxStages, tfull = ctl + 16 * kMaxStages,
                   done = tfull + 8;
    uint8_t *ctl_p = smem_raw + (ctl - raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl_p + 16 * kMaxStages + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ctl_p + 16 * kMaxStages + 20);
    volatile int *ok_flag = reinterpret_cast<volatile int *>(ctl_p + 16 * kMaxStages + 24);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = (int)(blockIdx.x % KS);  // the CTA's rank in its cluster
    const int r0 = (int)(blockIdx.x / KS) * nt, e0 = blockIdx.y * kM;
    const int kc_n = d / kBK, kc0 = kc_n * ks / KS, kc1 = kc_n * (ks + 1) / KS;
    clear_check_word(flags);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(done, 1);
        *abort_flag = 0;
        *ok_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&maps.w);
        prefetch_map(&maps.x);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(nt)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // x is written by the previous kernel
    const uint32_t tmem = *tmem_slot;

    uint32_t issued = 0, last_par = 0;  // producer: stages with a load in flight, parity
    bool mma_issued = false;
    if (warp == 0) {
        if (lane == 0) {
            for (int kc = kc0; kc < kc1; ++kc) {
                const int j = kc - kc0, s = j % S;
                const uint32_t ph = (uint32_t)(j / S) & 1u;
                if (!mbar_wait(empty + 8 * s, ph ^ 1u, abort_flag, flags)) break;
                mbar_expect_tx(full + 8 * s, kABytes + b_bytes);
                tma_load_2d(sA + s * kABytes, &maps.w, kc * kBK, e0, full + 8 * s);
                tma_load_2d(sB + s * b_bytes, &maps.x, kc * kBK, r0, full + 8 * s);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kM, (uint32_t)nt);
            bool ok = true;
            for (int kc = kc0; kc < kc1; ++kc) {
                const int j = kc - kc0, s = j % S;
                if (!mbar_wait(full + 8 * s, (uint32_t)(j / S) & 1u, abort_flag, flags)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = sA + s * kABytes, b = sB + s * b_bytes;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    mma_bf16(tmem, sw128_desc(a + 32u * k), sw128_desc(b + 32u * k), idesc,
                             (j | k) != 0);
                mma_issued = true;
                mma_commit(empty + 8 * s);
            }
            if (ok) mma_commit(tfull);  // arrives once every MMA above has completed
        }
        __syncwarp();
    }
    if (threadIdx.x == 32) *ok_flag = mbar_wait(tfull, 0, abort_flag, flags) ? 1 : 0;
    __syncthreads();
    const bool ok = *ok_flag != 0;
    if (!ok) {
        if (threadIdx.x == 0 && flags) atomicOr(flags, FLAG_WAIT_TIMEOUT);
        // nothing may be in flight when the ring is reused or the CTA exits
        if (warp == 0 && lane == 0)
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait(full + 8 * s, (last_par >> s) & 1u, nullptr, flags);
        if (warp == 1 && lane == 0 && mma_issued) {
            mma_commit(done);  // arrives once every MMA issued has completed
            mbar_wait(done, 0, nullptr, flags);
        }
        __syncwarp();
        __syncthreads();
    }
    tc_fence_after();
    const int el = warp * 32 + lane;
    if (KS == 1) {
        const int e = e0 + el;
        for (int c0 = 0; c0 < nt; c0 += 16) {
            uint32_t v[16];
            if (ok) tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int r = r0 + c0 + c;
                if (r < R && e < E) logits[(size_t)r * E + e] = ok ? __uint_as_float(v[c]) : NAN;
            }
        }
    } else {
        // this CTA's partial logits [nt][kM] over its drained stage ring (every load and MMA
        // on it has completed)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        float *part = reinterpret_cast<float *>(smem_raw + (sA - raw));
        for (int c0 = 0; c0 < nt; c0 += 16) {
            uint32_t v[16];
            if (ok) tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int c = 0; c < 16; ++c) part[(c0 + c) * kM + el] = ok ? __uint_as_float(v[c]) : NAN;
        }
        cluster_sync_all();
        // groups of 4 experts: every rank's 16-byte piece is requested before the adds
        const int rows = nt / KS, groups = rows * (kM / 4);
        for (int i = threadIdx.x; i < groups; i += kThreads) {
            const int rl = ks * rows + i / (kM / 4), ei = (i % (kM / 4)) * 4;
            const uint32_t off = sA + (uint32_t)((rl * kM + ei) * 4);
            float4 p[KS];
#pragma unroll
            for (int c = 0; c < KS; ++c) p[c] = ld_cluster_f32x4(off, (uint32_t)c);
            float4 sum = p[0];
#pragma unroll
            for (int c = 1; c < KS; ++c) {
                sum.x += p[c].x;
                sum.y += p[c].y;
                sum.z += p[c].z;
                sum.w += p[c].w;
            }
            const int r = r0 + rl, e = e0 + ei;
            if (r < R) {
                float *lr = logits + (size_t)r * E;
                if (e + 0 < E) lr[e + 0] = sum.x;
                if (e + 1 < E) lr[e + 1] = sum.y;
                if (e + 2 < E) lr[e + 2] = sum.z;
                if (e + 3 < E) lr[e + 3] = sum.w;
            }
        }
        cluster_sync_all();  // no CTA leaves while another still reads its partial
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(nt)
                     : "memory");
}

}  // namespace rtc

// From this many rows on, bf16 scores go to the tensor cores.
constexpr int kTcRows = 192;

// Up to this many rows the split-hidden shape is used.
constexpr int kSplitRows = 1024;

}  // namespace

bool router_tc_ok(const moe_layer_desc &L, int R) {
    if (L.dtype != MOE_DTYPE_BF16 || L.d % 64 != 0 || R < kTcRows) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    return major >= 10 && tc::encode_fn() != nullptr;
}

namespace {

// Raises the kernel's shared-memory limit once and returns how many of its KS-CTA clusters
// the device runs at once (one CTA per SM at any tile height; 0 if a query fails).
template <int KS>
int router_capacity(cudaError_t *err) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    static int clusters = 0;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(rtc::router_tc_kernel<KS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)rtc::kSmemBudget);
        if (attr != cudaSuccess) return;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(KS);
        cfg.blockDim = dim3(rtc::kThreads);
        cfg.dynamicSmemBytes = rtc::smem_bytes(32);
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = KS;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, rtc::router_tc_kernel<KS>, &cfg) !=
            cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
        }
    });
    *err = attr;
    return clusters;
}

// The tile height nt (tokens per CTA) and the clusters' split KS of the hidden dimension:
// among nt = 32 .. 256 and KS = 1 .. 8 (each CTA keeping at least 4 chunks of 64), the pair
// that puts the fewest bytes through one CTA ((128 + nt) rows of d / KS elements) with all
// of its clusters running at once; when no pair fits one wave, 256-row tiles without a
// split.
cudaError_t router_shape(int R, int E, int d, int &nt, int &ks) {
    const int et = (E + rtc::kM - 1) / rtc::kM, kc_n = d / rtc::kBK;
    cudaError_t err = cudaSuccess, e1;
    const int cap[4] = {router_capacity<1>(&e1), router_capacity<2>(&err),
                        router_capacity<4>(&err), router_capacity<8>(&err)};
    if (e1 != cudaSuccess) return e1;
    nt = 256;
    ks = 1;
    long best = -1;
    for (int t = 32; t <= 256; t *= 2)
        for (int k = 1, ki = 0; k <= 8 && kc_n / k >= 4; k *= 2, ++ki) {
            if (cap[ki] <= 0) continue;  // that split's clusters did not fit or the query failed
            const long clusters = (long)((R + t - 1) / t) * et;
            if (clusters > cap[ki]) continue;
            const long bytes = (long)(rtc::kM + t) * (d / k);
            if (best < 0 || bytes < best) {
                best = bytes;
                nt = t;
                ks = k;
            }
        }
    return cudaSuccess;
}

template <int KS>
cudaError_t launch_router_ks(const rtc::Maps &m, int R, const moe_layer_desc &L, int nt,
                             float *logits, int *flags, cudaStream_t s) {
    cudaError_t attr;
    router_capacity<KS>(&attr);
    if (attr != cudaSuccess) return attr;
    const dim3 grid((unsigned)(((R + nt - 1) / nt) * KS), (L.E + rtc::kM - 1) / rtc::kM);
    return launch_pdl(rtc::router_tc_kernel<KS>, grid, dim3(rtc::kThreads), rtc::smem_bytes(nt),
                      s, m, R, L.E, L.d, nt, logits, flags);
}

}  // namespace

cudaError_t launch_router_tc(const moe_layer_desc &L, const void *x, const void *Wr, int R,
                             float *logits, int *flags, cudaStream_t s) {
    int nt, ks;
    const cudaError_t err = router_shape(R, L.E, L.d, nt, ks);
    if (err != cudaSuccess) return err;
    rtc::Maps m{};
    const uint64_t wd[2] = {(uint64_t)L.d, (uint64_t)L.E}, xd[2] = {(uint64_t)L.d, (uint64_t)R};
    const uint64_t st[1] = {(uint64_t)L.d * 2};
    const uint32_t wb[2] = {(uint32_t)rtc::kBK, (uint32_t)rtc::kM};
    const uint32_t xb[2] = {(uint32_t)rtc::kBK, (uint32_t)nt};
    if (!tc::encode(&m.w, Wr, 2, wd, st, wb) || !tc::encode(&m.x, x, 2, xd, st, xb))
        return cudaErrorInvalidValue;
    switch (ks) {
    case 8: return launch_router_ks<8>(m, R, L, nt, logits, flags, s);
    case 4: return launch_router_ks<4>(m, R, L, nt, logits, flags, s);
    case 2: return launch_router_ks<2>(m, R, L, nt, logits, flags, s);
    default: return launch_router_ks<1>(m, R, L, nt, logits, flags, s);
    }
}

cudaError_t launch_router(const moe_layer_desc &L, const void *x, const void *Wr, int R,
                          float *logits, int *flags, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (router_tc_ok(L, R)) return launch_router_tc(L, x, Wr, R, logits, flags, s);
    if (R <= kSplitRows) {
        dim3 g((R + kRows - 1) / kRows, (L.E + kExp - 1) / kExp);
        if (L.dtype == MOE_DTYPE_BF16)
            return launch_pdl(router_splitd_kernel<__nv_bfloat16>, g, dim3(kWarps * 32), 0, s,
                              (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wr, R, L.d, L.E,
                              logits, flags);
        return launch_pdl(router_splitd_kernel<float>, g, dim3(kWarps * 32), 0, s,
                          (const float *)x, (const float *)Wr, R, L.d, L.E, logits, flags);
    }
    dim3 grid((R + kWarps * kRows - 1) / (kWarps * kRows), (L.E + kExp - 1) / kExp);
    if (L.dtype == MOE_DTYPE_BF16)
        return launch_pdl(router_kernel<__nv_bfloat16>, grid, dim3(kWarps * 32), 0, s,
                          (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wr, R, L.d, L.E,
                          logits, flags);
    return launch_pdl(router_kernel<float>, grid, dim3(kWarps * 32), 0, s, (const float *)x,
                      (const float *)Wr, R, L.d, L.E, logits, flags);
}

}  // namespace moe
