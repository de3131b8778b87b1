// Grouped SwiGLU experts on the 5th-generation tensor cores (tcgen05 + TMA + TMEM)
// ("MoE and speculative decoding" blog, "grouped GEMM for active experts"):
//   phase 1  h   = silu(X_e W_gate[e]^T) * (X_e W_up[e]^T)      (bf16 out)
//   phase 2  O_e = h W_down[e]^T                                (bf16 out)
// for every expert e with assignments, X_e its token rows in permuted order.
//
// A verification block routes only ~4-20 tokens to an expert, so the weights are
// the large operand: each unit of work streams one 128-row weight tile through
// shared memory once and multiplies it by all of the expert's tokens (up to 256).
// The weight tile is the MMA's A operand (M = 128 rows: 64 W_gate rows stacked on
// the same 64 W_up rows in phase 1, 128 W_down rows in phase 2), the token rows are
// the B operand (N = tokens rounded up to 16), and the fp32 accumulator lives in
// tensor memory. Both operands are K-major bf16 tiles of 64 elements (one 128-byte
// swizzle atom) loaded by TMA with 128-byte swizzling, which is the layout the
// tcgen05 shared-memory descriptors describe.
//
// Both phases run in one persistent launch, one CTA per SM (320 threads,
// warp-specialised):
//   warp 0       TMA producer (one lane): takes unit tickets from a global counter
//                (every phase-1 unit before any phase-2 unit), passes each ticket to
//                the other roles through a small shared-memory queue, and fills a ring
//                of `stages` buffers
//   warp 1       TMEM allocator and MMA issuer (one lane)
//   warps 2..9   epilogue, two teams of four (warps 2-5, 6-9) taking alternate
//                16-column chunks of the accumulator: tcgen05.ld (each warp may read
//                the 32 TMEM lanes of its quadrant, warp % 4), apply SwiGLU or store O;
//                each warp turns its 32 outputs x 16 tokens around in a 1 KB staging
//                buffer and writes them as 16-byte pieces of the output rows
// At the start the epilogue warps copy the row-tile list (expert, first permuted row,
// tokens, slot) into shared memory, so looking up a unit between two units costs no
// global round trip. Two 256-column accumulators alternate so the epilogue of one unit
// overlaps the MMAs of the next. A unit is one weight tile x one row tile (<= 256
// tokens of one expert); when every row tile of a launch has 32 or more tokens (and the
// launch has enough units per CTA) a unit is two weight tiles x one row tile instead,
// whose two MMAs per k-step share the stage's token rows, so each token row crosses into
// shared memory half as often: tiles of up to 128 tokens fill the two 128-column halves of
// one accumulator (two units still alternate), taller tiles one accumulator each. In
// phase 1 a pair's first MMA takes the 128 gate rows of both weight tiles and the second
// their 128 up rows, so every TMEM lane holds a gate row and its up row and each warp
// forms h alone; in phase 2 each epilogue team stores one tile. A phase-2 unit needs the
// whole h of its row tile: the epilogue that finishes a phase-1 unit publishes it with a
// release increment of the row tile's counter, and the producer of a phase-2 unit waits
// for the count with acquire loads before its TMA reads h. Tickets are handed out in
// order, so every phase-1 unit is owned by a running CTA before any CTA waits on one: no
// deadlock even when fewer CTAs than SMs are resident.
//
// Every wait is bounded: after 2 s a wait gives up, sets the workspace check bit
// FLAG_WAIT_TIMEOUT and makes the CTA stop; the CTA then waits (again bounded) for
// its TMA loads and MMAs in flight, frees its tensor memory and exits.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kEpiWarps = 8;                // two teams of four, one warp per TMEM quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kBK = 64;                     // K elements per stage: one 128-B swizzle atom
constexpr int kM = 128;                     // MMA M: weight rows per unit
constexpr int kAccCols = 256;               // TMEM columns per accumulator (max N)
constexpr int kTmemCols = 2 * kAccCols;     // two accumulators
constexpr uint32_t kABytes = kM * kBK * 2;  // 16 KB weight tile per stage
constexpr int kBoxes = 16;                  // token-row boxes of 16, 32, 48, ..., 256 rows
constexpr int kSgStride = 17;               // padded row of the silu(gate) exchange buffer
constexpr int kSgFloats = 64 * kSgStride;   // one buffer; two per team (double-buffered)
constexpr int kStageBytes = 16 * 64;        // per epilogue warp: 16 tokens x 32 bf16 outputs
constexpr int kMaxStages = 12;              // pipeline stages at most
constexpr int kCtlBytes = 512;              // barriers and slots (16 * kMaxStages + 152 bytes)

struct Maps {
    CUtensorMap wg;           // W_gate [S][f][d], box 64 x 64 x 1
    CUtensorMap wu;           // W_up   [S][f][d], box 64 x 64 x 1
    CUtensorMap wd;           // W_down [S][d][f], box 64 x 128 x 1
    CUtensorMap bx[kBoxes];   // gathered token rows x [A][d], box 64 x 16 (i + 1)
    CUtensorMap bh[kBoxes];   // activations h [A][f], box 64 x 16 (i + 1)
};

struct Params {
    int d, f;
    int mt1, mt2;  // weight tiles per expert: f / 64 (phase 1), ceil(d / 128) (phase 2)
    int smem;      // dynamic shared memory of the launch (bytes)
    int tbl_cap;   // row tiles described in the shared-memory table (the rest: global reads)
    int slots;     // expert slots in the weight pool
    int pair_min;    // row-tile heights from this up to 128 tokens take weight-tile pairs,
    int pair_units;  // when the launch has at least this many single-tile units per CTA
    int pair_max;    // tallest row tile that takes pairs (up to 128 tokens: the halves of one
                     // accumulator; up to 256: one accumulator per tile, both for one unit)
    const int *rowtiles, *slot;
    const uint8_t *pass;  // experts computed by this launch (null: all)
    int *flags;
    int *sched;    // [0] ticket counter, [1 + rt] finished phase-1 units of row tile rt
    __nv_bfloat16 *h, *o;
};

// Named barriers (bar.sync is warp-aligned: reconverge first): one per epilogue team of
// four warps (ids 1, 2), and one over all eight epilogue warps (id 3).
__device__ __forceinline__ void team_bar(int team) {
    __syncwarp();
    asm volatile("bar.sync %0, 128;" ::"r"(1 + team) : "memory");
}
__device__ __forceinline__ void epi_bar() {
    __syncwarp();
    asm volatile("bar.sync 3, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Stores one warp's outputs of a 16-token chunk. Lane l holds output column col0 + l of
// tokens c0 .. c0 + 15 (val[c], fp32); the warp writes them, rounded to bf16, into its
// staging buffer in token-major order and reads them back as 16-byte pieces (token c,
// columns col0 + 8 g .. + 8), so each store instruction writes 8 tokens x 64 contiguous
// bytes instead of one 2-byte element per lane. out points at token c0's row, column col0;
// ld is the row stride in elements; tokens from `left` on, or a column block past the
// output's width (cols_ok false), are not written.
__device__ __forceinline__ void store_chunk(uint8_t *stg, const float (&val)[16], int lane,
                                            __nv_bfloat16 *out, size_t ld, int left,
                                            bool cols_ok) {
    __nv_bfloat16 *sb = reinterpret_cast<__nv_bfloat16 *>(stg);
    __syncwarp();  // the previous chunk's reads of the buffer are done
#pragma unroll
    for (int c = 0; c < 16; ++c) sb[c * 32 + lane] = __float2bfloat16_rn(val[c]);
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int piece = h * 32 + lane, c = piece >> 2, g = piece & 3;
        const uint4 v = *reinterpret_cast<const uint4 *>(stg + c * 64 + g * 16);
        if (cols_ok && c < left) *reinterpret_cast<uint4 *>(out + (size_t)c * ld + g * 8) = v;
    }
}

struct Unit {
    int phase, rt, m, e, row0, ntok, slot;  // row0: the row tile's first permuted row
    int nm;                                 // weight tiles m, m + 1, ... of this unit (1 or 2)
    int group;                              // tiles of this expert (they share its weights)
};

// Row tile rt -> {expert, first permuted row, tokens | index in the expert's group << 12 |
// group size << 22, code}; code is the expert's slot, -1 for an expert outside this
// launch's expert pass, -2 for a slot outside the pool. (tokens <= 256, groups < 1024.)
__device__ __forceinline__ int4 row_tile(const Params &p, int rt) {
    const int *t = p.rowtiles + kRowTileHeader + 4 * rt;
    const int e = t[0], row0 = t[1], ntok = t[2];
    const int jg = (t[3] >> 16) & 1023, g = max(1, min(t[3] & 0xffff, 1023));
    int code;
    if (p.pass && !p.pass[e]) {
        code = -1;
    } else {
        const int sl = p.slot ? p.slot[e] : e;
        code = (sl >= 0 && sl < p.slots && ntok > 0) ? sl : -2;
    }
    return make_int4(e, row0, ntok | (jg << 12) | (g << 22), code);
}

__device__ __forceinline__ int4 tile_at(const Params &p, int rt, const int4 *tbl) {
    return (tbl && rt < p.tbl_cap) ? tbl[rt] : row_tile(p, rt);
}

// Ticket u -> unit. A unit is W consecutive weight tiles (W = 1, or 2 when the launch pairs
// them) of one row tile: mu = ceil(mt / W) units per row tile and phase, the last one short
// when W does not divide mt. Tickets [0, U1) are phase 1, the rest phase 2; within a phase the
// tickets of an expert's row tiles [f, f + g) form one block of g * mu tickets taken unit
// by unit: ticket f * mu + i * g + j is unit i of row tile f + j, so the g tiles that read
// the same weights are handed out together and run at the same time (the second read of
// those weights hits L2). The row tile's entry comes from the
// shared-memory table when it holds it (tbl != nullptr). Returns 0 for a unit to compute,
// 1 for one outside this launch's expert pass, 2 for an expert whose slot is outside the
// pool (skipped and flagged).
__device__ __forceinline__ int decode(const Params &p, int U1, int u, int W, Unit &w,
                                      const int4 *tbl) {
    const bool ph1 = u < U1;
    const int v = ph1 ? u : u - U1, mt = ph1 ? p.mt1 : p.mt2;
    const int mu = (mt + W - 1) / W;
    const int rt0 = v / mu;  // a tile of the right group (the order within differs)
    int4 t = tile_at(p, rt0, tbl);
    const int jg = (t.z >> 12) & 1023, g = ((unsigned)t.z >> 22) & 1023;
    w.phase = ph1 ? 1 : 2;
    int i;
    if (g <= 1) {  // an expert in one tile (every expert of small blocks)
        w.rt = rt0;
        i = v - rt0 * mu;
    } else {
        const int f = rt0 - jg;
        const int local = v - f * mu;
        i = local / g;
        w.rt = f + (local - i * g);
        if (w.rt != rt0) t = tile_at(p, w.rt, tbl);
    }
    w.m = i * W;
    w.nm = min(W, mt - w.m);
    w.e = t.x;
    w.row0 = t.y;
    w.ntok = t.z & 4095;
    w.group = g;
    w.slot = t.w;
    return t.w >= 0 ? 0 : (t.w == -1 ? 1 : 2);
}

constexpr int kQ = 4;  // ticket queue depth

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kThreads, 1)
ffn_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    // layout: control block, exchange buffers, row-tile table, then the ring of stages
    // (sized after the previous kernel has finished, from the row-tile height)
    uint8_t *ctl = gbase;
    const uint32_t ctl_s = base;
    // control block: full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2], done,
    // qfull[kQ], qempty[kQ], then tmem slot, abort, epilogue verdict[2], epilogue
    // ticket[2], ticket queue[kQ], then the table barrier
    const uint32_t full = ctl_s, empty = ctl_s + 8 * kMaxStages, tfull = ctl_s + 16 * kMaxStages,
                   tempty = tfull + 16, done = tempty + 16, qfull = done + 8,
                   qempty = qfull + 8 * kQ;
    int *ints = reinterpret_cast<int *>(ctl + 16 * kMaxStages + 40 + 16 * kQ);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ints);
    volatile int *abort_flag = ints + 1;
    volatile int *epi_ok = ints + 2;    // [2]
    volatile int *epi_u = ints + 4;     // [2]
    volatile int *queue = ints + 6;     // [kQ]
    const uint32_t tbl_bar = ctl_s + 16 * kMaxStages + 144;  // the row-tile table is filled
    // per epilogue warp, its outputs of one 16-token chunk in token-major order, so that
    // they leave for global memory as 16-byte pieces of the output rows
    uint8_t *stage_all = ctl + kCtlBytes;
    int4 *tbl = reinterpret_cast<int4 *>(stage_all + kEpiWarps * kStageBytes);  // [tbl_cap]
    // the silu(gate) exchange buffers, [team][2][64][kSgStride]: only launches of single
    // weight tiles have them (a pair keeps gate and up in the same TMEM lanes)
    float *sg_all = reinterpret_cast<float *>(tbl + p.tbl_cap);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + 8 * a, 1);
            mbar_init(tempty + 8 * a, 32 * kEpiWarps);
        }
        mbar_init(done, 1);
        mbar_init(tbl_bar, 32 * kEpiWarps);
        for (int q = 0; q < kQ; ++q) {
            mbar_init(qfull + 8 * q, 1);
            mbar_init(qempty + 8 * q, 2);  // the MMA lane and one epilogue thread
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&maps.wg);
        prefetch_map(&maps.wu);
        prefetch_map(&maps.wd);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // everything above only touched this CTA's own resources: wait for the previous
    // kernel before reading the routing tables it wrote
    pdl_wait();
    const uint32_t tmem = *tmem_slot;
    const int n_rt = p.rowtiles[0];
    // the ring: as many stages as fit of W 16 KB weight tiles + a token buffer of the
    // row-tile height (every row tile of this launch has at most that many tokens). With
    // row tiles of pair_min to pair_max tokens a unit takes two weight tiles (W = 2): two
    // MMAs per k-step read the same token tile, so the token rows cross into shared memory
    // once per two weight tiles. Only with enough units per CTA: a small union in units
    // twice as long leaves CTAs idle at the end.
    const int height = p.rowtiles[1];
    const uint32_t b_bytes = (uint32_t)height * 128u;
    const uint32_t pre = base + kCtlBytes + kEpiWarps * kStageBytes + (uint32_t)p.tbl_cap * 16u;
    const uint32_t end = raw + (uint32_t)p.smem;
    const uint32_t ring2 = (pre + 1023u) & ~1023u;
    const int W = (p.pair_min > 0 && height >= p.pair_min && height <= p.pair_max &&
                   n_rt * (p.mt1 + p.mt2) >= p.pair_units * (int)gridDim.x &&
                   end - ring2 >= 2u * (2u * kABytes + b_bytes))
                      ? 2
                      : 1;
    const uint32_t ring = W == 2 ? ring2 : (pre + 2 * 2 * kSgFloats * 4 + 1023u) & ~1023u;
    const uint32_t avail = end - ring;
    // accumulators in rotation and the column offset of a unit's second weight tile: pairs
    // over tiles of up to 128 tokens share one 256-column accumulator and two units
    // alternate; taller pairs take both accumulators, so a unit's MMAs wait for the
    // previous unit's epilogue (the ring keeps filling meanwhile)
    const int nacc = (W == 2 && height > kAccCols / 2) ? 1 : 2;
    const uint32_t sub_cols = nacc == 1 ? (uint32_t)kAccCols : (uint32_t)(kAccCols / 2);
    const uint32_t a_bytes = (uint32_t)W * kABytes;  // weight bytes of a stage
    const int S = max(1, min(kMaxStages, (int)(avail / (a_bytes + b_bytes))));
    const uint32_t sA = ring, sB = ring + (uint32_t)S * a_bytes;
    const int U1 = n_rt * ((p.mt1 + W - 1) / W), U = U1 + n_rt * ((p.mt2 + W - 1) / W);
    // the epilogue warps copy the row-tile list into shared memory (expert, first row,
    // tokens, slot), so that a unit's lookup costs no global round trips
    if (warp >= 2) {
        for (int rt = threadIdx.x - 64; rt < min(n_rt, p.tbl_cap); rt += 32 * kEpiWarps)
            tbl[rt] = row_tile(p, rt);
        mbar_arrive(tbl_bar);
    }

    uint32_t issued = 0, last_par = 0;  // producer: stages with a load issued, parity of it
    bool mma_issued = false;

    if (warp == 0) {
        if (lane == 0) {
            // weights read by one row tile stream through L2 once (evict first); weights
            // that the sibling tiles of a group read at the same time stay in L2 for them
            const uint64_t pol_once = evict_first_policy(), pol_shared = evict_normal_policy();
            int s = 0, qs = 0;
            uint32_t ph = 0, qph = 0;
            bool ok = mbar_wait(tbl_bar, 0, abort_flag, p.flags);
            while (ok) {
                int u = atomicAdd(p.sched, 1);
                if (u >= U) u = -1;
                if (!mbar_wait(qempty + 8 * qs, qph ^ 1u, abort_flag, p.flags)) break;
                queue[qs] = u;
                mbar_arrive(qfull + 8 * qs);
                if (++qs == kQ) {
                    qs = 0;
                    qph ^= 1u;
                }
                if (u < 0) break;
                Unit w;
                const int dc = decode(p, U1, u, W, w, tbl);
                if (dc != 0) {
                    if (dc == 2) atomicOr(p.flags, FLAG_BAD_EXPERT);
                    continue;
                }
                if (w.phase == 2) {  // wait until the row tile's h is complete
                    const unsigned long long t0 = now_ns();
                    while (ld_acquire(p.sched + 1 + w.rt) < p.mt1) {
                        __nanosleep(64);
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        if (now_ns() - t0 > kTimeoutNs) {
                            *abort_flag = 1;
                            atomicOr(p.flags, FLAG_WAIT_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                // one box of exactly the row tile's tokens rounded up to 16 rows
                const int bxi = ((w.ntok + 15) >> 4) - 1;
                const uint32_t bb = (uint32_t)(bxi + 1) * 16u * 128u;
                const int brow = w.row0;
                const int kchunks = (w.phase == 1 ? p.d : p.f) / kBK;
                const CUtensorMap *bmap = w.phase == 1 ? &maps.bx[bxi] : &maps.bh[bxi];
                const uint64_t pol = w.group > 1 ? pol_shared : pol_once;
                for (int kc = 0; kc < kchunks; ++kc) {
                    if (!mbar_wait(empty + 8 * s, ph ^ 1u, abort_flag, p.flags)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full + 8 * s;
                    const uint32_t a = sA + (uint32_t)s * a_bytes;
                    if (w.phase == 1 && W == 2) {
                        // a pair: the gate rows of both tiles (128) in the stage's first
                        // tile, their up rows in the second; a missing second tile (past f)
                        // reads as zeros
                        mbar_expect_tx(fb, 2u * kABytes + bb);
                        tma_load_3d(a, &maps.wg, kc * kBK, w.m * 64, w.slot, fb, pol);
                        tma_load_3d(a + kABytes / 2, &maps.wg, kc * kBK, w.m * 64 + 64, w.slot,
                                    fb, pol);
                        tma_load_3d(a + kABytes, &maps.wu, kc * kBK, w.m * 64, w.slot, fb, pol);
                        tma_load_3d(a + kABytes + kABytes / 2, &maps.wu, kc * kBK,
                                    w.m * 64 + 64, w.slot, fb, pol);
                    } else if (w.phase == 1) {
                        // one tile: 64 gate rows over the same 64 up rows
                        mbar_expect_tx(fb, kABytes + bb);
                        tma_load_3d(a, &maps.wg, kc * kBK, w.m * 64, w.slot, fb, pol);
                        tma_load_3d(a + kABytes / 2, &maps.wu, kc * kBK, w.m * 64, w.slot, fb,
                                    pol);
                    } else {
                        mbar_expect_tx(fb, (uint32_t)w.nm * kABytes + bb);
                        for (int t = 0; t < w.nm; ++t)
                            tma_load_3d(a + (uint32_t)t * kABytes, &maps.wd, kc * kBK,
                                        (w.m + t) * kM, w.slot, fb, pol);
                    }
                    tma_load_2d(sB + (uint32_t)s * b_bytes, bmap, kc * kBK, brow, fb);
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0, it = 0, qs = 0;
            uint32_t ph = 0, qph = 0;
            bool ok = mbar_wait(tbl_bar, 0, abort_flag, p.flags);
            while (ok) {
                if (!mbar_wait(qfull + 8 * qs, qph, abort_flag, p.flags)) break;
                const int u = queue[qs];
                mbar_arrive(qempty + 8 * qs);
                if (++qs == kQ) {
                    qs = 0;
                    qph ^= 1u;
                }
                if (u < 0) break;
                Unit w;
                if (decode(p, U1, u, W, w, tbl) != 0) continue;
                const int acc = nacc == 2 ? it & 1 : 0;
                const uint32_t aph = (uint32_t)(nacc == 2 ? it >> 1 : it) & 1u;
                ++it;
                if (!mbar_wait(tempty + 8 * acc, aph ^ 1u, abort_flag, p.flags)) break;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(kM, (uint32_t)((w.ntok + 15) & ~15));
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kAccCols);
                const int kchunks = (w.phase == 1 ? p.d : p.f) / kBK;
                for (int kc = 0; kc < kchunks; ++kc) {
                    if (!mbar_wait(full + 8 * s, ph, abort_flag, p.flags)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b = sB + (uint32_t)s * b_bytes;
                    // tile t of the stage accumulates into columns [t sub_cols, + N): in phase
                    // 1 of a pair the gate and the up rows, else weight tile m + t
                    const int ntiles = (W == 2 && w.phase == 1) ? 2 : w.nm;
                    for (int t = 0; t < ntiles; ++t) {
                        const uint32_t a = sA + (uint32_t)s * a_bytes + (uint32_t)t * kABytes;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k)
                            mma_bf16(d_tmem + (uint32_t)t * sub_cols, sw128_desc(a + 32u * k),
                                     sw128_desc(b + 32u * k), idesc, (kc | k) != 0);
                    }
                    mma_issued = true;
                    mma_commit(empty + 8 * s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) mma_commit(tfull + 8 * acc);
            }
        }
        __syncwarp();
    } else {
        const int q = warp & 3;            // TMEM lane quadrant of this warp
        const int team = (warp - 2) >> 2;  // epilogue team: warps 2-5 or 6-9
        const int row = q * 32 + lane;     // accumulator row
        float *sg = sg_all + team * 2 * kSgFloats;
        uint8_t *stg = stage_all + (warp - 2) * kStageBytes;
        int it = 0, qs = 0, turn = 0;
        uint32_t qph = 0;
        for (;; turn ^= 1) {
            // thread 64 takes the next ticket and the named barrier hands it to the
            // others; the slots alternate so a fast thread cannot overwrite a value a
            // slow one has yet to read
            if (threadIdx.x == 64) {
                int u = -1;
                if (mbar_wait(qfull + 8 * qs, qph, abort_flag, p.flags)) {
                    u = queue[qs];
                    mbar_arrive(qempty + 8 * qs);
                }
                epi_u[turn] = u;
            }
            if (++qs == kQ) {
                qs = 0;
                qph ^= 1u;
            }
            epi_bar();
            const int u = epi_u[turn];
            if (u < 0) break;
            Unit w;
            if (decode(p, U1, u, W, w, tbl) != 0) continue;
            const int acc = nacc == 2 ? it & 1 : 0;
            const uint32_t aph = (uint32_t)(nacc == 2 ? it >> 1 : it) & 1u;
            ++it;
            if (threadIdx.x == 64)
                epi_ok[acc] = mbar_wait(tfull + 8 * acc, aph, abort_flag, p.flags);
            epi_bar();
            if (!epi_ok[acc]) break;  // uniform over the eight warps
            tc_fence_after();
            const int N = (w.ntok + 15) & ~15;
            // one weight tile per unit: the two teams take alternate 16-column chunks of the
            // accumulator; a pair of weight tiles: team t takes all of tile t's columns
            const int sub = W == 2 ? team : 0;           // the weight tile this team stores
            const int c_first = W == 2 ? 0 : team * 16, c_step = W == 2 ? 16 : 32;
            const int m = w.m + sub;
            const uint32_t taddr = tmem + (uint32_t)(acc * kAccCols) + (uint32_t)sub * sub_cols +
                                   ((uint32_t)(q * 32) << 16);
            const size_t row0 = (size_t)w.row0;
            if (w.phase == 1 && W == 2) {
                // a pair: lane r of the accumulator holds gate row w.m * 64 + r in the first
                // tile's columns and the same up row in the second's, so each warp forms
                // h for its 32 rows by itself; the teams take alternate 16-token chunks
                const uint32_t tg = tmem + (uint32_t)(acc * kAccCols) + ((uint32_t)(q * 32) << 16);
                const int frow = w.m * 64 + q * 32;  // this warp's first h column
                for (int c0 = team * 16; c0 < N; c0 += 32) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tg + (uint32_t)c0, g);
                    tmem_ld16(tg + sub_cols + (uint32_t)c0, u);
                    float hv[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float gv = __uint_as_float(g[c]);
                        hv[c] = __fdividef(gv, 1.f + __expf(-gv)) * __uint_as_float(u[c]);
                    }
                    store_chunk(stg, hv, lane, p.h + (row0 + (size_t)c0) * p.f + frow,
                                (size_t)p.f, w.ntok - c0, frow < p.f);
                }
                tc_fence_before();
                mbar_arrive(tempty + 8 * acc);
                epi_bar();
                if (threadIdx.x == 64) {
                    __threadfence();
                    atomicAdd(p.sched + 1 + w.rt, w.nm);
                }
            } else if (w.phase == 1) {
                // within a team the gate warps (quadrants 0, 1) hand silu(gate) to the up
                // warps (quadrants 2, 3) through a double-buffered exchange buffer: one
                // team barrier per chunk (a buffer is rewritten two chunks later, after
                // the up warps have passed the barrier in between)
                int j = 0;
                for (int c0 = c_first; sub < w.nm && c0 < N; c0 += c_step, ++j) {
                    float *buf = sg + (j & 1) * kSgFloats;
                    uint32_t v[16];
                    tmem_ld16(taddr + (uint32_t)c0, v);
                    if (q < 2) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const float g = __uint_as_float(v[c]);
                            buf[row * kSgStride + c] = __fdividef(g, 1.f + __expf(-g));
                        }
                    }
                    team_bar(team);
                    if (q >= 2) {
                        const int i = row - 64;
                        float hv[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            hv[c] = buf[i * kSgStride + c] * __uint_as_float(v[c]);
                        store_chunk(stg, hv, lane,
                                    p.h + (row0 + (size_t)c0) * p.f + (size_t)m * 64 + (q - 2) * 32,
                                    (size_t)p.f, w.ntok - c0, true);
                    }
                }
                // the accumulator is read: hand it back to the MMA issuer first, then
                // publish h (every h store of this unit precedes the barrier)
                tc_fence_before();
                mbar_arrive(tempty + 8 * acc);
                epi_bar();
                if (threadIdx.x == 64) {
                    __threadfence();
                    atomicAdd(p.sched + 1 + w.rt, w.nm);
                }
            } else {
                // this warp's 32 output columns: all inside d or all past it (d is a
                // multiple of 64)
                const int col0 = m * kM + q * 32;
                for (int c0 = c_first; sub < w.nm && c0 < N; c0 += c_step) {
                    uint32_t v[16];
                    tmem_ld16(taddr + (uint32_t)c0, v);
                    float ov[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) ov[c] = __uint_as_float(v[c]);
                    store_chunk(stg, ov, lane, p.o + (row0 + (size_t)c0) * p.d + col0,
                                (size_t)p.d, w.ntok - c0, col0 < p.d);
                }
                tc_fence_before();
                mbar_arrive(tempty + 8 * acc);
            }
        }
    }

    // ---- teardown: nothing may be in flight when the CTA frees TMEM and exits ----
    __syncthreads();
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; ++s)
            if (issued & (1u << s)) mbar_wait(full + 8 * s, (last_par >> s) & 1u, nullptr, p.flags);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
        mma_commit(done);
        mbar_wait(done, 0, nullptr, p.flags);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// Gathers the token rows of every assignment into permuted order: xp[pos[a]] = x[a / k]
// for assignment a (row a / k, slot a % k), a warp per assignment, strided over the grid.
// The source row needs no lookup, so the row's loads (all of a lane's pieces of a chunk of
// 256 16-byte pieces at once) and the destination's lookup are in flight together. Block 0
// also zeroes the expert kernel's ticket counter and row-tile counters.
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32)
gather_rows_kernel(const __nv_bfloat16 *__restrict__ x, const int *__restrict__ pos, int A,
                   int k, int d, __nv_bfloat16 *__restrict__ xp, int *__restrict__ sched,
                   int n_sched) {
    pdl_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_sched; i += blockDim.x) sched[i] = 0;
    const int lane = threadIdx.x & 31;
    const int vec = d / 8;  // 16-byte pieces of a row
    for (int a = blockIdx.x * kGatherWarps + (threadIdx.x >> 5); a < A;
         a += gridDim.x * kGatherWarps) {
        const int p = pos[a];  // -1: a skipped (bad or repeated) expert id
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(a / k) * d);
        uint4 *dst = reinterpret_cast<uint4 *>(xp + (size_t)max(p, 0) * d);
        for (int i0 = 0; i0 < vec; i0 += 256) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + lane + 32 * j < vec) v[j] = __ldg(src + i0 + lane + 32 * j);
            if (p < 0) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + lane + 32 * j < vec) dst[i0 + lane + 32 * j] = v[j];
        }
    }
}

// ------------------------------------------------------------------- host

// Weight pool [S][rows][K] as a 3-D map with a 64 x box_rows x 1 box.
bool encode_weights(CUtensorMap *m, const void *w, int S, int rows, int K, int box_rows) {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)rows, (uint64_t)S};
    const uint64_t st[2] = {(uint64_t)K * 2, (uint64_t)rows * K * 2};
    const uint32_t box[3] = {(uint32_t)kBK, (uint32_t)box_rows, 1};
    return encode(m, w, 3, dims, st, box);
}

// Token rows [A][K] as 2-D maps with 64 x 16 (i + 1) boxes, for the row-tile heights up to
// `cap` rows that a launch can meet.
bool encode_rows(CUtensorMap *maps, const void *t, int A, int K, int cap) {
    for (int i = 0; i < kBoxes && 16 * i < cap; ++i) {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)A};
        const uint64_t st[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {(uint32_t)kBK, (uint32_t)(16 * (i + 1))};
        if (!encode(&maps[i], t, 2, dims, st, box)) return false;
    }
    return true;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Shared memory besides the ring and the table: alignment slack, control block,
// exchange buffers.
constexpr size_t kFixedSmem =
    1024 + kCtlBytes + 2 * 2 * kSgFloats * sizeof(float) + kEpiWarps * kStageBytes;
constexpr size_t kSmemBudget = 227 * 1024;
// Row tiles of at least kPairMinRows tokens (and at most kPairMaxRows) take weight-tile
// pairs: below it the token rows are a small part of a stage and single tiles balance the
// CTAs better.
// A launch on every SM pairs only with this many single-tile units per CTA (a union of ~26
// experts of the Qwen3-shaped layer has about 5, and units twice as long would leave CTAs
// idle at the end); a launch held to fewer CTAs runs beside other work, which fills the
// SMs its CTAs leave at the end, and pairs at any unit count.
constexpr int kPairMinRows = 32;
constexpr int kPairMaxRows = 256;
constexpr int kPairMinUnitsPerCta = 8;

}  // namespace

bool ffn_tc_supported(const moe_layer_desc &L) {
    if (L.dtype != MOE_DTYPE_BF16 || L.d % 64 != 0 || L.f % 64 != 0) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    return major >= 10 && encode_fn() != nullptr;
}

cudaError_t launch_ffn_tc(const FfnArgs &a, cudaStream_t s) {
    const int A = a.R * a.k;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    // the tallest row tile a launch can meet: kMaxRowTile tokens, or R if fewer (a row
    // picks an expert at most once), rounded up to 16; the kernel sizes its stages from
    // the height the permute kernel chose
    const int box_cap = ((std::min(a.R, kMaxRowTile) + 15) / 16) * 16;
    // the row-tile table takes what two stages of the tallest tiles leave (a stage of two
    // weight tiles when the tiles can pair); row tiles past it are read from global memory
    const size_t two_stages =
        2 * std::max(kABytes + (size_t)box_cap * 128,
                     box_cap >= kPairMinRows
                         ? 2 * kABytes + (size_t)std::min(box_cap, kPairMaxRows) * 128
                         : 0);
    const int tbl_cap = (int)std::min<size_t>((size_t)max_rowtiles(a.E, A),
                                              (kSmemBudget - kFixedSmem - two_stages) / 16);
    const size_t smem = kSmemBudget;
    const int S = a.slots;

    Maps m{};
    if (!encode_weights(&m.wg, a.Wg, S, a.f, a.d, 64) ||
        !encode_weights(&m.wu, a.Wu, S, a.f, a.d, 64) ||
        !encode_weights(&m.wd, a.Wd, S, a.d, a.f, kM) ||
        !encode_rows(m.bx, a.xp, A, a.d, box_cap) || !encode_rows(m.bh, a.h, A, a.f, box_cap))
        return cudaErrorInvalidValue;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(ffn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemBudget);
    });
    if (attr_err != cudaSuccess) return attr_err;

    const int n_sched = 1 + max_rowtiles(a.E, A);
    const int gather_ctas =
        std::max(1, std::min((A + kGatherWarps - 1) / kGatherWarps, 16 * nsm));
    cudaError_t err = launch_pdl(gather_rows_kernel, dim3(gather_ctas), dim3(kGatherWarps * 32),
                                 0, s, (const __nv_bfloat16 *)a.x, a.pos, A, a.k, a.d,
                                 (__nv_bfloat16 *)a.xp, a.sched, n_sched);
    if (err != cudaSuccess) return err;
    Params p{};
    p.d = a.d;
    p.f = a.f;
    p.mt1 = a.f / 64;
    p.mt2 = (a.d + kM - 1) / kM;
    p.smem = (int)smem;
    p.tbl_cap = tbl_cap;
    p.slots = S;
    p.pair_min = kPairMinRows;
    p.pair_units = a.max_ctas > 0 && a.max_ctas < nsm ? 0 : kPairMinUnitsPerCta;
    p.pair_max = kPairMaxRows;
    p.rowtiles = a.rowtiles;
    p.slot = a.slot;
    p.pass = a.pass;
    p.flags = a.flags;
    p.sched = a.sched;
    p.h = (__nv_bfloat16 *)a.h;
    p.o = (__nv_bfloat16 *)a.o;
    const int ctas = a.max_ctas > 0 ? std::min(nsm, a.max_ctas) : nsm;
    return launch_pdl(ffn_tc_kernel, dim3(ctas), dim3(kThreads), smem, s, m, p);
}

}  // namespace moe
