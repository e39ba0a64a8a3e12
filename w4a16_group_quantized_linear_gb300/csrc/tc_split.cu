// Tensor-core GEMM of the W4A16 layer for group-32 weights: the routed-expert
// layer of the LLM170 page's "g32, MoE resident" models, and dense layers of
// group 32 (sm_103a: TMA, tcgen05 MMA, TMEM).
//
// At group 32 the group-partial design of tc_linear.cu (one fp32 TMEM partial
// per scale group, scaled by the epilogue) pays one TMEM round trip per 32 k,
// which takes longer than the group's two MMAs. Here the scale goes into the A
// operand instead, exactly. For a scale s (fp16) and an integer q in [-8, 7]
// the product s*q has at most 15 significant bits, so it splits into two fp16
// values with no rounding at all:
//
//     hi = fp16_rn(s*q),   lo = s*q - hi   (one fused fp16 multiply-add; exact)
//
// lo is exact because s*q - hi is a multiple of ulp(s) (q is an integer) and
// smaller than ulp(hi), so it has at most 4 significant bits; it is never
// below the fp16 subnormal step because ulp(s) is not. Then
//
//     y[m, n] = sum_k x[m, k] * (hi[n, k] + lo[n, k])
//
// with every product x*hi, x*lo exact in fp32: two MMAs per 16 k into one fp32
// TMEM accumulator over all of K, and no per-group epilogue. hi overflows
// fp16 only when |s| > 8188 (|s q| > 65504); a row whose largest scale is that
// large is computed with its scales multiplied by a power of two 2^-e (exact
// while they stay normal fp16 numbers) and its result multiplied by 2^e.
//
// Formulation ("swap AB", as in tc_linear.cu): D[n, m] = sum_k W^[n, k] x[m, k].
// Persistent: one CTA per SM walks the tiles (expert, token tile, 128-row
// weight tile) t = blockIdx.x, blockIdx.x + gridDim.x, ... with the weight-row
// tile fastest (the tiles that share an x tile run side by side). A token tile
// holds up to 256 tokens: the MMA issue rate, not the tensor math, bounds
// narrow MMAs, so each expert's rows are split evenly over as few tiles as
// possible (260 rows: 144 + 116, not 256 + 4) and each tile's MMAs are only as
// wide as its rows (rounded up to 16). TMEM is allocated once; the producer
// and the dequant warps run ahead across tile boundaries; the epilogue reads
// the accumulator into registers and releases it before it stores, so the
// next tile's MMAs start at once.
//
//   warp 0      TMA producer: the packed weights of each 128-k stage
//               (128 rows x 64 B, 64-byte swizzle) into a 4-deep ring, and
//               the stage's x (two boxes of 256 tokens x 64 k, 128-byte
//               swizzle) into a 2-deep ring.
//   warp 1      TMEM allocation and the MMA issuer (one lane).
//   warps 2-5   dequant: thread = TMEM lane = weight row; turns each 32-k
//               group into hi and lo and writes them to the stage's TMEM A
//               columns (tcgen05.st); the scales of the next stage are loaded
//               one stage ahead.
//   warps 6-13  epilogue: two threads per weight row (= TMEM lane), each
//               reading half of the tile's tokens from the accumulator,
//               times 2^e, rounded once to fp16, stored.
// Every mbarrier wait is bounded in time; a wait that gives up records
// W4A16_ERR_TIMEOUT and the CTA unwinds (drains its copies and MMAs, frees TMEM).
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kG = 32;                               // scale group of this kernel
constexpr int kRows = 128;                           // weight rows per tile: MMA M, TMEM lanes
constexpr int kBN = 256;                             // tokens per tile: MMA N at most
constexpr int kKS = 128;                             // k per pipeline stage
constexpr int kGroupsPerStage = kKS / kG;            // 4
constexpr int kPStages = 4;                          // packed-weight ring
constexpr int kXStages = 2;                          // x ring (shared memory)
constexpr int kAStages = 2;                          // TMEM A stages
constexpr int kPBytes = kRows * kKS / 2;             // 8 KB
constexpr int kXBoxBytes = kBN * 128;                // 64 k x 256 tokens, 128-byte swizzle
constexpr int kXBytes = (kKS / 64) * kXBoxBytes;     // 32 KB
constexpr int kMaxE = 4096;                          // experts (two ints each in shared memory)
constexpr int kDeqWarps = 4;                         // one thread per weight row
constexpr int kDeqParts = kDeqWarps / 4;
constexpr int kPartGroups = kGroupsPerStage / kDeqParts;  // groups of a stage per dequant thread
constexpr int kEpiWarps = 8;                         // two threads per weight row
constexpr int kEpiCols = kBN / (kEpiWarps / 4);      // accumulator columns per epilogue thread
constexpr int kThreads = (2 + kDeqWarps + kEpiWarps) * 32;
// TMEM columns: the accumulator [0, 256); A stage s at 256 + 128 s: hi in its
// first 64 columns, lo in the next 64 (two fp16 k per column)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAColBase = kBN;
constexpr uint32_t kAStageCols = kKS;
constexpr uint32_t kAHalfCols = kKS / 2;
constexpr float kMaxUnshifted = 8188.0f;             // |s| <= 8188 keeps |s q| <= 65504 for |q| <= 8
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;    // 1 s

#ifdef W4A16_TEST_HOOKS
__device__ TestHooks g_hooks = {kWaitLimitNs, -1};
__device__ TestCounters g_counters = {0ull, 0ull};
__device__ __forceinline__ uint64_t wait_limit() { return g_hooks.wait_limit_ns; }
__device__ __forceinline__ bool may_issue(int64_t issued) {
    return g_hooks.issue_limit < 0 || issued < g_hooks.issue_limit;
}
#define W4A16_COUNT_TMEM(field) atomicAdd(&g_counters.field, 1ull)
#else
__device__ __forceinline__ constexpr uint64_t wait_limit() { return kWaitLimitNs; }
__device__ __forceinline__ constexpr bool may_issue(int64_t) { return true; }
#define W4A16_COUNT_TMEM(field) ((void)0)
#endif

struct SplitArgs {
    const uint16_t* s;
    uint16_t* y;
    const int32_t* offsets;  // routed experts; nullptr: dense, one expert of M rows
    int64_t M, N, K;
    int E;
    unsigned int* err;
};

struct SplitSmem {
    uint64_t pfull[kPStages];   // a packed-weight stage landed
    uint64_t pempty[kPStages];  // the dequant warps finished reading it
    uint64_t xfull[kXStages];   // an x stage landed
    uint64_t xempty[kXStages];  // the MMAs reading an x stage finished
    uint64_t afull[kAStages];   // a TMEM A stage was written
    uint64_t aempty[kAStages];  // the MMAs reading a TMEM A stage finished
    uint64_t dfull;             // the accumulator holds a finished tile
    uint64_t dempty;            // the epilogue has read the accumulator
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    int tiles;                        // token tiles over all experts (0: invalid offsets)
    int first_tile[kMaxE + 1];        // token tiles of the experts before e
    int row_start[kMaxE + 1];         // expert_offsets
};

struct Tile {
    int e, row0, rows, n0;
};

__device__ __forceinline__ void fail(const SplitArgs& a, SplitSmem* sm, unsigned code) {
    raise_device_error(a.err, code);
    *reinterpret_cast<volatile int*>(&sm->abort) = 1;
}

// An expert's token tiles: as few as hold its rows (at most kBN each), all of
// one size, a multiple of 16 (the last one takes what remains).
__device__ __forceinline__ int tile_tokens(int rows, int tiles) {
    return ((rows + tiles - 1) / tiles + 15) & ~15;
}

// Tile t: token tile t / ntn (over the experts in order), weight-row tile t % ntn.
__device__ __forceinline__ Tile decode_tile(const SplitSmem* sm, int t, int ntn, int E) {
    const int tt = t / ntn;
    int lo = 0, hi = E - 1;  // the last expert whose first token tile is <= tt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm->first_tile[mid] <= tt) lo = mid;
        else hi = mid - 1;
    }
    const int rows_e = sm->row_start[lo + 1] - sm->row_start[lo];
    const int size = tile_tokens(rows_e, sm->first_tile[lo + 1] - sm->first_tile[lo]);
    Tile r;
    r.e = lo;
    r.row0 = sm->row_start[lo] + (tt - sm->first_tile[lo]) * size;
    r.rows = min(size, sm->row_start[lo + 1] - r.row0);
    r.n0 = (t % ntn) * kRows;
    return r;
}

// Warp 0, at start: each expert's first token tile and first row, from the
// device offsets (dense: one expert of M rows); an invalid partition is
// reported and leaves no tile.
__device__ void plan_tiles(const SplitArgs& a, SplitSmem* sm, int lane) {
    int base = 0;
    bool ok = true;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0, tiles = 0;
        if (e < a.E) {
            int hi;
            if (a.offsets) {
                lo = __ldg(a.offsets + e);
                hi = __ldg(a.offsets + e + 1);
            } else {
                lo = 0;
                hi = (int)a.M;
            }
            if (hi < lo || lo < 0 || (int64_t)hi > a.M) ok = false;
            tiles = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;  // as few as hold its rows
        }
        int incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (e < a.E) {
            sm->first_tile[e] = base + incl - tiles;
            sm->row_start[e] = lo;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    ok = __all_sync(0xffffffffu, ok);
    const int end = a.offsets ? __ldg(a.offsets + a.E) : (int)a.M;
    const bool ends_ok = (a.offsets ? __ldg(a.offsets) == 0 : true) && (int64_t)end == a.M;
    if (lane == 0) {
        sm->first_tile[a.E] = base;
        sm->row_start[a.E] = end;
        sm->tiles = (ok && ends_ok) ? base : 0;
        if (!ok || !ends_ok) raise_device_error(a.err, W4A16_ERR_BAD_OFFSETS);
    }
}

// 2^-e for the row's scales: 1 unless the row's largest |s| exceeds 8188.
__device__ __forceinline__ float row_shift(const uint16_t* srow, int gk, bool ok) {
    uint32_t mx = 0;  // largest |s| as fp16 bits (ordered like the values)
    if (ok) {
        if ((gk & 7) == 0 && ((reinterpret_cast<uintptr_t>(srow) & 15) == 0)) {
            for (int g = 0; g < gk; g += 8) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(srow + g));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
            }
        } else {
            for (int g = 0; g < gk; ++g) mx = max(mx, (uint32_t)__ldg(srow + g) & 0x7fffu);
        }
    }
    const float ms = __half2float(__ushort_as_half((unsigned short)mx));
    float f = 1.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)  // fp16 scales stay below 65520: three halvings at most
        if (ms * f > kMaxUnshifted) f *= 0.5f;
    return f;
}

// Byte offset of 16-byte chunk c of row r in a 64-byte-swizzled packed box.
__device__ __forceinline__ int packed_offset(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                 const SplitArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* pring = base;                              // packed-weight stages
    uint8_t* xring = base + kPStages * kPBytes;          // x stages
    SplitSmem* sm = reinterpret_cast<SplitSmem*>(xring + kXStages * kXBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        plan_tiles(a, sm, lane);
        if (lane == 0) {
            for (int i = 0; i < kPStages; ++i) {
                ptx::mbar_init(&sm->pfull[i], 1);
                ptx::mbar_init(&sm->pempty[i], kDeqWarps * 32);
            }
            for (int i = 0; i < kXStages; ++i) {
                ptx::mbar_init(&sm->xfull[i], 1);
                ptx::mbar_init(&sm->xempty[i], 1);
            }
            for (int i = 0; i < kAStages; ++i) {
                ptx::mbar_init(&sm->afull[i], kDeqWarps * 32);
                ptx::mbar_init(&sm->aempty[i], 1);
            }
            ptx::mbar_init(&sm->dfull, 1);
            ptx::mbar_init(&sm->dempty, kEpiWarps * 32);
            ptx::mbar_init(&sm->mma_done, 1);
            sm->abort = 0;
            ptx::fence_mbar_init();
            ptx::prefetch_tensormap(&tmap_x);
            ptx::prefetch_tensormap(&tmap_w);
        }
    }
    __syncthreads();
    const int ntn = (int)((a.N + kRows - 1) / kRows);   // weight-row tiles
    const int total = sm->tiles * ntn;
    if ((int)blockIdx.x >= total) return;                // nothing for this CTA (uniform)
    if (warp == 1) {
        ptx::tmem_alloc(&sm->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
        if (lane == 0) W4A16_COUNT_TMEM(tmem_allocs);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int* abort = &sm->abort;
    const int nst = (int)((a.K + kKS - 1) / kKS);      // stages per tile
    const int gk = (int)(a.K / kG);                     // scale groups per row
    const int my_tiles = (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            const int64_t stages = (int64_t)my_tiles * nst;
            int64_t ix = 0, ip = 0;  // stages issued on each ring
            int jx = -1, jp = -1;    // the tile each ring is on
            Tile tx{}, tp{};
            bool ok = true;
            uint64_t idle_since = 0;
            while (ix < stages || ip < stages) {
                bool moved = false;
                if (ix < stages && may_issue(ix + ip)) {
                    const int st = (int)(ix % kXStages);
                    const int64_t round = ix / kXStages;
                    if (round == 0 || ptx::mbar_try_wait(&sm->xempty[st], (uint32_t)((round - 1) & 1))) {
                        const int j = (int)(ix / nst), s = (int)(ix % nst);
                        if (j != jx) {
                            tx = decode_tile(sm, (int)blockIdx.x + j * (int)gridDim.x, ntn, a.E);
                            jx = j;
                        }
                        ptx::mbar_arrive_expect_tx(&sm->xfull[st], kXBytes);
#pragma unroll
                        for (int b = 0; b < kKS / 64; ++b)
                            ptx::tma_load_2d(xring + st * kXBytes + b * kXBoxBytes, &tmap_x, &sm->xfull[st],
                                             s * kKS + 64 * b, tx.row0);
                        ++ix;
                        moved = true;
                    }
                }
                if (ip < stages && may_issue(ix + ip)) {
                    const int st = (int)(ip % kPStages);
                    const int64_t round = ip / kPStages;
                    if (round == 0 || ptx::mbar_try_wait(&sm->pempty[st], (uint32_t)((round - 1) & 1))) {
                        const int j = (int)(ip / nst), s = (int)(ip % nst);
                        if (j != jp) {
                            tp = decode_tile(sm, (int)blockIdx.x + j * (int)gridDim.x, ntn, a.E);
                            jp = j;
                        }
                        ptx::mbar_arrive_expect_tx(&sm->pfull[st], kPBytes);
                        if (a.offsets == nullptr)
                            ptx::tma_load_2d(pring + st * kPBytes, &tmap_w, &sm->pfull[st], s * (kKS / 2), tp.n0);
                        else
                            ptx::tma_load_3d(pring + st * kPBytes, &tmap_w, &sm->pfull[st], s * (kKS / 2), tp.n0,
                                             tp.e);
                        ++ip;
                        moved = true;
                    }
                }
                if (moved) {
                    idle_since = 0;
                    continue;
                }
                const uint64_t now = ptx::globaltimer_ns();
                if (idle_since == 0) idle_since = now;
                if (*abort || now - idle_since > wait_limit()) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                if (!*abort) fail(a, sm, W4A16_ERR_TIMEOUT);
                volatile int never = 0;  // let our own loads land before the CTA exits
                for (int64_t i = ip > kPStages ? ip - kPStages : 0; i < ip; ++i)
                    ptx::mbar_wait(&sm->pfull[i % kPStages], (uint32_t)((i / kPStages) & 1), &never, kDrainLimitNs);
                for (int64_t i = ix > kXStages ? ix - kXStages : 0; i < ix; ++i)
                    ptx::mbar_wait(&sm->xfull[i % kXStages], (uint32_t)((i / kXStages) & 1), &never, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            bool ok = true;
            int64_t c = 0;
            for (int j = 0; ok && j < my_tiles; ++j) {
                const Tile tl = decode_tile(sm, (int)blockIdx.x + j * (int)gridDim.x, ntn, a.E);
                if (j >= 1 && !ptx::mbar_wait(&sm->dempty, (uint32_t)((j - 1) & 1), abort, wait_limit())) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t idesc = ptx::idesc_f16_f32(kRows, (tl.rows + 15) & ~15);
                const uint32_t d = tmem;
                for (int s = 0; s < nst; ++s, ++c) {
                    const int xs = (int)(c % kXStages), as = (int)(c % kAStages);
                    if (!ptx::mbar_wait(&sm->xfull[xs], (uint32_t)((c / kXStages) & 1), abort, wait_limit()) ||
                        !ptx::mbar_wait(&sm->afull[as], (uint32_t)((c / kAStages) & 1), abort, wait_limit())) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int64_t kc = (int64_t)s * kKS;
                    const int nk = (int)((a.K - kc < kKS ? a.K - kc : kKS) >> 4);
                    const uint64_t bdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(xring + xs * kXBytes));
                    const uint32_t a_hi = tmem + kAColBase + (uint32_t)as * kAStageCols;
                    const uint32_t a_lo = a_hi + kAHalfCols;
#pragma unroll
                    for (int kk = 0; kk < kKS / 16; ++kk) {
                        if (kk >= nk) break;
                        const uint64_t bdesc = bdesc0 + (uint64_t)((((kk >> 2) * kXBoxBytes) + (kk & 3) * 32) >> 4);
                        ptx::mma_f16_ts(d, a_hi + (uint32_t)(kk * 8), bdesc, idesc, (s | kk) ? 1u : 0u);
                        ptx::mma_f16_ts(d, a_lo + (uint32_t)(kk * 8), bdesc, idesc, 1u);
                    }
                    ptx::mma_commit(&sm->xempty[xs]);  // the x slot is free again
                    ptx::mma_commit(&sm->aempty[as]);  // and the TMEM A stage
                }
                if (!ok) break;
                ptx::mma_commit(&sm->dfull);  // the tile's accumulator is complete
            }
            if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
            ptx::mma_commit(&sm->mma_done);
            volatile int never = 0;
            ptx::mbar_wait(&sm->mma_done, 0, &never, kDrainLimitNs);
        }
    } else if (warp < 2 + kDeqWarps) {
        // -------------------------------------------------------------- dequant
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int part = (warp - 2) >> 2;         // which groups of each stage
        const int r = quad * 32 + lane;           // weight row in the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        int64_t c = 0;
        for (int j = 0; ok && j < my_tiles; ++j) {
            const Tile tl = decode_tile(sm, (int)blockIdx.x + j * (int)gridDim.x, ntn, a.E);
            const int64_t n = (int64_t)tl.n0 + r;
            const bool n_ok = n < a.N;
            const uint16_t* srow = a.s + ((int64_t)tl.e * a.N + (n_ok ? n : 0)) * gk;
            const float f = row_shift(srow, gk, n_ok);
            // this thread's scales of a stage (0 past the row), one stage ahead
            auto load_scales = [&](int s_, uint32_t (&dst)[kPartGroups]) {
#pragma unroll
                for (int i = 0; i < kPartGroups; ++i) {
                    const int g = s_ * kGroupsPerStage + part * kPartGroups + i;
                    dst[i] = (s_ < nst && g < gk) ? (uint32_t)__ldg(srow + g) : 0u;
                }
            };
            uint32_t sc[kPartGroups], sc_next[kPartGroups];
            load_scales(0, sc);
            for (int s = 0; s < nst; ++s, ++c) {
                const int ps = (int)(c % kPStages), as = (int)(c % kAStages);
                load_scales(s + 1, sc_next);
                const int g0 = s * kGroupsPerStage + part * kPartGroups;
                const int ng = min(kPartGroups, gk - g0);  // this thread's groups in the stage
                const bool got =
                    ptx::mbar_wait(&sm->pfull[ps], (uint32_t)((c / kPStages) & 1), abort, wait_limit()) &&
                    (c < kAStages ||
                     ptx::mbar_wait(&sm->aempty[as], (uint32_t)((c / kAStages - 1) & 1), abort, wait_limit()));
                if (!__all_sync(0xffffffffu, got)) {  // warp-uniform: the TMEM stores are .sync.aligned
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint8_t* prow = pring + ps * kPBytes;
                const uint32_t acol = lane_base + kAColBase + (uint32_t)as * kAStageCols;
#pragma unroll
                for (int i = 0; i < kPartGroups; ++i) {
                    if (i >= ng) break;  // uniform: every lane has the same groups
                    const int gi = part * kPartGroups + i;  // group within the stage
                    const uint4 pk = *reinterpret_cast<const uint4*>(prow + packed_offset(r, gi));
                    const uint32_t words[4] = {pk.x, pk.y, pk.z, pk.w};
                    // exact: a (shifted) fp16 scale
                    const __half2 s2 = __float2half2_rn(__half2float(__ushort_as_half((unsigned short)sc[i])) * f);
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {  // word w holds k = 8w .. 8w+7 of the group
                        uint32_t h04, h15, h26, h37;
                        nibbles_to_half2(words[w], h04, h15, h26, h37);
                        const uint32_t q[4] = {__byte_perm(h04, h15, 0x5410), __byte_perm(h26, h37, 0x5410),
                                               __byte_perm(h04, h15, 0x7632), __byte_perm(h26, h37, 0x7632)};
#pragma unroll
                        for (int k2 = 0; k2 < 4; ++k2) {
                            const __half2 qh = *reinterpret_cast<const __half2*>(&q[k2]);
                            const __half2 h = __hmul2(s2, qh);                 // fp16_rn(s q)
                            const __half2 l = __hfma2(s2, qh, __hneg2(h));     // s q - hi, exact
                            hi[4 * w + k2] = *reinterpret_cast<const uint32_t*>(&h);
                            lo[4 * w + k2] = *reinterpret_cast<const uint32_t*>(&l);
                        }
                    }
                    ptx::tmem_st_32x32b_x16(acol + (uint32_t)(gi * 16), hi);
                    ptx::tmem_st_32x32b_x16(acol + kAHalfCols + (uint32_t)(gi * 16), lo);
                }
                ptx::mbar_arrive(&sm->pempty[ps]);  // this thread has read its packed bytes
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&sm->afull[as]);
#pragma unroll
                for (int i = 0; i < kPartGroups; ++i) sc[i] = sc_next[i];
            }
        }
        if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int half = (warp - 2 - kDeqWarps) >> 2;  // which tokens of the tile
        const int r = quad * 32 + lane;                // weight row in the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * kEpiCols);
        bool ok = true;
        for (int j = 0; ok && j < my_tiles; ++j) {
            const Tile tl = decode_tile(sm, (int)blockIdx.x + j * (int)gridDim.x, ntn, a.E);
            const int64_t n = (int64_t)tl.n0 + r;
            const bool n_ok = n < a.N;
            const int m0 = half * kEpiCols;                          // first token of this thread's share
            const int mine = max(0, min(kEpiCols, tl.rows - m0));    // tokens of the tile in that share
            // the row's 2^e, found while the tile's MMAs run
            const float mult = 1.0f / row_shift(a.s + ((int64_t)tl.e * a.N + (n_ok ? n : 0)) * gk, gk, n_ok);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm->dfull, (uint32_t)(j & 1), abort, wait_limit()))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // read the accumulator (rounded to fp16 pairs), then release it for the next tile
            uint32_t packed[kEpiCols / 2];
#pragma unroll
            for (int ch = 0; ch < kEpiCols / 32; ++ch) {
                if (ch * 32 < mine) {  // uniform: same tile in every lane
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(lane_base + (uint32_t)(ch * 32), v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const __half2 h = __floats2half2_rn(__uint_as_float(v[2 * i]) * mult,
                                                            __uint_as_float(v[2 * i + 1]) * mult);
                        packed[ch * 16 + i] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm->dempty);
            if (n_ok) {
                uint16_t* yrow = a.y + ((int64_t)tl.row0 + m0) * a.N + n;
#pragma unroll
                for (int i = 0; i < kEpiCols; ++i)
                    if (i < mine) yrow[(int64_t)i * a.N] = (uint16_t)(packed[i >> 1] >> (16 * (i & 1)));
            }
        }
        if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) {
        ptx::tmem_dealloc(tmem, kTmemCols);
        if (lane == 0) W4A16_COUNT_TMEM(tmem_frees);
    }
}

// ------------------------------------------------------------------- host --

constexpr size_t kSmem = 1024 + kPStages * kPBytes + kXStages * kXBytes + ((sizeof(SplitSmem) + 127) & ~(size_t)127);

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

bool split_supports(int group, int E) { return group == kG && E >= 1 && E <= kMaxE; }

w4a16_status split_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                          int64_t M, int64_t N, int64_t K, const int32_t* offsets, int E, cudaStream_t st) {
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    if (kSmem > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cuda_status(cudaErrorNotSupported, "gemm g32: cuTensorMapEncodeTiled entry point");
    CUtensorMap mx, mw;
    {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kBN};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm g32: cuTensorMapEncodeTiled (x)");
    }
    if (offsets == nullptr) {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        cuuint32_t box[2] = {kKS / 2, (cuuint32_t)kRows};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm g32: cuTensorMapEncodeTiled (weights)");
    } else {
        cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)(N * (K / 2))};
        cuuint32_t box[3] = {kKS / 2, (cuuint32_t)kRows, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm g32: cuTensorMapEncodeTiled (weights)");
    }
    SplitArgs a{};
    a.s = s;
    a.y = y;
    a.offsets = offsets;
    a.M = M;
    a.N = N;
    a.K = K;
    a.E = offsets ? E : 1;
    a.err = dev.error_word;
    // an upper bound on the tiles (each expert adds at most one partial token tile)
    const int64_t ntn = (N + kRows - 1) / kRows;
    const int64_t tiles = ((M + kBN - 1) / kBN + (offsets ? E : 0)) * ntn;
    if (tiles > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const unsigned grid = (unsigned)(tiles < dev.sms ? tiles : dev.sms);
    static PerDeviceOnce once;
    const cudaError_t attr = once.run(dev.device, [] {
        return cudaFuncSetAttribute(split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    });
    if (attr != cudaSuccess) return cuda_status(attr, "gemm g32: cudaFuncSetAttribute");
    split_kernel<<<grid, kThreads, kSmem, st>>>(mx, mw, a);
    return cuda_status(cudaGetLastError(), "gemm g32: kernel launch");
}

#ifdef W4A16_TEST_HOOKS
cudaError_t split_set_test_hooks(const TestHooks& h) { return cudaMemcpyToSymbol(g_hooks, &h, sizeof(h)); }
cudaError_t split_get_test_counters(TestCounters* c) { return cudaMemcpyFromSymbol(c, g_counters, sizeof(*c)); }
#endif

}  // namespace w4a16
