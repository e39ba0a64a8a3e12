// Tensor-core GEMM of the W4A16 layer with the scale folded into the A
// operand: the routed-expert layer (the LLM170 page's "g32, MoE resident"
// models) and dense layers past 64 tokens, at groups 32, 64 and 128 (sm_103a:
// TMA, tcgen05 MMA, TMEM).
//
// The group-partial design of tc_linear.cu (one fp32 TMEM partial per scale
// group, scaled by the epilogue) pays one TMEM round trip and one wait for its
// buffer per group; at group 32 that takes longer than the group's two MMAs,
// and at any group it keeps the MMAs at 128 tokens. Here the scale goes into
// the A operand instead, exactly. For a scale s (fp16) and an integer q in [-8, 7]
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
// Pipeline stages of KS k (Pipe<KS>): 128 for long K (two TMEM A stages, a
// 3-deep x ring of 64 KB stages and a 3-deep packed ring where the tile plan
// leaves room for them, else 2 and 4), 64 for short K, where a tile has few
// stages and a deeper pipeline hides its fill (four A stages, a 4-deep x ring
// of 32 KB, an 8-deep packed ring). Measured on the routed-expert layer:
// gate/up (K = 2048) 119 us at 128-k stages against 139 us at 64, and 109
// against 115 us with the third x stage; down (K = 512) 177 us at 64-k stages
// against 205 us at 128 with two x stages, but 121.4 against 126.8 us at 128
// once the third x stage is in, so plain GEMMs take 128-k stages from K = 512.
//
//   warp 0      TMA producer: the packed weights of each stage (128 rows x
//               KS/2 bytes, swizzled) and the stage's x (KS/64 boxes of 256
//               tokens x 64 k, 128-byte swizzle) into their rings (x not with
//               a row gather, below).
//   warp 1      TMEM allocation and the MMA issuer (one lane).
//   warps 2-5   dequant: thread = TMEM lane = weight row; turns each 32-k
//               chunk into hi and lo with the scale of its group and writes
//               them to the stage's TMEM A columns (tcgen05.st); the scales of
//               the next stage are loaded one stage ahead.
//   warps 6-13  epilogue: two threads per weight row (= TMEM lane), each
//               reading half of the tile's tokens from the accumulator,
//               times 2^e, rounded once to fp16, stored. With a row gather
//               (routed experts read straight from the token-major x) these
//               warps also fill the x ring while the tile's MMAs run: each
//               copies 32 rows of a stage, x[token_of_row[r]], 16 bytes at a
//               time into the swizzled layout a TMA box would have, and each
//               lane's arrival on the stage's barrier fires when its copies
//               land (nothing waits for them). The MMA thread fences them over
//               to the async proxy before it reads them.
// Every mbarrier wait is bounded in time; a wait that gives up records
// W4A16_ERR_TIMEOUT and the CTA unwinds (drains its copies and MMAs, frees TMEM).
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kChunk = 32;                           // k per dequant chunk: one scale each
constexpr int kRows = 128;                           // weight rows per tile: MMA M, TMEM lanes
constexpr int kBN = 256;                             // tokens per tile: MMA N at most
constexpr int kXBoxBytes = kBN * 128;                // 64 k x 256 tokens, 128-byte swizzle
constexpr int kMaxE = 4096;                          // experts (two ints each in shared memory)
constexpr int kDeqWarps = 4;                         // one thread per weight row
constexpr int kEpiWarps = 8;                         // two threads per weight row
constexpr int kEpiCols = kBN / (kEpiWarps / 4);      // accumulator columns per epilogue thread
constexpr int kThreads = (2 + kDeqWarps + kEpiWarps) * 32;
// TMEM columns: the accumulator [0, 256), then the A stages: hi of a stage in
// its first KS/2 columns, lo in the next KS/2 (two fp16 k per column)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAColBase = kBN;
constexpr int kStageTokens = 16;                     // tokens per epilogue store round
constexpr int kStageBytes = kStageTokens * 32 * 2;   // one warp's 32 rows x 16 tokens of fp16
constexpr float kMaxUnshifted = 8188.0f;             // |s| <= 8188 keeps |s q| <= 65504 for |q| <= 8
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;    // 1 s

// The rings of a pipeline of KS-k stages.
template <int KS, int XS = (KS == 128 ? 2 : 4)>
struct Pipe {
    static constexpr int kKS = KS;
    static constexpr int kChunksPerStage = KS / kChunk;
    static constexpr int kPStages = KS == 128 ? (XS >= 3 ? 3 : 4) : 8;  // packed-weight ring
    static constexpr int kXStages = XS;                                // x ring (shared memory)
    static constexpr int kAStages = KS == 128 ? 2 : 4;   // TMEM A stages
    static constexpr int kPBytes = kRows * KS / 2;        // packed weights of a stage
    static constexpr int kXBoxes = KS / 64;
    static constexpr int kXBytes = kXBoxes * kXBoxBytes;
    static constexpr uint32_t kAStageCols = KS;          // hi (KS fp16 = KS/2 columns), then lo
    static constexpr uint32_t kAHalfCols = KS / 2;
    static constexpr CUtensorMapSwizzle kPSwizzle = KS == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    static_assert(KS == 64 || KS == 128, "stage");
    static_assert(kAColBase + kAStages * kAStageCols <= kTmemCols, "TMEM budget");

    // byte offset of 16-byte chunk c of row r in a packed stage (rows of KS/2 bytes, swizzled)
    __device__ static __forceinline__ int packed_offset(int r, int c) {
        if constexpr (KS == 128) return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);  // 64-byte swizzle
        else return r * 32 + ((c ^ ((r >> 2) & 1)) << 4);                     // 32-byte swizzle
    }
};

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
    const uint16_t* s2;      // gated: the up projection's scales (s holds the gate's)
    uint16_t* y;
    const int32_t* offsets;  // routed experts; nullptr: dense, one expert of M rows
    const int32_t* gather;   // token of each row: x rows come from xg [T, K]; nullptr: x by TMA
    const uint16_t* xg;
    int64_t T;
    int64_t M, N, K;
    int E;
    int gshift;  // scale group = 32 << gshift
    unsigned int* err;
};

// The tile plan (filled once per CTA) in shared memory, after the store
// staging: E + 1 entries each, sized at launch.
struct TilePlan {
    int* first_tile;  // token tiles of the experts before e
    int* row_start;   // expert_offsets
};

template <class P>
struct SplitSmem {
    uint64_t pfull[P::kPStages];   // a packed-weight stage landed
    uint64_t pempty[P::kPStages];  // the dequant warps finished reading it
    uint64_t xfull[P::kXStages];   // an x stage landed
    uint64_t xempty[P::kXStages];  // the MMAs reading an x stage finished
    uint64_t afull[P::kAStages];   // a TMEM A stage was written
    uint64_t aempty[P::kAStages];  // the MMAs reading a TMEM A stage finished
    uint64_t dfull;                // the accumulator holds a finished tile
    uint64_t dempty;               // the epilogue has read the accumulator
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    int plan_tiles;                // token tiles over all experts (0: invalid offsets)
};

// Shared memory ahead of the rings: the store staging, the tile plan of E
// experts and the barrier block, rounded up to the rings' 1024-byte alignment.
// (Of the orders of these regions measured, this one ran the routed down
// projection, K = 512, fastest: 127 us against up to 138.)
template <class P>
constexpr int kBarrierBytes = (int)((sizeof(SplitSmem<P>) + 127) & ~(size_t)127);
template <class P>
__host__ __device__ constexpr int front_bytes(int E) {
    return (kBarrierBytes<P> + kEpiWarps * kStageBytes + 2 * (E + 1) * (int)sizeof(int) + 1023) & ~1023;
}

struct Tile {
    int e, row0, rows, n0;
};

__device__ __forceinline__ void fail(const SplitArgs& a, int* abort, unsigned code) {
    raise_device_error(a.err, code);
    *reinterpret_cast<volatile int*>(abort) = 1;
}

// An expert's token tiles: as few as hold its rows (at most kBN each), all of
// one size, a multiple of 16 (the last one takes what remains).
__device__ __forceinline__ int tile_tokens(int rows, int tiles) {
    return ((rows + tiles - 1) / tiles + 15) & ~15;
}

// Tile t: token tile t / ntn (over the experts in order), weight-row tile t % ntn
// of out_rows output rows.
__device__ __forceinline__ Tile decode_tile(const TilePlan& pl, int t, int ntn, int E, int out_rows) {
    const int tt = t / ntn;
    int lo = 0, hi = E - 1;  // the last expert whose first token tile is <= tt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pl.first_tile[mid] <= tt) lo = mid;
        else hi = mid - 1;
    }
    const int rows_e = pl.row_start[lo + 1] - pl.row_start[lo];
    const int size = tile_tokens(rows_e, pl.first_tile[lo + 1] - pl.first_tile[lo]);
    Tile r;
    r.e = lo;
    r.row0 = pl.row_start[lo] + (tt - pl.first_tile[lo]) * size;
    r.rows = min(size, pl.row_start[lo + 1] - r.row0);
    r.n0 = (t % ntn) * out_rows;
    return r;
}

// Warp 0, at start: each expert's first token tile and first row, from the
// device offsets (dense: one expert of M rows); an invalid partition is
// reported and leaves no tile.
__device__ void plan_tiles(const SplitArgs& a, const TilePlan& pl, int* tiles_out, int lane) {
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
            pl.first_tile[e] = base + incl - tiles;
            pl.row_start[e] = lo;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    ok = __all_sync(0xffffffffu, ok);
    const int end = a.offsets ? __ldg(a.offsets + a.E) : (int)a.M;
    const bool ends_ok = (a.offsets ? __ldg(a.offsets) == 0 : true) && (int64_t)end == a.M;
    if (lane == 0) {
        pl.first_tile[a.E] = base;
        pl.row_start[a.E] = end;
        *tiles_out = (ok && ends_ok) ? base : 0;
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

// GATED (dense only): each tile's 128 weight rows are 64 rows of Wg and the same
// 64 rows of Wu (tmap_w, tmap_w2), interleaved in TMEM as gated_out_row /
// gated_smem_row describe; the epilogue forms y = silu(g) * u from the fp32 sums.
template <int KS, bool GATED, int XS>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_w2, const SplitArgs a) {
    using P = Pipe<KS, XS>;
    constexpr int kOut = GATED ? kRows / 2 : kRows;  // output rows per tile
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    // the epilogue warps' store staging (kStageBytes each), the tile plan and
    // the barrier block come first; the rings start at the next 1024 bytes
    uint8_t* ystage = base;
    TilePlan plan;
    plan.first_tile = reinterpret_cast<int*>(ystage + kEpiWarps * kStageBytes);
    plan.row_start = plan.first_tile + (a.E + 1);
    SplitSmem<P>* sm = reinterpret_cast<SplitSmem<P>*>(plan.row_start + (a.E + 1));  // 8-byte aligned
    uint8_t* pring = base + front_bytes<P>(a.E);           // packed-weight stages
    uint8_t* xring = pring + P::kPStages * P::kPBytes;     // x stages (1024-byte aligned)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        plan_tiles(a, plan, &sm->plan_tiles, lane);
        if (lane == 0) {
            for (int i = 0; i < P::kPStages; ++i) {
                ptx::mbar_init(&sm->pfull[i], 1);
                ptx::mbar_init(&sm->pempty[i], kDeqWarps * 32);
            }
            for (int i = 0; i < P::kXStages; ++i) {
                // TMA: one arrival with the byte count; row gather: every epilogue lane
                ptx::mbar_init(&sm->xfull[i], a.gather ? kEpiWarps * 32 : 1);
                ptx::mbar_init(&sm->xempty[i], 1);
            }
            for (int i = 0; i < P::kAStages; ++i) {
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
            if (GATED) ptx::prefetch_tensormap(&tmap_w2);
        }
    }
    __syncthreads();
    const int ntn = (int)((a.N + kOut - 1) / kOut);     // weight-row tiles
    const int total = sm->plan_tiles * ntn;
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
    const int nst = (int)((a.K + KS - 1) / KS);         // stages per tile
    const int gk = (int)(a.K >> (5 + a.gshift));        // scale groups per row
    const int nck = (int)(a.K / kChunk);                // 32-k chunks per row
    const int my_tiles = (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int64_t stages = (int64_t)my_tiles * nst;
    auto tile_of = [&](int j) {
        return decode_tile(plan, (int)blockIdx.x + j * (int)gridDim.x, ntn, a.E, kOut);
    };

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        // the warp polls together; lane 0 issues the copies
        int64_t ix = a.gather ? stages : 0, ip = 0;  // stages issued on each ring (x: none with a gather)
        int jx = 0, sx = 0, jp = 0, sp = 0;          // each ring's tile and stage in it (no division per stage)
        int jtx = -1, jtp = -1;                      // the tile decoded for each ring
        Tile tx{}, tp{};
        bool ok = true;
        uint64_t idle_since = 0;
        while (ix < stages || ip < stages) {
            bool moved = false;
            if (ix < stages && may_issue(ix + ip)) {
                const int st = (int)(ix % P::kXStages);
                const int64_t round = ix / P::kXStages;
                bool free = round == 0;
                if (!free && lane == 0) free = ptx::mbar_try_wait(&sm->xempty[st], (uint32_t)((round - 1) & 1));
                if (__shfl_sync(0xffffffffu, free, 0)) {
                    const int j = jx, s = sx;
                    if (++sx == nst) {
                        sx = 0;
                        ++jx;
                    }
                    if (j != jtx) {
                        tx = tile_of(j);
                        jtx = j;
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(&sm->xfull[st], P::kXBytes);
#pragma unroll
                        for (int b = 0; b < P::kXBoxes; ++b)
                            ptx::tma_load_2d(xring + st * P::kXBytes + b * kXBoxBytes, &tmap_x, &sm->xfull[st],
                                             s * KS + 64 * b, tx.row0);
                    }
                    ++ix;
                    moved = true;
                }
            }
            if (ip < stages && may_issue(ix + ip)) {
                const int st = (int)(ip % P::kPStages);
                const int64_t round = ip / P::kPStages;
                bool free = round == 0;
                if (!free && lane == 0) free = ptx::mbar_try_wait(&sm->pempty[st], (uint32_t)((round - 1) & 1));
                if (__shfl_sync(0xffffffffu, free, 0)) {
                    const int j = jp, s = sp;
                    if (++sp == nst) {
                        sp = 0;
                        ++jp;
                    }
                    if (j != jtp) {
                        tp = tile_of(j);
                        jtp = j;
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(&sm->pfull[st], P::kPBytes);
                        if (GATED) {
                            ptx::tma_load_2d(pring + st * P::kPBytes, &tmap_w, &sm->pfull[st], s * (KS / 2), tp.n0);
                            ptx::tma_load_2d(pring + st * P::kPBytes + P::kPBytes / 2, &tmap_w2, &sm->pfull[st],
                                             s * (KS / 2), tp.n0);
                        } else if (a.offsets == nullptr)
                            ptx::tma_load_2d(pring + st * P::kPBytes, &tmap_w, &sm->pfull[st], s * (KS / 2), tp.n0);
                        else
                            ptx::tma_load_3d(pring + st * P::kPBytes, &tmap_w, &sm->pfull[st], s * (KS / 2), tp.n0,
                                             tp.e);
                    }
                    ++ip;
                    moved = true;
                }
            }
            if (moved) {
                idle_since = 0;
                continue;
            }
            bool quit = false;
            if (lane == 0) {
                const uint64_t now = ptx::globaltimer_ns();
                if (idle_since == 0) idle_since = now;
                quit = *abort || now - idle_since > wait_limit();
            }
            if (__shfl_sync(0xffffffffu, quit, 0)) {
                ok = false;
                break;
            }
        }
        if (!ok && lane == 0) {
            if (!*abort) fail(a, &sm->abort, W4A16_ERR_TIMEOUT);
            volatile int never = 0;  // let our own loads land before the CTA exits
            for (int64_t i = ip > P::kPStages ? ip - P::kPStages : 0; i < ip; ++i)
                ptx::mbar_wait(&sm->pfull[i % P::kPStages], (uint32_t)((i / P::kPStages) & 1), &never, kDrainLimitNs);
            if (!a.gather)
                for (int64_t i = ix > P::kXStages ? ix - P::kXStages : 0; i < ix; ++i)
                    ptx::mbar_wait(&sm->xfull[i % P::kXStages], (uint32_t)((i / P::kXStages) & 1), &never,
                                   kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            bool ok = true;
            int64_t c = 0;
            for (int j = 0; ok && j < my_tiles; ++j) {
                const Tile tl = tile_of(j);
                if (j >= 1 && !ptx::mbar_wait(&sm->dempty, (uint32_t)((j - 1) & 1), abort, wait_limit())) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t idesc = ptx::idesc_f16_f32(kRows, (tl.rows + 15) & ~15);
                const uint32_t d = tmem;
                for (int s = 0; s < nst; ++s, ++c) {
                    const int xs = (int)(c % P::kXStages), as = (int)(c % P::kAStages);
                    if (!ptx::mbar_wait(&sm->xfull[xs], (uint32_t)((c / P::kXStages) & 1), abort, wait_limit()) ||
                        !ptx::mbar_wait(&sm->afull[as], (uint32_t)((c / P::kAStages) & 1), abort, wait_limit())) {
                        ok = false;
                        break;
                    }
                    // gathered x was written through the generic proxy; the MMAs read it through the async one
                    if (a.gather) ptx::fence_proxy_async_shared();
                    ptx::tc_fence_after();
                    const int64_t kc = (int64_t)s * KS;
                    const int nk = (int)((a.K - kc < KS ? a.K - kc : KS) >> 4);
                    const uint64_t bdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(xring + xs * P::kXBytes));
                    const uint32_t a_hi = tmem + kAColBase + (uint32_t)as * P::kAStageCols;
                    const uint32_t a_lo = a_hi + P::kAHalfCols;
#pragma unroll
                    for (int kk = 0; kk < KS / 16; ++kk) {
                        if (kk >= nk) break;
                        // next 64-k box every 4 MMAs; 32 bytes per 16 k inside the swizzle atom
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
            if (!ok) fail(a, &sm->abort, W4A16_ERR_TIMEOUT);
            ptx::mma_commit(&sm->mma_done);
            volatile int never = 0;
            ptx::mbar_wait(&sm->mma_done, 0, &never, kDrainLimitNs);
        }
    } else if (warp < 2 + kDeqWarps) {
        // -------------------------------------------------------------- dequant
        constexpr int GPS = P::kChunksPerStage;
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;           // weight row in the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const bool up_row = GATED && ((r >> 3) & 1);
        const int prow_r = GATED ? gated_smem_row(r) : r;  // shared-memory row of this TMEM lane
        bool ok = true;
        int64_t c = 0;
        for (int j = 0; ok && j < my_tiles; ++j) {
            const Tile tl = tile_of(j);
            const int64_t n = (int64_t)tl.n0 + (GATED ? gated_out_row(r) : r);
            const bool n_ok = n < a.N;
            const uint16_t* srow = (up_row ? a.s2 : a.s) + ((int64_t)tl.e * a.N + (n_ok ? n : 0)) * gk;
            const float f = row_shift(srow, gk, n_ok);
            // the scale of each 32-k chunk of a stage (0 past the row), one stage ahead
            auto load_scales = [&](int s_, uint32_t (&dst)[GPS]) {
#pragma unroll
                for (int i = 0; i < GPS; ++i) {
                    const int ck = s_ * GPS + i;
                    dst[i] = (s_ < nst && ck < nck) ? (uint32_t)__ldg(srow + (ck >> a.gshift)) : 0u;
                }
            };
            uint32_t sc[GPS], sc_next[GPS];
            load_scales(0, sc);
            for (int s = 0; s < nst; ++s, ++c) {
                const int ps = (int)(c % P::kPStages), as = (int)(c % P::kAStages);
                load_scales(s + 1, sc_next);
                const int ng = min(GPS, nck - s * GPS);  // chunks in the stage
                const bool got =
                    ptx::mbar_wait(&sm->pfull[ps], (uint32_t)((c / P::kPStages) & 1), abort, wait_limit()) &&
                    (c < P::kAStages ||
                     ptx::mbar_wait(&sm->aempty[as], (uint32_t)((c / P::kAStages - 1) & 1), abort, wait_limit()));
                if (!__all_sync(0xffffffffu, got)) {  // warp-uniform: the TMEM stores are .sync.aligned
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint8_t* prow = pring + ps * P::kPBytes;
                const uint32_t acol = lane_base + kAColBase + (uint32_t)as * P::kAStageCols;
#pragma unroll
                for (int gi = 0; gi < GPS; ++gi) {
                    if (gi >= ng) break;  // uniform: every lane has the same chunks
                    const uint4 pk = *reinterpret_cast<const uint4*>(prow + P::packed_offset(prow_r, gi));
                    const uint32_t words[4] = {pk.x, pk.y, pk.z, pk.w};
                    // exact: a (shifted) fp16 scale
                    const __half2 s2 = __float2half2_rn(__half2float(__ushort_as_half((unsigned short)sc[gi])) * f);
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
                    ptx::tmem_st_32x32b_x16(acol + P::kAHalfCols + (uint32_t)(gi * 16), lo);
                }
                ptx::mbar_arrive(&sm->pempty[ps]);  // this thread has read its packed bytes
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&sm->afull[as]);
#pragma unroll
                for (int i = 0; i < GPS; ++i) sc[i] = sc_next[i];
            }
        }
        if (!ok) fail(a, &sm->abort, W4A16_ERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------- epilogue
        const int ew = warp - 2 - kDeqWarps;           // epilogue warp 0..7
        const int quad = warp & 3;
        const int half = ew >> 2;                      // which tokens of the tile
        const int r = quad * 32 + lane;                // weight row in the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * kEpiCols);
        const bool up_row = GATED && ((r >> 3) & 1);
        // tile j's results: the accumulator read as fp16 pairs (times the row's
        // 2^e), the accumulator released, then y stored. Gated: lanes r and r ^ 8
        // hold g and u of one output; the gate lane finishes the even tokens of
        // each pair and the up lane the odd ones, each handing the other the
        // operand it lacks (one shuffle), and y = fp16(silu(g) * u).
        auto finish_tile = [&](const Tile& tl, float mult) {
            const int64_t n = (int64_t)tl.n0 + (GATED ? gated_out_row(r) : r);
            const int m0 = half * kEpiCols;                          // first token of this thread's share
            const int mine = max(0, min(kEpiCols, tl.rows - m0));    // tokens of the tile in that share
            ptx::tc_fence_after();
            uint32_t packed[kEpiCols / 2];
#pragma unroll
            for (int ch = 0; ch < kEpiCols / 32; ++ch) {
                if (ch * 32 < mine) {  // uniform: same tile in every lane
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(lane_base + (uint32_t)(ch * 32), v);
                    ptx::tmem_ld_wait();
                    if constexpr (GATED) {
                        float yv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float e0 = __uint_as_float(v[2 * i]) * mult, e1 = __uint_as_float(v[2 * i + 1]) * mult;
                            const float other = __shfl_xor_sync(0xffffffffu, up_row ? e0 : e1, 8);
                            const float g = up_row ? other : e0, u = up_row ? e1 : other;
                            yv[i] = __fdividef(g, 1.0f + __expf(-g)) * u;
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const __half2 h = __floats2half2_rn(yv[2 * i], yv[2 * i + 1]);
                            packed[ch * 8 + i] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const __half2 h = __floats2half2_rn(__uint_as_float(v[2 * i]) * mult,
                                                                __uint_as_float(v[2 * i + 1]) * mult);
                            packed[ch * 16 + i] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm->dempty);
            if constexpr (GATED) {  // this lane's tokens: 2 i + (up lane)
                if (n < a.N) {
                    const int u0 = up_row ? 1 : 0;
                    uint16_t* yrow = a.y + ((int64_t)tl.row0 + m0 + u0) * a.N + n;
#pragma unroll
                    for (int i = 0; i < kEpiCols / 2; ++i)
                        if (2 * i + u0 < mine)
                            yrow[(int64_t)(2 * i) * a.N] = (uint16_t)(packed[i >> 1] >> (16 * (i & 1)));
                }
            } else if ((a.N & 7) == 0) {
                // Through this warp's staging area, 16 tokens at a time: the warp's 32
                // rows of a token are 64 contiguous bytes of y, so each lane then stores
                // 16 bytes (8 rows of one token) instead of 2: 8 times fewer store
                // instructions. Warp-local (every lane takes part; rows past N are
                // skipped 8 at a time, N being a multiple of 8): only __syncwarp orders it.
                uint16_t* stg = reinterpret_cast<uint16_t*>(ystage + ew * kStageBytes);
                const int64_t nw = (int64_t)tl.n0 + quad * 32;  // the warp's first row
#pragma unroll
                for (int q = 0; q < kEpiCols / kStageTokens; ++q) {
                    const int q0 = q * kStageTokens;
                    if (q0 >= mine) break;  // uniform in the warp
#pragma unroll
                    for (int j = 0; j < kStageTokens; ++j) {
                        const int i = q0 + j;
                        stg[j * 32 + lane] = (uint16_t)(packed[i >> 1] >> (16 * (i & 1)));
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int c = lane + 32 * k;  // 16-byte chunk: token c / 4, rows 8 (c % 4) ..
                        const int tok = q0 + (c >> 2);
                        const uint4 v = *reinterpret_cast<const uint4*>(stg + (c >> 2) * 32 + (c & 3) * 8);
                        if (tok < mine && nw + (c & 3) * 8 < a.N)
                            *reinterpret_cast<uint4*>(a.y + ((int64_t)tl.row0 + m0 + tok) * a.N + nw + (c & 3) * 8) = v;
                    }
                    __syncwarp();
                }
            } else if (n < a.N) {
                uint16_t* yrow = a.y + ((int64_t)tl.row0 + m0) * a.N + n;
#pragma unroll
                for (int i = 0; i < kEpiCols; ++i)
                    if (i < mine) yrow[(int64_t)i * a.N] = (uint16_t)(packed[i >> 1] >> (16 * (i & 1)));
            }
        };
        auto row_mult = [&](const Tile& tl) {  // the row's 2^e
            const int64_t n = (int64_t)tl.n0 + (GATED ? gated_out_row(r) : r);
            const bool n_ok = n < a.N;
            return 1.0f / row_shift((up_row ? a.s2 : a.s) + ((int64_t)tl.e * a.N + (n_ok ? n : 0)) * gk, gk, n_ok);
        };
        bool ok = true;
        if (!a.gather) {
            for (int j = 0; ok && j < my_tiles; ++j) {
                const Tile tl = tile_of(j);
                const float mult = row_mult(tl);  // found while the tile's MMAs run
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm->dfull, (uint32_t)(j & 1), abort, wait_limit()))) {
                    ok = false;
                    break;
                }
                finish_tile(tl, mult);
            }
        } else {
            // Row gather: between tile epilogues these warps fill the x ring, each with
            // 32 rows of every stage. Lane l copies 16-byte chunk l % CPR of rows
            // 32 ew + l / CPR + (32 / CPR) i, written where the 128-byte swizzle of a TMA
            // box puts it; rows past the tile, k past K and tokens outside [0, T) read
            // zeros. Each lane's arrival fires when its copies land.
            constexpr int CPR = KS / 8;              // 16-byte chunks of a row per stage
            constexpr int RPI = 32 / CPR;            // rows per warp instruction
            int64_t gx = 0;                          // x stages this warp has gathered its rows of
            int jg = -1;
            Tile tg{};
            int jm = -1;
            Tile tl{};
            float mult = 0.0f;
            uint64_t idle_since = 0;
            for (int j = 0; ok && j < my_tiles;) {
                if (jm != j) {
                    tl = tile_of(j);
                    mult = row_mult(tl);
                    jm = j;
                }
                if (gx < stages) {
                    const int st = (int)(gx % P::kXStages);
                    const int64_t round = gx / P::kXStages;
                    bool free = round == 0;
                    if (!free && lane == 0)
                        free = ptx::mbar_try_wait(&sm->xempty[st], (uint32_t)((round - 1) & 1));
                    if (__shfl_sync(0xffffffffu, free, 0)) {
                        const int jx = (int)(gx / nst), sx = (int)(gx % nst);
                        if (jx != jg) {
                            tg = tile_of(jx);
                            jg = jx;
                        }
                        const uint32_t xdst = ptx::smem_u32(xring + st * P::kXBytes);
                        const int c16 = lane % CPR;
                        const int64_t k = (int64_t)sx * KS + c16 * 8;
                        const int n_mma = (tg.rows + 15) & ~15;
#pragma unroll
                        for (int i = 0; i < CPR; ++i) {
                            const int row = 32 * ew + lane / CPR + RPI * i;
                            if (row >= n_mma) continue;
                            int t = row < tg.rows ? __ldg(a.gather + tg.row0 + row) : -1;
                            if (row < tg.rows && (t < 0 || (int64_t)t >= a.T)) {
                                if (sx == 0 && c16 == 0) raise_device_error(a.err, W4A16_ERR_BAD_ROUTING);
                                t = -1;
                            }
                            const bool v = t >= 0 && k < a.K;
                            const uint32_t dst = xdst + (uint32_t)((c16 >> 3) * kXBoxBytes + row * 128 +
                                                                   (((c16 & 7) ^ (row & 7)) << 4));
                            ptx::cp_async_16(dst, v ? a.xg + (int64_t)t * a.K + k : a.xg, v ? 16u : 0u);
                        }
                        ptx::cp_async_mbar_arrive_noinc(&sm->xfull[st]);
                        ++gx;
                        idle_since = 0;
                        continue;
                    }
                }
                bool ready = false;
                if (lane == 0) ready = ptx::mbar_try_wait(&sm->dfull, (uint32_t)(j & 1));
                if (__shfl_sync(0xffffffffu, ready, 0)) {
                    finish_tile(tl, mult);
                    ++j;
                    idle_since = 0;
                    continue;
                }
                bool quit = false;
                if (lane == 0) {
                    const uint64_t now = ptx::globaltimer_ns();
                    if (idle_since == 0) idle_since = now;
                    quit = *abort || now - idle_since > wait_limit();
                }
                if (__shfl_sync(0xffffffffu, quit, 0)) ok = false;
            }
            ptx::cp_async_wait_all();  // this lane's copies land before the CTA exits
        }
        if (!ok) fail(a, &sm->abort, W4A16_ERR_TIMEOUT);
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

template <class P>
constexpr size_t smem_bytes(int E) {
    return 1024 + front_bytes<P>(E) + P::kPStages * P::kPBytes + P::kXStages * P::kXBytes;
}

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

template <int KS, bool GATED = false>
w4a16_status launch_split(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                          uint16_t* y, int64_t M, int64_t N, int64_t K, int gshift, const int32_t* offsets, int E,
                          const int32_t* gather, int64_t T, cudaStream_t st, const uint8_t* qw2 = nullptr,
                          const uint16_t* s2 = nullptr) {
    constexpr int kOut = GATED ? kRows / 2 : kRows;
    // 128-k stages take a third x stage (and one packed stage less) when the
    // tile plan leaves room for it: the MMA thread then rarely waits for x
    using P = Pipe<KS>;
    using P3 = Pipe<KS, 3>;
    const int ne = offsets ? E : 1;
    const bool x3 = KS == 128 && smem_bytes<P3>(ne) <= dev.smem_optin;
    const size_t smem = x3 ? smem_bytes<P3>(ne) : smem_bytes<P>(ne);
    if (smem > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cuda_status(cudaErrorNotSupported, "gemm split: cuTensorMapEncodeTiled entry point");
    CUtensorMap mx, mw, mw2;
    {  // x [M, K] (with a row gather: x [T, K]; the map is then never loaded from)
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(gather ? T : M)};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kBN};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm split: cuTensorMapEncodeTiled (x)");
    }
    auto encode_w2d = [&](CUtensorMap* m, const uint8_t* w) {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        cuuint32_t box[2] = {KS / 2, (cuuint32_t)kOut};  // gated: 64 rows of each matrix per stage
        cuuint32_t es[2] = {1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, P::kPSwizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (GATED && (offsets != nullptr || gather != nullptr || qw2 == nullptr || s2 == nullptr))
        return W4A16_ERR_INVALID_ARG;
    if (offsets == nullptr) {
        if (!encode_w2d(&mw, qw) || (GATED && !encode_w2d(&mw2, qw2)))
            return cuda_status(cudaErrorInvalidValue, "gemm split: cuTensorMapEncodeTiled (weights)");
        if (!GATED) mw2 = mw;
    } else {
        cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)(N * (K / 2))};
        cuuint32_t box[3] = {KS / 2, (cuuint32_t)kRows, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, P::kPSwizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm split: cuTensorMapEncodeTiled (weights)");
        mw2 = mw;
    }
    SplitArgs a{};
    a.s = s;
    a.s2 = s2;
    a.y = y;
    a.offsets = offsets;
    a.gather = gather;
    a.xg = x;
    a.T = T;
    a.M = M;
    a.N = N;
    a.K = K;
    a.E = offsets ? E : 1;
    a.gshift = gshift;
    a.err = dev.error_word;
    // an upper bound on the tiles (each expert adds at most one partial token tile)
    const int64_t ntn = (N + kOut - 1) / kOut;
    const int64_t tiles = ((M + kBN - 1) / kBN + (offsets ? E : 0)) * ntn;
    if (tiles > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const unsigned grid = (unsigned)(tiles < dev.sms ? tiles : dev.sms);
    static PerDeviceOnce once;
    const cudaError_t attr = once.run(dev.device, [&dev] {
        cudaError_t e = cudaFuncSetAttribute(split_kernel<KS, GATED, P::kXStages>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev.smem_optin);
        if constexpr (KS == 128) {
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(split_kernel<KS, GATED, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dev.smem_optin);
        }
        return e;
    });
    if (attr != cudaSuccess) return cuda_status(attr, "gemm split: cudaFuncSetAttribute");
    if constexpr (KS == 128) {
        if (x3) {
            split_kernel<KS, GATED, 3><<<grid, kThreads, smem, st>>>(mx, mw, mw2, a);
            return cuda_status(cudaGetLastError(), "gemm split: kernel launch");
        }
    }
    split_kernel<KS, GATED, P::kXStages><<<grid, kThreads, smem, st>>>(mx, mw, mw2, a);
    return cuda_status(cudaGetLastError(), "gemm split: kernel launch");
}

}  // namespace

bool split_supports(int group, int E) {
    return (group == 32 || group == 64 || group == 128) && E >= 1 && E <= kMaxE;
}

w4a16_status split_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                          int64_t M, int64_t N, int64_t K, int group, const int32_t* offsets, int E,
                          const int32_t* gather, int64_t T, cudaStream_t st) {
    if (!split_supports(group, offsets ? E : 1)) return W4A16_ERR_UNSUPPORTED;
    const int gshift = group == 32 ? 0 : group == 64 ? 1 : 2;
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL || T > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    // long K: 128-k stages; short K: 64-k stages and a deeper pipeline for the tile's fill
    // 128-k stages from K = 512: with the third x stage they beat 64-k stages on
    // the routed down projection too (K = 512: 121.4 against 126.8 us)
    if (K >= 512) return launch_split<128>(dev, x, qw, s, y, M, N, K, gshift, offsets, E, gather, T, st);
    return launch_split<64>(dev, x, qw, s, y, M, N, K, gshift, offsets, E, gather, T, st);
}

w4a16_status split_gated_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw_gate,
                                const uint16_t* s_gate, const uint8_t* qw_up, const uint16_t* s_up, uint16_t* y,
                                int64_t M, int64_t N, int64_t K, int group, cudaStream_t st) {
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    if (!split_supports(group, 1)) return W4A16_ERR_UNSUPPORTED;
    const int gshift = group == 32 ? 0 : group == 64 ? 1 : 2;
    if (K >= 1024)
        return launch_split<128, true>(dev, x, qw_gate, s_gate, y, M, N, K, gshift, nullptr, 1, nullptr, 0, st,
                                       qw_up, s_up);
    return launch_split<64, true>(dev, x, qw_gate, s_gate, y, M, N, K, gshift, nullptr, 1, nullptr, 0, st, qw_up,
                                  s_up);
}

#ifdef W4A16_TEST_HOOKS
cudaError_t split_set_test_hooks(const TestHooks& h) { return cudaMemcpyToSymbol(g_hooks, &h, sizeof(h)); }
cudaError_t split_get_test_counters(TestCounters* c) { return cudaMemcpyFromSymbol(c, g_counters, sizeof(*c)); }
#endif

}  // namespace w4a16
