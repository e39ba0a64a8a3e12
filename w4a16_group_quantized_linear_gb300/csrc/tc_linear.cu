// Tensor-core GEMM of the W4A16 layer (sm_103a: TMA, tcgen05 MMA, TMEM) for
// prefill (LLM170 page: pp512..pp4096) and the routed-expert layer (LLM170
// page: "MoE resident" g32 models).
//
// Formulation ("swap AB"): D[n, m] = sum_k W^[n, k] x[m, k]. A CTA owns 128
// weight rows n (the 128 TMEM lanes) and BN tokens m (TMEM columns), over all
// of K, in stages of KSTAGE k.
//
//   warp 0       TMA producer. Two rings: the packed weights of a stage
//                (128 rows x KSTAGE/2 bytes, swizzled) in a PSTAGES-deep ring,
//                and the stage's x (KSTAGE/64 boxes of BN rows x 64 fp16,
//                128-byte swizzle) in an XSTAGES-deep ring. The packed ring is
//                deeper, so the dequant warps do not wait on a load once a
//                TMEM A stage frees up.
//   warp 1       TMEM allocation and the MMA issuer: one lane issues
//                tcgen05.mma.kind::f16 with A (the dequantized weights) read
//                from TMEM and B (x) from shared memory; per stage one commit
//                releases the x slot and one the TMEM A stage (the two rings
//                may differ in depth).
//   DEQW warps   dequant: thread = TMEM lane = weight row; expands its row's
//                nibbles of the stage into the exact fp16 integers q (natural
//                k order) and writes them into the TMEM A stage (tcgen05.st).
//   EPIW warps   epilogue: every scale group gets its own fp32 partial in one
//                of two TMEM buffers; per group the epilogue reads it
//                (tcgen05.ld), multiplies by the row's fp32 scale and adds
//                into fp32 registers: acc += s[n, grp] * sum_{k in grp} x q.
//                Finally it rounds once to fp16 and stores y.
// All products x*q are exact, group sums are fp32 and the scale is applied
// in fp32; no fp16 rounding of s*q happens.
//
// The routed-expert variant derives (expert, token tile) from the device-side
// offsets. Every mbarrier wait is bounded in time; a wait that gives up
// records W4A16_ERR_TIMEOUT in the device error word and the CTA unwinds (it
// drains its own TMA loads and MMAs first, then frees TMEM).
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s
constexpr int kRowsPerTile = 128;

#ifdef W4A16_TEST_HOOKS
__device__ TestHooks g_hooks = {kWaitLimitNs, -1};
__device__ TestCounters g_counters = {0ull, 0ull};
__device__ __forceinline__ uint64_t wait_limit() { return g_hooks.wait_limit_ns; }
__device__ __forceinline__ bool may_issue(int64_t issued) {
    return g_hooks.issue_limit < 0 || issued < g_hooks.issue_limit;
}
__device__ __forceinline__ void count_tmem(unsigned long long* c) { atomicAdd(c, 1ull); }
#define W4A16_COUNT_TMEM(field) count_tmem(&g_counters.field)
#else
__device__ __forceinline__ constexpr uint64_t wait_limit() { return kWaitLimitNs; }
__device__ __forceinline__ constexpr bool may_issue(int64_t) { return true; }
#define W4A16_COUNT_TMEM(field) ((void)0)
#endif

template <int G_, int BN_, int KSTAGE_, int PSTAGES_, int XSTAGES_, int DEQW_, int EPIW_, bool SRUNS_ = false,
          int ASTAGES_ = XSTAGES_, int MMAW_ = 1>
struct Cfg {
    static constexpr int G = G_;              // scale group
    static constexpr int BN = BN_;            // tokens per tile (MMA N)
    static constexpr int KSTAGE = KSTAGE_;    // k per pipeline stage
    static constexpr int PSTAGES = PSTAGES_;  // packed-weight ring depth
    static constexpr int XSTAGES = XSTAGES_;  // x ring depth
    static constexpr int ASTAGES = ASTAGES_;  // TMEM A ring depth
    static constexpr int MMAW = MMAW_;        // MMA-issuing warps (2: one per partial buffer)
    static constexpr int DEQW = DEQW_;        // dequant warps (multiple of 4)
    static constexpr int EPIW = EPIW_;        // epilogue warps (multiple of 4)
    static constexpr bool SRUNS = SRUNS_;     // scales in 16-byte runs, 16-24 groups ahead

    static constexpr int THREADS = (2 + DEQW + EPIW + MMAW - 1) * 32;
    static constexpr int PBYTES = kRowsPerTile * KSTAGE / 2;  // packed weights per stage
    static constexpr int XBOXES = KSTAGE / 64;                 // x boxes of 64 k per stage
    static constexpr int XBOX_BYTES = BN * 128;
    static constexpr int XBYTES = XBOXES * XBOX_BYTES;
    static constexpr int ACOLS = KSTAGE / 2;                   // TMEM columns per A stage
    static constexpr int DCOLS = 2 * BN;                       // two group-partial buffers
    static constexpr int TMEM_COLS = 512;
    static constexpr int NPART = DEQW / 4;                     // dequant threads per row
    static constexpr int PART_K = KSTAGE / NPART;              // k per dequant thread per stage
    static constexpr int NCP = EPIW / 4;                       // epilogue threads per row
    static constexpr int BNP = BN / NCP;                       // tokens per epilogue thread
    static constexpr int XOFF = PSTAGES * PBYTES;              // x ring after the packed ring
    static constexpr int SMEM = XOFF + XSTAGES * XBYTES + 1024 + 512;
    // packed rows of KSTAGE/2 bytes are stored with the swizzle of that width
    static constexpr CUtensorMapSwizzle PSWIZZLE =
        KSTAGE == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : (KSTAGE == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);

    static_assert(KSTAGE % 64 == 0 && KSTAGE <= 256, "stage shape");
    static_assert(DCOLS + ASTAGES * ACOLS <= TMEM_COLS, "TMEM budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(PART_K % 64 == 0 && BNP % 16 == 0, "per-thread shares");
    static_assert(PSTAGES <= 8 && XSTAGES <= 8 && ASTAGES <= 4 && PSTAGES >= ASTAGES, "ring depths");
    static_assert(MMAW == 1 || (MMAW == 2 && KSTAGE >= G), "a second issuer takes whole groups");
    static_assert(PBYTES % 1024 == 0 && XBYTES % 1024 == 0, "1024-byte aligned stages");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// 128-token tiles (the fused gate+up pair and experts outside the split-scale
// kernel's range): 256-k stages amortise the MMA thread's per-stage waits and
// commits over 16 MMAs.
template <int G>
using PrefillCfg = Cfg<G, 128, 256, 4, 2, 4, 8>;
// Small batches (M <= 64): narrower token tiles waste fewer MMA columns; four
// epilogue warps cover the tile. The MMA issue rate bounds these tiles (about
// 60 ns per instruction whatever the width), and a second issuing warp takes
// every other scale group: M = 32 runs in 30.8 instead of 32.8 us.
template <int G>
using Narrow64Cfg = Cfg<G, 64, 256, 4, 2, 4, 4, false, 2, 2>;
template <int G>
using Narrow32Cfg = Cfg<G, 32, 256, 4, 2, 4, 4, false, 2, 2>;
// Routed experts: the prefill tile, with the scales fetched further ahead. At group 32 a
// stage holds 8 groups, so scalar loads a few groups ahead leave the epilogue waiting on HBM.
template <int G>
using MoeCfg = Cfg<G, 128, 256, 4, 2, 4, 8, true>;

struct Args {
    const uint16_t* s;
    const uint16_t* s2;      // gated: the up projection's scales (s holds the gate's)
    uint16_t* y;
    const int32_t* offsets;  // routed experts; nullptr: dense
    int64_t M, N, K;
    int64_t mt, tiles;  // dense: token tiles, and tiles in all (token tile fastest)
    int E;
    int n_fast;  // routed experts: 1 if blockIdx.x is the weight-row tile and blockIdx.y the token tile
    unsigned int* err;
};

struct Smem {
    uint64_t pfull[8];   // a packed-weight stage landed
    uint64_t pempty[8];  // the dequant warps finished reading a packed stage
    uint64_t xfull[8];   // an x stage landed
    uint64_t xempty[8];  // the MMAs reading an x stage finished
    uint64_t afull[4];   // a TMEM A stage was written
    uint64_t aempty[4];  // the MMAs reading a TMEM A stage finished
    uint64_t dfull[2];   // group partial ready in TMEM buffer b
    uint64_t dempty[2];  // epilogue done reading TMEM buffer b
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    int expert, row0, row_end, valid;
};
static_assert(sizeof(Smem) <= 512, "barrier block");

__device__ __forceinline__ void fail(const Args& a, Smem* sm, unsigned code) {
    raise_device_error(a.err, code);
    *reinterpret_cast<volatile int*>(&sm->abort) = 1;
}

// Routed experts: the CTA's token tile from the device offsets. One warp.
template <int BN>
__device__ void find_tile(const Args& a, Smem* sm, int lane, int t) {
    int base = 0;
    bool ok = true;
    int found = -1, f_row0 = 0, f_end = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0, hi = 0, tiles = 0;
        if (e < a.E) {
            lo = __ldg(a.offsets + e);
            hi = __ldg(a.offsets + e + 1);
            if (hi < lo || lo < 0 || (int64_t)hi > a.M) ok = false;
            tiles = hi > lo ? (hi - lo + BN - 1) / BN : 0;
        }
        int incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        const int start = base + incl - tiles;
        if (e < a.E && t >= start && t < start + tiles) {
            found = e;
            f_row0 = lo + (t - start) * BN;
            f_end = hi;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    ok = __all_sync(0xffffffffu, ok);
    const bool ends_ok = __ldg(a.offsets) == 0 && (int64_t)__ldg(a.offsets + a.E) == a.M;
    if (lane == 0) {
        sm->valid = 0;
        if (!ok || !ends_ok) raise_device_error(a.err, W4A16_ERR_BAD_OFFSETS);
    }
    __syncwarp();
    if (ok && ends_ok && found >= 0) {  // tiles are disjoint: at most one lane
        sm->expert = found;
        sm->row0 = f_row0;
        sm->row_end = f_end;
        sm->valid = 1;
    }
}

// Byte offset of 16-byte chunk c of row r in a swizzled packed box.
template <int KSTAGE>
__device__ __forceinline__ int packed_offset(int r, int c) {
    if constexpr (KSTAGE == 256) return r * 128 + ((c ^ (r & 7)) << 4);          // 128-byte swizzle
    else if constexpr (KSTAGE == 128) return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); // 64-byte swizzle
    else return r * 32 + ((c ^ ((r >> 2) & 1)) << 4);                             // 32-byte swizzle
}

// GATED: the tile's 128 weight rows are 64 rows of Wg and the same 64 rows of
// Wu, loaded as two boxes of 64 rows into one packed stage (tmap_w, tmap_w2;
// shared-memory rows 0-63 and 64-127); the CTA forms y = silu(g) * u for its
// 64 outputs from the fp32 sums. TMEM lane r holds output o = 8 (r / 16) +
// r % 8 of the gate (bit 3 of r clear) or of the up projection (bit 3 set), so
// the g and u of one output sit in lanes r and r ^ 8 of the same warp and meet
// through one shuffle; each run of 8 lanes reads 8 distinct swizzle rows.

template <class C, bool GATED>
__global__ void __launch_bounds__(C::THREADS, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
              const __grid_constant__ CUtensorMap tmap_w2, const Args a) {
    constexpr int kOutRows = GATED ? kRowsPerTile / 2 : kRowsPerTile;  // outputs n per tile
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* pring = base;                // packed-weight stages
    uint8_t* xring = base + C::XOFF;      // x stages
    Smem* sm = reinterpret_cast<Smem*>(xring + C::XSTAGES * C::XBYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nst = (a.K + C::KSTAGE - 1) / C::KSTAGE;  // stages over K per tile
    const int nst32 = (int)nst;                             // K < 2^31
    // Dense: a persistent grid; this CTA takes tiles blockIdx.x, + gridDim.x, ...
    // and its rings, TMEM and group counters run on from one tile into the next,
    // so a tile's epilogue overlaps the next tile's loads and MMAs. Routed
    // experts: one tile per CTA, found from the device offsets.
    const bool dense = a.offsets == nullptr;
    const int64_t my_tiles = dense ? (a.tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 1;
    const int64_t my_stages = my_tiles * nst;

    if (warp == 0) {
        if (!dense) {
            find_tile<C::BN>(a, sm, lane, (int)(a.n_fast ? blockIdx.y : blockIdx.x));
        } else if (lane == 0) {
            sm->expert = 0;
            sm->row0 = 0;
            sm->row_end = (int)a.M;
            sm->valid = 1;
        }
        if (lane == 0) {
            for (int i = 0; i < C::PSTAGES; ++i) {
                ptx::mbar_init(&sm->pfull[i], 1);
                ptx::mbar_init(&sm->pempty[i], C::DEQW * 32);
            }
            for (int i = 0; i < C::XSTAGES; ++i) {
                ptx::mbar_init(&sm->xfull[i], 1);
                ptx::mbar_init(&sm->xempty[i], C::MMAW);
            }
            for (int i = 0; i < C::ASTAGES; ++i) {
                ptx::mbar_init(&sm->afull[i], C::DEQW * 32);
                ptx::mbar_init(&sm->aempty[i], C::MMAW);
            }
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(&sm->dfull[b], 1);
                ptx::mbar_init(&sm->dempty[b], C::EPIW * 32);
            }
            ptx::mbar_init(&sm->mma_done, C::MMAW);
            sm->abort = 0;
            ptx::fence_mbar_init();
            ptx::prefetch_tensormap(&tmap_x);
            ptx::prefetch_tensormap(&tmap_w);
            if (GATED) ptx::prefetch_tensormap(&tmap_w2);
        }
    }
    __syncthreads();
    if (!sm->valid) return;
    if (warp == 1) {
        ptx::tmem_alloc(&sm->tmem_base, C::TMEM_COLS);
        ptx::tmem_relinquish();
        if (lane == 0) W4A16_COUNT_TMEM(tmem_allocs);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    const int expert = sm->expert, row_end = sm->row_end;
    volatile int* abort = &sm->abort;
    // tile j of this CTA: its first token and its weight-row tile
    auto tile_row0 = [&](int64_t j) -> int {
        return dense ? (int)(((int64_t)blockIdx.x + j * gridDim.x) % a.mt * C::BN) : sm->row0;
    };
    auto tile_n = [&](int64_t j) -> int64_t {
        return dense ? ((int64_t)blockIdx.x + j * gridDim.x) / a.mt : (a.n_fast ? blockIdx.x : blockIdx.y);
    };

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int64_t ip = 0, ix = 0;  // stages issued on each ring
            // each ring's position in its current tile (kept incrementally: no 64-bit
            // division per stage on this thread)
            int sx = 0, sp = 0;
            int64_t jx = 0, jp = 0;
            int row0x = tile_row0(0);
            int n0p = (int)(tile_n(0) * kOutRows);
            // Both rings are polled, so a full ring never holds up the other one.
            bool ok = true;
            uint64_t idle_since = 0;
            while (ip < my_stages || ix < my_stages) {
                bool moved = false;
                if (ix < my_stages && may_issue(ip + ix)) {
                    const int st = (int)(ix % C::XSTAGES);
                    const int64_t round = ix / C::XSTAGES;
                    if (round == 0 || ptx::mbar_try_wait(&sm->xempty[st], (uint32_t)((round - 1) & 1))) {
                        ptx::mbar_arrive_expect_tx(&sm->xfull[st], C::XBYTES);
                        const int kc = sx * C::KSTAGE;
#pragma unroll
                        for (int b = 0; b < C::XBOXES; ++b)
                            ptx::tma_load_2d(xring + st * C::XBYTES + b * C::XBOX_BYTES, &tmap_x, &sm->xfull[st],
                                             kc + 64 * b, row0x);
                        ++ix;
                        if (++sx == nst32) {
                            sx = 0;
                            if (++jx < my_tiles) row0x = tile_row0(jx);
                        }
                        moved = true;
                    }
                }
                if (ip < my_stages && may_issue(ip + ix)) {
                    const int st = (int)(ip % C::PSTAGES);
                    const int64_t round = ip / C::PSTAGES;
                    if (round == 0 || ptx::mbar_try_wait(&sm->pempty[st], (uint32_t)((round - 1) & 1))) {
                        ptx::mbar_arrive_expect_tx(&sm->pfull[st], C::PBYTES);
                        const int kc = sp * C::KSTAGE, n0 = n0p;
                        if (GATED) {
                            ptx::tma_load_2d(pring + st * C::PBYTES, &tmap_w, &sm->pfull[st], kc / 2, n0);
                            ptx::tma_load_2d(pring + st * C::PBYTES + C::PBYTES / 2, &tmap_w2, &sm->pfull[st],
                                             kc / 2, n0);
                        } else if (a.offsets == nullptr) {
                            ptx::tma_load_2d(pring + st * C::PBYTES, &tmap_w, &sm->pfull[st], kc / 2, n0);
                        } else {
                            ptx::tma_load_3d(pring + st * C::PBYTES, &tmap_w, &sm->pfull[st], kc / 2, n0, expert);
                        }
                        ++ip;
                        if (++sp == nst32) {
                            sp = 0;
                            if (++jp < my_tiles) n0p = (int)(tile_n(jp) * kOutRows);
                        }
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
                for (int64_t i = ip > C::PSTAGES ? ip - C::PSTAGES : 0; i < ip; ++i)
                    ptx::mbar_wait(&sm->pfull[i % C::PSTAGES], (uint32_t)((i / C::PSTAGES) & 1), &never, kDrainLimitNs);
                for (int64_t i = ix > C::XSTAGES ? ix - C::XSTAGES : 0; i < ix; ++i)
                    ptx::mbar_wait(&sm->xfull[i % C::XSTAGES], (uint32_t)((i / C::XSTAGES) & 1), &never, kDrainLimitNs);
            }
        }
    } else if (warp == 1 || (C::MMAW == 2 && warp == 2 + C::DEQW + C::EPIW)) {
        // ----------------------------------------------------------- MMA issue
        // With two issuers, issuer mi takes the scale groups whose partial goes to
        // TMEM buffer mi: the instruction issue of one thread is the limit.
        const int mi = warp == 1 ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(kRowsPerTile, C::BN);
            constexpr int GPS = C::G / 16;  // MMAs per scale group
            int64_t grp = 0;
            int cur_b = 0;
            bool ok = true;
            int s_in = 0;  // stage within the current tile
            for (int64_t c = 0; ok && c < my_stages; ++c, s_in = s_in + 1 == nst32 ? 0 : s_in + 1) {
                const int xs = (int)(c % C::XSTAGES), as = (int)(c % C::ASTAGES);
                if (!ptx::mbar_wait(&sm->xfull[xs], (uint32_t)((c / C::XSTAGES) & 1), abort, wait_limit()) ||
                    !ptx::mbar_wait(&sm->afull[as], (uint32_t)((c / C::ASTAGES) & 1), abort, wait_limit())) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const int64_t kc = (int64_t)s_in * C::KSTAGE;
                const uint64_t bdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(xring + xs * C::XBYTES));
                const uint32_t a_col = tmem + (uint32_t)(C::DCOLS + as * C::ACOLS);
                const int nk = (int)((a.K - kc < C::KSTAGE ? a.K - kc : C::KSTAGE) >> 4);
                const bool stage_opens = C::KSTAGE >= C::G || (kc % C::G) == 0;
                const bool stage_closes = C::KSTAGE >= C::G || ((kc + C::KSTAGE) % C::G) == 0;
#pragma unroll
                for (int kk = 0; kk < C::KSTAGE / 16; ++kk) {
                    if (kk >= nk) break;
                    const bool first = C::KSTAGE >= C::G ? (kk % GPS == 0) : (kk == 0 && stage_opens);
                    const bool last = C::KSTAGE >= C::G ? (kk % GPS == GPS - 1)
                                                        : (kk == C::KSTAGE / 16 - 1 && stage_closes);
                    const bool mine = C::MMAW == 1 || (int)(grp & 1) == mi;
                    if (first && mine) {
                        cur_b = (int)(grp & 1);
                        if (grp >= 2) {
                            if (!ptx::mbar_wait(&sm->dempty[cur_b], (uint32_t)(((grp >> 1) - 1) & 1), abort,
                                                wait_limit())) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                        }
                    }
                    if (mine) {
                        const uint64_t bdesc =
                            bdesc0 + (uint64_t)((((kk >> 2) * C::XBOX_BYTES) + (kk & 3) * 32) >> 4);
                        ptx::mma_f16_ts(tmem + (uint32_t)(cur_b * C::BN), a_col + (uint32_t)(kk * 8), bdesc, idesc,
                                        first ? 0u : 1u);
                        if (last) ptx::mma_commit(&sm->dfull[cur_b]);
                    }
                    if (last) ++grp;
                }
                if (!ok) break;
                ptx::mma_commit(&sm->xempty[xs]);  // the x slot is free again
                ptx::mma_commit(&sm->aempty[as]);  // and so is the TMEM A stage
            }
            if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
            ptx::mma_commit(&sm->mma_done);
            volatile int never = 0;
            ptx::mbar_wait(&sm->mma_done, 0, &never, kDrainLimitNs);
        }
    } else if (warp < 2 + C::DEQW) {
        // -------------------------------------------------------------- dequant
        const int dw = warp - 2;
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int part = dw >> 2;                  // which share of the stage's k
        const int r = quad * 32 + lane;            // weight row in the tile = TMEM lane
        constexpr int CH = C::PART_K / 32;         // 16-byte packed chunks (32 k each) per thread
        bool ok = true;
        for (int64_t c = 0; c < my_stages; ++c) {
            const int ps = (int)(c % C::PSTAGES), as = (int)(c % C::ASTAGES);
            const int64_t around = c / C::ASTAGES;
            // warp-uniform outcome: the TMEM stores below are .sync.aligned
            const bool got = ptx::mbar_wait(&sm->pfull[ps], (uint32_t)((c / C::PSTAGES) & 1), abort, wait_limit()) &&
                             (around == 0 ||
                              ptx::mbar_wait(&sm->aempty[as], (uint32_t)((around - 1) & 1), abort, wait_limit()));
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint8_t* prow = pring + ps * C::PBYTES;
            const int prow_r = GATED ? gated_smem_row(r) : r;  // shared-memory row of this TMEM lane
            const uint32_t tcol = tmem + ((uint32_t)(quad * 32) << 16) +
                                  (uint32_t)(C::DCOLS + as * C::ACOLS + part * (C::PART_K / 2));
#pragma unroll
            for (int h = 0; h < CH; h += 2) {  // two chunks = 64 k = 32 columns per store
                uint32_t v[32];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint4 p =
                        *reinterpret_cast<const uint4*>(prow + packed_offset<C::KSTAGE>(prow_r, part * CH + h + q));
                    const uint32_t words[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {  // word j holds k = 8j .. 8j+7 of this chunk
                        uint32_t h04, h15, h26, h37;
                        nibbles_to_half2(words[j], h04, h15, h26, h37);
                        v[q * 16 + 4 * j + 0] = __byte_perm(h04, h15, 0x5410);  // (k0, k1)
                        v[q * 16 + 4 * j + 1] = __byte_perm(h26, h37, 0x5410);  // (k2, k3)
                        v[q * 16 + 4 * j + 2] = __byte_perm(h04, h15, 0x7632);  // (k4, k5)
                        v[q * 16 + 4 * j + 3] = __byte_perm(h26, h37, 0x7632);  // (k6, k7)
                    }
                }
                ptx::tmem_st_32x32b_x32(tcol + (uint32_t)(h * 16), v);
            }
            ptx::mbar_arrive(&sm->pempty[ps]);  // this thread has read its packed bytes
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm->afull[as]);
        }
        if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------- epilogue
        const int ew = warp - 2 - C::DEQW;
        const int quad = warp & 3;
        const int cp = ew >> 2;                    // which share of the BN tokens
        const int r = quad * 32 + lane;            // weight row in the tile
        const int gk = (int)(a.K / C::G);          // groups per row
        int64_t grp = 0;
        bool ok = true;  // warp-uniform: every failed wait below is agreed on by the whole warp
        const bool up_row = GATED && ((r >> 3) & 1);
        int64_t n = 0;                  // this thread's output row in the current tile
        bool n_ok = false;
        const uint16_t* srow = a.s;     // and its scale row
        float acc[C::BNP];
        // Scales are streamed from HBM once. Dense tiles keep SB..2 SB groups of them in flight
        // (scalar loads); with SRUNS they come in runs of 8 groups (one 16-byte load when a
        // scale row is a multiple of 16 bytes), three runs in flight, 16 to 24 groups ahead.
        constexpr int SB = C::SRUNS ? 8 : (C::BNP > 32 ? 4 : 8);
        using Run = std::conditional_t<C::SRUNS, uint4, float[SB]>;
        const bool svec = (gk % 8) == 0;
        Run run0, run1, run2;
        auto load_run = [&](Run& dst, int gb) {
            if constexpr (C::SRUNS) {
                dst = make_uint4(0u, 0u, 0u, 0u);
                if (!n_ok || gb >= gk) return;
                if (svec) {
                    dst = __ldg(reinterpret_cast<const uint4*>(srow + gb));
                } else {
                    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int i = 0; i < SB; ++i)
                        if (gb + i < gk) w[i >> 1] |= (uint32_t)__ldg(srow + gb + i) << (16 * (i & 1));
                    dst = make_uint4(w[0], w[1], w[2], w[3]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < SB; ++i)
                    dst[i] = (n_ok && gb + i < gk) ? __half2float(__ushort_as_half(__ldg(srow + gb + i))) : 0.0f;
            }
        };
        auto scale_of = [&](const Run& run, int i) -> float {
            if constexpr (C::SRUNS) {
                const uint32_t w = i < 2 ? run.x : i < 4 ? run.y : i < 6 ? run.z : run.w;
                return __half2float(__ushort_as_half((unsigned short)(w >> (16 * (i & 1)))));
            } else {
                return run[i];
            }
        };
        auto run_groups = [&](const Run& run, int gb) {
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                if (gb + i >= gk || !ok) break;
                const int b = (int)(grp & 1);
                if (!__all_sync(0xffffffffu,
                                ptx::mbar_wait(&sm->dfull[b], (uint32_t)((grp >> 1) & 1), abort, wait_limit()))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * C::BN + cp * C::BNP);
                const float sv = scale_of(run, i);
                // The buffer goes back to the MMA thread as soon as the partial is in
                // registers; the multiply-adds follow.
                if constexpr (C::BNP == 16) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(taddr, v);
                    ptx::tmem_ld_wait();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(&sm->dempty[b]);
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = fmaf(sv, __uint_as_float(v[j]), acc[j]);
                } else {
#pragma unroll
                    for (int ch = 0; ch < C::BNP / 32; ++ch) {
                        uint32_t v[32];
                        ptx::tmem_ld_32x32b_x32(taddr + ch * 32, v);
                        ptx::tmem_ld_wait();
                        if (ch == C::BNP / 32 - 1) {
                            ptx::tc_fence_before();
                            ptx::mbar_arrive(&sm->dempty[b]);
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) acc[ch * 32 + j] = fmaf(sv, __uint_as_float(v[j]), acc[ch * 32 + j]);
                    }
                }
                ++grp;
            }
        };
        for (int64_t jt = 0; ok && jt < my_tiles; ++jt) {
        n = tile_n(jt) * kOutRows + (GATED ? gated_out_row(r) : r);
        n_ok = n < a.N;
        srow = (up_row ? a.s2 : a.s) + ((int64_t)expert * a.N + (n_ok ? n : 0)) * gk;
#pragma unroll
        for (int j = 0; j < C::BNP; ++j) acc[j] = 0.0f;
        load_run(run0, 0);
        load_run(run1, SB);
        if constexpr (C::SRUNS) {
            load_run(run2, 2 * SB);
            for (int gb = 0; ok && gb < gk; gb += 3 * SB) {
                run_groups(run0, gb);
                load_run(run0, gb + 3 * SB);
                if (ok) run_groups(run1, gb + SB);
                load_run(run1, gb + 4 * SB);
                if (ok) run_groups(run2, gb + 2 * SB);
                load_run(run2, gb + 5 * SB);
            }
        } else {
            for (int gb = 0; ok && gb < gk; gb += 2 * SB) {
                run_groups(run0, gb);
                load_run(run0, gb + 2 * SB);
                if (ok) run_groups(run1, gb + SB);
                load_run(run1, gb + 3 * SB);
            }
        }
        if (!ok) break;
        const int m0 = tile_row0(jt) + cp * C::BNP;  // first token of this thread's share
        if constexpr (GATED) {
            // Lanes r and r ^ 8 hold g and u of output n: the gate lane finishes the even
            // tokens of each pair and the up lane the odd ones, each handing the other
            // the operand it lacks (the whole warp is here: ok is warp-uniform).
            {
#pragma unroll
                for (int j = 0; j < C::BNP; j += 2) {
                    const float mine = up_row ? acc[j] : acc[j + 1];
                    const float other = __shfl_xor_sync(0xffffffffu, mine, 8);
                    const float g = up_row ? other : acc[j], u = up_row ? acc[j + 1] : other;
                    const int m = m0 + j + (up_row ? 1 : 0);
                    if (n_ok && m < row_end) {
                        const float silu = __fdividef(g, 1.0f + __expf(-g));
                        a.y[(int64_t)m * a.N + n] = __half_as_ushort(__float2half_rn(silu * u));
                    }
                }
            }
        } else {
            if (n_ok) {
#pragma unroll
                for (int j = 0; j < C::BNP; ++j)
                    if (m0 + j < row_end) a.y[(int64_t)(m0 + j) * a.N + n] = __half_as_ushort(__float2half_rn(acc[j]));
            }
        }
        }
        if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) {
        ptx::tmem_dealloc(tmem, C::TMEM_COLS);
        if (lane == 0) W4A16_COUNT_TMEM(tmem_frees);
    }
}

// ------------------------------------------------------------------- host --

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

template <class C>
w4a16_status make_maps(const uint16_t* x, const uint8_t* qw, int64_t M, int64_t N, int64_t K, int E, bool grouped,
                       CUtensorMap* mx, CUtensorMap* mw, int w_rows = kRowsPerTile) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cuda_status(cudaErrorNotSupported, "gemm: cuTensorMapEncodeTiled entry point");
    {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)C::BN};
        cuuint32_t es[2] = {1, 1};
        if (enc(mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm: cuTensorMapEncodeTiled");
    }
    if (!grouped) {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        cuuint32_t box[2] = {(cuuint32_t)(C::KSTAGE / 2), (cuuint32_t)w_rows};
        cuuint32_t es[2] = {1, 1};
        if (enc(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, C::PSWIZZLE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm: cuTensorMapEncodeTiled");
    } else {
        cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)(N * (K / 2))};
        cuuint32_t box[3] = {(cuuint32_t)(C::KSTAGE / 2), (cuuint32_t)kRowsPerTile, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, C::PSWIZZLE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemm: cuTensorMapEncodeTiled");
    }
    return W4A16_OK;
}

// A dense launch is a persistent grid of one CTA per SM: each CTA holds all of
// an SM's TMEM for its lifetime, so a second CTA on the same SM would only
// wait. Configurations whose shared memory would let two CTAs share an SM ask
// for just over half of the SM's shared memory instead.
template <class C>
size_t dense_smem(const DeviceInfo& dev) {
    const size_t half = dev.smem_optin / 2 + 1024;
    return (size_t)C::SMEM > half ? (size_t)C::SMEM : half;
}

template <class C, bool GATED = false>
w4a16_status launch(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mw2,
                    const Args& a, dim3 grid, size_t smem, cudaStream_t st) {
    static PerDeviceOnce once;
    const cudaError_t attr_err = once.run(dev.device, [&dev] {
        return cudaFuncSetAttribute(tc_kernel<C, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)dev.smem_optin);
    });
    if (attr_err != cudaSuccess) return cuda_status(attr_err, "gemm: cudaFuncSetAttribute");
    tc_kernel<C, GATED><<<grid, C::THREADS, smem, st>>>(mx, mw, mw2, a);
    return cuda_status(cudaGetLastError(), "gemm: kernel launch");
}

template <class C>
w4a16_status gemm_g(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                    int64_t M, int64_t N, int64_t K, const int32_t* offsets, int E, cudaStream_t st) {
    if ((size_t)C::SMEM > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    CUtensorMap mx, mw;
    const w4a16_status ms = make_maps<C>(x, qw, M, N, K, E, offsets != nullptr, &mx, &mw);
    if (ms != W4A16_OK) return ms;
    Args a{};
    a.s = s;
    a.y = y;
    a.offsets = offsets;
    a.M = M;
    a.N = N;
    a.K = K;
    a.E = E;
    a.err = dev.error_word;
    const int64_t mt = offsets ? (M + C::BN - 1) / C::BN + E : (M + C::BN - 1) / C::BN;
    const int64_t nt = (N + kRowsPerTile - 1) / kRowsPerTile;
    if (mt > 0x7fffffffLL || nt > 65535) return W4A16_ERR_UNSUPPORTED;
    a.mt = mt;
    a.tiles = mt * nt;
    if (!offsets) {  // persistent: token tiles of one weight-row tile are consecutive, sharing it in L2
        const int64_t grid = a.tiles < dev.sms ? a.tiles : dev.sms;
        return launch<C>(dev, mx, mw, mw, a, dim3((unsigned)grid), dense_smem<C>(dev), st);
    }
    // Routed experts: the weight-row tiles of one token tile run side by side, so
    // they share that x tile in L2 instead of streaming x from HBM once per
    // weight-row tile (x_sorted is larger than L2 at the routed workloads).
    if (mt <= 65535) {
        a.n_fast = 1;
        return launch<C>(dev, mx, mw, mw, a, dim3((unsigned)nt, (unsigned)mt), C::SMEM, st);
    }
    return launch<C>(dev, mx, mw, mw, a, dim3((unsigned)mt, (unsigned)nt), C::SMEM, st);
}

// Gated pair: each CTA covers 64 outputs n with the 64 matching rows of Wg and Wu.
template <class C>
w4a16_status gemm_gated_g(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qg, const uint16_t* sg,
                          const uint8_t* qu, const uint16_t* su, uint16_t* y, int64_t M, int64_t N, int64_t K,
                          cudaStream_t st) {
    if ((size_t)C::SMEM > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    CUtensorMap mx, mg, mu, unused;
    w4a16_status ms = make_maps<C>(x, qg, M, N, K, 1, false, &mx, &mg, kRowsPerTile / 2);
    if (ms == W4A16_OK) ms = make_maps<C>(x, qu, M, N, K, 1, false, &unused, &mu, kRowsPerTile / 2);
    if (ms != W4A16_OK) return ms;
    Args a{};
    a.s = sg;
    a.s2 = su;
    a.y = y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.E = 1;
    a.err = dev.error_word;
    const int64_t mt = (M + C::BN - 1) / C::BN;
    const int64_t nt = (N + kRowsPerTile / 2 - 1) / (kRowsPerTile / 2);
    if (mt > 0x7fffffffLL || nt > 0x7fffffffLL / mt) return W4A16_ERR_UNSUPPORTED;
    a.mt = mt;
    a.tiles = mt * nt;
    const int64_t grid = a.tiles < dev.sms ? a.tiles : dev.sms;
    return launch<C, true>(dev, mx, mg, mu, a, dim3((unsigned)grid), dense_smem<C>(dev), st);
}

}  // namespace

w4a16_status gemm_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                         int64_t M, int64_t N, int64_t K, int group, const int32_t* expert_offsets, int E,
                         cudaStream_t st) {
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    // routed experts, and dense layers past the narrow tiles: the scale goes into
    // the A operand as an exact fp16 pair (tc_split.cu), with no per-group
    // epilogue round trip and 256-token MMAs (measured at M = 4096, 5120 -> 17408:
    // group 128 742 against 858 us on the tiles below, group 64 747 against 1066)
    if (split_supports(group, expert_offsets != nullptr ? E : 1) && (expert_offsets != nullptr || M > 64))
        return split_launch(dev, x, qw, s, y, M, N, K, group, expert_offsets, E, nullptr, 0, st);
    const int bn = expert_offsets != nullptr ? 0 : (M > 64 ? 128 : (M > 32 ? 64 : 32));
#define W4A16_GEMM(CFG)                                                                              \
    switch (group) {                                                                                 \
        case 32: return gemm_g<CFG<32>>(dev, x, qw, s, y, M, N, K, expert_offsets, E, st);           \
        case 64: return gemm_g<CFG<64>>(dev, x, qw, s, y, M, N, K, expert_offsets, E, st);           \
        case 128: return gemm_g<CFG<128>>(dev, x, qw, s, y, M, N, K, expert_offsets, E, st);         \
        default: return W4A16_ERR_UNSUPPORTED;                                                       \
    }
    if (bn == 0) W4A16_GEMM(MoeCfg)
    if (bn == 32) W4A16_GEMM(Narrow32Cfg)
    if (bn == 64) W4A16_GEMM(Narrow64Cfg)
    W4A16_GEMM(PrefillCfg)
#undef W4A16_GEMM
}

w4a16_status gemm_gated_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qweight_gate,
                               const uint16_t* scales_gate, const uint8_t* qweight_up, const uint16_t* scales_up,
                               uint16_t* y, int64_t M, int64_t N, int64_t K, int group, cudaStream_t st) {
    if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    // past the narrow tiles the pair runs on the split-scale kernel, as the plain layer does
    if (M > 64 && split_supports(group, 1))
        return split_gated_launch(dev, x, qweight_gate, scales_gate, qweight_up, scales_up, y, M, N, K, group, st);
    const int bn = M > 64 ? 128 : (M > 32 ? 64 : 32);
#define W4A16_GEMM(CFG)                                                                                    \
    switch (group) {                                                                                       \
        case 32: return gemm_gated_g<CFG<32>>(dev, x, qweight_gate, scales_gate, qweight_up, scales_up, y, \
                                              M, N, K, st);                                                \
        case 64: return gemm_gated_g<CFG<64>>(dev, x, qweight_gate, scales_gate, qweight_up, scales_up, y, \
                                              M, N, K, st);                                                \
        case 128: return gemm_gated_g<CFG<128>>(dev, x, qweight_gate, scales_gate, qweight_up, scales_up,  \
                                                y, M, N, K, st);                                           \
        default: return W4A16_ERR_UNSUPPORTED;                                                             \
    }
    if (bn == 32) W4A16_GEMM(Narrow32Cfg)
    if (bn == 64) W4A16_GEMM(Narrow64Cfg)
    W4A16_GEMM(PrefillCfg)
#undef W4A16_GEMM
}

#ifdef W4A16_TEST_HOOKS
cudaError_t gemm_set_test_hooks(const TestHooks& h) { return cudaMemcpyToSymbol(g_hooks, &h, sizeof(h)); }
cudaError_t gemm_get_test_counters(TestCounters* c) { return cudaMemcpyFromSymbol(c, g_counters, sizeof(*c)); }
#endif

}  // namespace w4a16
