// Tensor-core kernels of the W4A16 layer (sm_103a: TMA, tcgen05 MMA, TMEM).
//
// One warp-specialised kernel template serves the decode GEMV (M <= 16 rows
// of x, LLM170 page: "CUDA-graph decode", np4) and the prefill / routed-expert
// GEMM (LLM170 page: pp512..pp4096, "MoE resident" g32 models).
//
// Formulation ("swap AB"): D[n, m] = sum_k W^[n, k] x[m, k]. A CTA owns 128
// weight rows n (the 128 TMEM lanes) and BN tokens m (TMEM columns).
//
//   warp 0       TMA producer: for each K-stage, the packed weight box
//                (128 rows x KSTAGE/2 bytes, swizzled) and KSTAGE/64 boxes of
//                x (BN rows x 64 fp16, 128-byte swizzle) into a smem ring.
//   warp 1       TMEM allocation and the MMA issuer: one lane issues
//                tcgen05.mma.kind::f16 with A (the dequantized weights) read
//                from TMEM and B (x) from shared memory.
//   DEQW warps   dequant: thread = TMEM lane = weight row; expands its row's
//                nibbles of the stage into the exact fp16 integers q (natural
//                k order) and writes them into a TMEM A stage (tcgen05.st).
//   EPIW warps   epilogue: every scale group gets its own fp32 partial in one
//                of two TMEM buffers; per group the epilogue reads it
//                (tcgen05.ld), multiplies by the row's fp32 scale and adds
//                into fp32 registers: acc += s[n, grp] * sum_{k in grp} x q.
//                Finally it rounds once to fp16 and stores y.
// All products x*q are exact, group sums are fp32 and the scale is applied
// in fp32; no fp16 rounding of s*q happens.
//
// Schedules. TILES: one (128-row, BN-token) tile per CTA over all of K; the
// routed-expert variant derives (expert, token tile) from the device-side
// offsets. STREAM-K (decode): the (128-row tile, KSTAGE unit) space is split
// into equal contiguous ranges, one per CTA (a persistent grid of one CTA per
// SM); a CTA's range is a sequence of segments, one per row tile. A segment
// that covers all of K stores y directly; partial segments store fp32 partials
// in the workspace and the last CTA to arrive at a row tile (counter per
// tile) adds all partials in CTA order - deterministic - and stores y.
//
// Every mbarrier wait is bounded in time; a wait that gives up records
// W4A16_ERR_TIMEOUT in the device error word and the CTA unwinds (it drains
// its own TMA loads and MMAs first, then frees TMEM).
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s
constexpr int kRowsPerTile = 128;

template <int G_, int BN_, int KSTAGE_, int STAGES_, int ASTAGES_, int DEQW_, int EPIW_, bool STREAMK_, int ND_ = 2>
struct Cfg {
    static constexpr int G = G_;              // scale group
    static constexpr int BN = BN_;            // tokens per tile (MMA N)
    static constexpr int KSTAGE = KSTAGE_;    // k per pipeline stage
    static constexpr int STAGES = STAGES_;    // smem ring depth
    static constexpr int ASTAGES = ASTAGES_;  // TMEM A ring depth
    static constexpr int DEQW = DEQW_;        // dequant warps (multiple of 4)
    static constexpr int EPIW = EPIW_;        // epilogue warps (multiple of 4)
    static constexpr bool STREAMK = STREAMK_;
    static constexpr int ND = ND_;            // group-partial buffers in TMEM

    static constexpr int THREADS = (2 + DEQW + EPIW) * 32;
    static constexpr int PBYTES = kRowsPerTile * KSTAGE / 2;  // packed weights per stage
    static constexpr int XBOXES = KSTAGE / 64;                 // x boxes of 64 k per stage
    static constexpr int XBOX_BYTES = BN * 128;
    static constexpr int XBYTES = XBOXES * XBOX_BYTES;
    static constexpr int STAGE_BYTES = PBYTES + XBYTES;        // both multiples of 1024
    static constexpr int ACOLS = KSTAGE / 2;                   // TMEM columns per A stage
    static constexpr int DCOLS = ND * BN;                      // group-partial buffers
    static constexpr int TMEM_COLS = 512;
    static constexpr int NPART = DEQW / 4;                     // dequant threads per row
    static constexpr int PART_K = KSTAGE / NPART;              // k per dequant thread per stage
    static constexpr int NCP = EPIW / 4;                       // epilogue threads per row
    static constexpr int BNP = BN / NCP;                       // tokens per epilogue thread
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 512;
    // packed rows of KSTAGE/2 bytes are stored with the swizzle of that width
    static constexpr CUtensorMapSwizzle PSWIZZLE =
        KSTAGE == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : (KSTAGE == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);

    // stream-K segments start at stage boundaries, which must be group boundaries
    static_assert((!STREAMK || KSTAGE % G == 0) && KSTAGE % 64 == 0 && KSTAGE <= 256, "stage / group shape");
    static_assert(DCOLS + ASTAGES * ACOLS <= TMEM_COLS, "TMEM budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(PART_K % 64 == 0 && BNP % 16 == 0, "per-thread shares");
    static_assert(STAGES <= 8 && ASTAGES <= 8 && ND <= 4, "barrier arrays");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Prefill / routed experts: 128 tokens, 256-k stages, one tile per CTA. Large
// stages amortise the MMA thread's per-stage waits and commits over 16 MMAs.
template <int G>
using PrefillCfg = Cfg<G, 128, 256, 2, 2, 4, 8, false>;

struct Args {
    const uint16_t* s;
    uint16_t* y;
    const int32_t* offsets;  // routed experts; nullptr: dense
    int64_t M, N, K;
    int E;
    unsigned int* err;
    // stream-K
    float* partial;  // [CTAs][2][M][128] fp32
    int* counter;    // [row tiles]
    int64_t KU;      // KSTAGE units per row: ceil(K / KSTAGE)
    int64_t U;       // units: row tiles * KU
    int64_t P;       // CTAs taking part
};

struct Smem {
    uint64_t full[8];    // TMA bytes landed (packed + x)
    uint64_t empty[8];   // MMAs reading the stage finished
    uint64_t afull[8];   // TMEM A stage written
    uint64_t aempty[8];  // MMAs reading the TMEM A stage finished
    uint64_t dfull[4];   // group partial ready in TMEM buffer b
    uint64_t dempty[4];  // epilogue done reading TMEM buffer b
    uint64_t mma_done;
    uint64_t pstored;    // stream-K: every epilogue thread stored its partial
    uint64_t pflag;      // stream-K: last_flag is set
    uint32_t tmem_base;
    int abort;
    int expert, row0, row_end, valid;
    int last_flag;       // stream-K: this CTA finishes the row tile
};
static_assert(sizeof(Smem) <= 512, "barrier block");

// One stretch of work on one row tile: k in [k0, k1), tokens [row0, row_end).
struct Seg {
    int64_t n_tile, k0, k1;
    bool full;  // covers all of K: store y directly
    int slot;   // stream-K partial slot: 0 = first segment of the CTA, 1 = last
};

template <class C>
struct Schedule {
    int64_t u, u_end, first_tile;
    int64_t tile_y;  // TILES: row tile of this CTA
    bool done;

    __device__ __forceinline__ void init(const Args& a) {
        if constexpr (C::STREAMK) {
            u = blockIdx.x < a.P ? (int64_t)blockIdx.x * a.U / a.P : 0;
            u_end = blockIdx.x < a.P ? ((int64_t)blockIdx.x + 1) * a.U / a.P : 0;
            first_tile = u / a.KU;
            done = u >= u_end;
        } else {
            tile_y = blockIdx.y;
            done = false;
        }
    }
    __device__ __forceinline__ bool next(const Args& a, Seg& s) {
        if (done) return false;
        if constexpr (C::STREAMK) {
            const int64_t nt = u / a.KU, ku0 = u % a.KU;
            const int64_t tile_end = (nt + 1) * a.KU;
            const int64_t e = u_end < tile_end ? u_end : tile_end;
            s.n_tile = nt;
            s.k0 = ku0 * C::KSTAGE;
            s.k1 = (e - nt * a.KU) * C::KSTAGE;
            if (s.k1 > a.K) s.k1 = a.K;
            s.full = ku0 == 0 && e == tile_end;
            s.slot = nt == first_tile ? 0 : 1;
            u = e;
            done = u >= u_end;
        } else {
            s.n_tile = tile_y;
            s.k0 = 0;
            s.k1 = a.K;
            s.full = true;
            s.slot = 0;
            done = true;
        }
        return true;
    }
};

__device__ __forceinline__ void fail(const Args& a, Smem* sm, unsigned code) {
    raise_device_error(a.err, code);
    *reinterpret_cast<volatile int*>(&sm->abort) = 1;
}

// Routed experts: the CTA's token tile from the device offsets. One warp.
template <int BN>
__device__ void find_tile(const Args& a, Smem* sm, int lane) {
    const int t = blockIdx.x;
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

// Cross-CTA stream-K bookkeeping (same formulas on every CTA).
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, const Args& a) {
    return ((u + 1) * a.P + a.U - 1) / a.U - 1;  // largest c with c*U/P <= u
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w, const Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Smem* sm = reinterpret_cast<Smem*>(base + C::STAGES * C::STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        if (a.offsets != nullptr) {
            find_tile<C::BN>(a, sm, lane);
        } else if (lane == 0) {
            sm->expert = 0;
            sm->row0 = C::STREAMK ? 0 : (int)(blockIdx.x * C::BN);
            sm->row_end = (int)a.M;
            sm->valid = C::STREAMK ? (blockIdx.x < a.P) : 1;
        }
        if (lane == 0) {
            for (int i = 0; i < C::STAGES; ++i) {
                ptx::mbar_init(&sm->full[i], 1);
                ptx::mbar_init(&sm->empty[i], 1);
            }
            for (int i = 0; i < C::ASTAGES; ++i) {
                ptx::mbar_init(&sm->afull[i], C::DEQW * 32);
                ptx::mbar_init(&sm->aempty[i], 1);
            }
            for (int b = 0; b < C::ND; ++b) {
                ptx::mbar_init(&sm->dfull[b], 1);
                ptx::mbar_init(&sm->dempty[b], C::EPIW * 32);
            }
            ptx::mbar_init(&sm->mma_done, 1);
            ptx::mbar_init(&sm->pstored, C::EPIW * 32);
            ptx::mbar_init(&sm->pflag, 1);
            sm->abort = 0;
            ptx::fence_mbar_init();
            ptx::prefetch_tensormap(&tmap_x);
            ptx::prefetch_tensormap(&tmap_w);
        }
    }
    __syncthreads();
    if (!sm->valid) return;
    if (warp == 1) {
        ptx::tmem_alloc(&sm->tmem_base, C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    const int expert = sm->expert, row0 = sm->row0, row_end = sm->row_end;
    volatile int* abort = &sm->abort;
    Schedule<C> sched;
    sched.init(a);
    Seg seg;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int64_t c = 0;
            bool stop = false;
            while (!stop && sched.next(a, seg)) {
                for (int64_t kc = seg.k0; kc < seg.k1; kc += C::KSTAGE, ++c) {
                    const int st = (int)(c % C::STAGES);
                    const int64_t round = c / C::STAGES;
                    if (round > 0 && !ptx::mbar_wait(&sm->empty[st], (uint32_t)((round - 1) & 1), abort, kWaitLimitNs)) {
                        fail(a, sm, W4A16_ERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                    uint8_t* stage = base + st * C::STAGE_BYTES;
                    ptx::mbar_arrive_expect_tx(&sm->full[st], C::STAGE_BYTES);
                    const int n0 = (int)(seg.n_tile * kRowsPerTile);
                    if (a.offsets == nullptr)
                        ptx::tma_load_2d(stage, &tmap_w, &sm->full[st], (int)(kc / 2), n0);
                    else
                        ptx::tma_load_3d(stage, &tmap_w, &sm->full[st], (int)(kc / 2), n0, expert);
#pragma unroll
                    for (int b = 0; b < C::XBOXES; ++b)
                        ptx::tma_load_2d(stage + C::PBYTES + b * C::XBOX_BYTES, &tmap_x, &sm->full[st],
                                         (int)(kc + 64 * b), row0);
                }
            }
            if (*abort) {  // let our own loads land before the CTA exits
                volatile int never = 0;
                const int64_t first = c - C::STAGES < 0 ? 0 : c - C::STAGES;
                for (int64_t i = first; i < c; ++i)
                    ptx::mbar_wait(&sm->full[i % C::STAGES], (uint32_t)((i / C::STAGES) & 1), &never, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(kRowsPerTile, C::BN);
            int64_t c = 0, grp = 0;
            int cur_b = 0;
            bool ok = true;
            while (ok && sched.next(a, seg)) {
                for (int64_t kc = seg.k0; ok && kc < seg.k1; kc += C::KSTAGE, ++c) {
                    const int st = (int)(c % C::STAGES), as = (int)(c % C::ASTAGES);
                    // afull implies full: the dequant warps saw the stage's bytes land before arriving
                    if (!ptx::mbar_wait(&sm->afull[as], (uint32_t)((c / C::ASTAGES) & 1), abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // per stage: descriptors, the number of k16 steps and where groups start/end
                    const uint64_t bdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(base + st * C::STAGE_BYTES + C::PBYTES));
                    const uint32_t a_col = tmem + (uint32_t)(C::DCOLS + as * C::ACOLS);
                    const int nk = (int)((seg.k1 - kc < C::KSTAGE ? seg.k1 - kc : C::KSTAGE) >> 4);
                    constexpr int GPS = C::G / 16;  // MMAs per scale group
                    const bool stage_opens = C::KSTAGE >= C::G || (kc % C::G) == 0;
                    const bool stage_closes = C::KSTAGE >= C::G || ((kc + C::KSTAGE) % C::G) == 0;
#pragma unroll
                    for (int kk = 0; kk < C::KSTAGE / 16; ++kk) {
                        if (kk >= nk) break;
                        const bool first = C::KSTAGE >= C::G ? (kk % GPS == 0) : (kk == 0 && stage_opens);
                        const bool last = C::KSTAGE >= C::G ? (kk % GPS == GPS - 1)
                                                            : (kk == C::KSTAGE / 16 - 1 && stage_closes);
                        if (first) {
                            cur_b = (int)(grp % C::ND);
                            if (grp >= C::ND) {
                                if (!ptx::mbar_wait(&sm->dempty[cur_b], (uint32_t)((grp / C::ND - 1) & 1), abort,
                                                    kWaitLimitNs)) {
                                    ok = false;
                                    break;
                                }
                                ptx::tc_fence_after();
                            }
                        }
                        const uint64_t bdesc = bdesc0 + (uint64_t)((((kk >> 2) * C::XBOX_BYTES) + (kk & 3) * 32) >> 4);
                        ptx::mma_f16_ts(tmem + (uint32_t)(cur_b * C::BN), a_col + (uint32_t)(kk * 8), bdesc, idesc,
                                        first ? 0u : 1u);
                        if (last) {
                            ptx::mma_commit(&sm->dfull[cur_b]);
                            ++grp;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(&sm->empty[st]);
                    if (C::ASTAGES != C::STAGES) ptx::mma_commit(&sm->aempty[as]);
                }
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
        int64_t c = 0;
        bool ok = true;
        while (ok && sched.next(a, seg)) {
            for (int64_t kc = seg.k0; kc < seg.k1; kc += C::KSTAGE, ++c) {
                const int st = (int)(c % C::STAGES), as = (int)(c % C::ASTAGES);
                const int64_t around = c / C::ASTAGES;
                if (!ptx::mbar_wait(&sm->full[st], (uint32_t)((c / C::STAGES) & 1), abort, kWaitLimitNs) ||
                    (around > 0 &&
                     !ptx::mbar_wait(C::ASTAGES != C::STAGES ? &sm->aempty[as] : &sm->empty[st],
                                     (uint32_t)((around - 1) & 1), abort, kWaitLimitNs))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint8_t* prow = base + st * C::STAGE_BYTES;
                const uint32_t tcol = tmem + ((uint32_t)(quad * 32) << 16) +
                                      (uint32_t)(C::DCOLS + as * C::ACOLS + part * (C::PART_K / 2));
#pragma unroll
                for (int h = 0; h < CH; h += 2) {  // two chunks = 64 k = 32 columns per store
                    uint32_t v[32];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 p = *reinterpret_cast<const uint4*>(
                            prow + packed_offset<C::KSTAGE>(r, part * CH + h + q));
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
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&sm->afull[as]);
            }
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
        int npartial = 0;                          // partial segments so far (mbarrier parity)
        bool ok = true;
        while (ok && sched.next(a, seg)) {
            const int64_t n = seg.n_tile * kRowsPerTile + r;
            const bool n_ok = n < a.N;
            const uint16_t* srow = a.s + ((int64_t)expert * a.N + (n_ok ? n : 0)) * gk;
            float acc[C::BNP];
#pragma unroll
            for (int j = 0; j < C::BNP; ++j) acc[j] = 0.0f;
            const int g0 = (int)(seg.k0 / C::G), g1 = (int)(seg.k1 / C::G);
            // scales are streamed from HBM once: keep SB..2 SB groups of them in flight
            constexpr int SB = C::BNP > 32 ? 4 : 8;
            float scA[SB], scB[SB];
            auto load_scales = [&](float (&dst)[SB], int gb) {
#pragma unroll
                for (int i = 0; i < SB; ++i)
                    dst[i] = (n_ok && gb + i < g1) ? __half2float(__ushort_as_half(__ldg(srow + gb + i))) : 0.0f;
            };
            auto run_groups = [&](const float (&sc)[SB], int gb) {
#pragma unroll
                for (int i = 0; i < SB; ++i) {
                    if (gb + i >= g1 || !ok) break;
                    const int b = (int)(grp % C::ND);
                    if (!__all_sync(0xffffffffu,
                                    ptx::mbar_wait(&sm->dfull[b], (uint32_t)((grp / C::ND) & 1), abort, kWaitLimitNs))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t taddr =
                        tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * C::BN + cp * C::BNP);
                    const float sv = sc[i];
                    if constexpr (C::BNP == 16) {
                        uint32_t v[16];
                        ptx::tmem_ld_32x32b_x16(taddr, v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] = fmaf(sv, __uint_as_float(v[j]), acc[j]);
                    } else {
#pragma unroll
                        for (int ch = 0; ch < C::BNP / 32; ++ch) {
                            uint32_t v[32];
                            ptx::tmem_ld_32x32b_x32(taddr + ch * 32, v);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                acc[ch * 32 + j] = fmaf(sv, __uint_as_float(v[j]), acc[ch * 32 + j]);
                        }
                    }
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(&sm->dempty[b]);
                    ++grp;
                }
            };
            load_scales(scA, g0);
            load_scales(scB, g0 + SB);
            for (int gb = g0; ok && gb < g1; gb += 2 * SB) {
                run_groups(scA, gb);
                load_scales(scA, gb + 2 * SB);
                if (ok) run_groups(scB, gb + SB);
                load_scales(scB, gb + 3 * SB);
            }
            if (!ok) break;
            const int m0 = row0 + cp * C::BNP;  // first token of this thread's share
            if (seg.full) {
                if (n_ok) {
#pragma unroll
                    for (int j = 0; j < C::BNP; ++j)
                        if (m0 + j < row_end) a.y[(int64_t)(m0 + j) * a.N + n] = __half_as_ushort(__float2half_rn(acc[j]));
                }
            } else if constexpr (C::STREAMK) {
                // partial: slot of this CTA, fp32 [M][128]
                const int64_t slot_elems = (int64_t)a.M * kRowsPerTile;
                float* mine = a.partial + ((int64_t)blockIdx.x * 2 + seg.slot) * slot_elems;
#pragma unroll
                for (int j = 0; j < C::BNP; ++j)
                    if (m0 + j < a.M) __stcg(mine + (int64_t)(m0 + j) * kRowsPerTile + r, acc[j]);
                __threadfence();
                // handshake through mbarriers (bounded waits): all partials stored -> one
                // thread counts the arrival -> everyone learns whether this CTA is last
                ptx::mbar_arrive(&sm->pstored);
                const uint32_t ppar = (uint32_t)(npartial & 1);
                ++npartial;
                if (ew == 0 && lane == 0) {
                    if (!ptx::mbar_wait(&sm->pstored, ppar, abort, kWaitLimitNs)) {
                        fail(a, sm, W4A16_ERR_TIMEOUT);
                    } else {
                        const int old = atomicAdd(a.counter + seg.n_tile, 1);
                        const int64_t ca = cta_of_unit(seg.n_tile * a.KU, a);
                        const int64_t cb = cta_of_unit(seg.n_tile * a.KU + a.KU - 1, a);
                        sm->last_flag = (int64_t)old == cb - ca;
                    }
                    ptx::mbar_arrive(&sm->pflag);
                }
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm->pflag, ppar, abort, kWaitLimitNs)) || *abort) {
                    ok = false;
                    break;
                }
                if (sm->last_flag) {
                    __threadfence();
                    const int64_t ca = cta_of_unit(seg.n_tile * a.KU, a);
                    const int64_t cb = cta_of_unit(seg.n_tile * a.KU + a.KU - 1, a);
                    float sum[C::BNP];
#pragma unroll
                    for (int j = 0; j < C::BNP; ++j) sum[j] = 0.0f;
                    for (int64_t v = ca; v <= cb; ++v) {
                        // the tile is the first segment of every contributor except possibly ca
                        const bool ca_inside = (v * a.U / a.P) == seg.n_tile * a.KU;
                        const int slot = (v == ca && !ca_inside) ? 1 : 0;
                        const float* src = a.partial + (v * 2 + slot) * slot_elems;
#pragma unroll
                        for (int j = 0; j < C::BNP; ++j)
                            if (m0 + j < a.M) sum[j] += __ldcg(src + (int64_t)(m0 + j) * kRowsPerTile + r);
                    }
                    if (n_ok) {
#pragma unroll
                        for (int j = 0; j < C::BNP; ++j)
                            if (m0 + j < a.M) a.y[(int64_t)(m0 + j) * a.N + n] = __half_as_ushort(__float2half_rn(sum[j]));
                    }
                    if (ew == 0 && lane == 0) a.counter[seg.n_tile] = 0;
                }
            }
        }
        if (!ok) fail(a, sm, W4A16_ERR_TIMEOUT);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
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
                       CUtensorMap* mx, CUtensorMap* mw) {
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
        cuuint32_t box[2] = {(cuuint32_t)(C::KSTAGE / 2), (cuuint32_t)kRowsPerTile};
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

template <class C>
w4a16_status launch(const CUtensorMap& mx, const CUtensorMap& mw, const Args& a, dim3 grid, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (attr_err != cudaSuccess) return cuda_status(attr_err, "gemm: cudaFuncSetAttribute");
    tc_kernel<C><<<grid, C::THREADS, C::SMEM, st>>>(mx, mw, a);
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
    return launch<C>(mx, mw, a, dim3((unsigned)mt, (unsigned)nt), st);
}

}  // namespace

w4a16_status gemm_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                         int64_t M, int64_t N, int64_t K, int group, const int32_t* expert_offsets, int E,
                         cudaStream_t st) {
    if (M > 0x7fffffffLL || N > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    switch (group) {
        case 32: return gemm_g<PrefillCfg<32>>(dev, x, qw, s, y, M, N, K, expert_offsets, E, st);
        case 64: return gemm_g<PrefillCfg<64>>(dev, x, qw, s, y, M, N, K, expert_offsets, E, st);
        case 128: return gemm_g<PrefillCfg<128>>(dev, x, qw, s, y, M, N, K, expert_offsets, E, st);
        default: return W4A16_ERR_UNSUPPORTED;
    }
}

}  // namespace w4a16
