// Decode GEMV for the W4A16 layer, M <= 16 activation rows (LLM170 page:
// "CUDA-graph decode", np4 = four sequences per step).
//
// Decode streams every packed weight byte once and does little arithmetic per
// byte: the kernel is bound by HBM bandwidth, by the issue rate of its
// dequantization and legacy tensor-core MMAs, and by the latency of the
// kernel before it. Design (one block per SM: kConsumers compute warps and
// one producer warp):
//
// * Work unit = 16 weight rows x 512 input features (4 KB packed). Units are
//   ordered row-block major, k minor; every compute warp of a persistent grid
//   owns an equal contiguous range of them (stream-K split), so each SM
//   streams the same number of bytes whatever N and K are.
// * Each compute warp has a private ring of kSlots shared-memory slots. Lane c
//   of the producer warp keeps compute warp c's ring full: one TMA copy per
//   unit (a 3-D box that lands as [k-step][row][64 B], so the fragment reads
//   are free of bank conflicts; four 2-D boxes when K % 128 != 0) plus the
//   unit's box of scales, refilled as soon as the warp releases the slot on
//   its "empty" barrier. Compute warps neither issue copies nor compute
//   addresses for them, and no warp waits behind another.
// * The activations (M x K fp16, when small enough) are staged once per block
//   in shared memory, permuted into MMA fragment order; larger x is read
//   through the L1.
// * Nibbles become exact fp16 integers in registers (lop3 + one half2 op per
//   pair) and go straight into mma.sync m16n8k16 as the A operand (rows =
//   weight rows, columns = tokens padded to 8): the tensor core does the x*q
//   products (exact) and their fp32 sum within one scale group. The k order
//   inside a group is permuted identically on the activation side, which
//   leaves every group sum unchanged.
// * After each group the fp32 partial is multiplied by the group's scale and
//   added into fp32 accumulators: acc += s[n, grp] * sum_{k in grp} x q.
// * A row-block whose units span several warps is finished by the last warp
//   to arrive: each contributor stores its fp32 partial in the workspace,
//   bumps a per-row-block counter, and the last one sums all partials in
//   warp order (deterministic), rounds once to fp16 and resets the counter.
//   A warp publishes each partial as soon as its segment ends, with one
//   acquire-release atomic on the counter.
// * Programmatic dependent launch: each compute warp lets the next kernel on
//   the stream launch when it reaches its last unit, so that kernel's blocks
//   take each SM the moment this one's block leaves it. A block may start
//   while the kernel before it is still finishing. By default it reads
//   nothing (weights included, which that kernel may have written) before
//   griddepcontrol.wait returns. With static weights (the caller's promise
//   that no pending work writes them) the producer fills every ring with
//   weights and scales first and only x waits for the previous kernel. That
//   pays when the kernel before leaves SMs idle for a while; behind another
//   GEMV it measured 1.5 % slower, its copies competing with that GEMV's last
//   units.
//
// Every wait is bounded in time; one that gives up records W4A16_ERR_TIMEOUT in
// the device error word, and the block leaves only after the copies it issued
// have landed.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kConsumers = 8;    // compute warps per block (one block per SM; 2 per scheduler)
constexpr int kProducer = kConsumers;  // warp index of the block's TMA producer
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kConsumerThreads = kConsumers * 32;
constexpr int kSlots = 4;        // ring slots per compute warp (8 x 4 measured best of 4..16 x 2..8)
constexpr int kStepK = 128;      // k per step (one 64-byte piece of a row)
constexpr int kUnitSteps = 4;    // steps per unit
constexpr int kUnitK = kStepK * kUnitSteps;
constexpr int kRows = 16;        // weight rows per unit
constexpr int kWBytes = kUnitSteps * kRows * 64;  // packed weights of a unit: 4 KB
// Scales travel with the weights (TS) as one TMA box of 16 rows x kScaleBox<G>
// groups: the unit's groups, or 8 (16 bytes, the smallest box that starts on
// a 16-byte boundary) when a unit has fewer; then the box also holds the
// groups of neighbouring units.
template <int G>
constexpr int kScaleBox = kUnitK / G > 8 ? kUnitK / G : 8;
template <int G, bool TS>
constexpr int kSlotBytes = kWBytes + (TS ? kRows * kScaleBox<G> * 2 : 0);
constexpr int kMaxM = 16;        // activation rows handled by the GEMV
constexpr size_t kXSmemMax = 84 * 1024;  // x staged in shared memory up to this size (M = 8 at K = 5120)
constexpr int kXLoads = (int)((kXSmemMax / 16 + kConsumerThreads - 1) / kConsumerThreads);  // x loads per thread
constexpr uint64_t kWaitLimitNs = 2000000000ull;

#ifdef W4A16_TEST_HOOKS
__device__ TestHooks g_hooks = {kWaitLimitNs, -1};
__device__ __forceinline__ uint64_t wait_limit() { return g_hooks.wait_limit_ns; }
__device__ __forceinline__ bool may_issue(int issued) { return g_hooks.issue_limit < 0 || issued < g_hooks.issue_limit; }
#else
__device__ __forceinline__ constexpr uint64_t wait_limit() { return kWaitLimitNs; }
__device__ __forceinline__ constexpr bool may_issue(int) { return true; }
#endif

// GemvArgs::mode bits
constexpr int kMode3d = 1;      // the weight map is 3-D: one TMA box per unit
constexpr int kModeStatic = 2;  // weights and scales may be read before the dependency wait

struct GemvArgs {
    const uint16_t* x;
    const uint16_t* s;
    uint16_t* y;
    int M;
    int N, K;
    int64_t KU;  // 512-k units per row: ceil(K / 512)
    int64_t U;   // units: ceil(N / 16) * KU
    int64_t P;   // consumer warps taking part (each owns >= 1 unit)
    float* partial;  // [P][2][16 * M] fp32 partial sums (first / last segment)
    int* counter;    // [ceil(N/16)] arrivals per row-block, zero between calls
    unsigned int* err;
    int gpr;         // scale groups per row: K / G
    int svec;        // scale rows start 16-byte aligned (gpr % 8 == 0): whole units load as vectors
    int mode;        // kMode3d | kModeStatic
};

// Gated pair (gate and up projections of one MLP, fused; a parameter of the
// gated kernel only, which keeps the plain kernel's parameters as small as
// they measure fastest): row-block rb of the output is virtual row-blocks 2 rb
// (gate) and 2 rb + 1 (up); the second of the two to finish writes
// y = silu(gate) * up.
struct GatedArgs {
    const uint16_t* s2;  // scales of the up projection
    float* gres;         // [2][M][N] fp32 gate and up results
    int* pair;           // [ceil(N/16)] finished halves per row-block, zero between calls
};

struct Bars {
    uint64_t full[kConsumers][kSlots];   // a unit's bytes have landed in the slot
    uint64_t empty[kConsumers][kSlots];  // the compute warp has finished with the slot
    int abort;
    alignas(16) uint8_t zero[1024];  // x of one unit for lanes without a token
};

// Every input may have been written by the kernel just before this one on
// the stream (its completion is awaited with griddepcontrol.wait), so none is
// read through the non-coherent path. One-shot reads bypass L1 (.cg); x read
// repeatedly from global memory uses the L1 (.ca).
__device__ __forceinline__ uint4 ld_l2_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_l1_v4(const void* p) {
    uint4 v;
    asm("ld.global.ca.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_l2_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
// Shared-memory loads by shared address; volatile keeps them after the barrier
// wait that guards them (measured 0.15 us per GEMV faster than plain loads).
__device__ __forceinline__ uint4 lds_v4(const uint8_t* a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(ptx::smem_u32(a)));
    return v;
}
__device__ __forceinline__ uint2 lds_v2(const uint8_t* a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(ptx::smem_u32(a)));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(const uint8_t* a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(ptx::smem_u32(a)));
    return v;
}
__device__ __forceinline__ uint32_t ld_l2_u16(const uint16_t* p) {
    unsigned short v;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// (x0..x7) -> (x0,x4), (x1,x5), (x2,x6), (x3,x7): the pair order the nibble
// conversion produces for the weights.
__device__ __forceinline__ uint4 permute_x8(uint4 v) {
    return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                      __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

// Shared-memory activations: per token a row of 4 KU steps x 16 chunks of 16
// bytes (+64 B pad), each chunk pre-permuted by permute_x8 and placed so that
// the four threads of a quad read consecutive chunks.
__device__ __forceinline__ int xs_pos(int c_local, int G) {
    const int cpp = G / 8;  // chunks per group
    const int j = c_local / cpp, rem = c_local % cpp;
    const int t4 = rem / (G / 32), wi = rem % (G / 32);
    return (j * (G / 32) + wi) * 4 + t4;
}

// Scales of one unit for rows gid and gid+8 as raw fp16: word j of a row holds
// the unit's groups 2j (low half) and 2j+1 (high half). They are converted
// only when used, so the loads stay in flight during the previous unit.
template <int G>
struct UnitScales {
    static constexpr int W = kUnitK / G / 2;
    uint32_t lo[W], hi[W];
};

// The scale rows of this lane (rows gid and gid+8 of a row-block); a row past
// N reads row 0 and is zeroed.
struct ScaleRows {
    const uint16_t* r0;
    const uint16_t* r1;
    bool v0, v1;
};

template <bool GT>
__device__ __forceinline__ ScaleRows scale_rows(const GemvArgs& p, const GatedArgs& ga, int vrb, int gid) {
    const int64_t n0 = (int64_t)(GT ? vrb >> 1 : vrb) * kRows + gid, n1 = n0 + 8;
    const uint16_t* s = (GT && (vrb & 1)) ? ga.s2 : p.s;
    ScaleRows r;
    r.v0 = n0 < p.N;
    r.v1 = n1 < p.N;
    r.r0 = s + (r.v0 ? n0 : 0) * p.gpr;
    r.r1 = s + (r.v1 ? n1 : 0) * p.gpr;
    return r;
}

template <int G, class Args>
__device__ __forceinline__ void load_scales(UnitScales<G>& sc, const Args& p, const ScaleRows& sr, int ku) {
    constexpr int GPU = kUnitK / G;  // groups per unit: 4, 8 or 16
    const int g0 = ku * GPU;
    if (p.svec && g0 + GPU <= p.gpr) {  // whole unit from aligned rows: vector loads
        if constexpr (GPU == 4) {
            const uint2 a = sr.v0 ? ld_l2_v2(sr.r0 + g0) : make_uint2(0, 0);
            const uint2 b = sr.v1 ? ld_l2_v2(sr.r1 + g0) : make_uint2(0, 0);
            sc.lo[0] = a.x; sc.lo[1] = a.y;
            sc.hi[0] = b.x; sc.hi[1] = b.y;
        } else {
#pragma unroll
            for (int q = 0; q < GPU / 8; ++q) {
                const uint4 a = sr.v0 ? ld_l2_v4(sr.r0 + g0 + 8 * q) : make_uint4(0, 0, 0, 0);
                const uint4 b = sr.v1 ? ld_l2_v4(sr.r1 + g0 + 8 * q) : make_uint4(0, 0, 0, 0);
                sc.lo[4 * q] = a.x; sc.lo[4 * q + 1] = a.y; sc.lo[4 * q + 2] = a.z; sc.lo[4 * q + 3] = a.w;
                sc.hi[4 * q] = b.x; sc.hi[4 * q + 1] = b.y; sc.hi[4 * q + 2] = b.z; sc.hi[4 * q + 3] = b.w;
            }
        }
    } else {  // ragged or unaligned: one scale at a time, groups past K read as 0
#pragma unroll
        for (int w = 0; w < GPU / 2; ++w) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int g = g0 + 2 * w + h;
                const bool vg = g < p.gpr;
                lo |= ((sr.v0 && vg) ? ld_l2_u16(sr.r0 + g) : 0u) << (16 * h);
                hi |= ((sr.v1 && vg) ? ld_l2_u16(sr.r1 + g) : 0u) << (16 * h);
            }
            sc.lo[w] = lo;
            sc.hi[w] = hi;
        }
    }
}

// Scales from the unit's TMA box in its slot (rows and groups outside the
// tensor were filled with zeros by the copy).
template <int G>
__device__ __forceinline__ void load_scales_smem(UnitScales<G>& sc, const uint8_t* box, int ku, int gid) {
    constexpr int GPU = kUnitK / G;
    const uint8_t* r0 = box + gid * (kScaleBox<G> * 2) + ((ku * GPU) % kScaleBox<G>) * 2;
    const uint8_t* r1 = r0 + 8 * (kScaleBox<G> * 2);
    if constexpr (GPU == 4) {
        const uint2 a = lds_v2(r0), b = lds_v2(r1);
        sc.lo[0] = a.x; sc.lo[1] = a.y;
        sc.hi[0] = b.x; sc.hi[1] = b.y;
    } else {
#pragma unroll
        for (int q = 0; q < GPU / 8; ++q) {
            const uint4 a = lds_v4(r0 + 16 * q), b = lds_v4(r1 + 16 * q);
            sc.lo[4 * q] = a.x; sc.lo[4 * q + 1] = a.y; sc.lo[4 * q + 2] = a.z; sc.lo[4 * q + 3] = a.w;
            sc.hi[4 * q] = b.x; sc.hi[4 * q + 1] = b.y; sc.hi[4 * q + 2] = b.z; sc.hi[4 * q + 3] = b.w;
        }
    }
}

__device__ __forceinline__ float half_bits(uint32_t w, int h) {
    return __half2float(__ushort_as_half((unsigned short)(h ? (w >> 16) : (w & 0xffffu))));
}

// One unit from its ring slot: for every 128-k step and scale group, the
// quad's share of rows gid and gid+8. `wlane` points at this lane's first
// weight bytes in the slot (row gid, its quad's offset). XS: x comes from
// shared memory at xlane[t] (this lane's 16-byte chunk of the unit's x for
// token 8t+gid, or of the zero block for lanes without a token), so no load
// is predicated and every offset below is a constant.
template <int G, int NT, bool XS>
__device__ __forceinline__ void compute_unit(const uint8_t* wlane, const UnitScales<G>& sc, const GemvArgs& p,
                                             const uint8_t* const (&xlane)[NT], int ku, int gid, int t4,
                                             float (&acc)[NT][4]) {
    constexpr int WPP = G / 32;      // words per thread per row per group
    constexpr int GPS = kStepK / G;  // groups per step
#pragma unroll
    for (int step = 0; step < kUnitSteps; ++step) {
#pragma unroll
        for (int j = 0; j < GPS; ++j) {
            uint32_t wa[WPP], wb[WPP];
            const uint8_t* ra = wlane + step * (kRows * 64) + j * (G / 2);
            const uint8_t* rbp = ra + 8 * 64;
            if constexpr (WPP == 4) {
                const uint4 a = lds_v4(ra), b = lds_v4(rbp);
                wa[0] = a.x; wa[1] = a.y; wa[2] = a.z; wa[3] = a.w;
                wb[0] = b.x; wb[1] = b.y; wb[2] = b.z; wb[3] = b.w;
            } else if constexpr (WPP == 2) {
                const uint2 a = lds_v2(ra), b = lds_v2(rbp);
                wa[0] = a.x; wa[1] = a.y;
                wb[0] = b.x; wb[1] = b.y;
            } else {
                wa[0] = lds_u32(ra);
                wb[0] = lds_u32(rbp);
            }
            uint4 xv[WPP][NT];
#pragma unroll
            for (int wi = 0; wi < WPP; ++wi)
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (XS) {
                        xv[wi][t] = lds_v4(xlane[t] + step * (kStepK * 2) + (j * WPP + wi) * 64);
                    } else {
                        const int m = 8 * t + gid;
                        const int64_t k0 = ((int64_t)ku * kUnitSteps + step) * kStepK + j * G + t4 * (G / 4) + 8 * wi;
                        xv[wi][t] = make_uint4(0, 0, 0, 0);
                        if (m < p.M && k0 < p.K) xv[wi][t] = permute_x8(ld_l1_v4(p.x + (int64_t)m * p.K + k0));
                    }
                }
            float c[NT][4];  // this group's fp32 sum of x*q
#pragma unroll
            for (int wi = 0; wi < WPP; ++wi) {
                uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
                nibbles_to_half2(wa[wi], a04, a15, a26, a37);
                nibbles_to_half2(wb[wi], b04, b15, b26, b37);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (wi == 0) mma_16816_zero(c[t], a04, b04, a15, b15, xv[wi][t].x, xv[wi][t].y);
                    else mma_16816(c[t], a04, b04, a15, b15, xv[wi][t].x, xv[wi][t].y);
                    mma_16816(c[t], a26, b26, a37, b37, xv[wi][t].z, xv[wi][t].w);
                }
            }
            const int gi = step * GPS + j;
            const float s0 = half_bits(sc.lo[gi >> 1], gi & 1), s1 = half_bits(sc.hi[gi >> 1], gi & 1);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                acc[t][0] = fmaf(s0, c[t][0], acc[t][0]);
                acc[t][1] = fmaf(s0, c[t][1], acc[t][1]);
                acc[t][2] = fmaf(s1, c[t][2], acc[t][2]);
                acc[t][3] = fmaf(s1, c[t][3], acc[t][3]);
            }
        }
    }
}

// Accumulator element i of tile t: row gid + 8 (i >> 1), token 8 t + 2 t4 + (i & 1).
template <int NT>
__device__ __forceinline__ void store_y(const GemvArgs& p, int64_t rb, const float (&v)[NT][4], int gid, int t4) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * t4 + (i & 1);
            const int64_t n = rb * kRows + gid + 8 * (i >> 1);
            if (m < p.M && n < p.N) p.y[(int64_t)m * p.N + n] = __half_as_ushort(__float2half_rn(v[t][i]));
        }
}

// The finished fp32 sums of virtual row-block vrb. Plain: round once to fp16
// and store y. Gated: park them in the workspace; the second half of the pair
// to finish computes y = silu(gate) * up in fp32 and rounds once to fp16
// (rust-inference README, list of accuracy fixes, item 5: the SiLU-activated
// gate multiplies the up projection).
template <int NT, bool GT>
__device__ __forceinline__ void finish_row_block(const GemvArgs& p, const GatedArgs& ga, int vrb,
                                                 const float (&v)[NT][4], int gid, int t4, int lane) {
    if constexpr (!GT) {
        store_y<NT>(p, vrb, v, gid, t4);
        return;
    }
    const int rb = vrb >> 1, mat = vrb & 1;
    const int64_t half = (int64_t)p.M * p.N;
    float* mine = ga.gres + mat * half;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * t4 + (i & 1);
            const int64_t n = (int64_t)rb * kRows + gid + 8 * (i >> 1);
            if (m < p.M && n < p.N) __stcg(mine + (int64_t)m * p.N + n, v[t][i]);
        }
    __syncwarp();  // the lanes' stores happen before lane 0's release
    int old = 0;
    if (lane == 0) old = ptx::atom_add_acq_rel_gpu(ga.pair + rb, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == 0) return;  // the other half finishes the pair
    __syncwarp();  // every lane's loads below come after lane 0's acquire
    float* other = ga.gres + (mat ^ 1) * half;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * t4 + (i & 1);
            const int64_t n = (int64_t)rb * kRows + gid + 8 * (i >> 1);
            if (m < p.M && n < p.N) {
                const float o = __ldcg(other + (int64_t)m * p.N + n);
                const float g = mat == 0 ? v[t][i] : o, u = mat == 0 ? o : v[t][i];
                const float silu = g / (1.0f + expf(-g));
                p.y[(int64_t)m * p.N + n] = __half_as_ushort(__float2half_rn(silu * u));
                // both halves are consumed: return the parking area to zero, so the
                // workspace is all zero between calls (a plain GEMV may reuse it)
                __stcg(mine + (int64_t)m * p.N + n, 0.0f);
                __stcg(other + (int64_t)m * p.N + n, 0.0f);
            }
        }
    if (lane == 0) ga.pair[rb] = 0;
}

__device__ __forceinline__ int unit_begin(int w, const GemvArgs& p) { return (int)((int64_t)w * p.U / p.P); }

__device__ __forceinline__ int64_t warp_of_unit(int64_t u, const GemvArgs& p) {
    return ((u + 1) * p.P + p.U - 1) / p.U - 1;  // largest w with w*U/P <= u
}

template <int NT>
__device__ __forceinline__ void store_partial(const GemvArgs& p, int64_t w, int slot, const float (&acc)[NT][4],
                                              int gid, int t4) {
    float* mine = p.partial + (w * 2 + slot) * ((int64_t)kRows * p.M);
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * t4 + (i & 1);
            if (m < p.M) __stcg(mine + m * kRows + gid + 8 * (i >> 1), acc[t][i]);
        }
}

// Publishes this warp's fp32 partial of row-block rb (slot 0: the warp's first
// segment, 1: its last) and counts the arrival with one acquire-release
// atomic; the last contributor sums every contributor's partial in warp order,
// rounds once to fp16, stores y and resets the counter.
template <int NT, bool GT>
__device__ __noinline__ void publish_partial(const GemvArgs& p, const GatedArgs& ga, int64_t w, int slot, int64_t rb,
                                             const float (&acc)[NT][4], int gid, int t4, int lane) {
    store_partial<NT>(p, w, slot, acc, gid, t4);
    __syncwarp();  // the lanes' stores happen before lane 0's release
    int old = 0;
    if (lane == 0) old = ptx::atom_add_acq_rel_gpu(p.counter + rb, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int64_t wa = warp_of_unit(rb * p.KU, p);
    const int64_t wb = warp_of_unit(rb * p.KU + p.KU - 1, p);
    if ((int64_t)old != wb - wa) return;  // another warp finishes this row-block
    __syncwarp();  // every lane's loads of the other partials come after lane 0's acquire
    const int64_t slot_elems = (int64_t)kRows * p.M;
    // rb is the first segment of every contributor except possibly wa
    const bool wa_started_inside = (wa * p.U / p.P) == rb * p.KU;
    float sum[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) sum[t][0] = sum[t][1] = sum[t][2] = sum[t][3] = 0.0f;
    // kBatch contributors' partials are loaded at once, then added in warp
    // order: one L2 round trip per batch instead of one per contributor
    constexpr int kBatch = NT == 1 ? 8 : 4;
    for (int64_t v0 = wa; v0 <= wb; v0 += kBatch) {
        float part[kBatch][NT][4];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int64_t v = v0 + b;
            const int sl = (v == wa && !wa_started_inside) ? 1 : 0;
            const float* src = p.partial + (v * 2 + sl) * slot_elems;
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = 8 * t + 2 * t4 + (i & 1);
                    part[b][t][i] = (v <= wb && m < p.M) ? __ldcg(src + m * kRows + gid + 8 * (i >> 1)) : 0.0f;
                }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (v0 + b <= wb) sum[t][i] += part[b][t][i];
    }
    if (lane == 0) p.counter[rb] = 0;
    finish_row_block<NT, GT>(p, ga, (int)rb, sum, gid, t4, lane);
}

// The tensor maps of one launch (kernel parameters): weights and scales, and
// for a gated pair the up projection's as well.
struct MapPtrs {
    const CUtensorMap* w;
    const CUtensorMap* s;
    const CUtensorMap* w2;
    const CUtensorMap* s2;
};

// The producer warp: lane c streams compute warp c's units into that warp's
// ring, refilling a slot as soon as the warp releases it. The lanes issue
// their copies side by side, so no compute warp waits behind another.
template <int G, bool TS, bool GT>
__device__ __forceinline__ void produce(const MapPtrs& maps, const GemvArgs& p,
                                        Bars* bars, uint8_t* ring, volatile int* abort, int lane) {
    constexpr int SLOT = kSlotBytes<G, TS>;
    const int KU = (int)p.KU;
    const int c = lane < kConsumers ? lane : 0;
    const int w = blockIdx.x * kConsumers + c;
    const int ub = (lane < kConsumers && w < p.P) ? unit_begin(w, p) : 0;
    const int n = (lane < kConsumers && w < p.P) ? unit_begin(w + 1, p) - ub : 0;
    int ri = 0;  // units issued into the ring
    // first group of the box holding unit ku's groups (a multiple of 8: 16-byte aligned)
    auto scale_x = [](int ku) { return (ku * (kUnitK / G)) / kScaleBox<G> * kScaleBox<G>; };
    auto issue = [&](int sl, int u) {
        const int vrb = u / KU, ku = u % KU;
        int rb = vrb;
        const CUtensorMap* mw = maps.w;
        const CUtensorMap* ms = maps.s;
        if constexpr (GT) {
            rb = vrb >> 1;
            if (vrb & 1) {
                mw = maps.w2;
                ms = maps.s2;
            }
        }
        uint64_t* bar = &bars->full[c][sl];
        uint8_t* dst = ring + (c * kSlots + sl) * SLOT;
        ptx::mbar_arrive_expect_tx(bar, SLOT);
        if (p.mode & kMode3d) {
            ptx::tma_load_3d(dst, mw, bar, 0, rb * kRows, ku * kUnitSteps);
        } else {
#pragma unroll
            for (int step = 0; step < kUnitSteps; ++step)
                ptx::tma_load_2d(dst + step * (kRows * 64), mw, bar, (ku * kUnitSteps + step) * 64, rb * kRows);
        }
        if (TS) ptx::tma_load_2d(dst + kWBytes, ms, bar, scale_x(ku), rb * kRows);
    };

    // By default every input, the weights included, may come from the kernel
    // before this one on the stream, which may still be running: nothing is
    // read before griddepcontrol.wait returns. (Prefetching the first units
    // into L2 before the wait is safe, but measured slower: the extra traffic
    // delays the previous kernel's completion and this kernel's x loads.) With
    // static weights the producer reads only what no pending kernel writes, so
    // it fills the rings at once and never waits.
    if (!(p.mode & kModeStatic)) ptx::grid_dependency_wait();
    for (; ri < kSlots && ri < n && may_issue(ri); ++ri) issue(ri, ub + ri);
    uint64_t idle_since = 0;
    bool failed = false;
    while (__any_sync(0xffffffffu, ri < n && !failed)) {
        bool moved = false;
        if (ri < n && !failed && may_issue(ri)) {
            const int sl = ri % kSlots;
            // the slot's previous unit (ri - kSlots) completed phase ri / kSlots - 1
            if (ptx::mbar_try_wait(&bars->empty[c][sl], (uint32_t)((ri / kSlots + 1) & 1))) {
                issue(sl, ub + ri);
                ++ri;
                moved = true;
            }
        }
        if (__any_sync(0xffffffffu, moved)) {
            idle_since = 0;
            continue;
        }
        const uint64_t now = ptx::globaltimer_ns();
        if (idle_since == 0) idle_since = now;
        if (*abort || now - idle_since > wait_limit()) {
            if (lane == 0 && !*abort) {
                raise_device_error(p.err, W4A16_ERR_TIMEOUT);
                *abort = 1;
            }
            failed = true;
        }
    }
    // leave only when every load issued has landed (the block's shared memory
    // must not be released under an outstanding copy)
    volatile int never = 0;
    for (int q = ri > kSlots ? ri - kSlots : 0; q < ri; ++q)
        ptx::mbar_wait(&bars->full[c][q % kSlots], (uint32_t)((q / kSlots) & 1), &never, kWaitLimitNs);
}

template <int G, int NT, bool XS, bool TS, bool GT>
__device__ __forceinline__ void gemv_body(const MapPtrs& maps, const GemvArgs& p, const GatedArgs& ga) {
    constexpr int SLOT = kSlotBytes<G, TS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned start, by pointer arithmetic so the pointers stay shared-space
    uint8_t* ring = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    Bars* bars = reinterpret_cast<Bars*>(ring + kConsumers * kSlots * SLOT);
    uint8_t* xs = reinterpret_cast<uint8_t*>(bars) + ((sizeof(Bars) + 127) & ~(size_t)127);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int xsteps = (int)p.KU * kUnitSteps;     // staged steps per token (whole units)
    const int xstride = xsteps * (kStepK * 2) + 64;  // bytes per token row of staged x
    volatile int* abort = &bars->abort;

    if (threadIdx.x == 0) {
        for (int w = 0; w < kConsumers; ++w)
            for (int sl = 0; sl < kSlots; ++sl) {
                ptx::mbar_init(&bars->full[w][sl], 1);
                ptx::mbar_init(&bars->empty[w][sl], 1);
            }
        bars->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(maps.w);
        if (TS) ptx::prefetch_tensormap(maps.s);
        if constexpr (GT) {
            ptx::prefetch_tensormap(maps.w2);
            if (TS) ptx::prefetch_tensormap(maps.s2);
        }
    }
    if (threadIdx.x < 64) reinterpret_cast<uint4*>(bars->zero)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    if (warp == kProducer) {
        produce<G, TS, GT>(maps, p, bars, ring, abort, lane);
        return;
    }

    // ------------------------------------------------------------ compute warps
    const int cw = warp;
    const int w = blockIdx.x * kConsumers + cw;
    const int u_begin = w < p.P ? unit_begin(w, p) : 0;
    const int n_units = w < p.P ? unit_begin(w + 1, p) - u_begin : 0;
    int rb = u_begin / (int)p.KU, ku = u_begin % (int)p.KU;
    ptx::grid_dependency_wait();
    // the first unit's scales (global path) and x go out at once
    ScaleRows sr = scale_rows<GT>(p, ga, rb, gid);
    UnitScales<G> sc;
    if (!TS && n_units > 0) load_scales<G>(sc, p, sr, ku);
    if (XS) {
        // chunk c = threadIdx.x + i * kConsumerThreads is token m, chunk cc of its
        // row (16 bytes, zero past K); (m, cc) advance without division
        const int per_tok = xsteps * 16;
        uint4 xv[kXLoads];
        int m = 0, cc = threadIdx.x;
        while (cc >= per_tok) cc -= per_tok, ++m;
#pragma unroll
        for (int i = 0; i < kXLoads; ++i) {
            xv[i] = make_uint4(0, 0, 0, 0);
            if (m < p.M && cc * 8 < p.K) xv[i] = ld_l2_v4(p.x + (int64_t)m * p.K + cc * 8);
            cc += kConsumerThreads;
            while (cc >= per_tok) cc -= per_tok, ++m;
        }
        m = 0;
        cc = threadIdx.x;
        while (cc >= per_tok) cc -= per_tok, ++m;
#pragma unroll
        for (int i = 0; i < kXLoads; ++i) {
            if (m < p.M)
                *reinterpret_cast<uint4*>(xs + m * xstride + (cc >> 4) * (kStepK * 2) + xs_pos(cc & 15, G) * 16) =
                    permute_x8(xv[i]);
            cc += kConsumerThreads;
            while (cc >= per_tok) cc -= per_tok, ++m;
        }
        ptx::named_bar_sync(1, kConsumerThreads);  // compute warps only; the producer runs on
    }
    if (n_units == 0) return;

    const int first_rb = rb, KU = (int)p.KU;
    int seg_ku0 = ku;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    // shared address of this lane's x chunk in unit 0 (the zero block for lanes
    // without a token) and its stride per unit
    const uint8_t* xlane0[NT];
    int xunit[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const bool has = 8 * t + gid < p.M;
        xlane0[t] = (has ? xs + (8 * t + gid) * xstride : bars->zero) + t4 * 16;
        xunit[t] = has ? kUnitSteps * kStepK * 2 : 0;
    }
    const uint8_t* slot0 = ring + cw * (kSlots * SLOT);
    const int wlane = gid * 64 + t4 * (G / 8);

    int sl = 0;
    uint32_t phase = 0;
    for (int r = 0; r < n_units; ++r) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars->full[cw][sl], phase, abort, wait_limit()))) {
            if (!*abort) raise_device_error(p.err, W4A16_ERR_TIMEOUT);
            *abort = 1;  // the producer stops and waits for the loads it issued
            return;
        }
        int nrb = rb, nku = ku + 1;
        if (nku == KU) {
            nku = 0;
            ++nrb;
        }
        const uint8_t* slot = slot0 + sl * SLOT;
        UnitScales<G> sc_next;
        ScaleRows nsr = sr;
        if (TS) {
            load_scales_smem<G>(sc, slot + kWBytes, ku, gid);
        } else {
            if (nku == 0) nsr = scale_rows<GT>(p, ga, nrb, gid);
            if (r + 1 < n_units) load_scales<G>(sc_next, p, nsr, nku);
        }
        const uint8_t* xlane[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) xlane[t] = xlane0[t] + ku * xunit[t];
        compute_unit<G, NT, XS>(slot + wlane, sc, p, xlane, ku, gid, t4, acc);
        // only this warp's epilogue remains: the next kernel on the stream may
        // launch (its blocks take each SM as this kernel's block there leaves).
        // Measured against a trigger right after set-up: 15.6 against 16.0 us
        // per GEMV in the back-to-back decode step.
        if (r == n_units - 1) ptx::launch_dependents();
        __syncwarp();  // every lane has read the slot
        if (lane == 0) ptx::mbar_arrive(&bars->empty[cw][sl]);
        if (!TS) {
            if (r + 1 < n_units) sc = sc_next;
            sr = nsr;
        }

        const bool seg_end = (ku == KU - 1) || (r == n_units - 1);
        if (seg_end) {
            if (seg_ku0 == 0 && ku == KU - 1)
                finish_row_block<NT, GT>(p, ga, rb, acc, gid, t4, lane);  // whole row-block in this warp
            else  // partial: published now, so its latency overlaps the units that follow
                publish_partial<NT, GT>(p, ga, w, rb == first_rb ? 0 : 1, rb, acc, gid, t4, lane);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
        }
        rb = nrb;
        ku = nku;
        if (seg_end) seg_ku0 = ku;
        if (++sl == kSlots) {
            sl = 0;
            phase ^= 1u;
        }
    }
}

template <int G, int NT, bool XS, bool TS>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
                const GemvArgs p) {
    const MapPtrs maps{&tmap_w, &tmap_s, &tmap_w, &tmap_s};
    const GatedArgs none{nullptr, nullptr, nullptr};
    gemv_body<G, NT, XS, TS, false>(maps, p, none);
}

template <int G, int NT, bool XS, bool TS>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_gated_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
                      const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_s2,
                      const GemvArgs p, const GatedArgs ga) {
    const MapPtrs maps{&tmap_w, &tmap_s, &tmap_w2, &tmap_s2};
    gemv_body<G, NT, XS, TS, true>(maps, p, ga);
}

// ============================================================================
// Cluster kernel: group 128, M <= 8, one weight matrix.
//
// * A cluster of C blocks (one per SM, kCWarps compute warps each) owns an
//   equal share of whole row-blocks, and its C x kCWarps warps split the
//   cluster's units into equal contiguous ranges (stream-K inside the
//   cluster). Every split row-block is therefore summed inside one cluster.
// * Each lane loads its own 16-byte pieces of a unit (rows gid and gid + 8,
//   the k its mma fragments take) straight into registers, one unit ahead of
//   the unit it computes: no copy engine, no ring, no wait per unit. (Against
//   the TMA ring above, with the same arithmetic: 14.9 against 15.7 us per
//   GEMV in the back-to-back decode step.)
// * x: for M <= 2 each warp stages the x of its next unit in a two-slot ring
//   of its own, so no block-wide barrier delays the first unit; larger M is
//   staged once per block, as above.
// * A split row-block: each contributor leaves its fp32 partial in its own
//   block's shared memory and counts its arrival with one cluster-scope
//   acquire-release atomic on a counter in the first contributor's block; the
//   last to arrive sums every contributor's partial in warp order through
//   distributed shared memory (deterministic), rounds once to fp16 and stores
//   y. No partial crosses L2: summing split row-blocks through L2 (a partial
//   store, a release fence and an atomic per contributor, then the last
//   arriver's loads) cost about 4 us of each 15 us launch, almost all of it at
//   the end of the launch, where every warp finishes its last row-block.
// * Blocks meet on the cluster barrier at the start (the counters are zeroed
//   before any remote atomic) and before they leave (no block's partials
//   vanish while another may read them). Neither barrier waits on anything
//   but the cluster's own blocks, all resident together.
constexpr int kCWarps = 12;                    // compute warps per block
constexpr int kCThreads = kCWarps * 32;

// Shared memory of the cluster kernel for x staged per warp (MX = 1 or 2
// tokens) or per block (MX = 8): zero x (1 KB), the partials, the counters,
// then x. The footprint is kept small on purpose: the shared-memory carveout
// comes out of the L1, which also holds the in-flight weight loads (a 65 KB
// footprint against a 27 KB one measured 0.3 us slower per GEMV).
template <int MX>
struct CLayout {
    static constexpr int kPart = kRows * MX;                           // floats per partial
    static constexpr int kXTok = MX == 1 ? kUnitK * 2 : kUnitK * 2 + 64;  // a token's unit of x (+pad against bank conflicts)
    static constexpr int kXSlot = MX * kXTok;                           // one unit of x
    static constexpr int kFixed = 1024 + kCWarps * 2 * kPart * 4 + 128;
    static constexpr int kXWarp = MX <= 2 ? kCWarps * 2 * kXSlot : 0;  // per-warp rings
};

static_assert(CLayout<1>::kFixed + CLayout<1>::kXWarp <= 48 * 1024, "M = 1 within the default shared memory");

struct ClusterArgs {
    const uint16_t* x;
    const uint8_t* qw;
    const uint16_t* s;
    uint16_t* y;
    int M, N, K;
    int KU;    // 512-k units per row
    int RB;    // row-blocks: ceil(N / 16)
    int gpr;   // scale groups per row
    int svec;  // scale rows start 16-byte aligned
    int mode;  // kModeStatic
    unsigned int* err;  // device error word (a summing wait that gave up)
};

// A lane's share of one unit: rows gid and gid + 8, bytes 64 step + 16 t4 of
// the unit's 256 per row ([step][row half]).
struct Pieces {
    uint4 w[2 * kUnitSteps];
};

// Weights: read once, through L1 without allocating there (measured 0.3 us
// per GEMV faster than bypassing L1 with .cg). Read after griddepcontrol.wait
// (or, with static weights, with nothing pending that writes them), so they
// are the current contents.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// x and scales: plain (not volatile) loads, free to be scheduled with the rest
__device__ __forceinline__ uint4 ld_l2_v4_nv(const void* p) {
    uint4 v;
    asm("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_l2_v2_nv(const void* p) {
    uint2 v;
    asm("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// EXACT (N % 16 == 0, K % 512 == 0): every piece lies inside the matrix.
// Otherwise rows past N read row N - 1 (their sums are never stored) and
// pieces past K are zero (K is a multiple of 32: a piece is wholly in or out).
template <bool EXACT>
__device__ __forceinline__ void load_pieces(Pieces& u, const ClusterArgs& p, int rb, int ku, int gid, int t4) {
    const int64_t hk = p.K / 2;
    int64_t r0 = (int64_t)rb * kRows + gid, r1 = r0 + 8;
    if (!EXACT) {
        if (r0 >= p.N) r0 = p.N - 1;
        if (r1 >= p.N) r1 = p.N - 1;
    }
    const int64_t c = (int64_t)ku * (kUnitK / 2) + t4 * 16;
    const uint8_t* a = p.qw + r0 * hk + c;
    const uint8_t* b = p.qw + r1 * hk + c;
#pragma unroll
    for (int step = 0; step < kUnitSteps; ++step) {
        const bool in = EXACT || c + step * 64 < hk;
        u.w[2 * step] = in ? ld_stream_v4(a + step * 64) : make_uint4(0, 0, 0, 0);
        u.w[2 * step + 1] = in ? ld_stream_v4(b + step * 64) : make_uint4(0, 0, 0, 0);
    }
}

// The unit's four scales of rows gid and gid + 8 (EXACT: whole 16-byte aligned
// scale rows, no row past N).
template <bool EXACT>
__device__ __forceinline__ void load_unit_scales(UnitScales<128>& sc, const ClusterArgs& p, const ScaleRows& sr,
                                                 int ku) {
    if (EXACT) {
        const uint2 a = ld_l2_v2_nv(sr.r0 + ku * 4), b = ld_l2_v2_nv(sr.r1 + ku * 4);
        sc.lo[0] = a.x; sc.lo[1] = a.y;
        sc.hi[0] = b.x; sc.hi[1] = b.y;
    } else {
        load_scales<128>(sc, p, sr, ku);
    }
}

__device__ __forceinline__ ScaleRows plain_scale_rows(const ClusterArgs& p, int rb, int gid) {
    const int64_t n0 = (int64_t)rb * kRows + gid, n1 = n0 + 8;
    ScaleRows r;
    r.v0 = n0 < p.N;
    r.v1 = n1 < p.N;
    r.r0 = p.s + (r.v0 ? n0 : 0) * p.gpr;
    r.r1 = p.s + (r.v1 ? n1 : 0) * p.gpr;
    return r;
}

// One unit from registers (group 128: one group per 128-k step); x as in
// compute_unit, at xl (this lane's 16-byte chunk of the unit's x).
__device__ __forceinline__ void compute_pieces(const Pieces& u, const UnitScales<128>& sc, const uint8_t* xl,
                                               float (&acc)[4]) {
#pragma unroll
    for (int step = 0; step < kUnitSteps; ++step) {
        const uint32_t wa[4] = {u.w[2 * step].x, u.w[2 * step].y, u.w[2 * step].z, u.w[2 * step].w};
        const uint32_t wb[4] = {u.w[2 * step + 1].x, u.w[2 * step + 1].y, u.w[2 * step + 1].z,
                                u.w[2 * step + 1].w};
        float c[4];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const uint4 xv = lds_v4(xl + step * (kStepK * 2) + wi * 64);
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            nibbles_to_half2(wa[wi], a04, a15, a26, a37);
            nibbles_to_half2(wb[wi], b04, b15, b26, b37);
            if (wi == 0) mma_16816_zero(c, a04, b04, a15, b15, xv.x, xv.y);
            else mma_16816(c, a04, b04, a15, b15, xv.x, xv.y);
            mma_16816(c, a26, b26, a37, b37, xv.z, xv.w);
        }
        const float s0 = half_bits(sc.lo[step >> 1], step & 1), s1 = half_bits(sc.hi[step >> 1], step & 1);
        acc[0] = fmaf(s0, c[0], acc[0]);
        acc[1] = fmaf(s0, c[1], acc[1]);
        acc[2] = fmaf(s1, c[2], acc[2]);
        acc[3] = fmaf(s1, c[3], acc[3]);
    }
}

// Two 128-k steps (one group each) from pieces base .. base + 3 ([step][row
// half]); sl / sh hold the two groups' scales of rows gid and gid + 8.
__device__ __forceinline__ void compute_half_pieces(const Pieces& u, int base, uint32_t sl, uint32_t sh,
                                                    const uint8_t* xl, float (&acc)[4]) {
#pragma unroll
    for (int step = 0; step < kUnitSteps / 2; ++step) {
        const uint4 A = u.w[base + 2 * step], B = u.w[base + 2 * step + 1];
        const uint32_t wa[4] = {A.x, A.y, A.z, A.w};
        const uint32_t wb[4] = {B.x, B.y, B.z, B.w};
        float c[4];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const uint4 xv = lds_v4(xl + step * (kStepK * 2) + wi * 64);
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            nibbles_to_half2(wa[wi], a04, a15, a26, a37);
            nibbles_to_half2(wb[wi], b04, b15, b26, b37);
            if (wi == 0) mma_16816_zero(c, a04, b04, a15, b15, xv.x, xv.y);
            else mma_16816(c, a04, b04, a15, b15, xv.x, xv.y);
            mma_16816(c, a26, b26, a37, b37, xv.z, xv.w);
        }
        const float s0 = half_bits(sl, step), s1 = half_bits(sh, step);
        acc[0] = fmaf(s0, c[0], acc[0]);
        acc[1] = fmaf(s0, c[1], acc[1]);
        acc[2] = fmaf(s1, c[2], acc[2]);
        acc[3] = fmaf(s1, c[3], acc[3]);
    }
}

__device__ __forceinline__ uint32_t ld_l2_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void store_y_cluster(const ClusterArgs& p, int rb, const float (&v)[4], int gid, int t4,
                                                int m0 = 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + 2 * t4 + (i & 1);
        const int64_t n = (int64_t)rb * kRows + gid + 8 * (i >> 1);
        if (m < p.M && n < p.N) p.y[(int64_t)m * p.N + n] = __half_as_ushort(__float2half_rn(v[i]));
    }
}

// A split row-block as one contributor sees it: the cluster warps ga..gb
// contribute, and the row-block is ga's first segment or its last.
struct SplitSeg {
    int ga, gb;
    bool ga_first;
};

// MX: x staged per warp for M <= MX (1 or 2), or once per block (MX = 8);
// C: blocks per cluster.
template <int MX, bool EXACT, int C>
__global__ void __launch_bounds__(kCThreads, 1) gemv_cluster_kernel(const ClusterArgs p) {
    using L = CLayout<MX>;
    constexpr bool XW = MX <= 2;
    constexpr int XC = XW ? 2 * MX : 1;  // x chunks per lane per unit (per-warp staging)
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* zero = smem_raw;                                         // 1 KB of zero x
    float* part = reinterpret_cast<float*>(smem_raw + 1024);          // [warp][2][L::kPart]
    int* counter = reinterpret_cast<int*>(part + kCWarps * 2 * L::kPart);  // [warp]
    uint8_t* xs = smem_raw + L::kFixed;                               // per-warp rings, or the block's x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int rank = (int)ptx::cluster_rank();
    const int NC = (int)gridDim.x / C, cid = (int)blockIdx.x / C;
    const int KU = p.KU;
    const int rb0 = (int)((int64_t)p.RB * cid / NC), rb1 = (int)((int64_t)p.RB * (cid + 1) / NC);
    const int64_t Tc = (int64_t)(rb1 - rb0) * KU;  // the cluster's units
    // warps taking part: every one owns at least one unit, so the contributors
    // to a row-block are consecutive warps
    const int GW = (int)(Tc < C * kCWarps ? Tc : C * kCWarps), g = rank * kCWarps + warp;
    const int q0 = g < GW ? (int)(Tc * g / GW) : 0, n = g < GW ? (int)(Tc * (g + 1) / GW) - q0 : 0;
    // the cluster warp whose range holds the cluster's unit q
    auto warp_of = [&](int64_t q) { return (int)(((q + 1) * GW + Tc - 1) / Tc - 1); };
    int lrb = q0 / KU, ku = q0 % KU;  // row-block (from rb0) and unit of the next unit
    // Only a warp's first and last row-blocks can be split with other warps:
    // their contributors are worked out here, before the dependency wait,
    // rather than by divisions at the end of the launch.
    auto split_seg = [&](int lrb_) {
        const int64_t qa = (int64_t)lrb_ * KU;
        SplitSeg sg;
        sg.ga = warp_of(qa);
        sg.gb = warp_of(qa + KU - 1);
        sg.ga_first = Tc * sg.ga / GW >= qa;
        return sg;
    };
    SplitSeg seg_first = {0, 0, false}, seg_last = {0, 0, false};
    if (n > 0) {
        seg_first = split_seg(lrb);
        seg_last = split_seg((q0 + n - 1) / KU);
    }
    const int xstride = (int)KU * (kUnitSteps * kStepK * 2) + 64;  // block-staged x: bytes per token

    Pieces cur, nxt;
    if ((p.mode & kModeStatic) && n > 0) load_pieces<EXACT>(cur, p, rb0 + lrb, ku, gid, t4);
    if (threadIdx.x < 64) reinterpret_cast<uint4*>(zero)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x < kCWarps) counter[threadIdx.x] = 0;
    ptx::cluster_sync();  // the counters of every block are zero before any arrival
    ptx::grid_dependency_wait();
    if (!(p.mode & kModeStatic) && n > 0) load_pieces<EXACT>(cur, p, rb0 + lrb, ku, gid, t4);
    // the first unit's scales go out before x is staged
    ScaleRows sr = plain_scale_rows(p, rb0 + lrb, gid);
    UnitScales<128> sc;
    if (n > 0) load_unit_scales<EXACT>(sc, p, sr, ku);

    // per-warp x: this lane's chunks c = lane + 32 i of a unit (token c / 64,
    // 16-byte chunk c % 64 of its 1 KB), zero past K
    uint8_t* xw = xs + warp * (2 * L::kXSlot);
    auto load_x = [&](int ku_, uint4 (&v)[XC]) {
#pragma unroll
        for (int i = 0; i < XC; ++i) {
            const int c = lane + 32 * i, m = c >> 6, j = c & 63;
            const int64_t k = (int64_t)ku_ * kUnitK + j * 8;
            v[i] = ((EXACT || k < p.K) && (MX == 1 || m < p.M)) ? ld_l2_v4_nv(p.x + (int64_t)m * p.K + k)
                                                                 : make_uint4(0, 0, 0, 0);
        }
    };
    auto store_x = [&](uint8_t* slot, const uint4 (&v)[XC]) {
#pragma unroll
        for (int i = 0; i < XC; ++i) {
            const int c = lane + 32 * i, m = c >> 6, j = c & 63;
            if (MX == 1 || m < p.M)
                *reinterpret_cast<uint4*>(slot + m * L::kXTok + (j >> 4) * (kStepK * 2) + xs_pos(j & 15, 128) * 16) =
                    permute_x8(v[i]);
        }
    };
    if constexpr (XW) {
        if (n > 0) {
            uint4 v[XC];
            load_x(ku, v);
            store_x(xw, v);
            __syncwarp();
        }
    } else {  // the whole x, once per block (as gemv_body does)
        const int per_tok = KU * kUnitSteps * 16;
        for (int c = threadIdx.x; c < p.M * per_tok; c += kCThreads) {
            const int m = c / per_tok, cc = c % per_tok;
            const uint4 v = cc * 8 < p.K ? ld_l2_v4(p.x + (int64_t)m * p.K + cc * 8) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(xs + m * xstride + (cc >> 4) * (kStepK * 2) + xs_pos(cc & 15, 128) * 16) =
                permute_x8(v);
        }
        __syncthreads();
    }

    if (n > 0) {
        const bool has = gid < p.M;
        const int first_lrb = lrb;
        int seg_ku0 = ku;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < n; ++r) {
            int nlrb = lrb, nku = ku + 1;
            if (nku == KU) {
                nku = 0;
                ++nlrb;
            }
            UnitScales<128> sc_next = sc;
            uint4 xv[XC];
            if (r + 1 < n) {  // the next unit's weights, scales and x go out before this one's arithmetic
                load_pieces<EXACT>(nxt, p, rb0 + nlrb, nku, gid, t4);
                if (nku == 0) sr = plain_scale_rows(p, rb0 + nlrb, gid);
                load_unit_scales<EXACT>(sc_next, p, sr, nku);
                if constexpr (XW) load_x(nku, xv);
            }
            const uint8_t* xl;
            if constexpr (XW) xl = (has ? xw + (r & 1) * L::kXSlot + gid * L::kXTok : zero) + t4 * 16;
            else xl = (has ? xs + gid * xstride + ku * (kUnitSteps * kStepK * 2) : zero) + t4 * 16;
            compute_pieces(cur, sc, xl, acc);
            if constexpr (XW) {
                if (r + 1 < n) {
                    store_x(xw + ((r + 1) & 1) * L::kXSlot, xv);
                    __syncwarp();  // every lane's chunks before any lane reads the slot
                }
            }
            // only this warp's last sums remain: the next kernel on the stream may launch
            if (r == n - 1) ptx::launch_dependents();
            if (ku == KU - 1 || r == n - 1) {
                const int rb = rb0 + lrb;
                if (seg_ku0 == 0 && ku == KU - 1) {
                    store_y_cluster(p, rb, acc, gid, t4);  // the whole row-block in this warp
                } else {
                    // the row-block's contributors: cluster warps ga..gb; this one
                    // is at slot 0 if the row-block is its first segment
                    const int sl = lrb == first_lrb ? 0 : 1;
                    float* mine = part + (warp * 2 + sl) * L::kPart;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = 2 * t4 + (i & 1);
                        if (m < p.M) mine[m * kRows + gid + 8 * (i >> 1)] = acc[i];
                    }
                    __syncwarp();  // the lanes' partials before lane 0's release
                    const SplitSeg sg = sl == 0 ? seg_first : seg_last;
                    const int ga = sg.ga, gb = sg.gb;
                    int old = 0;
                    if (lane == 0)
                        old = ptx::atom_add_acq_rel_cluster(
                            ptx::cluster_map(ptx::smem_u32(counter + ga % kCWarps), (uint32_t)(ga / kCWarps)), 1);
                    old = __shfl_sync(0xffffffffu, old, 0);
                    if (old == gb - ga) {  // the last contributor: sum them all in warp order
                        __syncwarp();      // every lane's loads after lane 0's acquire
                        const bool ga_first = sg.ga_first;  // the row-block is ga's first segment
                        float sum[4] = {0.f, 0.f, 0.f, 0.f};
                        constexpr int kBatch = 8;  // partials loaded at once
                        for (int v0 = ga; v0 <= gb; v0 += kBatch) {
                            float pv[kBatch][4];
#pragma unroll
                            for (int b = 0; b < kBatch; ++b) {
                                const int v = v0 + b;
                                const int slv = (v == ga && !ga_first) ? 1 : 0;
                                const uint32_t base = ptx::cluster_map(
                                    ptx::smem_u32(part + ((v % kCWarps) * 2 + slv) * L::kPart),
                                    (uint32_t)(v / kCWarps));
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int m = 2 * t4 + (i & 1);
                                    pv[b][i] = (v <= gb && m < p.M)
                                                   ? ptx::ld_cluster_f32(base + 4u * (m * kRows + gid + 8 * (i >> 1)))
                                                   : 0.f;
                                }
                            }
#pragma unroll
                            for (int b = 0; b < kBatch; ++b)
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (v0 + b <= gb) sum[i] += pv[b][i];
                        }
                        store_y_cluster(p, rb, sum, gid, t4);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = 0.f;
                seg_ku0 = nku;
            }
            lrb = nlrb;
            ku = nku;
            cur = nxt;
            sc = sc_next;
        }
    } else {
        ptx::launch_dependents();
    }
    ptx::cluster_sync();  // no block leaves while another may still read its partials
}

// The decode case of gemv_cluster_kernel, written out for it: M = 1, N % 16 ==
// 0, K % 512 == 0, every cluster with at least C x kCWarps units (so every
// warp takes part) and at most kMail + 1 contributors to a row-block. The same
// arithmetic in the same order, with the general kernel's index arithmetic
// (cluster size and warp count known only at run time, rows and pieces
// checked against N and K, a scale-row record) taken out: that cost 0.6 to
// 1.1 us per GEMV in the back-to-back decode step.
//
// Split row-blocks are summed without any contributor waiting: the first
// contributor ga of a row-block (for which it is its last segment) finishes
// it. Every other contributor sends its 16 fp32 sums into ga's mailbox with
// one-way st.async stores, which complete the transaction count of ga's
// mbarrier as they land; ga arms that barrier with the bytes it expects at the
// start of the launch, waits on it (with a time limit) after its own units,
// and adds the sums in warp order: the same order, and the same result, as
// the general kernel's. (A cluster-scope acquire-release atomic per
// contributor, whose release waits for the contributor's in-flight weight
// loads, then loads by the last arriver, cost 1.8 us of a 13.0 us launch.)
constexpr int kMail = 8;  // contributors besides the finisher, per row-block

template <int C>
__global__ void __launch_bounds__(kCThreads, 1) gemv_decode_kernel(const ClusterArgs p) {
    constexpr int GW = C * kCWarps;  // the cluster's warps, all taking part
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* zero = smem_raw;                                              // 1 KB of zero x
    uint8_t* xr = smem_raw + 1024;                                         // [warp][2 slots][1 KB]
    float* mail = reinterpret_cast<float*>(smem_raw + 1024 + kCWarps * 2048);  // [warp][kMail][16]
    uint64_t* bar = reinterpret_cast<uint64_t*>(mail + kCWarps * kMail * kRows);  // [warp]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int rank = (int)ptx::cluster_rank();
    const int cid = (int)blockIdx.x / C, NC = (int)gridDim.x / C;
    const int KU = p.KU;
    const int rb0 = (int)((int64_t)p.RB * cid / NC), rb1 = (int)((int64_t)p.RB * (cid + 1) / NC);
    const int Tc = (rb1 - rb0) * KU;
    const int g = rank * kCWarps + warp;
    const int q0 = (int)((int64_t)Tc * g / GW), n = (int)((int64_t)Tc * (g + 1) / GW) - q0;
    auto warp_of = [&](int q) { return (int)(((int64_t)(q + 1) * GW + Tc - 1) / Tc - 1); };
    int lrb = q0 / KU, ku = q0 % KU;
    const int hk = p.K / 2;
    const uint8_t* lane_base = p.qw + (int64_t)gid * hk + t4 * 16;  // row gid of row-block 0, this lane's bytes
    auto load_unit = [&](Pieces& u, int rb_, int ku_) {
        const uint8_t* a = lane_base + (int64_t)rb_ * kRows * hk + ku_ * (kUnitK / 2);
#pragma unroll
        for (int step = 0; step < kUnitSteps; ++step) {
            u.w[2 * step] = ld_stream_v4(a + step * 64);
            u.w[2 * step + 1] = ld_stream_v4(a + 8 * hk + step * 64);
        }
    };
    Pieces cur, nxt;
    if ((p.mode & kModeStatic) && n > 0) load_unit(cur, rb0 + lrb, ku);
    // this warp's first and last row-blocks: its only segments that may be split
    const int lrb_first = lrb, lrb_last = (q0 + n - 1) / KU;
    const int fa = warp_of(lrb_first * KU), fb = warp_of(lrb_first * KU + KU - 1);  // contributors, first
    const int la = warp_of(lrb_last * KU), lb = warp_of(lrb_last * KU + KU - 1);    // contributors, last
    if (threadIdx.x < 64) reinterpret_cast<uint4*>(zero)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    if (lane == 0) {
        ptx::mbar_init(&bar[warp], 1);
        // the finisher of its last row-block expects the others' 64 bytes each
        if (la == g && lb > la) ptx::mbar_arrive_expect_tx(&bar[warp], (uint32_t)(lb - la) * kRows * 4);
        ptx::fence_mbar_init();
    }
    ptx::cluster_sync();  // every mailbox barrier is set up before any store lands
    ptx::grid_dependency_wait();
    if (!(p.mode & kModeStatic)) load_unit(cur, rb0 + lrb, ku);
    // the unit's four scales of rows gid and gid + 8 (rows 16-byte aligned)
    auto load_sc = [&](int rb_, int ku_, uint2& a, uint2& b) {
        const uint16_t* r0 = p.s + (int64_t)(rb_ * kRows + gid) * p.gpr + ku_ * 4;
        a = ld_l2_v2(r0);
        b = ld_l2_v2(r0 + 8 * p.gpr);
    };
    // this lane's two 16-byte chunks (lane, lane + 32) of a unit's x
    auto load_x = [&](int ku_, uint4& a, uint4& b) {
        const uint16_t* xp = p.x + ku_ * kUnitK;
        a = ld_l2_v4_nv(xp + lane * 8);
        b = ld_l2_v4_nv(xp + (lane + 32) * 8);
    };
    uint8_t* xw = xr + warp * 2048;
    auto store_x = [&](uint8_t* slot, uint4 a, uint4 b) {
        const int j0 = lane, j1 = lane + 32;
        *reinterpret_cast<uint4*>(slot + (j0 >> 4) * 256 + xs_pos(j0 & 15, 128) * 16) = permute_x8(a);
        *reinterpret_cast<uint4*>(slot + (j1 >> 4) * 256 + xs_pos(j1 & 15, 128) * 16) = permute_x8(b);
    };
    uint2 sa, sb;
    load_sc(rb0 + lrb, ku, sa, sb);
    {
        uint4 a, b;
        load_x(ku, a, b);
        store_x(xw, a, b);
        __syncwarp();
    }
    const bool has = gid == 0;  // the token's lanes; the others read zero x
    int seg_ku0 = ku;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < n; ++r) {
        int nlrb = lrb, nku = ku + 1;
        if (nku == KU) {
            nku = 0;
            ++nlrb;
        }
        uint2 na = sa, nb = sb;
        uint4 xa, xb;
        if (r + 1 < n) {
            load_unit(nxt, rb0 + nlrb, nku);
            load_sc(rb0 + nlrb, nku, na, nb);
            load_x(nku, xa, xb);
        }
        UnitScales<128> sc;
        sc.lo[0] = sa.x;
        sc.lo[1] = sa.y;
        sc.hi[0] = sb.x;
        sc.hi[1] = sb.y;
        compute_pieces(cur, sc, (has ? xw + (r & 1) * 1024 : zero) + t4 * 16, acc);
        if (r + 1 < n) {
            store_x(xw + ((r + 1) & 1) * 1024, xa, xb);
            __syncwarp();  // every lane's chunks before any lane reads the slot
        }
        if (r == n - 1) ptx::launch_dependents();
        const bool seg_end = (ku == KU - 1) || (r == n - 1);
        if (seg_end) {
            const int rb = rb0 + lrb;
            if (seg_ku0 == 0 && ku == KU - 1) {
                store_y_cluster(p, rb, acc, gid, t4);  // the whole row-block in this warp
            } else {
                const bool first = lrb == lrb_first;
                const int ga = first ? fa : la, gb = first ? fb : lb;
                if (g != ga) {
                    // into slot g - ga - 1 of ga's mailbox; ga's barrier counts the bytes
                    // (a test build can hold the sums back to make ga's wait run out)
                    if (t4 == 0 && may_issue(0)) {
                        const uint32_t rk = (uint32_t)(ga / kCWarps);
                        const uint32_t dst = ptx::cluster_map(
                            ptx::smem_u32(mail + ((ga % kCWarps) * kMail + (g - ga - 1)) * kRows + gid), rk);
                        const uint32_t rbar = ptx::cluster_map(ptx::smem_u32(&bar[ga % kCWarps]), rk);
                        ptx::st_async_cluster_f32(dst, acc[0], rbar);
                        ptx::st_async_cluster_f32(dst + 32, acc[2], rbar);
                    }
                } else {
                    // this warp finishes the row-block: the others' sums, then all in warp order
                    volatile int never = 0;
                    const bool ok = ptx::mbar_wait(&bar[warp], 0, &never, wait_limit());
                    if (ok) {
                        float sum0 = 0.f + acc[0], sum1 = 0.f + acc[2];
                        if (t4 == 0) {
                            const float* box = mail + warp * kMail * kRows + gid;
                            for (int v = 1; v <= gb - ga; ++v) {
                                sum0 += box[(v - 1) * kRows];
                                sum1 += box[(v - 1) * kRows + 8];
                            }
                        }
                        const float sv[4] = {sum0, 0.f, sum1, 0.f};
                        store_y_cluster(p, rb, sv, gid, t4);
                    } else if (lane == 0) {
                        raise_device_error(p.err, W4A16_ERR_TIMEOUT);
                    }
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            seg_ku0 = nku;
        }
        lrb = nlrb;
        ku = nku;
        cur = nxt;
        sa = na;
        sb = nb;
    }
    ptx::cluster_sync();  // no block leaves while a store into its mailbox may be on the way
}

constexpr size_t kDecodeSmem = 1024 + kCWarps * 2048 + kCWarps * kMail * kRows * 4 + kCWarps * 8;

// The fused gate+up decode (M = 1, group 128, N % 16 == 0, K % 512 == 0) on
// the same design. A unit here is a pair: 16 rows of Wg and the same 16 rows
// of Wu over 256 k (2 + 2 KB, so a lane holds what it holds in the plain
// kernel: 8 pieces of 16 bytes). A row-block is one 16-row block of the
// output; its units run over K / 256. A warp keeps the gate and the up sums of
// its segment apart; a split row-block's finisher gets both from every other
// contributor (32 fp32 values by st.async), adds them in warp order and forms
// y = silu(g) * u in fp32, rounded once to fp16 (rust-inference README, list
// of accuracy fixes, item 5). g and u never leave the cluster.
struct GatedClusterArgs {
    ClusterArgs a;        // x, Wg, sg, y, M, N, K; KU counts 256-k units
    const uint8_t* qw2;   // Wu
    const uint16_t* s2;   // su
};

constexpr int kGMail = 8;                 // contributors besides the finisher, per row-block
constexpr int kGPart = 2 * kRows;         // floats of one contributor's sums: 16 g, then 16 u
constexpr int kGMailOff = 1024 + kCWarps * 1024;  // after zero x and the per-warp x rings (2 x 512 B)
constexpr int kGBarOff = kGMailOff + kCWarps * kGMail * kGPart * 4;
constexpr size_t kGatedDecodeSmem = kGBarOff + kCWarps * 8;

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.0f + expf(-g)) * u; }

template <int C>
__global__ void __launch_bounds__(kCThreads, 1) gemv_gated_decode_kernel(const GatedClusterArgs ga_) {
    const ClusterArgs& p = ga_.a;
    constexpr int GW = C * kCWarps;
    constexpr int kHalf = kUnitSteps / 2;  // 128-k steps per matrix in a pair unit
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* zero = smem_raw;                                            // 1 KB of zero x
    uint8_t* xr = smem_raw + 1024;                                       // [warp][2 slots][512 B]
    float* mail = reinterpret_cast<float*>(smem_raw + kGMailOff);       // [warp][kGMail][kGPart]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + kGBarOff);   // [warp]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int rank = (int)ptx::cluster_rank();
    const int cid = (int)blockIdx.x / C, NC = (int)gridDim.x / C;
    const int KU = p.KU;  // 256-k pair units per row-block
    const int rb0 = (int)((int64_t)p.RB * cid / NC), rb1 = (int)((int64_t)p.RB * (cid + 1) / NC);
    const int Tc = (rb1 - rb0) * KU;
    const int g = rank * kCWarps + warp;
    const int q0 = (int)((int64_t)Tc * g / GW), n = (int)((int64_t)Tc * (g + 1) / GW) - q0;
    auto warp_of = [&](int q) { return (int)(((int64_t)(q + 1) * GW + Tc - 1) / Tc - 1); };
    int lrb = q0 / KU, ku = q0 % KU;
    const int hk = p.K / 2;
    const int64_t lane_off = (int64_t)gid * hk + t4 * 16;  // row gid, this lane's bytes
    // pieces [step][row half] of Wg (0..3), then of Wu (4..7)
    auto load_unit = [&](Pieces& u, int rb_, int ku_) {
        const int64_t o = lane_off + (int64_t)rb_ * kRows * hk + ku_ * (kUnitK / 4);
#pragma unroll
        for (int step = 0; step < kHalf; ++step) {
            u.w[2 * step] = ld_stream_v4(p.qw + o + step * 64);
            u.w[2 * step + 1] = ld_stream_v4(p.qw + o + 8 * hk + step * 64);
            u.w[4 + 2 * step] = ld_stream_v4(ga_.qw2 + o + step * 64);
            u.w[4 + 2 * step + 1] = ld_stream_v4(ga_.qw2 + o + 8 * hk + step * 64);
        }
    };
    Pieces cur, nxt;
    if ((p.mode & kModeStatic) && n > 0) load_unit(cur, rb0 + lrb, ku);
    const int lrb_first = lrb, lrb_last = (q0 + n - 1) / KU;
    const int fa = warp_of(lrb_first * KU), fb = warp_of(lrb_first * KU + KU - 1);
    const int la = warp_of(lrb_last * KU), lb = warp_of(lrb_last * KU + KU - 1);
    if (threadIdx.x < 64) reinterpret_cast<uint4*>(zero)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    if (lane == 0) {
        ptx::mbar_init(&bar[warp], 1);
        if (la == g && lb > la) ptx::mbar_arrive_expect_tx(&bar[warp], (uint32_t)(lb - la) * kGPart * 4);
        ptx::fence_mbar_init();
    }
    ptx::cluster_sync();  // every mailbox barrier is set up before any store lands
    ptx::grid_dependency_wait();
    if (!(p.mode & kModeStatic)) load_unit(cur, rb0 + lrb, ku);
    // a pair unit's scales: two groups of rows gid and gid + 8, of Wg and of Wu
    auto load_sc = [&](int rb_, int ku_, uint32_t (&sv)[4]) {
        const int64_t o = (int64_t)(rb_ * kRows + gid) * p.gpr + ku_ * 2;
        sv[0] = ld_l2_u32(p.s + o);
        sv[1] = ld_l2_u32(p.s + o + 8 * p.gpr);
        sv[2] = ld_l2_u32(ga_.s2 + o);
        sv[3] = ld_l2_u32(ga_.s2 + o + 8 * p.gpr);
    };
    // this lane's 16-byte chunk of a pair unit's x (256 k = 32 chunks)
    auto load_x = [&](int ku_) { return ld_l2_v4_nv(p.x + ku_ * (kUnitK / 2) + lane * 8); };
    uint8_t* xw = xr + warp * 1024;
    auto store_x = [&](uint8_t* slot, uint4 a) {
        *reinterpret_cast<uint4*>(slot + (lane >> 4) * 256 + xs_pos(lane & 15, 128) * 16) = permute_x8(a);
    };
    uint32_t sv[4];
    load_sc(rb0 + lrb, ku, sv);
    store_x(xw, load_x(ku));
    __syncwarp();
    const bool has = gid == 0;
    int seg_ku0 = ku;
    float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < n; ++r) {
        int nlrb = lrb, nku = ku + 1;
        if (nku == KU) {
            nku = 0;
            ++nlrb;
        }
        uint32_t nsv[4] = {sv[0], sv[1], sv[2], sv[3]};
        uint4 xa;
        if (r + 1 < n) {
            load_unit(nxt, rb0 + nlrb, nku);
            load_sc(rb0 + nlrb, nku, nsv);
            xa = load_x(nku);
        }
        const uint8_t* xl = (has ? xw + (r & 1) * 512 : zero) + t4 * 16;
        compute_half_pieces(cur, 0, sv[0], sv[1], xl, accg);
        compute_half_pieces(cur, 4, sv[2], sv[3], xl, accu);
        if (r + 1 < n) {
            store_x(xw + ((r + 1) & 1) * 512, xa);
            __syncwarp();  // every lane's chunk before any lane reads the slot
        }
        if (r == n - 1) ptx::launch_dependents();
        const bool seg_end = (ku == KU - 1) || (r == n - 1);
        if (seg_end) {
            const int rb = rb0 + lrb;
            if (seg_ku0 == 0 && ku == KU - 1) {
                const float yv[4] = {silu_times(accg[0], accu[0]), 0.f, silu_times(accg[2], accu[2]), 0.f};
                store_y_cluster(p, rb, yv, gid, t4);  // the whole row-block in this warp
            } else {
                const bool first = lrb == lrb_first;
                const int ga = first ? fa : la, gb = first ? fb : lb;
                if (g != ga) {
                    if (t4 == 0 && may_issue(0)) {
                        const uint32_t rk = (uint32_t)(ga / kCWarps);
                        const uint32_t dst = ptx::cluster_map(
                            ptx::smem_u32(mail + ((ga % kCWarps) * kGMail + (g - ga - 1)) * kGPart + gid), rk);
                        const uint32_t rbar = ptx::cluster_map(ptx::smem_u32(&bar[ga % kCWarps]), rk);
                        ptx::st_async_cluster_f32(dst, accg[0], rbar);
                        ptx::st_async_cluster_f32(dst + 32, accg[2], rbar);
                        ptx::st_async_cluster_f32(dst + 64, accu[0], rbar);
                        ptx::st_async_cluster_f32(dst + 96, accu[2], rbar);
                    }
                } else {
                    volatile int never = 0;
                    const bool ok = ptx::mbar_wait(&bar[warp], 0, &never, wait_limit());
                    if (ok) {
                        float g0 = 0.f + accg[0], g1 = 0.f + accg[2], u0 = 0.f + accu[0], u1 = 0.f + accu[2];
                        if (t4 == 0) {
                            const float* box = mail + warp * kGMail * kGPart + gid;
                            for (int v = 1; v <= gb - ga; ++v) {
                                g0 += box[(v - 1) * kGPart];
                                g1 += box[(v - 1) * kGPart + 8];
                                u0 += box[(v - 1) * kGPart + 16];
                                u1 += box[(v - 1) * kGPart + 24];
                            }
                        }
                        const float yv[4] = {silu_times(g0, u0), 0.f, silu_times(g1, u1), 0.f};
                        store_y_cluster(p, rb, yv, gid, t4);
                    } else if (lane == 0) {
                        raise_device_error(p.err, W4A16_ERR_TIMEOUT);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) accg[i] = accu[i] = 0.f;
            seg_ku0 = nku;
        }
        lrb = nlrb;
        ku = nku;
        cur = nxt;
#pragma unroll
        for (int i = 0; i < 4; ++i) sv[i] = nsv[i];
    }
    ptx::cluster_sync();  // no block leaves while a store into its mailbox may be on the way
}

// The decode kernel for 2 to 8 tokens (MT = 8): the same partition and
// mailbox sum, x staged once per block (a unit's x for 8 tokens does not fit
// the registers of a warp that also holds two units of weights), each
// contributor sending its 16 x M sums. (A single kernel for both token counts
// measured 0.1 to 0.25 us slower at M = 1, so the one-token kernel above keeps
// its own code.)
template <int MT>
struct DLayout {
    static constexpr int kMail = 4;            // contributors besides the finisher, per row-block
    static constexpr int kPart = kRows * MT;   // floats of one contributor's sums
    static constexpr int kMailOff = 1024;
    static constexpr int kBarOff = kMailOff + kCWarps * kMail * kPart * 4;
    static constexpr int kFixed = (kBarOff + kCWarps * 8 + 127) & ~127;  // then the block's x
};

// One unit from registers for NT tiles of 8 tokens: each weight word is turned
// into fp16 once and feeds NT MMAs (x of tile t at xl[t]).
template <int NT>
__device__ __forceinline__ void compute_pieces_nt(const Pieces& u, const UnitScales<128>& sc,
                                                  const uint8_t* const (&xl)[NT], float (&acc)[NT][4]) {
#pragma unroll
    for (int step = 0; step < kUnitSteps; ++step) {
        const uint32_t wa[4] = {u.w[2 * step].x, u.w[2 * step].y, u.w[2 * step].z, u.w[2 * step].w};
        const uint32_t wb[4] = {u.w[2 * step + 1].x, u.w[2 * step + 1].y, u.w[2 * step + 1].z,
                                u.w[2 * step + 1].w};
        float c[NT][4];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            nibbles_to_half2(wa[wi], a04, a15, a26, a37);
            nibbles_to_half2(wb[wi], b04, b15, b26, b37);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4 xv = lds_v4(xl[t] + step * (kStepK * 2) + wi * 64);
                if (wi == 0) mma_16816_zero(c[t], a04, b04, a15, b15, xv.x, xv.y);
                else mma_16816(c[t], a04, b04, a15, b15, xv.x, xv.y);
                mma_16816(c[t], a26, b26, a37, b37, xv.z, xv.w);
            }
        }
        const float s0 = half_bits(sc.lo[step >> 1], step & 1), s1 = half_bits(sc.hi[step >> 1], step & 1);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(s0, c[t][0], acc[t][0]);
            acc[t][1] = fmaf(s0, c[t][1], acc[t][1]);
            acc[t][2] = fmaf(s1, c[t][2], acc[t][2]);
            acc[t][3] = fmaf(s1, c[t][3], acc[t][3]);
        }
    }
}

// MT tokens at most (8 or 16): NT = MT / 8 tiles of the mma's 8 columns.
template <int C, int MT>
__global__ void __launch_bounds__(kCThreads, 1) gemv_decode_tokens_kernel(const ClusterArgs p) {
    using L = DLayout<MT>;
    constexpr int NT = MT / 8;
    constexpr int GW = C * kCWarps;  // the cluster's warps, all taking part
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* zero = smem_raw;                                          // 1 KB of zero x
    float* mail = reinterpret_cast<float*>(smem_raw + L::kMailOff);   // [warp][kMail][kPart]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + L::kBarOff);  // [warp]
    uint8_t* xs = smem_raw + L::kFixed;                                // the block's x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int rank = (int)ptx::cluster_rank();
    const int cid = (int)blockIdx.x / C, NC = (int)gridDim.x / C;
    const int KU = p.KU;
    const int rb0 = (int)((int64_t)p.RB * cid / NC), rb1 = (int)((int64_t)p.RB * (cid + 1) / NC);
    const int Tc = (rb1 - rb0) * KU;
    const int g = rank * kCWarps + warp;
    const int q0 = (int)((int64_t)Tc * g / GW), n = (int)((int64_t)Tc * (g + 1) / GW) - q0;
    auto warp_of = [&](int q) { return (int)(((int64_t)(q + 1) * GW + Tc - 1) / Tc - 1); };
    int lrb = q0 / KU, ku = q0 % KU;
    const int hk = p.K / 2;
    const int M = p.M;
    const uint8_t* lane_base = p.qw + (int64_t)gid * hk + t4 * 16;  // row gid of row-block 0, this lane's bytes
    auto load_unit = [&](Pieces& u, int rb_, int ku_) {
        const uint8_t* a = lane_base + (int64_t)rb_ * kRows * hk + ku_ * (kUnitK / 2);
#pragma unroll
        for (int step = 0; step < kUnitSteps; ++step) {
            u.w[2 * step] = ld_stream_v4(a + step * 64);
            u.w[2 * step + 1] = ld_stream_v4(a + 8 * hk + step * 64);
        }
    };
    Pieces cur, nxt;
    if ((p.mode & kModeStatic) && n > 0) load_unit(cur, rb0 + lrb, ku);
    // this warp's first and last row-blocks: its only segments that may be split
    const int lrb_first = lrb, lrb_last = (q0 + n - 1) / KU;
    const int fa = warp_of(lrb_first * KU), fb = warp_of(lrb_first * KU + KU - 1);  // contributors, first
    const int la = warp_of(lrb_last * KU), lb = warp_of(lrb_last * KU + KU - 1);    // contributors, last
    if (threadIdx.x < 64) reinterpret_cast<uint4*>(zero)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    if (lane == 0) {
        ptx::mbar_init(&bar[warp], 1);
        // the finisher of its last row-block expects the others' sums: 16 rows x M tokens each
        if (la == g && lb > la) ptx::mbar_arrive_expect_tx(&bar[warp], (uint32_t)(lb - la) * kRows * M * 4);
        ptx::fence_mbar_init();
    }
    ptx::cluster_sync();  // every mailbox barrier is set up before any store lands
    ptx::grid_dependency_wait();
    if (!(p.mode & kModeStatic)) load_unit(cur, rb0 + lrb, ku);
    // the unit's four scales of rows gid and gid + 8 (rows 16-byte aligned)
    auto load_sc = [&](int rb_, int ku_, uint2& a, uint2& b) {
        const uint16_t* r0 = p.s + (int64_t)(rb_ * kRows + gid) * p.gpr + ku_ * 4;
        a = ld_l2_v2(r0);
        b = ld_l2_v2(r0 + 8 * p.gpr);
    };
    const int xstride = KU * (kUnitSteps * kStepK * 2) + 64;  // bytes per token of the block's x
    uint2 sa, sb;
    load_sc(rb0 + lrb, ku, sa, sb);
    {  // the whole x, once per block, in fragment order
        const int per_tok = KU * kUnitSteps * 16;
        for (int c = threadIdx.x; c < M * per_tok; c += kCThreads) {
            const int m = c / per_tok, cc = c % per_tok;
            const uint4 v = ld_l2_v4(p.x + (int64_t)m * p.K + cc * 8);
            *reinterpret_cast<uint4*>(xs + m * xstride + (cc >> 4) * (kStepK * 2) + xs_pos(cc & 15, 128) * 16) =
                permute_x8(v);
        }
        __syncthreads();
    }
    int seg_ku0 = ku;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    for (int r = 0; r < n; ++r) {
        int nlrb = lrb, nku = ku + 1;
        if (nku == KU) {
            nku = 0;
            ++nlrb;
        }
        uint2 na = sa, nb = sb;
        if (r + 1 < n) {
            load_unit(nxt, rb0 + nlrb, nku);
            load_sc(rb0 + nlrb, nku, na, nb);
        }
        UnitScales<128> sc;
        sc.lo[0] = sa.x;
        sc.lo[1] = sa.y;
        sc.hi[0] = sb.x;
        sc.hi[1] = sb.y;
        const uint8_t* xl[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t)
            xl[t] = (8 * t + gid < M ? xs + (8 * t + gid) * xstride + ku * (kUnitSteps * kStepK * 2) : zero) + t4 * 16;
        compute_pieces_nt<NT>(cur, sc, xl, acc);
        if (r == n - 1) ptx::launch_dependents();
        const bool seg_end = (ku == KU - 1) || (r == n - 1);
        if (seg_end) {
            const int rb = rb0 + lrb;
            if (seg_ku0 == 0 && ku == KU - 1) {
#pragma unroll
                for (int t = 0; t < NT; ++t) store_y_cluster(p, rb, acc[t], gid, t4, 8 * t);  // whole row-block
            } else {
                const bool first = lrb == lrb_first;
                const int ga = first ? fa : la, gb = first ? fb : lb;
                if (g != ga) {
                    // into slot g - ga - 1 of ga's mailbox ([token][row]); ga's barrier
                    // counts the bytes (a test build can hold the sums back to make
                    // ga's wait run out)
                    if (may_issue(0)) {
                        const uint32_t rk = (uint32_t)(ga / kCWarps);
                        const uint32_t dst = ptx::cluster_map(
                            ptx::smem_u32(mail + ((ga % kCWarps) * L::kMail + (g - ga - 1)) * L::kPart), rk);
                        const uint32_t rbar = ptx::cluster_map(ptx::smem_u32(&bar[ga % kCWarps]), rk);
#pragma unroll
                        for (int t = 0; t < NT; ++t)
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int m = 8 * t + 2 * t4 + (i & 1);
                                if (m < M)
                                    ptx::st_async_cluster_f32(dst + 4u * (m * kRows + gid + 8 * (i >> 1)), acc[t][i],
                                                              rbar);
                            }
                    }
                } else {
                    // this warp finishes the row-block: the others' sums, then all in warp order
                    volatile int never = 0;
                    const bool ok = ptx::mbar_wait(&bar[warp], 0, &never, wait_limit());
                    if (ok) {
                        const float* box = mail + warp * L::kMail * L::kPart;
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            float sum[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int m = 8 * t + 2 * t4 + (i & 1);
                                sum[i] = 0.f + acc[t][i];
                                if (m < M)
                                    for (int v = 1; v <= gb - ga; ++v)
                                        sum[i] += box[(v - 1) * L::kPart + m * kRows + gid + 8 * (i >> 1)];
                            }
                            store_y_cluster(p, rb, sum, gid, t4, 8 * t);
                        }
                    } else if (lane == 0) {
                        raise_device_error(p.err, W4A16_ERR_TIMEOUT);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            seg_ku0 = nku;
        }
        lrb = nlrb;
        ku = nku;
        cur = nxt;
        sa = na;
        sb = nb;
    }
    ptx::cluster_sync();  // no block leaves while a store into its mailbox may be on the way
}


int64_t max_warps(const DeviceInfo& dev) { return (int64_t)dev.sms * kConsumers; }

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
    });
    return fn;
}

int scale_box(int group) { return kUnitK / group > 8 ? kUnitK / group : 8; }  // = kScaleBox<group>

size_t smem_bytes(size_t slot_bytes, bool xs, int64_t M, int64_t steps) {
    size_t b = 1024 + (size_t)kConsumers * kSlots * slot_bytes + ((sizeof(Bars) + 127) & ~(size_t)127);
    if (xs) b += (size_t)M * (size_t)(steps * kStepK * 2 + 64);
    return b;
}

template <int G, int NT, bool XS, bool TS, bool GT>
w4a16_status launch_one(const DeviceInfo& dev, const CUtensorMap (&map)[4], const GemvArgs& a, const GatedArgs& ga,
                        unsigned blocks, size_t smem, cudaStream_t st) {
    static PerDeviceOnce once;
    const cudaError_t attr = once.run(dev.device, [&dev] {
        const void* fn = GT ? reinterpret_cast<const void*>(gemv_gated_kernel<G, NT, XS, TS>)
                            : reinterpret_cast<const void*>(gemv_kernel<G, NT, XS, TS>);
        // the device's opt-in maximum (each launch checks its own size); the
        // shared-memory carveout stays the driver's choice (forcing the largest
        // cost 0.5 us per GEMV in the back-to-back decode step)
        return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev.smem_optin);
    });
    if (attr != cudaSuccess) return cuda_status(attr, "gemv: cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    const cudaError_t e = GT ? cudaLaunchKernelEx(&cfg, gemv_gated_kernel<G, NT, XS, TS>, map[0], map[1], map[2],
                                                  map[3], a, ga)
                             : cudaLaunchKernelEx(&cfg, gemv_kernel<G, NT, XS, TS>, map[0], map[1], a);
    return cuda_status(e, "gemv: kernel launch");
}

template <int G, int NT, bool GT>
w4a16_status launch_xt(const DeviceInfo& dev, const CUtensorMap (&map)[4], const GemvArgs& a, const GatedArgs& ga,
                       unsigned blocks, bool xs, bool ts, size_t smem, cudaStream_t st) {
    if (xs) return ts ? launch_one<G, NT, true, true, GT>(dev, map, a, ga, blocks, smem, st)
                      : launch_one<G, NT, true, false, GT>(dev, map, a, ga, blocks, smem, st);
    return ts ? launch_one<G, NT, false, true, GT>(dev, map, a, ga, blocks, smem, st)
              : launch_one<G, NT, false, false, GT>(dev, map, a, ga, blocks, smem, st);
}

template <int G, int NT>
w4a16_status launch_group(const DeviceInfo& dev, const CUtensorMap (&map)[4], const GemvArgs& a, const GatedArgs& ga,
                          unsigned blocks, bool xs, bool ts, bool gated, size_t smem, cudaStream_t st) {
    return gated ? launch_xt<G, NT, true>(dev, map, a, ga, blocks, xs, ts, smem, st)
                 : launch_xt<G, NT, false>(dev, map, a, ga, blocks, xs, ts, smem, st);
}

bool encode(CUtensorMap* map, CUtensorMapDataType type, const void* base, cuuint32_t rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(map, type, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Workspace layout: [partials, sized for the largest M, at offset 0][counters].
// The partial region has the same size for every call, so the counters of any
// call never overlap partial sums that an earlier call (any shape) left behind;
// each call leaves its counters at zero.
size_t partial_region_bytes(const DeviceInfo& dev) {
    return align256((size_t)max_warps(dev) * 2 * kRows * kMaxM * sizeof(float));
}

// Gated layout after the counters: [pair counters, one per row-block][gate and
// up fp32 results, [2][M][N]].
size_t gemv_workspace_bytes(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K, bool gated) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const int64_t RB = (N + kRows - 1) / kRows;
    size_t b = partial_region_bytes(dev) + align256((size_t)RB * (gated ? 2 : 1) * sizeof(int));
    if (gated) b += align256((size_t)RB * sizeof(int)) + align256((size_t)2 * M * N * sizeof(float));
    return b;
}

namespace {

// Clusters of 2 and of 4 blocks that are resident at once on a device (0 when
// none can be), found once per device; every instance of the cluster kernel
// has the same registers and block size, so one answer serves them all.
struct ClusterFit {
    int count[2];
};

// The opt-in shared-memory limit, for the instances that may need more than
// the default 48 KB (M > 1); the M = 1 instances (27 KB) keep the default.
template <int MX>
cudaError_t cluster_attrs(const DeviceInfo& dev) {
    if (MX == 1) return cudaSuccess;
    const void* fns[4] = {reinterpret_cast<const void*>(gemv_cluster_kernel<MX, true, 2>),
                          reinterpret_cast<const void*>(gemv_cluster_kernel<MX, false, 2>),
                          reinterpret_cast<const void*>(gemv_cluster_kernel<MX, true, 4>),
                          reinterpret_cast<const void*>(gemv_cluster_kernel<MX, false, 4>)};
    for (const void* fn : fns) {
        const cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev.smem_optin);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

const ClusterFit& cluster_fit(const DeviceInfo& dev, cudaError_t* err) {
    static ClusterFit fit[kMaxDevices];
    static PerDeviceOnce once;
    *err = once.run(dev.device, [&dev] {
        cudaError_t e = cluster_attrs<1>(dev);
        if (e == cudaSuccess) e = cluster_attrs<2>(dev);
        if (e == cudaSuccess) e = cluster_attrs<8>(dev);
        for (const void* fn : {reinterpret_cast<const void*>(gemv_decode_tokens_kernel<2, 8>),
                               reinterpret_cast<const void*>(gemv_decode_tokens_kernel<4, 8>),
                               reinterpret_cast<const void*>(gemv_decode_tokens_kernel<2, 16>),
                               reinterpret_cast<const void*>(gemv_decode_tokens_kernel<4, 16>)})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev.smem_optin);
        if (e != cudaSuccess) return e;
        for (int i = 0; i < 2; ++i) {
            const int c = 2 << i;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(dev.sms / c * c));
            cfg.blockDim = dim3(kCThreads);
            cfg.dynamicSmemBytes = CLayout<1>::kFixed + CLayout<1>::kXWarp;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)c;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int m = 0;
            const cudaError_t q = c == 2 ? cudaOccupancyMaxActiveClusters(&m, gemv_cluster_kernel<1, true, 2>, &cfg)
                                         : cudaOccupancyMaxActiveClusters(&m, gemv_cluster_kernel<1, true, 4>, &cfg);
            if (q != cudaSuccess) {
                (void)cudaGetLastError();  // not a sticky error: this cluster size is just not used
                m = 0;
            }
            fit[dev.device].count[i] = m;
        }
        return cudaSuccess;
    });
    return fit[dev.device];
}

template <int MX>
cudaError_t cluster_launch(const cudaLaunchConfig_t& cfg, const ClusterArgs& a, bool exact, int c) {
    if (c == 2)
        return exact ? cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<MX, true, 2>, a)
                     : cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<MX, false, 2>, a);
    return exact ? cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<MX, true, 4>, a)
                 : cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<MX, false, 4>, a);
}

// Launches the cluster kernel when it applies (group 128, M <= 8, one matrix,
// x within shared memory); *used is false when the caller must take the ring
// kernel instead.
w4a16_status cluster_run(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                         int64_t M, int64_t N, int64_t K, int group, bool static_weights, cudaStream_t st,
                         bool* used) {
    *used = false;
    if (group != 128 || M > 16) return W4A16_OK;  // 9..16 tokens: the decode kernel only
    const int64_t KU = (K + kUnitK - 1) / kUnitK, RB = (N + kRows - 1) / kRows;
    if (RB * KU > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const int mx = M == 1 ? 1 : M == 2 ? 2 : 8;
    size_t smem = 0;
    if (mx == 1) smem = CLayout<1>::kFixed + CLayout<1>::kXWarp;
    else if (mx == 2) smem = CLayout<2>::kFixed + CLayout<2>::kXWarp;
    else smem = CLayout<8>::kFixed + (size_t)M * (size_t)(KU * kUnitSteps * kStepK * 2 + 64);
    if (smem > dev.smem_optin && M <= 8) return W4A16_OK;
    cudaError_t e = cudaSuccess;
    const ClusterFit& fit = cluster_fit(dev, &e);
    if (e != cudaSuccess) return cuda_status(e, "gemv cluster: cudaFuncSetAttribute");
    // the cluster size whose busiest warp has the fewest units
    int c = 0, nc = 0;
    int64_t best = 0;
    for (int i = 0; i < 2; ++i) {
        const int ci = 2 << i, ni = fit.count[i];
        if (ni <= 0) continue;
        const int64_t per_warp = ((RB + ni - 1) / ni * KU + ci * kCWarps - 1) / (ci * kCWarps);
        if (c == 0 || per_warp < best) {
            c = ci;
            nc = ni;
            best = per_warp;
        }
    }
    if (c == 0) return W4A16_OK;
    ClusterArgs a;
    a.x = x;
    a.qw = qw;
    a.s = s;
    a.y = y;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.KU = (int)KU;
    a.RB = (int)RB;
    a.gpr = (int)(K / group);
    a.svec = a.gpr % 8 == 0;
    a.mode = static_weights ? kModeStatic : 0;
    a.err = dev.error_word;
    const bool exact = N % kRows == 0 && K % kUnitK == 0;  // then gpr % 4 == 0: a unit's scales are one 8-byte load
    // the decode kernel wants every warp of every cluster busy, no row-block
    // split over more than kMail + 1 of them, and (M > 1) the block's x in
    // shared memory
    const int64_t slice = (RB / nc) * KU / (c * kCWarps);  // the fewest units a warp gets
    const int mail = M == 1 ? kMail : DLayout<8>::kMail;
    const size_t xblock = (size_t)M * (size_t)(KU * kUnitSteps * kStepK * 2 + 64);
    const size_t dsmem = M == 1 ? kDecodeSmem : (M <= 8 ? DLayout<8>::kFixed : DLayout<16>::kFixed) + xblock;
    const bool decode = exact && slice >= 1 && (KU - 1 + slice - 1) / slice <= mail && dsmem <= dev.smem_optin;
    if (M > 8 && !decode) return W4A16_OK;  // the general kernel stops at 8 tokens
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nc * c));
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = decode ? dsmem : smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)c;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    *used = true;
    if (decode && M == 1)
        e = c == 2 ? cudaLaunchKernelEx(&cfg, gemv_decode_kernel<2>, a)
                   : cudaLaunchKernelEx(&cfg, gemv_decode_kernel<4>, a);
    else if (decode)
        e = M <= 8 ? (c == 2 ? cudaLaunchKernelEx(&cfg, gemv_decode_tokens_kernel<2, 8>, a)
                             : cudaLaunchKernelEx(&cfg, gemv_decode_tokens_kernel<4, 8>, a))
                   : (c == 2 ? cudaLaunchKernelEx(&cfg, gemv_decode_tokens_kernel<2, 16>, a)
                             : cudaLaunchKernelEx(&cfg, gemv_decode_tokens_kernel<4, 16>, a));
    else
        e = mx == 1 ? cluster_launch<1>(cfg, a, exact, c) : mx == 2 ? cluster_launch<2>(cfg, a, exact, c)
                                                                    : cluster_launch<8>(cfg, a, exact, c);
    return cuda_status(e, "gemv cluster: kernel launch");
}

// The fused gate+up decode on clusters when it applies (group 128, M = 1,
// N % 16 == 0, K % 512 == 0, the pair units spread so that every warp has
// one and no row-block has more than kGMail + 1 contributors); *used is false
// when the caller must take the ring kernel instead.
w4a16_status gated_cluster_run(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                               const uint8_t* qw2, const uint16_t* s2, uint16_t* y, int64_t M, int64_t N, int64_t K,
                               int group, bool static_weights, cudaStream_t st, bool* used) {
    *used = false;
    if (group != 128 || M != 1 || N % kRows != 0 || K % kUnitK != 0) return W4A16_OK;
    const int64_t KU = K / (kUnitK / 2), RB = N / kRows;  // 256-k pair units per row-block
    if (RB * KU > 0x7fffffffLL) return W4A16_OK;
    cudaError_t e = cudaSuccess;
    const ClusterFit& fit = cluster_fit(dev, &e);
    if (e != cudaSuccess) return cuda_status(e, "gemv cluster: cudaFuncSetAttribute");
    int c = 0, nc = 0;
    int64_t best = 0;
    for (int i = 0; i < 2; ++i) {
        const int ci = 2 << i, ni = fit.count[i];
        if (ni <= 0) continue;
        const int64_t slice = (RB / ni) * KU / (ci * kCWarps);
        if (slice < 1 || (KU - 1 + slice - 1) / slice > kGMail) continue;
        const int64_t per_warp = ((RB + ni - 1) / ni * KU + ci * kCWarps - 1) / (ci * kCWarps);
        if (c == 0 || per_warp < best) {
            c = ci;
            nc = ni;
            best = per_warp;
        }
    }
    if (c == 0) return W4A16_OK;
    GatedClusterArgs g;
    g.a.x = x;
    g.a.qw = qw;
    g.a.s = s;
    g.a.y = y;
    g.a.M = 1;
    g.a.N = (int)N;
    g.a.K = (int)K;
    g.a.KU = (int)KU;
    g.a.RB = (int)RB;
    g.a.gpr = (int)(K / group);
    g.a.svec = 1;
    g.a.mode = static_weights ? kModeStatic : 0;
    g.a.err = dev.error_word;
    g.qw2 = qw2;
    g.s2 = s2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nc * c));
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = kGatedDecodeSmem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)c;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    *used = true;
    e = c == 2 ? cudaLaunchKernelEx(&cfg, gemv_gated_decode_kernel<2>, g)
               : cudaLaunchKernelEx(&cfg, gemv_gated_decode_kernel<4>, g);
    return cuda_status(e, "gemv gated cluster: kernel launch");
}

bool encode_weights(CUtensorMap (&map)[4], int slot, const uint8_t* qw, const uint16_t* s, int64_t N, int64_t K,
                    int group, bool ts, bool* w3d) {
    const int64_t gpr = K / group;
    // the ring's weight boxes: one 3-D box per unit ([step][row][64 B] in shared
    // memory) when every 64-byte step piece lies inside its row, else four 2-D
    // boxes of 16 rows x 64 B; then the scales' 16-row boxes
    *w3d = false;
    if ((K / 2) % 64 == 0) {
        const cuuint64_t dims[3] = {64, (cuuint64_t)N, (cuuint64_t)(K / 128)};
        const cuuint64_t strides[2] = {(cuuint64_t)(K / 2), 64};
        const cuuint32_t box[3] = {64, (cuuint32_t)kRows, (cuuint32_t)kUnitSteps};
        *w3d = encode(&map[slot], CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, 3, dims, strides, box);
    }
    if (!*w3d) {
        const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        const cuuint32_t box[2] = {64, (cuuint32_t)kRows};
        if (!encode(&map[slot], CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, 2, dims, strides, box)) return false;
    }
    if (ts) {
        const cuuint64_t dims[2] = {(cuuint64_t)gpr, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)(gpr * 2)};
        const cuuint32_t box[2] = {(cuuint32_t)scale_box(group), (cuuint32_t)kRows};
        if (!encode(&map[slot + 1], CU_TENSOR_MAP_DATA_TYPE_UINT16, s, 2, dims, strides, box)) return false;
    }
    return true;
}

w4a16_status gemv_run(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                      const uint8_t* qw2, const uint16_t* s2, uint16_t* y, int64_t M, int64_t N, int64_t K, int group,
                      void* workspace, size_t workspace_bytes, const GemvOptions& opt, cudaStream_t st) {
    const bool gated = qw2 != nullptr;
    const size_t need = gemv_workspace_bytes(dev, M, N, K, gated);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return W4A16_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255) != 0) return W4A16_ERR_MISALIGNED;
    if (M > kMaxM || N > 0x7fffffffLL || K > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    {
        bool used = false;
        const w4a16_status r =
            gated ? gated_cluster_run(dev, x, qw, s, qw2, s2, y, M, N, K, group, opt.static_weights, st, &used)
                  : cluster_run(dev, x, qw, s, y, M, N, K, group, opt.static_weights, st, &used);
        if (used || r != W4A16_OK) return r;
    }
    if (!encode_fn()) return cuda_status(cudaErrorNotSupported, "gemv: cuTensorMapEncodeTiled entry point");
    const int64_t gpr = K / group;
    const bool ts = (gpr * 2) % 16 == 0;  // scale rows can be TMA boxes
    // [0, 1] weights and scales; [2, 3] the up projection's (gated), else a copy of [0, 1]
    CUtensorMap map[4];
    memset(map, 0, sizeof(map));
    bool w3d = false, w3d2 = false;
    if (!encode_weights(map, 0, qw, s, N, K, group, ts, &w3d) ||
        (gated && !encode_weights(map, 2, qw2, s2, N, K, group, ts, &w3d2)))
        return cuda_status(cudaErrorInvalidValue, "gemv: cuTensorMapEncodeTiled");
    if (!gated) {
        map[2] = map[0];
        map[3] = map[1];
        w3d2 = w3d;
    }
    if (w3d != w3d2) return W4A16_ERR_UNSUPPORTED;  // same shape, so the same choice
    GemvArgs a;
    a.x = x;
    a.s = s;
    a.y = y;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.KU = (K + kUnitK - 1) / kUnitK;
    const int64_t RB = (N + kRows - 1) / kRows;
    a.U = RB * (gated ? 2 : 1) * a.KU;
    if (a.U > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    int64_t blocks = (a.U + kConsumers - 1) / kConsumers;
    if (blocks > dev.sms) blocks = dev.sms;
    a.P = blocks * kConsumers < a.U ? blocks * kConsumers : a.U;
    char* ws = reinterpret_cast<char*>(workspace);
    a.partial = reinterpret_cast<float*>(ws);
    a.counter = reinterpret_cast<int*>(ws + partial_region_bytes(dev));
    a.err = dev.error_word;
    a.gpr = (int)gpr;
    a.svec = gpr % 8 == 0;
    a.mode = (w3d ? kMode3d : 0) | (opt.static_weights ? kModeStatic : 0);
    GatedArgs ga{s2, nullptr, nullptr};
    if (gated) {
        char* after = ws + partial_region_bytes(dev) + align256((size_t)RB * 2 * sizeof(int));
        ga.pair = reinterpret_cast<int*>(after);
        ga.gres = reinterpret_cast<float*>(after + align256((size_t)RB * sizeof(int)));
    }
    const size_t slot = (size_t)kWBytes + (ts ? (size_t)kRows * scale_box(group) * 2 : 0);
    const int64_t xsteps = a.KU * kUnitSteps;
    const size_t xbytes = (size_t)M * (size_t)(xsteps * kStepK * 2 + 64);
    const bool xs = xbytes <= kXSmemMax && smem_bytes(slot, true, M, xsteps) <= dev.smem_optin;
    const size_t smem = smem_bytes(slot, xs, M, xsteps);
    if (smem > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    const unsigned nb = (unsigned)blocks;
    if (M <= 8) {
        if (group == 128) return launch_group<128, 1>(dev, map, a, ga, nb, xs, ts, gated, smem, st);
        if (group == 64) return launch_group<64, 1>(dev, map, a, ga, nb, xs, ts, gated, smem, st);
        return launch_group<32, 1>(dev, map, a, ga, nb, xs, ts, gated, smem, st);
    }
    if (group == 128) return launch_group<128, 2>(dev, map, a, ga, nb, xs, ts, gated, smem, st);
    if (group == 64) return launch_group<64, 2>(dev, map, a, ga, nb, xs, ts, gated, smem, st);
    return launch_group<32, 2>(dev, map, a, ga, nb, xs, ts, gated, smem, st);
}

}  // namespace

w4a16_status gemv_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                         uint16_t* y, int64_t M, int64_t N, int64_t K, int group, void* workspace,
                         size_t workspace_bytes, const GemvOptions& opt, cudaStream_t st) {
    return gemv_run(dev, x, qw, s, nullptr, nullptr, y, M, N, K, group, workspace, workspace_bytes, opt, st);
}

w4a16_status gemv_gated_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw_gate,
                               const uint16_t* s_gate, const uint8_t* qw_up, const uint16_t* s_up, uint16_t* y,
                               int64_t M, int64_t N, int64_t K, int group, void* workspace, size_t workspace_bytes,
                               const GemvOptions& opt, cudaStream_t st) {
    if (qw_up == nullptr || s_up == nullptr) return W4A16_ERR_INVALID_ARG;
    return gemv_run(dev, x, qw_gate, s_gate, qw_up, s_up, y, M, N, K, group, workspace, workspace_bytes, opt, st);
}

#ifdef W4A16_TEST_HOOKS
cudaError_t gemv_set_test_hooks(const TestHooks& h) { return cudaMemcpyToSymbol(g_hooks, &h, sizeof(h)); }
#endif

}  // namespace w4a16
