// Decode GEMV for the W4A16 layer, M <= 16 activation rows (LLM170 page:
// "CUDA-graph decode", np4 = four sequences per step).
//
// Decode streams every packed weight byte once and does little arithmetic per
// byte: the kernel is bound by HBM bandwidth, and on the instruction budget
// of its dequantization. Design (one block of kConsumers warps per SM):
//
// * Work unit = 16 weight rows x 512 input features (4 KB packed). Units are
//   ordered row-block major, k minor; every consumer warp of a persistent
//   grid owns an equal contiguous range of them (stream-K split), so each SM
//   streams the same number of bytes whatever N and K are.
// * Every warp streams its units through a private ring of kSlots shared-
//   memory slots with TMA, refilling a slot as soon as it has consumed it (no
//   coupling between warps): a unit is four 16-row x 64-byte boxes issued back
//   to back, i.e. 256 contiguous bytes per weight row per unit. Slots are laid
//   out [k-step][row][64 B], so the fragment reads below are free of bank
//   conflicts.
// * The activations (M x K fp16, when small enough) are staged once per block
//   in shared memory, permuted into MMA fragment order, while the first weight
//   boxes are in flight; larger x is read through the L1.
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
// * Programmatic dependent launch: the block starts while the kernel before it
//   is still finishing. Until griddepcontrol.wait returns it only prefetches
//   the weights of its first units into L2 (L2 is the point of coherence, so
//   this is safe even if that kernel wrote them); after it, x is loaded first
//   and the ring's TMA loads then hit L2.
//
// Waits on the slot barriers are bounded in time; one that gives up records
// W4A16_ERR_TIMEOUT in the device error word and the block unwinds after its
// own TMA loads land.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kConsumers = 12;   // warps per block (one block per SM; 3 per scheduler)
constexpr int kThreads = kConsumers * 32;
constexpr int kSlots = 3;        // ring slots per consumer warp
constexpr int kStepK = 128;      // k per step (one 64-byte piece of a row)
constexpr int kUnitSteps = 4;    // steps per unit
constexpr int kUnitK = kStepK * kUnitSteps;
constexpr int kRows = 16;        // weight rows per unit
constexpr int kSlotBytes = kUnitSteps * kRows * 64;  // 4 KB
constexpr int kRingBytes = kConsumers * kSlots * kSlotBytes;
constexpr int kMaxM = 16;        // activation rows handled by the GEMV
constexpr size_t kXSmemMax = 80 * 1024;  // x staged in shared memory up to this size
constexpr int kXLoads = (int)((kXSmemMax / 16 + kThreads - 1) / kThreads);  // x loads per thread
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct GemvArgs {
    const uint16_t* x;
    const uint16_t* s;
    uint16_t* y;
    int M;
    int64_t N, K;
    int64_t KS;  // 128-k steps per row: ceil(K / 128)
    int64_t KU;  // 512-k units per row: ceil(K / 512)
    int64_t U;   // units: ceil(N / 16) * KU
    int64_t P;   // consumer warps taking part (each owns >= 1 unit)
    float* partial;  // [P][2][16 * M] fp32 partial sums (first / last segment)
    int* counter;    // [ceil(N/16)] arrivals per row-block, zero between calls
    unsigned int* err;
    int gpr;         // scale groups per row: K / G
    int svec;        // scale rows start 16-byte aligned (gpr % 8 == 0): whole units load as vectors
};

struct Bars {
    uint64_t full[kConsumers][kSlots];
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
// Shared-memory loads by 32-bit shared address (the offsets fold into the
// instruction); volatile keeps them after the barrier wait that guards them.
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
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

__device__ __forceinline__ ScaleRows scale_rows(const GemvArgs& p, int rb, int gid) {
    const int64_t n0 = (int64_t)rb * kRows + gid, n1 = n0 + 8;
    ScaleRows r;
    r.v0 = n0 < p.N;
    r.v1 = n1 < p.N;
    r.r0 = p.s + (r.v0 ? n0 : 0) * p.gpr;
    r.r1 = p.s + (r.v1 ? n1 : 0) * p.gpr;
    return r;
}

template <int G>
__device__ __forceinline__ void load_scales(UnitScales<G>& sc, const GemvArgs& p, const ScaleRows& sr, int ku) {
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

__device__ __forceinline__ float half_bits(uint32_t w, int h) {
    return __half2float(__ushort_as_half((unsigned short)(h ? (w >> 16) : (w & 0xffffu))));
}

// One unit from its ring slot: for every 128-k step and scale group, the
// quad's share of rows gid and gid+8. `wlane` is the shared address of this
// lane's first weight bytes in the slot (row gid, its quad's offset). XS: x
// comes from shared memory at xlane[t] (this lane's 16-byte chunk of the
// unit's x for token 8t+gid, or of the zero block for lanes without a token),
// so no load is predicated and every offset below is a constant.
template <int G, int NT, bool XS>
__device__ __forceinline__ void compute_unit(uint32_t wlane, const UnitScales<G>& sc, const GemvArgs& p,
                                             const uint32_t (&xlane)[NT], int ku, int gid, int t4,
                                             float (&acc)[NT][4]) {
    constexpr int WPP = G / 32;      // words per thread per row per group
    constexpr int GPS = kStepK / G;  // groups per step
#pragma unroll
    for (int step = 0; step < kUnitSteps; ++step) {
#pragma unroll
        for (int j = 0; j < GPS; ++j) {
            uint32_t wa[WPP], wb[WPP];
            const uint32_t ra = wlane + step * (kRows * 64) + j * (G / 2);
            const uint32_t rbp = ra + 8 * 64;
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
template <int NT>
__device__ __noinline__ void publish_partial(const GemvArgs& p, int64_t w, int slot, int64_t rb,
                                             const float (&acc)[NT][4], int gid, int t4, int lane) {
    store_partial<NT>(p, w, slot, acc, gid, t4);
    __syncwarp();  // the lanes' stores happen before lane 0's release
    int old = 0;
    if (lane == 0) old = ptx::atom_add_acq_rel_gpu(p.counter + rb, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int64_t wa = warp_of_unit(rb * p.KU, p);
    const int64_t wb = warp_of_unit(rb * p.KU + p.KU - 1, p);
    if ((int64_t)old != wb - wa) return;  // another warp finishes this row-block
    const int64_t slot_elems = (int64_t)kRows * p.M;
    float sum[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) sum[t][0] = sum[t][1] = sum[t][2] = sum[t][3] = 0.0f;
    for (int64_t v = wa; v <= wb; ++v) {
        // rb is the first segment of every contributor except possibly wa
        const bool wa_started_inside = (v * p.U / p.P) == rb * p.KU;
        const int sl = (v == wa && !wa_started_inside) ? 1 : 0;
        const float* src = p.partial + (v * 2 + sl) * slot_elems;
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * t + 2 * t4 + (i & 1);
                if (m < p.M) sum[t][i] += __ldcg(src + m * kRows + gid + 8 * (i >> 1));
            }
    }
    store_y<NT>(p, rb, sum, gid, t4);
    if (lane == 0) p.counter[rb] = 0;
}

template <int G, int NT, bool XS>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmap_w, const GemvArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Bars* bars = reinterpret_cast<Bars*>(ring + kRingBytes);
    uint8_t* xs = reinterpret_cast<uint8_t*>(bars) + ((sizeof(Bars) + 127) & ~(size_t)127);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int64_t xsteps = p.KU * kUnitSteps;             // staged steps per token (whole units)
    const int64_t xstride = xsteps * (kStepK * 2) + 64;  // bytes per token row of staged x
    volatile int* abort = &bars->abort;

    if (threadIdx.x == 0) {
        for (int w = 0; w < kConsumers; ++w)
            for (int sl = 0; sl < kSlots; ++sl) ptx::mbar_init(&bars->full[w][sl], 1);
        bars->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&tmap_w);
    }
    if (threadIdx.x < 64) reinterpret_cast<uint4*>(bars->zero)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    // unit range of every consumer warp of this block
    auto range = [&](int cw, int64_t& ub, int64_t& ue) {
        const int64_t w = (int64_t)blockIdx.x * kConsumers + cw;
        ub = w < p.P ? w * p.U / p.P : 0;
        ue = w < p.P ? (w + 1) * p.U / p.P : 0;
    };
    auto issue = [&](int cw, int64_t rb, int64_t ku, int sl) {  // one unit: four 16-row x 64-byte boxes
        uint64_t* bar = &bars->full[cw][sl];
        uint8_t* dst = ring + (cw * kSlots + sl) * kSlotBytes;
        ptx::mbar_arrive_expect_tx(bar, kSlotBytes);
#pragma unroll
        for (int step = 0; step < kUnitSteps; ++step)
            ptx::tma_load_2d(dst + step * (kRows * 64), &tmap_w, bar, (int)((ku * kUnitSteps + step) * 64),
                             (int)(rb * kRows));
    };

    const int cw = warp;
    int64_t u_begin, u_end;
    range(cw, u_begin, u_end);
    // refill cursor: the next unit to load into this warp's ring
    int64_t f_rb = u_begin / p.KU, f_ku = u_begin % p.KU;
    auto advance = [&](int64_t& rb_, int64_t& ku_) {
        if (++ku_ == p.KU) {
            ku_ = 0;
            ++rb_;
        }
    };
    // Every input, the weights included, may come from the kernel before this
    // one on the stream, which may still be running: until griddepcontrol.wait
    // returns, the first units of this warp are only prefetched into L2.
    if (lane == 0) {
        int64_t rb_ = f_rb, ku_ = f_ku;
        for (int r = 0; r < kSlots && u_begin + r < u_end; ++r) {
#pragma unroll
            for (int step = 0; step < kUnitSteps; ++step)
                ptx::tma_prefetch_l2_2d(&tmap_w, (int)((ku_ * kUnitSteps + step) * 64), (int)(rb_ * kRows));
            advance(rb_, ku_);
        }
    }
    ptx::grid_dependency_wait();
    // x loads first (every unit waits for them), then the ring, then the x stores
    const int64_t chunks = XS ? (int64_t)p.M * xsteps * 16 : 0;  // 16-byte chunks, zero past K
    uint4 xv[XS ? kXLoads : 1];
    if (XS) {
#pragma unroll
        for (int i = 0; i < kXLoads; ++i) {
            const int64_t c = threadIdx.x + i * kThreads;
            xv[i] = make_uint4(0, 0, 0, 0);
            if (c < chunks) {
                const int64_t m = c / (xsteps * 16), k0 = (c % (xsteps * 16)) * 8;
                if (k0 < p.K) xv[i] = ld_l2_v4(p.x + m * p.K + k0);
            }
        }
    }
    for (int r = 0; r < kSlots && u_begin + r < u_end; ++r) {
        if (lane == 0) issue(cw, f_rb, f_ku, r);
        advance(f_rb, f_ku);
    }
    if (XS) {
#pragma unroll
        for (int i = 0; i < kXLoads; ++i) {
            const int64_t c = threadIdx.x + i * kThreads;
            if (c < chunks) {
                const int64_t m = c / (xsteps * 16), cc = c % (xsteps * 16);
                *reinterpret_cast<uint4*>(xs + m * xstride + (cc >> 4) * (kStepK * 2) +
                                          xs_pos((int)(cc & 15), G) * 16) = permute_x8(xv[i]);
            }
        }
        __syncthreads();
    }

    // ------------------------------------------------------------ consumers
    const int64_t w = (int64_t)blockIdx.x * kConsumers + cw;
    if (w >= p.P) return;

    const int n_units = (int)(u_end - u_begin);
    int rb = (int)(u_begin / p.KU), ku = (int)(u_begin % p.KU);
    const int first_rb = rb, KU = (int)p.KU;
    int seg_ku0 = ku;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    ScaleRows sr = scale_rows(p, rb, gid);
    UnitScales<G> sc;
    load_scales<G>(sc, p, sr, ku);
    // shared address of this lane's x chunk in unit 0 (the zero block for lanes
    // without a token) and its stride per unit
    uint32_t xlane0[NT], xunit[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const bool has = 8 * t + gid < p.M;
        xlane0[t] = (has ? ptx::smem_u32(xs) + (8 * t + gid) * (uint32_t)xstride : ptx::smem_u32(bars->zero)) + t4 * 16;
        xunit[t] = has ? kUnitSteps * kStepK * 2 : 0;
    }
    const uint32_t wlane0 = ptx::smem_u32(ring) + cw * (kSlots * kSlotBytes) + gid * 64 + t4 * (G / 8);

    int sl = 0;
    uint32_t phase = 0;
    for (int r = 0; r < n_units; ++r) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars->full[cw][sl], phase, abort, kWaitLimitNs))) {
            raise_device_error(p.err, W4A16_ERR_TIMEOUT);
            *abort = 1;
            if (lane == 0) {  // this warp's own loads still in flight land before it exits
                volatile int never = 0;
                for (int q = r + 1; q < r + kSlots && q < n_units; ++q)
                    ptx::mbar_wait(&bars->full[cw][q % kSlots], (uint32_t)((q / kSlots) & 1), &never, kWaitLimitNs);
            }
            return;
        }
        int nrb = rb, nku = ku + 1;
        if (nku == KU) {
            nku = 0;
            ++nrb;
        }
        const ScaleRows nsr = nku == 0 ? scale_rows(p, nrb, gid) : sr;
        UnitScales<G> sc_next;
        if (r + 1 < n_units) load_scales<G>(sc_next, p, nsr, nku);
        uint32_t xlane[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) xlane[t] = xlane0[t] + ku * xunit[t];
        compute_unit<G, NT, XS>(wlane0 + sl * kSlotBytes, sc, p, xlane, ku, gid, t4, acc);
        __syncwarp();  // every lane has read the slot
        if (r + kSlots < n_units) {
            if (lane == 0) issue(cw, f_rb, f_ku, sl);
            advance(f_rb, f_ku);
        }
        if (r + 1 < n_units) sc = sc_next;
        sr = nsr;

        const bool seg_end = (ku == KU - 1) || (r == n_units - 1);
        if (seg_end) {
            if (r == n_units - 1) ptx::launch_dependents();  // only the epilogue of this warp remains
            if (seg_ku0 == 0 && ku == KU - 1)
                store_y<NT>(p, rb, acc, gid, t4);  // whole row-block in this warp
            else  // partial: published now, so its latency overlaps the units that follow
                publish_partial<NT>(p, w, rb == first_rb ? 0 : 1, rb, acc, gid, t4, lane);
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

size_t smem_bytes(bool xs, int64_t M, int64_t steps) {
    size_t b = 1024 + kRingBytes + ((sizeof(Bars) + 127) & ~(size_t)127);
    if (xs) b += (size_t)M * (size_t)(steps * kStepK * 2 + 64);
    return b;
}

template <int G, int NT, bool XS>
w4a16_status launch_one(const DeviceInfo& dev, const CUtensorMap& map, const GemvArgs& a, unsigned blocks,
                        size_t smem, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&dev] {  // the device's opt-in maximum; each launch checks its own size
        attr = cudaFuncSetAttribute(gemv_kernel<G, NT, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)dev.smem_optin);
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
    return cuda_status(cudaLaunchKernelEx(&cfg, gemv_kernel<G, NT, XS>, map, a), "gemv: kernel launch");
}

}  // namespace

// Workspace layout: [partials, sized for the largest M, at offset 0][counters].
// The partial region has the same size for every call, so the counters of any
// call never overlap partial sums that an earlier call (any shape) left behind;
// each call leaves its counters at zero.
size_t partial_region_bytes(const DeviceInfo& dev) {
    return align256((size_t)max_warps(dev) * 2 * kRows * kMaxM * sizeof(float));
}

size_t gemv_workspace_bytes(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const int64_t RB = (N + kRows - 1) / kRows;
    return partial_region_bytes(dev) + align256((size_t)RB * sizeof(int));
}

w4a16_status gemv_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                         uint16_t* y, int64_t M, int64_t N, int64_t K, int group, void* workspace,
                         size_t workspace_bytes, cudaStream_t st) {
    const size_t need = gemv_workspace_bytes(dev, M, N, K);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return W4A16_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255) != 0) return W4A16_ERR_MISALIGNED;
    if (M > kMaxM || N > 0x7fffffffLL || K / 2 > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cuda_status(cudaErrorNotSupported, "gemv: cuTensorMapEncodeTiled entry point");
    CUtensorMap map;
    {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        cuuint32_t box[2] = {64, (cuuint32_t)kRows};
        cuuint32_t es[2] = {1, 1};
        if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_status(cudaErrorInvalidValue, "gemv: cuTensorMapEncodeTiled");
    }
    GemvArgs a;
    a.x = x;
    a.s = s;
    a.y = y;
    a.M = (int)M;
    a.N = N;
    a.K = K;
    a.KS = (K + kStepK - 1) / kStepK;
    a.KU = (K + kUnitK - 1) / kUnitK;
    const int64_t RB = (N + kRows - 1) / kRows;
    a.U = RB * a.KU;
    int64_t blocks = (a.U + kConsumers - 1) / kConsumers;
    if (blocks > dev.sms) blocks = dev.sms;
    a.P = blocks * kConsumers < a.U ? blocks * kConsumers : a.U;
    a.partial = reinterpret_cast<float*>(workspace);
    a.counter = reinterpret_cast<int*>(reinterpret_cast<char*>(workspace) + partial_region_bytes(dev));
    a.err = dev.error_word;
    a.gpr = (int)(K / group);
    a.svec = (K / group) % 8 == 0;
    const int64_t xsteps = a.KU * kUnitSteps;
    const size_t xbytes = (size_t)M * (size_t)(xsteps * kStepK * 2 + 64);
    const bool xs = xbytes <= kXSmemMax && smem_bytes(true, M, xsteps) <= dev.smem_optin;
    const size_t smem = smem_bytes(xs, M, xsteps);
    if (smem > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    const int nt = M <= 8 ? 1 : 2;
    w4a16_status r = W4A16_OK;
#define W4A16_GEMV(G_, NT_)                                                           \
    r = xs ? launch_one<G_, NT_, true>(dev, map, a, (unsigned)blocks, smem, st)       \
           : launch_one<G_, NT_, false>(dev, map, a, (unsigned)blocks, smem, st)
    if (nt == 1) {
        if (group == 128) W4A16_GEMV(128, 1);
        else if (group == 64) W4A16_GEMV(64, 1);
        else W4A16_GEMV(32, 1);
    } else {
        if (group == 128) W4A16_GEMV(128, 2);
        else if (group == 64) W4A16_GEMV(64, 2);
        else W4A16_GEMV(32, 2);
    }
#undef W4A16_GEMV
    return r;
}

}  // namespace w4a16
