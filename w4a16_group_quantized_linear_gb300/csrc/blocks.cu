// GGUF block-format weights: the decode GEMV y = x * W^T and the dequantizer.
//
// The formats are two of the GGUF block types the infr README lists among its
// validated formats ("Also validated for correctness": on-device decode
// byte-identical to the CPU dequant; footnote 3: routed expert banks stored as
// Q5_1) and the LLM170 README's status names ("q5_1 down", "q4_K" tiles).
// Their layouts are ggml's block types as GGUF files carry them:
//
//   Q4_K  256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes of 6-bit
//         sub-block scales sc[8] and minimums mn[8], 128 bytes of nibbles;
//         weight 64c + l (l < 32) is the low nibble of qs[32c + l], weight
//         64c + 32 + l its high nibble; W^ = d sc[i/32] q - dmin mn[i/32].
//   Q5_1  32 weights in 24 bytes: fp16 d, fp16 m, 32 fifth bits qh, 16 bytes
//         of nibbles (weight i < 16: low nibble of byte i, else high nibble
//         of byte i - 16; bit i of qh on top); W^ = d q + m.
//
// GEMV design. A warp's unit is 256 k of 16 weight rows (Q4_K: one block a
// row) or of 8 rows (Q5_1: eight blocks a row). Each warp copies its units
// with cp.async into a ring of three stages in shared memory, two units ahead
// of the one it computes; each lane reads its pieces of a stage and turns
// nibbles into exact fp16 integers. mma.sync m16n8k16 takes them as A and up
// to 8 tokens of x as B; an A of constant ones (a second mma for Q4_K, A rows
// 8-15 for Q5_1) gives the sums X = sum x over
// each 32-weight sub-block beside the integer dot products S = sum x q, so the
// sub-block adds a S + b X (W^ = a q + b) in fp32 with no extra pass over x.
// The grid is persistent: each thread-block cluster (1 to 8 blocks of 8 warps)
// owns a run of whole row-blocks and its warps stream equal shares of their
// units; the partial sums meet in the shared memory of the cluster's first
// block and are added in a fixed order, so results are deterministic.
#include <type_traits>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr int kBWarps = 8;             // warps per block
constexpr int kBThreads = kBWarps * 32;
constexpr int kBUnitK = 256;           // k per unit
constexpr int kBTokens = 8;            // tokens per launch


__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    return __byte_perm(a, b, sel);
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                        *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
}

constexpr uint32_t kMagic = 0x64006400u;     // fp16 1024 in both halves
constexpr uint32_t k1024 = 0x64006400u;      // 1024
constexpr uint32_t kSixteenth = 0x2C002C00u; // 1/16
constexpr uint32_t kMinus64 = 0xD400D400u;   // -64
constexpr uint32_t kOnes = 0x3C003C00u;      // 1.0

// Byte e of a uint32 as an exact float: the byte becomes the low mantissa
// bits of 2^23 and 2^23 is subtracted.
__device__ __forceinline__ float byte_to_float(uint32_t v, int e) {
    const uint32_t f = __byte_perm(v, 0x4B000000u, 0x7650u | (uint32_t)e);
    return __uint_as_float(f) - 8388608.0f;
}

// x fragments for one 16-k step: b0 = (x[k0], x[k0+2]), b1 = (x[k0+1], x[k0+3])
// from the four consecutive fp16 values in (u0, u1); this pairs with A
// registers built from bytes (0, 2) and (1, 3) of a 32-bit weight word.
__device__ __forceinline__ void x_pairs(uint32_t u0, uint32_t u1, uint32_t& b0, uint32_t& b1) {
    b0 = prmt(u0, u1, 0x5410);
    b1 = prmt(u0, u1, 0x7632);
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Stores into the shared memory of another block of the cluster.
__device__ __forceinline__ void st_cluster_f32(uint32_t caddr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}

// ------------------------------------------------------------------ Q4_K --
// A Q4_K unit is 16 rows x 256 k: the lane holds rows gid and gid + 8 (A rows
// of one mma); a second mma with constant-one A rows gives the sub-block sums
// of x.

struct Q4KRow {
    uint4 head;      // d, dmin, 12 scale bytes
    uint2 qs[4];     // bytes 8 t4 .. 8 t4 + 7 of each 32-byte chunk
};
struct Q4KUnit {
    Q4KRow r[2];     // rows gid and gid + 8
};

// Scale (sc) and minimum (mn) bytes of a row's eight sub-blocks: j < 4 in the
// low six bits of scale bytes 0-3 and 4-7; j >= 4 low four bits from bytes
// 8-11, top two bits from the top of bytes 0-3 (sc) and 4-7 (mn).
struct Q4KScales {
    uint32_t s03, m03, s47, m47;
};

__device__ __forceinline__ Q4KScales q4k_scales(const uint4& h) {
    Q4KScales q;
    q.s03 = h.y & 0x3F3F3F3Fu;
    q.m03 = h.z & 0x3F3F3F3Fu;
    q.s47 = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    q.m47 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    return q;
}

// Nibbles of bytes (0, 2) and (1, 3) of w (low or high nibbles) as exact fp16 pairs.
template <int HI>
__device__ __forceinline__ void q4_pairs(uint32_t w, uint32_t w8, uint32_t& p02, uint32_t& p13) {
    if (HI) {
        p02 = hfma2_u32(lop3_and_or(w, 0x00F000F0u, kMagic), kSixteenth, kMinus64);
        p13 = hfma2_u32(lop3_and_or(w8, 0x00F000F0u, kMagic), kSixteenth, kMinus64);
    } else {
        p02 = hsub2_u32(lop3_and_or(w, 0x000F000Fu, kMagic), k1024);
        p13 = hsub2_u32(lop3_and_or(w8, 0x000F000Fu, kMagic), k1024);
    }
}

// One Q4_K unit: acc[r][t] (row gid + 8 r, token 2 t4 + t) += sum over the
// unit's 256 k of x W^.
__device__ __forceinline__ void compute_unit(const Q4KUnit& u, const uint16_t* xk, float (&acc)[2][2]) {
    const Q4KScales q0 = q4k_scales(u.r[0].head), q1 = q4k_scales(u.r[1].head);
    float sacc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}}, macc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // x for sub-blocks 2c (low nibbles) and 2c + 1 (high nibbles): eight
        // consecutive values each, at 32 j + 8 t4
        const uint4 xl = *reinterpret_cast<const uint4*>(xk + 64 * c);
        const uint4 xh = *reinterpret_cast<const uint4*>(xk + 64 * c + 32);
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            const uint4 xv = hi ? xh : xl;
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f}, xs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const uint32_t w0 = s ? u.r[0].qs[c].y : u.r[0].qs[c].x;
                const uint32_t w1 = s ? u.r[1].qs[c].y : u.r[1].qs[c].x;
                uint32_t a0, a1, a2, a3;
                if (hi) {
                    q4_pairs<1>(w0, w0 >> 8, a0, a2);
                    q4_pairs<1>(w1, w1 >> 8, a1, a3);
                } else {
                    q4_pairs<0>(w0, w0 >> 8, a0, a2);
                    q4_pairs<0>(w1, w1 >> 8, a1, a3);
                }
                uint32_t b0, b1;
                x_pairs(s ? xv.z : xv.x, s ? xv.w : xv.y, b0, b1);
                mma_16816(d, a0, a1, a2, a3, b0, b1);
                mma_16816(xs, kOnes, kOnes, kOnes, kOnes, b0, b1);
            }
            const int j = 2 * c + hi, e = j & 3;
            const float sc0 = byte_to_float(j < 4 ? q0.s03 : q0.s47, e), mn0 = byte_to_float(j < 4 ? q0.m03 : q0.m47, e);
            const float sc1 = byte_to_float(j < 4 ? q1.s03 : q1.s47, e), mn1 = byte_to_float(j < 4 ? q1.m03 : q1.m47, e);
            sacc[0][0] = fmaf(sc0, d[0], sacc[0][0]);
            sacc[0][1] = fmaf(sc0, d[1], sacc[0][1]);
            sacc[1][0] = fmaf(sc1, d[2], sacc[1][0]);
            sacc[1][1] = fmaf(sc1, d[3], sacc[1][1]);
            macc[0][0] = fmaf(mn0, xs[0], macc[0][0]);
            macc[0][1] = fmaf(mn0, xs[1], macc[0][1]);
            macc[1][0] = fmaf(mn1, xs[0], macc[1][0]);
            macc[1][1] = fmaf(mn1, xs[1], macc[1][1]);
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float2 df = __half22float2(*reinterpret_cast<const __half2*>(&u.r[r].head.x));   // (d, dmin)
        acc[r][0] = fmaf(df.x, sacc[r][0], fmaf(-df.y, macc[r][0], acc[r][0]));
        acc[r][1] = fmaf(df.x, sacc[r][1], fmaf(-df.y, macc[r][1], acc[r][1]));
    }
}

// ------------------------------------------------------------------ Q5_1 --

struct Q51Unit {
    uint2 head[8];   // d, m, qh of each of the row's eight blocks
    uint32_t qs[8];  // bytes 4 t4 .. 4 t4 + 3 of each block's nibbles
};

// Two fp16 pairs (bytes 0, 2) and (bytes 1, 3) of the nibbles in v (bits
// 0-3 of each byte) with fifth bits f (bit e = byte e's), as exact integers.
__device__ __forceinline__ void q5_pairs(uint32_t v, uint32_t f, uint32_t& p02, uint32_t& p13) {
    // bit 0 of f to bit 4 and bit 2 to bit 20; bit 1 to bit 4 and bit 3 to bit 20
    const uint32_t f02 = lop3_and_or(f * 0x00040010u, 0x00100010u, kMagic);
    const uint32_t f13 = lop3_and_or(f * 0x00020008u, 0x00100010u, kMagic);
    p02 = hsub2_u32(lop3_and_or(v, 0x000F000Fu, f02), k1024);
    p13 = hsub2_u32(lop3_and_or(v >> 8, 0x000F000Fu, f13), k1024);
}

__device__ __forceinline__ void compute_unit(const Q51Unit& r, const uint16_t* xk, int t4, int nb,
                                             float (&acc)[2]) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        uint2 xl = make_uint2(0, 0), xh = make_uint2(0, 0);
        if (b < nb) {
            xl = *reinterpret_cast<const uint2*>(xk + 32 * b);        // weights 4 t4 .. + 3
            xh = *reinterpret_cast<const uint2*>(xk + 32 * b + 16);   // weights 16 + 4 t4 .. + 3
        }
        const uint32_t qh = r.head[b].y;
        const uint32_t flo = (qh >> (4 * t4)) & 0xFu, fhi = (qh >> (16 + 4 * t4)) & 0xFu;
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t a0, a2, b0, b1;
        q5_pairs(r.qs[b], flo, a0, a2);
        x_pairs(xl.x, xl.y, b0, b1);
        mma_16816(d, a0, kOnes, a2, kOnes, b0, b1);
        q5_pairs(r.qs[b] >> 4, fhi, a0, a2);
        x_pairs(xh.x, xh.y, b0, b1);
        mma_16816(d, a0, kOnes, a2, kOnes, b0, b1);
        const __half2 dm = *reinterpret_cast<const __half2*>(&r.head[b].x);
        const float2 f = __half22float2(dm);   // (d, m)
        acc[0] = fmaf(f.x, d[0], fmaf(f.y, d[2], acc[0]));
        acc[1] = fmaf(f.x, d[1], fmaf(f.y, d[3], acc[1]));
    }
}

// ---------------------------------------------------------------- kernel --

template <int FMT>
struct Fmt;
template <>
struct Fmt<W4A16_FORMAT_Q4_K> {
    using Unit = Q4KUnit;
    static constexpr int kRows = 16;       // rows per row-block (two per lane)
    static constexpr int kUnitBytes = 144; // bytes of a unit in one row
    static constexpr int kPiece = 16;      // bytes per cp.async
    static constexpr int kStride = 160;    // shared-memory bytes per row of a stage (conflict-free 8-byte reads)
    static constexpr int kXStep = 8;       // x offset of lane t4 inside a sub-block, per t4
};
template <>
struct Fmt<W4A16_FORMAT_Q5_1> {
    using Unit = Q51Unit;
    static constexpr int kRows = 8;        // one row per lane, constant ones in A rows 8-15
    static constexpr int kUnitBytes = 192;
    static constexpr int kPiece = 8;       // rows of 24-byte blocks need not start 16-byte aligned
    static constexpr int kStride = 208;
    static constexpr int kXStep = 4;
};

constexpr int kStages = 3;   // units in flight per warp (a ring in shared memory)

template <int FMT>
constexpr int stage_bytes() {
    return Fmt<FMT>::kRows * Fmt<FMT>::kStride;
}

__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src, uint32_t src_size) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_size) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
}

// The lane's part of a unit from its shared-memory stage (rows kStride apart).
__device__ __forceinline__ void read_unit(Q4KUnit& u, uint32_t st, int gid, int t4) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const uint32_t row = st + (uint32_t)(gid + 8 * r) * Fmt<W4A16_FORMAT_Q4_K>::kStride;
        u.r[r].head = lds128(row);
#pragma unroll
        for (int c = 0; c < 4; ++c) u.r[r].qs[c] = lds64(row + 16 + 32 * c + 8 * t4);
    }
}
__device__ __forceinline__ void read_unit(Q51Unit& u, uint32_t st, int gid, int t4) {
    const uint32_t row = st + (uint32_t)gid * Fmt<W4A16_FORMAT_Q5_1>::kStride;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        u.head[b] = lds64(row + 24 * b);
        u.qs[b] = lds32(row + 24 * b + 8 + 4 * t4);
    }
}

// Work split. Row-block r covers rows [kRows r, kRows (r + 1)); its units are
// the KU = ceil(K / 256) stretches of 256 k. Cluster cl owns the row-blocks
// [nrb cl / ncl, nrb (cl + 1) / ncl) and lists their units row-block by
// row-block; warp v of the cluster's V takes the contiguous run [T v / V,
// T (v + 1) / V) of that list (T units), so every warp streams the same
// number of units, give or take one, across row-block boundaries. Each run
// leaves one partial sum per row-block it touches (at most J) in the shared
// memory of the cluster's first block.
struct StreamArgs {
    const uint16_t* x;   // fp16 [M, K]
    const uint8_t* w;    // blocks [N, row_bytes]
    uint16_t* y;         // fp16 [M, N]
    int64_t N, K, row_bytes;
    int M;               // tokens of this launch, 1..8
    int KU;              // units per row-block
    int tail;            // Q5_1 blocks in a row's last unit (8 when K % 256 == 0)
    int64_t rb_first;    // first row-block of this launch
    int nrb, ncl, J;     // row-blocks, clusters, partial slots per warp
};

__host__ __device__ __forceinline__ int64_t run_begin(int64_t T, int v, int V) { return T * v / V; }

template <int FMT, int C>
__global__ void __launch_bounds__(kBThreads, 2) blocks_gemv_kernel(const StreamArgs a) {
    using F = Fmt<FMT>;
    constexpr int RL = F::kRows / 8;   // rows per lane
    constexpr int V = C * kBWarps;
    // [V][J][32][2 RL] partial sums (used in the cluster's first block), then
    // each warp's ring of weight stages
    extern __shared__ __align__(16) float part[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, t4 = lane & 3;
    const int rank = C > 1 ? (int)cluster_rank() : 0;
    const int cl = blockIdx.x / C;
    const int64_t rb0 = a.rb_first + (int64_t)cl * a.nrb / a.ncl, rb1 = a.rb_first + (int64_t)(cl + 1) * a.nrb / a.ncl;
    const int64_t T = (rb1 - rb0) * a.KU;
    const int v = rank * kBWarps + warp;
    const int64_t i0 = run_begin(T, v, V), i1 = run_begin(T, v + 1, V);
    const int KU = a.KU;
    // the lane's x: token gid, at kXStep * t4 inside each sub-block. Lanes past
    // the last token read the last token instead: their columns of the
    // product are never stored, and no load is predicated.
    const int tok = gid < a.M ? gid : a.M - 1;
    const uint16_t* xrow = a.x + (int64_t)tok * a.K + F::kXStep * t4;
    // this lane's first partial slot, in the shared memory of the cluster's first block
    const uint32_t own = (uint32_t)(v * a.J * 32 + lane) * (8 * RL);
    const uint32_t part_base = (C > 1 ? cluster_map(smem_u32(part), 0) : smem_u32(part)) + own;

    // weights: a ring of kStages units per warp in shared memory, filled by
    // cp.async kStages - 1 units ahead of the unit being computed; the load
    // position (row-block lr, unit ls) runs ahead of the compute position (cr, cs)
    const uint32_t ring = smem_u32(part) + (uint32_t)a.J * V * 32 * (8 * RL) +
                          (uint32_t)(warp * kStages) * stage_bytes<FMT>();
    int lr = (int)(i0 / KU), ls = (int)(i0 % KU);
    int cr = lr, cs = ls;
    const int first = cr;
    constexpr int P = F::kUnitBytes / F::kPiece;   // pieces per row of a unit
    auto issue = [&](int stage) {
        const uint32_t dst0 = ring + (uint32_t)stage * stage_bytes<FMT>();
        const int valid = FMT == W4A16_FORMAT_Q4_K ? F::kUnitBytes : (ls == KU - 1 ? a.tail : 8) * 24;
#pragma unroll
        for (int i = 0; i < (F::kRows * P + 31) / 32; ++i) {
            const int idx = i * 32 + lane;
            if (idx < F::kRows * P) {
                const int r = idx / P, pc = idx % P;
                const int64_t row = (rb0 + lr) * F::kRows + r;
                const bool ok = row < a.N && pc * F::kPiece < valid;
                const uint8_t* src = a.w + (ok ? row * a.row_bytes + (int64_t)ls * F::kUnitBytes + pc * F::kPiece : 0);
                const uint32_t dst = dst0 + (uint32_t)(r * F::kStride + pc * F::kPiece);
                if constexpr (F::kPiece == 16)
                    cp_async_16(dst, src, ok ? 16u : 0u);
                else
                    cp_async_8(dst, src, ok ? 8u : 0u);
            }
        }
        if (++ls == KU) {
            ls = 0;
            ++lr;
        }
    };
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (i0 + i < i1) issue(i);
        cp_async_commit();
    }
    float acc[RL][2] = {};
    int stage = 0;
    for (int64_t i = i0; i < i1; ++i) {
        if (i + kStages - 1 < i1) issue(stage == 0 ? kStages - 1 : stage - 1);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncwarp();
        typename F::Unit u;
        read_unit(u, ring + (uint32_t)stage * stage_bytes<FMT>(), gid, t4);
        __syncwarp();   // the stage is refilled next round
        if constexpr (FMT == W4A16_FORMAT_Q4_K)
            compute_unit(u, xrow + (int64_t)cs * kBUnitK, acc);
        else
            compute_unit(u, xrow + (int64_t)cs * kBUnitK, t4, cs == KU - 1 ? a.tail : 8, acc[0]);
        // the run leaves this row-block: park its partial sum
        if (cs == KU - 1 || i + 1 == i1) {
            const uint32_t p = part_base + (uint32_t)((cr - first) * 32) * (8 * RL);
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                if constexpr (C > 1) {
                    st_cluster_f32(p + 8 * r, acc[r][0]);
                    st_cluster_f32(p + 8 * r + 4, acc[r][1]);
                } else {
                    st_shared_f32(p + 8 * r, acc[r][0]);
                    st_shared_f32(p + 8 * r + 4, acc[r][1]);
                }
                acc[r][0] = acc[r][1] = 0.0f;
            }
        }
        if (++cs == KU) {
            cs = 0;
            ++cr;
        }
        if (++stage == kStages) stage = 0;
    }
    cp_async_wait<0>();

    if constexpr (C > 1)
        cluster_sync();
    else
        __syncthreads();
    if (rank != 0) return;
    // the first block adds each row-block's partial sums in warp order
    for (int64_t r = warp; r < rb1 - rb0; r += kBWarps) {
        // the warps whose runs touch units [r KU, (r + 1) KU)
        const int64_t lo = r * KU, hi = (r + 1) * KU;
        int u = (int)(((lo + 1) * V + T - 1) / T) - 1;   // the run that holds unit lo
        float s[RL][2] = {};
        for (; u < V; ++u) {
            const int64_t b0 = run_begin(T, u, V), b1 = run_begin(T, u + 1, V);
            if (b0 >= hi) break;
            if (b1 <= b0 || b1 <= lo) continue;
            const float* p = part + ((int64_t)(u * a.J + (r - b0 / KU)) * 32 + lane) * (2 * RL);
#pragma unroll
            for (int q = 0; q < RL; ++q) {
                s[q][0] += p[2 * q];
                s[q][1] += p[2 * q + 1];
            }
        }
#pragma unroll
        for (int q = 0; q < RL; ++q) {
            const int64_t n = (rb0 + r) * F::kRows + gid + 8 * q;
            if (n >= a.N) continue;
            const int m0 = 2 * t4;
            if (m0 < a.M) a.y[(int64_t)m0 * a.N + n] = __half_as_ushort(__float2half_rn(s[q][0]));
            if (m0 + 1 < a.M) a.y[(int64_t)(m0 + 1) * a.N + n] = __half_as_ushort(__float2half_rn(s[q][1]));
        }
    }
}

// ------------------------------------------------------------- dequantize --

// One thread per 4 consecutive weights, so that a warp stores 512 contiguous
// bytes: W^ in fp32 with the step and offset exact in fp32, step * q exact,
// one rounding in the sum.
template <int FMT>
__global__ void __launch_bounds__(256) blocks_dequant_kernel(const uint8_t* __restrict__ w, float* __restrict__ out,
                                                             int64_t N, int64_t K, int64_t row_bytes) {
    const int64_t per_row = K / 4;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N * per_row) return;
    const int64_t n = t / per_row;
    const int k = (int)(t % per_row) * 4;
    float v[4];
    if constexpr (FMT == W4A16_FORMAT_Q4_K) {
        const uint8_t* blk = w + n * row_bytes + (int64_t)(k / 256) * 144;
        const int i = k % 256, j = i / 32, c = i / 64, r = i % 64;
        const uint4 head = __ldg(reinterpret_cast<const uint4*>(blk));
        const uint32_t s03 = head.y & 0x3F3F3F3Fu, m03 = head.z & 0x3F3F3F3Fu;
        const uint32_t s47 = (head.w & 0x0F0F0F0Fu) | ((head.y >> 2) & 0x30303030u);
        const uint32_t m47 = ((head.w >> 4) & 0x0F0F0F0Fu) | ((head.z >> 2) & 0x30303030u);
        const float sc = byte_to_float(j < 4 ? s03 : s47, j & 3), mn = byte_to_float(j < 4 ? m03 : m47, j & 3);
        const float2 df = __half22float2(*reinterpret_cast<const __half2*>(&head.x));
        const float step = __fmul_rn(df.x, sc), off = __fmul_rn(df.y, mn);
        // weights 64c + (r mod 32) .. + 3: four bytes, low nibbles if r < 32, else high
        const uint32_t q4 = __ldg(reinterpret_cast<const uint32_t*>(blk + 16 + 32 * c + (r % 32))) >> (r < 32 ? 0 : 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fsub_rn(__fmul_rn(step, (float)((q4 >> (8 * e)) & 0xFu)), off);
    } else {
        const uint8_t* blk = w + n * row_bytes + (int64_t)(k / 32) * 24;
        const int i = k % 32;
        const uint2 head = __ldg(reinterpret_cast<const uint2*>(blk));
        const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&head.x));
        const uint32_t q4 = __ldg(reinterpret_cast<const uint32_t*>(blk + 8 + (i % 16))) >> (i < 16 ? 0 : 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t q = ((q4 >> (8 * e)) & 0xFu) | (((head.y >> (i + e)) & 1u) << 4);
            v[e] = __fadd_rn(__fmul_rn(dm.x, (float)q), dm.y);
        }
    }
    *reinterpret_cast<float4*>(out + n * K + k) = make_float4(v[0], v[1], v[2], v[3]);
}

template <int FMT, int C>
cudaError_t launch_c(const StreamArgs& a, size_t smem, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.ncl * C));
    cfg.blockDim = dim3(kBThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = C > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, blocks_gemv_kernel<FMT, C>, a);
}

constexpr size_t kPartSmem = 32 * 1024;   // largest partial-sum area of a block

// Dynamic shared memory of a block: the partial-sum area, then the weight rings.
template <int FMT>
constexpr size_t ring_bytes() {
    return (size_t)kBWarps * kStages * stage_bytes<FMT>();
}
constexpr int kClusterSizes[4] = {1, 2, 4, 8};

// Per device and format: the dynamic shared-memory limit set once, and how
// many clusters of each size fit on the GPU at once with that much memory.
struct ClusterFit {
    int count[4];
};

template <int FMT>
const ClusterFit& cluster_fit(const DeviceInfo& dev, cudaError_t* err) {
    static PerDeviceOnce once;
    static ClusterFit fit[kMaxDevices];
    *err = once.run(dev.device, [&]() -> cudaError_t {
        cudaError_t e = cudaSuccess;
        e = cudaFuncSetAttribute(blocks_gemv_kernel<FMT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kPartSmem + ring_bytes<FMT>()));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(blocks_gemv_kernel<FMT, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kPartSmem + ring_bytes<FMT>()));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(blocks_gemv_kernel<FMT, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kPartSmem + ring_bytes<FMT>()));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(blocks_gemv_kernel<FMT, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kPartSmem + ring_bytes<FMT>()));
        if (e != cudaSuccess) return e;
        for (int i = 0; i < 4; ++i) {
            const int c = kClusterSizes[i];
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(c * dev.sms));
            cfg.blockDim = dim3(kBThreads);
            cfg.dynamicSmemBytes = kPartSmem + ring_bytes<FMT>();
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)c;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int m = 0;
            const cudaError_t q =
                c == 1 ? cudaOccupancyMaxActiveClusters(&m, blocks_gemv_kernel<FMT, 1>, &cfg)
                : c == 2 ? cudaOccupancyMaxActiveClusters(&m, blocks_gemv_kernel<FMT, 2>, &cfg)
                : c == 4 ? cudaOccupancyMaxActiveClusters(&m, blocks_gemv_kernel<FMT, 4>, &cfg)
                         : cudaOccupancyMaxActiveClusters(&m, blocks_gemv_kernel<FMT, 8>, &cfg);
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

// Runs the GEMV for up to 8 tokens. Rows go in chunks small enough that the
// partial sums of a cluster fit its first block's shared memory.
template <int FMT>
w4a16_status run_gemv(const DeviceInfo& dev, StreamArgs a, cudaStream_t st) {
    using F = Fmt<FMT>;
    constexpr int RL = F::kRows / 8;
    cudaError_t e = cudaSuccess;
    const ClusterFit& fit = cluster_fit<FMT>(dev, &e);
    if (e != cudaSuccess) return cuda_status(e, "blocks gemv: set-up");
    const int64_t nrb_all = (a.N + F::kRows - 1) / F::kRows;
    // the cluster size that gives the fewest units to the busiest warp
    int best = -1;
    double best_load = 0.0;
    int64_t best_per_cl = 0;
    for (int i = 0; i < 4; ++i) {
        const int c = kClusterSizes[i], m = fit.count[i], V = c * kBWarps;
        const size_t slot = (size_t)V * 32 * 2 * RL * sizeof(float);   // one partial slot of every warp
        const int64_t jmax = (int64_t)(kPartSmem / slot);
        // a run of L units touches at most (L - 1) / KU + 2 row-blocks, which
        // must not exceed jmax: a cluster takes at most per_cl row-blocks a launch
        const int64_t per_cl = jmax >= 2 ? ((jmax - 1) * a.KU - 1) * V / a.KU : 0;
        if (m <= 0 || per_cl < 1) continue;
        const int64_t ncl = nrb_all < m ? nrb_all : m;
        int64_t rbc = (nrb_all + ncl - 1) / ncl;
        if (rbc > per_cl) rbc = per_cl;
        const double load = (double)rbc * a.KU / V;
        if (best < 0 || load < best_load * 0.97) {
            best = i;
            best_load = load;
            best_per_cl = per_cl;
        }
    }
    if (best < 0) return W4A16_ERR_UNSUPPORTED;
    const int c = kClusterSizes[best], V = c * kBWarps;
    const int64_t maxcl = fit.count[best], per_cl = best_per_cl;
    const size_t slot = (size_t)V * 32 * 2 * RL * sizeof(float);
    for (int64_t r0 = 0; r0 < nrb_all;) {
        const int64_t nrb = nrb_all - r0 < maxcl * per_cl ? nrb_all - r0 : maxcl * per_cl;
        StreamArgs b = a;
        b.rb_first = r0;
        b.nrb = (int)nrb;
        b.ncl = (int)(nrb < maxcl ? nrb : maxcl);
        const int64_t T = (nrb + b.ncl - 1) / b.ncl * a.KU;   // the most units a cluster gets
        b.J = (int)((T + V - 1) / V / a.KU + 2);
        const size_t smem = (size_t)b.J * slot + ring_bytes<FMT>();
        e = c == 1 ? launch_c<FMT, 1>(b, smem, st)
            : c == 2 ? launch_c<FMT, 2>(b, smem, st)
            : c == 4 ? launch_c<FMT, 4>(b, smem, st)
                     : launch_c<FMT, 8>(b, smem, st);
        if (e != cudaSuccess) return cuda_status(e, "blocks gemv: kernel launch");
        r0 += nrb;
    }
    return W4A16_OK;
}

}  // namespace

int64_t blocks_row_bytes(int32_t format, int64_t K) {
    const int bw = format == W4A16_FORMAT_Q4_K ? 256 : format == W4A16_FORMAT_Q5_1 ? 32 : 0;
    const int bb = format == W4A16_FORMAT_Q4_K ? 144 : 24;
    if (bw == 0 || K < 0 || K % bw != 0) return -1;
    return K / bw * bb;
}

w4a16_status blocks_linear_launch(const DeviceInfo& dev, int32_t format, const uint16_t* x, const uint8_t* w,
                                  uint16_t* y, int64_t M, int64_t N, int64_t K, cudaStream_t st) {
    const int64_t units = (K + kBUnitK - 1) / kBUnitK;
    if (units > 0x7fffffffLL || (N + 7) / 8 > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    StreamArgs a;
    a.w = w;
    a.N = N;
    a.K = K;
    a.row_bytes = blocks_row_bytes(format, K);
    a.KU = (int)units;
    a.tail = K % kBUnitK ? (int)(K % kBUnitK) / 32 : 8;
    a.rb_first = 0;
    a.nrb = a.ncl = a.J = 0;
    for (int64_t m0 = 0; m0 < M; m0 += kBTokens) {
        a.x = x + m0 * K;
        a.y = y + m0 * N;
        a.M = (int)(M - m0 < kBTokens ? M - m0 : kBTokens);
        const w4a16_status r = format == W4A16_FORMAT_Q4_K ? run_gemv<W4A16_FORMAT_Q4_K>(dev, a, st)
                                                           : run_gemv<W4A16_FORMAT_Q5_1>(dev, a, st);
        if (r != W4A16_OK) return r;
    }
    return W4A16_OK;
}

w4a16_status blocks_dequant_launch(int32_t format, const uint8_t* w, int64_t N, int64_t K, float* out,
                                   cudaStream_t st) {
    const int64_t threads = N * (K / 4);
    if (threads == 0) return W4A16_OK;
    const int64_t grid = (threads + 255) / 256;
    if (grid > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const int64_t rb = blocks_row_bytes(format, K);
    if (format == W4A16_FORMAT_Q4_K)
        blocks_dequant_kernel<W4A16_FORMAT_Q4_K><<<(unsigned)grid, 256, 0, st>>>(w, out, N, K, rb);
    else
        blocks_dequant_kernel<W4A16_FORMAT_Q5_1><<<(unsigned)grid, 256, 0, st>>>(w, out, N, K, rb);
    return cuda_status(cudaGetLastError(), "blocks dequant: kernel launch");
}

}  // namespace w4a16
