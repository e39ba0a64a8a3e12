// Decode GEMV for the W4A16 layer, M <= 16 activation rows (LLM170 page:
// "CUDA-graph decode", np4 = four sequences per step).
//
// Decode streams every packed weight byte once and does almost no arithmetic
// per byte, so the kernel is bound by HBM bandwidth. Design:
//
// * Work unit = 16 output features (rows n of W) x 128 input features k:
//   1 KB of packed weights plus their scales. Units are ordered row-block
//   major, k minor, and each warp of a persistent grid takes an equal
//   contiguous range of units (stream-K split), so every SM streams the same
//   number of bytes whatever N and K are.
// * Each thread loads 16 B of two weight rows per unit with 128-bit
//   coalesced, L1-bypassing loads, kDepth units ahead of the math.
// * Nibbles become exact fp16 integers in registers (lop3 + one half2 op per
//   pair) and go straight into mma.sync m16n8k16 as the A operand (rows =
//   weight rows, columns = tokens padded to 8): the tensor core does the
//   x*q products (exact) and their fp32 sum within one scale group, which
//   keeps the ALU cost per weight near one instruction. The k order inside a
//   group is permuted identically on the activation side, which leaves every
//   group sum unchanged.
// * After each group the fp32 partial is multiplied by the group's scale and
//   added into fp32 accumulators: acc += s[n, grp] * sum_{k in grp} x q.
// * A row-block whose units span several warps is finished by the last warp
//   to arrive: each contributor stores its fp32 partial in the workspace,
//   bumps a per-row-block counter, and the last one sums all partials in
//   warp order (deterministic), rounds once to fp16 and resets the counter.
#include "internal.cuh"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;        // warps per block
constexpr int kBlocksPerSM = 2;  // resident blocks per SM (16 warps)
constexpr int kStepK = 128;      // input features per unit
constexpr int kRows = 16;        // output features per unit
constexpr int kDepth = 4;        // units in flight per warp

struct GemvArgs {
    const uint16_t* x;
    const uint8_t* qw;
    const uint16_t* s;
    uint16_t* y;
    int M;
    int64_t N, K;
    int64_t KS;  // k-steps per row: ceil(K / 128)
    int64_t U;   // units: ceil(N / 16) * KS
    int64_t P;   // active warps (each owns >= 1 unit)
    int* counter;    // [ceil(N/16)] arrivals per row-block, zero between calls
    float* partial;  // [P][2][16 * M] fp32 partial sums (first / last segment)
};

template <int G>
struct Unit {
    uint32_t wa[4], wb[4];     // rows gid and gid + 8: 32 nibbles each
    uint32_t sc[kStepK / G];   // per group: scale of row gid (low) and gid + 8 (high)
};

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_cached_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_cached_u16(const uint16_t* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Loads the thread's share of unit (rb, ks): for each scale group in the
// 128-k step, the quarter t4 of that group of rows gid and gid + 8.
template <int G>
__device__ __forceinline__ void load_unit(Unit<G>& u, const GemvArgs& p, int64_t rb, int64_t ks,
                                          int gid, int t4) {
    constexpr int WPP = G / 32;  // 32-bit words per thread per row per group
    const int64_t r0 = rb * kRows + gid, r1 = r0 + 8;
    const bool ok0 = r0 < p.N, ok1 = r1 < p.N;
    const int64_t rowbytes = p.K >> 1, gpr = p.K / G;
#pragma unroll
    for (int j = 0; j < kStepK / G; ++j) {
        const int64_t kg = ks * kStepK + j * G;  // first k of the group
        const bool vk = kg < p.K;
        const int64_t byte = (kg + t4 * (G / 4)) >> 1;
        const uint8_t* a = p.qw + r0 * rowbytes + byte;
        const uint8_t* b = p.qw + r1 * rowbytes + byte;
        if constexpr (WPP == 4) {
            const uint4 va = (vk && ok0) ? ld_stream_v4(a) : make_uint4(0, 0, 0, 0);
            const uint4 vb = (vk && ok1) ? ld_stream_v4(b) : make_uint4(0, 0, 0, 0);
            u.wa[0] = va.x; u.wa[1] = va.y; u.wa[2] = va.z; u.wa[3] = va.w;
            u.wb[0] = vb.x; u.wb[1] = vb.y; u.wb[2] = vb.z; u.wb[3] = vb.w;
        } else if constexpr (WPP == 2) {
            const uint2 va = (vk && ok0) ? ld_stream_v2(a) : make_uint2(0, 0);
            const uint2 vb = (vk && ok1) ? ld_stream_v2(b) : make_uint2(0, 0);
            u.wa[2 * j] = va.x; u.wa[2 * j + 1] = va.y;
            u.wb[2 * j] = vb.x; u.wb[2 * j + 1] = vb.y;
        } else {
            u.wa[j] = (vk && ok0) ? ld_stream_u32(a) : 0u;
            u.wb[j] = (vk && ok1) ? ld_stream_u32(b) : 0u;
        }
        const uint32_t s0 = (vk && ok0) ? ld_cached_u16(p.s + r0 * gpr + kg / G) : 0u;
        const uint32_t s1 = (vk && ok1) ? ld_cached_u16(p.s + r1 * gpr + kg / G) : 0u;
        u.sc[j] = s0 | (s1 << 16);
    }
}

template <int G, int NT>
__device__ __forceinline__ void compute_unit(const Unit<G>& u, const GemvArgs& p, int64_t ks, int gid,
                                             int t4, float (&acc)[NT][4]) {
    constexpr int WPP = G / 32;
#pragma unroll
    for (int j = 0; j < kStepK / G; ++j) {
        const int64_t kg = ks * kStepK + j * G;
        if (kg >= p.K) break;  // ragged last step (warp-uniform)
        float c[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) c[t][0] = c[t][1] = c[t][2] = c[t][3] = 0.0f;
#pragma unroll
        for (int wi = 0; wi < WPP; ++wi) {
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            nibbles_to_half2(u.wa[j * WPP + wi], a04, a15, a26, a37);
            nibbles_to_half2(u.wb[j * WPP + wi], b04, b15, b26, b37);
            const int64_t k0 = kg + t4 * (G / 4) + 8 * wi;  // x[k0 .. k0+7] matches this word
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int m = 8 * t + gid;
                uint4 xv = make_uint4(0, 0, 0, 0);
                if (m < p.M) xv = ld_cached_v4(p.x + (int64_t)m * p.K + k0);
                // (x0,x4), (x1,x5), (x2,x6), (x3,x7): the order of the weight pairs
                const uint32_t x04 = __byte_perm(xv.x, xv.z, 0x5410);
                const uint32_t x15 = __byte_perm(xv.x, xv.z, 0x7632);
                const uint32_t x26 = __byte_perm(xv.y, xv.w, 0x5410);
                const uint32_t x37 = __byte_perm(xv.y, xv.w, 0x7632);
                mma_16816(c[t], a04, b04, a15, b15, x04, x15);
                mma_16816(c[t], a26, b26, a37, b37, x26, x37);
            }
        }
        const float s0 = __half2float(__ushort_as_half((unsigned short)(u.sc[j] & 0xFFFFu)));
        const float s1 = __half2float(__ushort_as_half((unsigned short)(u.sc[j] >> 16)));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(s0, c[t][0], acc[t][0]);
            acc[t][1] = fmaf(s0, c[t][1], acc[t][1]);
            acc[t][2] = fmaf(s1, c[t][2], acc[t][2]);
            acc[t][3] = fmaf(s1, c[t][3], acc[t][3]);
        }
    }
}

// Accumulator element i of tile t: row gid + 8 (i >> 1), token 8 t + 2 t4 + (i & 1).
template <int NT>
__device__ __forceinline__ void store_y(const GemvArgs& p, int64_t rb, const float (&v)[NT][4], int gid,
                                        int t4) {
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
__device__ __noinline__ void finish_segment(const GemvArgs& p, int64_t w, int64_t rb, int64_t first_rb,
                                            bool full, float (&acc)[NT][4], int gid, int t4, int lane) {
    if (full) {
        store_y<NT>(p, rb, acc, gid, t4);
        return;
    }
    const int64_t slot_elems = (int64_t)kRows * p.M;
    float* mine = p.partial + (w * 2 + (rb == first_rb ? 0 : 1)) * slot_elems;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * t4 + (i & 1);
            if (m < p.M) __stcg(mine + m * kRows + gid + 8 * (i >> 1), acc[t][i]);
        }
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(p.counter + rb, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int64_t wa = warp_of_unit(rb * p.KS, p);
    const int64_t wb = warp_of_unit(rb * p.KS + p.KS - 1, p);
    if ((int64_t)old != wb - wa) return;  // another warp finishes this row-block
    __threadfence();
    float sum[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) sum[t][0] = sum[t][1] = sum[t][2] = sum[t][3] = 0.0f;
    for (int64_t v = wa; v <= wb; ++v) {
        // rb is the first segment of every contributor except possibly wa
        const bool wa_started_inside = (v * p.U / p.P) == rb * p.KS;
        const int slot = (v == wa && !wa_started_inside) ? 1 : 0;
        const float* src = p.partial + (v * 2 + slot) * slot_elems;
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

template <int G, int NT>
__global__ void __launch_bounds__(kWarps * 32, kBlocksPerSM) gemv_kernel(const GemvArgs p) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (w >= p.P) return;
    const int64_t u_begin = w * p.U / p.P, u_end = (w + 1) * p.U / p.P;

    Unit<G> buf[kDepth];
    int64_t lrb = u_begin / p.KS, lks = u_begin % p.KS;  // next unit to load
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
        if (u_begin + d < u_end) load_unit<G>(buf[d], p, lrb, lks, gid, t4);
        if (++lks == p.KS) { lks = 0; ++lrb; }
    }

    int64_t rb = u_begin / p.KS, ks = u_begin % p.KS;
    const int64_t first_rb = rb;
    int64_t seg_ks0 = ks;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

    for (int64_t u = u_begin; u < u_end; u += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            if (u + d < u_end) {
                compute_unit<G, NT>(buf[d], p, ks, gid, t4, acc);
                if (u + d + kDepth < u_end) load_unit<G>(buf[d], p, lrb, lks, gid, t4);
                if (++lks == p.KS) { lks = 0; ++lrb; }
                const bool seg_end = (ks == p.KS - 1) || (u + d == u_end - 1);
                if (seg_end) {
                    finish_segment<NT>(p, w, rb, first_rb, seg_ks0 == 0 && ks == p.KS - 1, acc, gid, t4,
                                       lane);
#pragma unroll
                    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
                }
                if (++ks == p.KS) { ks = 0; ++rb; }
                if (seg_end) seg_ks0 = ks;
            }
        }
    }
}

int64_t max_warps(const DeviceInfo& dev) { return (int64_t)dev.sms * kBlocksPerSM * kWarps; }

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t gemv_workspace_bytes(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const int64_t RB = (N + kRows - 1) / kRows;
    return align256((size_t)RB * sizeof(int)) + (size_t)max_warps(dev) * 2 * kRows * M * sizeof(float);
}

w4a16_status gemv_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                         uint16_t* y, int64_t M, int64_t N, int64_t K, int group, void* workspace,
                         size_t workspace_bytes, cudaStream_t st) {
    const size_t need = gemv_workspace_bytes(dev, M, N, K);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return W4A16_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255) != 0) return W4A16_ERR_MISALIGNED;
    GemvArgs a;
    a.x = x; a.qw = qw; a.s = s; a.y = y;
    a.M = (int)M; a.N = N; a.K = K;
    a.KS = (K + kStepK - 1) / kStepK;
    const int64_t RB = (N + kRows - 1) / kRows;
    a.U = RB * a.KS;
    int64_t blocks = (a.U + kWarps - 1) / kWarps;
    const int64_t max_blocks = (int64_t)dev.sms * kBlocksPerSM;
    if (blocks > max_blocks) blocks = max_blocks;
    a.P = blocks * kWarps < a.U ? blocks * kWarps : a.U;
    a.counter = reinterpret_cast<int*>(workspace);
    a.partial = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + align256((size_t)RB * sizeof(int)));
    const int nt = M <= 8 ? 1 : 2;
#define W4A16_GEMV(G_, NT_) gemv_kernel<G_, NT_><<<(unsigned)blocks, kWarps * 32, 0, st>>>(a)
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
    return cuda_status(cudaGetLastError());
}

}  // namespace w4a16
