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
// * The activations (M x K fp16, at most 200 KB) are copied once per block
//   into shared memory with bulk asynchronous copies while the first weight
//   loads are in flight; larger x is read through the L1 instead.
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
//   A warp publishes its (at most two) partials after its last load, so the
//   memory fence never waits on weight loads still in flight.
#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kWarps = 16;       // warps per block, one block per SM
constexpr int kBlocksPerSM = 1;
constexpr size_t kXSmemMax = 200 * 1024;  // x staged in shared memory up to this size
constexpr int kStepK = 128;      // input features per unit
constexpr int kRows = 16;        // output features per unit
constexpr int kDepth = 4;        // units in flight per warp
constexpr int kMaxM = 16;        // activation rows handled by the GEMV

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
    float* partial;  // [P][2][16 * M] fp32 partial sums (first / last segment)
    int* counter;    // [ceil(N/16)] arrivals per row-block, zero between calls
    unsigned int* err;
};

template <int G>
struct Unit {
    uint32_t wa[4], wb[4];     // rows gid and gid + 8: 32 nibbles each
    uint32_t sc[kStepK / G];   // per group: scale of row gid (low) and gid + 8 (high)
};

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_cached_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_cached_u16(const uint16_t* p) {
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// (x0..x7) -> (x0,x4), (x1,x5), (x2,x6), (x3,x7): the pair order the nibble
// conversion produces for the weights.
__device__ __forceinline__ uint4 permute_x8(uint4 v) {
    return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                      __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

// Load cursor: per-thread addresses of one unit (rows gid and gid + 8 of
// row-block rb, k-step ks). Rows past N point at row N-1 and get a zero
// scale, so the hot loop needs no predicates.
template <int G>
struct Cursor {
    const uint8_t* pa;
    const uint8_t* pb;
    const uint16_t* sa;
    const uint16_t* sb;
    int64_t rb, ks;
    bool va, vb;

    __device__ __forceinline__ void seek(const GemvArgs& p, int64_t rb_, int64_t ks_, int gid, int t4) {
        rb = rb_;
        ks = ks_;
        int64_t r0 = rb * kRows + gid, r1 = r0 + 8;
        va = r0 < p.N;
        vb = r1 < p.N;
        if (!va) r0 = p.N - 1;
        if (!vb) r1 = p.N - 1;
        const int64_t rowbytes = p.K >> 1, gpr = p.K / G;
        const int64_t byte = ks * (kStepK / 2) + t4 * (G / 8);
        pa = p.qw + r0 * rowbytes + byte;
        pb = p.qw + r1 * rowbytes + byte;
        sa = p.s + r0 * gpr + ks * (kStepK / G);
        sb = p.s + r1 * gpr + ks * (kStepK / G);
    }
    __device__ __forceinline__ void next(const GemvArgs& p, int gid, int t4) {
        if (++ks == p.KS) {
            seek(p, rb + 1, 0, gid, t4);
        } else {
            pa += kStepK / 2;
            pb += kStepK / 2;
            sa += kStepK / G;
            sb += kStepK / G;
        }
    }
};

template <int G>
__device__ __forceinline__ void load_unit(Unit<G>& u, const Cursor<G>& c, const GemvArgs& p) {
    constexpr int WPP = G / 32;  // 32-bit words per thread per row per group
#pragma unroll
    for (int j = 0; j < kStepK / G; ++j) {
        // a group past K (ragged last step, G < 128) re-reads group 0 with a zero scale
        const bool vk = (G == kStepK) || (c.ks * kStepK + j * G < p.K);
        const int off = vk ? j * (G / 2) : 0;
        if constexpr (WPP == 4) {
            const uint4 va = ld_stream_v4(c.pa + off);
            const uint4 vb = ld_stream_v4(c.pb + off);
            u.wa[0] = va.x; u.wa[1] = va.y; u.wa[2] = va.z; u.wa[3] = va.w;
            u.wb[0] = vb.x; u.wb[1] = vb.y; u.wb[2] = vb.z; u.wb[3] = vb.w;
        } else if constexpr (WPP == 2) {
            const uint2 va = ld_stream_v2(c.pa + off);
            const uint2 vb = ld_stream_v2(c.pb + off);
            u.wa[2 * j] = va.x; u.wa[2 * j + 1] = va.y;
            u.wb[2 * j] = vb.x; u.wb[2 * j + 1] = vb.y;
        } else {
            u.wa[j] = ld_stream_u32(c.pa + off);
            u.wb[j] = ld_stream_u32(c.pb + off);
        }
        const uint32_t s0 = ld_cached_u16(c.sa + (vk ? j : 0));
        const uint32_t s1 = ld_cached_u16(c.sb + (vk ? j : 0));
        u.sc[j] = ((c.va && vk) ? s0 : 0u) | ((c.vb && vk) ? (s1 << 16) : 0u);
    }
}

// Shared-memory activations: per token a row of ceil(K/128) units x 16 chunks
// of 16 bytes (+64 B pad), each chunk pre-permuted by permute_x8 and placed so
// that the four threads of a quad read consecutive chunks.
__device__ __forceinline__ int xs_pos(int c_local, int G) {
    const int cpp = G / 8;              // chunks per group
    const int j = c_local / cpp, rem = c_local % cpp;
    const int t4 = rem / (G / 32), wi = rem % (G / 32);
    return (j * (G / 32) + wi) * 4 + t4;
}

template <int G, int NT, bool XS>
__device__ __forceinline__ void compute_unit(const Unit<G>& u, const GemvArgs& p, const uint8_t* xs_unit,
                                             int64_t xstride, int64_t ks, int gid, int t4, float (&acc)[NT][4]) {
    constexpr int WPP = G / 32;
#pragma unroll
    for (int j = 0; j < kStepK / G; ++j) {
        float c0[NT][4], c1[NT][4];  // two independent MMA chains per group
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) c0[t][i] = c1[t][i] = 0.0f;
#pragma unroll
        for (int wi = 0; wi < WPP; ++wi) {
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            nibbles_to_half2(u.wa[j * WPP + wi], a04, a15, a26, a37);
            nibbles_to_half2(u.wb[j * WPP + wi], b04, b15, b26, b37);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int m = 8 * t + gid;
                uint4 xv = make_uint4(0, 0, 0, 0);
                if (XS) {
                    if (m < p.M)
                        xv = *reinterpret_cast<const uint4*>(xs_unit + m * xstride + ((j * WPP + wi) * 4 + t4) * 16);
                } else {
                    const int64_t k0 = ks * kStepK + j * G + t4 * (G / 4) + 8 * wi;
                    if (m < p.M && k0 < p.K) xv = permute_x8(ld_cached_v4(p.x + (int64_t)m * p.K + k0));
                }
                mma_16816(c0[t], a04, b04, a15, b15, xv.x, xv.y);
                mma_16816(c1[t], a26, b26, a37, b37, xv.z, xv.w);
            }
        }
        const float s0 = __half2float(__ushort_as_half((unsigned short)(u.sc[j] & 0xFFFFu)));
        const float s1 = __half2float(__ushort_as_half((unsigned short)(u.sc[j] >> 16)));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(s0, c0[t][0] + c1[t][0], acc[t][0]);
            acc[t][1] = fmaf(s0, c0[t][1] + c1[t][1], acc[t][1]);
            acc[t][2] = fmaf(s1, c0[t][2] + c1[t][2], acc[t][2]);
            acc[t][3] = fmaf(s1, c0[t][3] + c1[t][3], acc[t][3]);
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

// Stores a row-block's fp32 partial in this warp's slot (0: first segment,
// 1: last segment).
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

// After this warp's partial for row-block rb is visible: count the arrival;
// the last contributor sums every contributor's partial in warp order,
// rounds once to fp16, stores y and resets the counter.
template <int NT>
__device__ __noinline__ void arrive_row_block(const GemvArgs& p, int64_t rb, int gid, int t4, int lane) {
    int old = 0;
    if (lane == 0) old = atomicAdd(p.counter + rb, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int64_t wa = warp_of_unit(rb * p.KS, p);
    const int64_t wb = warp_of_unit(rb * p.KS + p.KS - 1, p);
    if ((int64_t)old != wb - wa) return;  // another warp finishes this row-block
    __threadfence();
    const int64_t slot_elems = (int64_t)kRows * p.M;
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

template <int G, int NT, bool XS>
__global__ void __launch_bounds__(kWarps * 32, kBlocksPerSM) gemv_kernel(const GemvArgs p) {
    extern __shared__ __align__(16) uint8_t xs[];
    const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const bool active = w < p.P;
    const int64_t u_begin = active ? w * p.U / p.P : 0, u_end = active ? (w + 1) * p.U / p.P : 0;

    // weight loads for the first kDepth units go out before anything else
    Unit<G> buf[kDepth];
    Cursor<G> lc;
    lc.seek(p, u_begin / p.KS, u_begin % p.KS, gid, t4);
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
        if (u_begin + d < u_end) {
            load_unit<G>(buf[d], lc, p);
            lc.next(p, gid, t4);
        }
    }

    const int64_t xstride = p.KS * (kStepK * 2) + 64;  // bytes per token row
    if (XS) {
        // stage x: coalesced 16-byte loads, permuted into MMA fragment order, zero past K
        const int64_t chunks = (int64_t)p.M * p.KS * 16;
        for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
            const int64_t m = c / (p.KS * 16), cc = c % (p.KS * 16);
            const int64_t k0 = cc * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k0 < p.K) v = permute_x8(ld_cached_v4(p.x + m * p.K + k0));
            const int unit = (int)(cc >> 4), pos = xs_pos((int)(cc & 15), G);
            *reinterpret_cast<uint4*>(xs + m * xstride + unit * (kStepK * 2) + pos * 16) = v;
        }
        __syncthreads();
    }
    if (!active) return;

    int64_t rb = u_begin / p.KS, ks = u_begin % p.KS;
    const int64_t first_rb = rb;
    int64_t seg_ks0 = ks;
    float acc[NT][4], acc_first[NT][4];
    bool has_first = false;
    int64_t last_rb = -1;
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

    for (int64_t u = u_begin; u < u_end; u += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            if (u + d < u_end) {
                compute_unit<G, NT, XS>(buf[d], p, xs + ks * (kStepK * 2), xstride, ks, gid, t4, acc);
                if (u + d + kDepth < u_end) {
                    load_unit<G>(buf[d], lc, p);
                    lc.next(p, gid, t4);
                }
                const bool seg_end = (ks == p.KS - 1) || (u + d == u_end - 1);
                if (seg_end) {
                    if (seg_ks0 == 0 && ks == p.KS - 1) {
                        store_y<NT>(p, rb, acc, gid, t4);  // whole row-block in this warp
                    } else if (rb == first_rb) {
                        // partial first segment: published after the last load (a fence
                        // here would wait for the loads in flight)
                        has_first = true;
#pragma unroll
                        for (int t = 0; t < NT; ++t)
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc_first[t][i] = acc[t][i];
                    } else {
                        store_partial<NT>(p, w, 1, acc, gid, t4);  // partial last segment
                        last_rb = rb;
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
                }
                if (++ks == p.KS) { ks = 0; ++rb; }
                if (seg_end) seg_ks0 = ks;
            }
        }
    }
    if (has_first) store_partial<NT>(p, w, 0, acc_first, gid, t4);
    if (has_first || last_rb >= 0) {
        __threadfence();
        __syncwarp();
        if (has_first) arrive_row_block<NT>(p, first_rb, gid, t4, lane);
        if (last_rb >= 0) arrive_row_block<NT>(p, last_rb, gid, t4, lane);
    }
}

int64_t max_warps(const DeviceInfo& dev) { return (int64_t)dev.sms * kBlocksPerSM * kWarps; }

template <int G, int NT, bool XS>
w4a16_status launch_one(const GemvArgs& a, unsigned blocks, size_t smem, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    if (XS)
        std::call_once(once, [] {
            attr = cudaFuncSetAttribute(gemv_kernel<G, NT, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kXSmemMax);
        });
    if (attr != cudaSuccess) return W4A16_ERR_CUDA;
    gemv_kernel<G, NT, XS><<<blocks, kWarps * 32, smem, st>>>(a);
    return cuda_status(cudaGetLastError());
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

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
    a.partial = reinterpret_cast<float*>(workspace);
    a.counter = reinterpret_cast<int*>(reinterpret_cast<char*>(workspace) + partial_region_bytes(dev));
    a.err = dev.error_word;
    const int nt = M <= 8 ? 1 : 2;
    const size_t xbytes = (size_t)M * (size_t)(a.KS * kStepK * 2 + 64);
    const bool xs = xbytes <= kXSmemMax && xbytes <= dev.smem_optin;
    w4a16_status st_ = W4A16_OK;
#define W4A16_GEMV(G_, NT_)                                                                  \
    st_ = xs ? launch_one<G_, NT_, true>(a, (unsigned)blocks, xbytes, st)                    \
             : launch_one<G_, NT_, false>(a, (unsigned)blocks, 0, st)
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
    return st_;
}

}  // namespace w4a16
