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
// GEMV design. A warp's unit is 8 weight rows x 256 k (one Q4_K block or
// eight Q5_1 blocks per row). Every lane loads its own pieces of the unit
// straight into registers, one unit ahead, and turns nibbles into exact fp16
// integers. One mma.sync m16n8k16 per 16 k takes weight rows as A rows 0-7,
// constant ones as A rows 8-15 and up to 8 tokens of x as B: C rows 0-7 are
// the integer dot products S = sum x q of a 32-weight sub-block and C rows
// 8-15 the sums X = sum x over the same k, so the sub-block adds a S + b X
// (W^ = a q + b) in fp32 with no extra pass over x. A block of 4 warps owns a
// row-block and splits its units over the warps (and, when row-blocks are
// few, over the 2 or 4 blocks of a thread-block cluster); the partial sums
// meet in the shared memory of the cluster's first block and are added in a
// fixed order, so results are deterministic.
#include <type_traits>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr int kBWarps = 4;             // warps per block
constexpr int kBThreads = kBWarps * 32;
constexpr int kBRows = 8;              // weight rows per row-block
constexpr int kBUnitK = 256;           // k per unit
constexpr int kBTokens = 8;            // tokens per launch

struct BlocksArgs {
    const uint16_t* x;   // fp16 [M, K]
    const uint8_t* w;    // blocks [N, row_bytes]
    uint16_t* y;         // fp16 [M, N]
    int64_t N, K, row_bytes;
    int M;               // tokens of this launch, 1..8
    int units;           // ceil(K / 256)
    int tail;            // Q5_1 blocks in the last unit when K % 256 != 0, else 8
};

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

// Stores into the shared memory of another block of the cluster.
__device__ __forceinline__ void st_cluster_f32(uint32_t caddr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}

// ------------------------------------------------------------------ Q4_K --

struct Q4KUnit {
    uint4 head;      // d, dmin, 12 scale bytes of the lane's row
    uint2 qs[4];     // bytes 8 t4 .. 8 t4 + 7 of each 32-byte chunk
};

__device__ __forceinline__ void load_unit(Q4KUnit& r, const uint8_t* blk, int t4, bool ok, int) {
    if (ok) {
        r.head = __ldg(reinterpret_cast<const uint4*>(blk));
#pragma unroll
        for (int c = 0; c < 4; ++c) r.qs[c] = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 32 * c + 8 * t4));
    } else {
        r.head = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 4; ++c) r.qs[c] = make_uint2(0, 0);
    }
}

// One Q4_K unit: acc[0..1] (row gid, tokens 2 t4 and 2 t4 + 1) += sum over the
// unit's 256 k of x W^.
__device__ __forceinline__ void compute_unit(const Q4KUnit& r, const uint16_t* xk, bool xok, float (&acc)[2]) {
    // sub-block scales sc[j] and minimums mn[j] as bytes: j < 4 in the low six
    // bits of scale bytes 0-3 and 4-7; j >= 4 low four bits from bytes 8-11,
    // top two bits from the top of bytes 0-3 (sc) and 4-7 (mn)
    const uint32_t s03 = r.head.y & 0x3F3F3F3Fu, m03 = r.head.z & 0x3F3F3F3Fu;
    const uint32_t s47 = (r.head.w & 0x0F0F0F0Fu) | ((r.head.y >> 2) & 0x30303030u);
    const uint32_t m47 = ((r.head.w >> 4) & 0x0F0F0F0Fu) | ((r.head.z >> 2) & 0x30303030u);
    float sacc[2] = {0.0f, 0.0f}, macc[2] = {0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // x for sub-blocks 2c (low nibbles) and 2c + 1 (high nibbles): eight
        // consecutive values each, at 32 j + 8 t4
        uint4 xl = make_uint4(0, 0, 0, 0), xh = make_uint4(0, 0, 0, 0);
        if (xok) {
            xl = *reinterpret_cast<const uint4*>(xk + 64 * c);
            xh = *reinterpret_cast<const uint4*>(xk + 64 * c + 32);
        }
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            const uint4 xv = hi ? xh : xl;
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const uint32_t w = s ? r.qs[c].y : r.qs[c].x;
                const uint32_t w8 = w >> 8;
                uint32_t a0, a2;
                if (hi) {
                    a0 = hfma2_u32(lop3_and_or(w, 0x00F000F0u, kMagic), kSixteenth, kMinus64);
                    a2 = hfma2_u32(lop3_and_or(w8, 0x00F000F0u, kMagic), kSixteenth, kMinus64);
                } else {
                    a0 = hsub2_u32(lop3_and_or(w, 0x000F000Fu, kMagic), k1024);
                    a2 = hsub2_u32(lop3_and_or(w8, 0x000F000Fu, kMagic), k1024);
                }
                uint32_t b0, b1;
                x_pairs(s ? xv.z : xv.x, s ? xv.w : xv.y, b0, b1);
                mma_16816(d, a0, kOnes, a2, kOnes, b0, b1);
            }
            const int j = 2 * c + hi;
            const float sc = byte_to_float(j < 4 ? s03 : s47, j & 3);
            const float mn = byte_to_float(j < 4 ? m03 : m47, j & 3);
            sacc[0] = fmaf(sc, d[0], sacc[0]);
            sacc[1] = fmaf(sc, d[1], sacc[1]);
            macc[0] = fmaf(mn, d[2], macc[0]);
            macc[1] = fmaf(mn, d[3], macc[1]);
        }
    }
    const __half2 dd = *reinterpret_cast<const __half2*>(&r.head.x);
    const float2 df = __half22float2(dd);   // (d, dmin)
    acc[0] = fmaf(df.x, sacc[0], fmaf(-df.y, macc[0], acc[0]));
    acc[1] = fmaf(df.x, sacc[1], fmaf(-df.y, macc[1], acc[1]));
}

// ------------------------------------------------------------------ Q5_1 --

struct Q51Unit {
    uint2 head[8];   // d, m, qh of each of the row's eight blocks
    uint32_t qs[8];  // bytes 4 t4 .. 4 t4 + 3 of each block's nibbles
};

__device__ __forceinline__ void load_unit(Q51Unit& r, const uint8_t* blk, int t4, bool ok, int nb) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        if (ok && b < nb) {
            r.head[b] = __ldg(reinterpret_cast<const uint2*>(blk + 24 * b));
            r.qs[b] = __ldg(reinterpret_cast<const uint32_t*>(blk + 24 * b + 8 + 4 * t4));
        } else {
            r.head[b] = make_uint2(0, 0);
            r.qs[b] = 0;
        }
    }
}

// Two fp16 pairs (bytes 0, 2) and (bytes 1, 3) of the nibbles in v (bits
// 0-3 of each byte) with fifth bits f (bit e = byte e's), as exact integers.
__device__ __forceinline__ void q5_pairs(uint32_t v, uint32_t f, uint32_t& p02, uint32_t& p13) {
    // bit 0 of f to bit 4 and bit 2 to bit 20; bit 1 to bit 4 and bit 3 to bit 20
    const uint32_t f02 = lop3_and_or(f * 0x00040010u, 0x00100010u, kMagic);
    const uint32_t f13 = lop3_and_or(f * 0x00020008u, 0x00100010u, kMagic);
    p02 = hsub2_u32(lop3_and_or(v, 0x000F000Fu, f02), k1024);
    p13 = hsub2_u32(lop3_and_or(v >> 8, 0x000F000Fu, f13), k1024);
}

__device__ __forceinline__ void compute_unit(const Q51Unit& r, const uint16_t* xk, int t4, bool xok, int nb,
                                             float (&acc)[2]) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        uint2 xl = make_uint2(0, 0), xh = make_uint2(0, 0);
        if (xok && b < nb) {
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

template <int FMT, int C>
__global__ void __launch_bounds__(kBThreads) blocks_gemv_kernel(const BlocksArgs a) {
    __shared__ float red[C * kBWarps][32][2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, t4 = lane & 3;
    const int rank = C > 1 ? (int)cluster_rank() : 0;
    const int64_t rb = blockIdx.x / C;
    const int64_t row = rb * kBRows + gid;
    const bool row_ok = row < a.N;
    const bool xok = gid < a.M;
    const int v = rank * kBWarps + warp, V = C * kBWarps;
    const uint8_t* wrow = a.w + (row_ok ? row : 0) * a.row_bytes;
    constexpr int kUnitBytes = FMT == W4A16_FORMAT_Q4_K ? 144 : 192;
    // the lane's x: token gid, at 8 t4 (Q4_K) or 4 t4 (Q5_1) inside each sub-block
    const uint16_t* xrow = a.x + (int64_t)(xok ? gid : 0) * a.K + (FMT == W4A16_FORMAT_Q4_K ? 8 * t4 : 4 * t4);

    float acc[2] = {0.0f, 0.0f};
    using Unit = typename std::conditional<FMT == W4A16_FORMAT_Q4_K, Q4KUnit, Q51Unit>::type;
    Unit cur, nxt;
    const int last = a.units - 1;
    if (v < a.units) load_unit(cur, wrow + (int64_t)v * kUnitBytes, t4, row_ok, v == last ? a.tail : 8);
    for (int u = v; u < a.units; u += V) {
        const int un = u + V;
        if (un < a.units) load_unit(nxt, wrow + (int64_t)un * kUnitBytes, t4, row_ok, un == last ? a.tail : 8);
        if constexpr (FMT == W4A16_FORMAT_Q4_K)
            compute_unit(cur, xrow + (int64_t)u * kBUnitK, xok, acc);
        else
            compute_unit(cur, xrow + (int64_t)u * kBUnitK, t4, xok, u == last ? a.tail : 8, acc);
        cur = nxt;
    }

    // partial sums of every warp of the cluster meet in the first block
    if constexpr (C == 1) {
        red[v][lane][0] = acc[0];
        red[v][lane][1] = acc[1];
        __syncthreads();
    } else {
        const uint32_t base = cluster_map(smem_u32(&red[v][lane][0]), 0);
        st_cluster_f32(base, acc[0]);
        st_cluster_f32(base + 4, acc[1]);
        cluster_sync();
    }
    if (rank != 0 || warp != 0) return;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int i = 0; i < C * kBWarps; ++i) {
        s0 += red[i][lane][0];
        s1 += red[i][lane][1];
    }
    if (!row_ok) return;
    const int m0 = 2 * t4;
    if (m0 < a.M) a.y[(int64_t)m0 * a.N + row] = __half_as_ushort(__float2half_rn(s0));
    if (m0 + 1 < a.M) a.y[(int64_t)(m0 + 1) * a.N + row] = __half_as_ushort(__float2half_rn(s1));
}

// ------------------------------------------------------------- dequantize --

// One thread per 32 weights (a Q4_K sub-block or a Q5_1 block): W^ in fp32,
// step and offset exact in fp32, step * q exact, one rounding in the sum.
template <int FMT>
__global__ void __launch_bounds__(256) blocks_dequant_kernel(const uint8_t* __restrict__ w, float* __restrict__ out,
                                                             int64_t N, int64_t K, int64_t row_bytes) {
    const int64_t per_row = K / 32;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N * per_row) return;
    const int64_t n = t / per_row, g = t % per_row;
    float v[32];
    if constexpr (FMT == W4A16_FORMAT_Q4_K) {
        const uint8_t* blk = w + n * row_bytes + (g / 8) * 144;
        const int j = (int)(g % 8), c = j / 2, hi = j % 2;
        const uint4 head = __ldg(reinterpret_cast<const uint4*>(blk));
        const uint32_t s03 = head.y & 0x3F3F3F3Fu, m03 = head.z & 0x3F3F3F3Fu;
        const uint32_t s47 = (head.w & 0x0F0F0F0Fu) | ((head.y >> 2) & 0x30303030u);
        const uint32_t m47 = ((head.w >> 4) & 0x0F0F0F0Fu) | ((head.z >> 2) & 0x30303030u);
        const float sc = byte_to_float(j < 4 ? s03 : s47, j & 3), mn = byte_to_float(j < 4 ? m03 : m47, j & 3);
        const float2 df = __half22float2(*reinterpret_cast<const __half2*>(&head.x));
        const float step = __fmul_rn(df.x, sc), off = __fmul_rn(df.y, mn);
        const uint4* qs = reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
        const uint4 q0 = __ldg(qs), q1 = __ldg(qs + 1);
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t q = (words[i / 4] >> (8 * (i % 4) + 4 * hi)) & 0xFu;
            v[i] = __fsub_rn(__fmul_rn(step, (float)q), off);
        }
    } else {
        const uint8_t* blk = w + n * row_bytes + g * 24;
        const uint2 head = __ldg(reinterpret_cast<const uint2*>(blk));
        const uint2 qa = __ldg(reinterpret_cast<const uint2*>(blk + 8)), qb = __ldg(reinterpret_cast<const uint2*>(blk + 16));
        const uint32_t words[4] = {qa.x, qa.y, qb.x, qb.y};
        const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&head.x));
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int byte = i % 16;
            const uint32_t nib = (words[byte / 4] >> (8 * (byte % 4) + (i < 16 ? 0 : 4))) & 0xFu;
            const uint32_t q = nib | (((head.y >> i) & 1u) << 4);
            v[i] = __fadd_rn(__fmul_rn(dm.x, (float)q), dm.y);
        }
    }
    float4* o = reinterpret_cast<float4*>(out + n * K + g * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <int FMT>
cudaError_t launch_gemv(const BlocksArgs& a, int c, cudaStream_t st) {
    const int64_t nrb = (a.N + kBRows - 1) / kBRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nrb * c));
    cfg.blockDim = dim3(kBThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)c;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = c > 1 ? 1 : 0;
    if (c == 1) return cudaLaunchKernelEx(&cfg, blocks_gemv_kernel<FMT, 1>, a);
    if (c == 2) return cudaLaunchKernelEx(&cfg, blocks_gemv_kernel<FMT, 2>, a);
    return cudaLaunchKernelEx(&cfg, blocks_gemv_kernel<FMT, 4>, a);
}

// Blocks per cluster: 1, or 2 / 4 when row-blocks are too few to give every SM
// about six blocks and each warp still gets two units or more.
int cluster_size(const DeviceInfo& dev, int64_t N, int64_t units) {
    const int64_t nrb = (N + kBRows - 1) / kBRows;
    int c = 1;
    while (c < 4 && nrb * c < 6LL * dev.sms && units >= 2LL * kBWarps * 2 * c) c *= 2;
    return c;
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
    if (units > 0x7fffffffLL || (N + kBRows - 1) / kBRows * 4 > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const int c = cluster_size(dev, N, units);
    BlocksArgs a;
    a.w = w;
    a.N = N;
    a.K = K;
    a.row_bytes = blocks_row_bytes(format, K);
    a.units = (int)units;
    a.tail = K % kBUnitK ? (int)(K % kBUnitK) / 32 : 8;
    for (int64_t m0 = 0; m0 < M; m0 += kBTokens) {
        a.x = x + m0 * K;
        a.y = y + m0 * N;
        a.M = (int)(M - m0 < kBTokens ? M - m0 : kBTokens);
        const cudaError_t e = format == W4A16_FORMAT_Q4_K ? launch_gemv<W4A16_FORMAT_Q4_K>(a, c, st)
                                                          : launch_gemv<W4A16_FORMAT_Q5_1>(a, c, st);
        if (e != cudaSuccess) return cuda_status(e, "blocks gemv: kernel launch");
    }
    return W4A16_OK;
}

w4a16_status blocks_dequant_launch(int32_t format, const uint8_t* w, int64_t N, int64_t K, float* out,
                                   cudaStream_t st) {
    const int64_t threads = N * (K / 32);
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
