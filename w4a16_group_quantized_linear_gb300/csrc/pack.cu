// Symmetric int4 group quantizer and unpacker (LLM170 page, introduction:
// "int4 sym g128"; group 32 for its MoE models).
//
// Quantizer, per row n and group of `G` consecutive k (one warp per group):
//   amax = max |w| (fp32, exact), s = fp16_rn(fp32(amax / 7)),
//   q = clamp(rint(w / s), -8, 7) with IEEE fp32 division and rint half-to-even,
//   all-zero group -> s = 0, q = 0; stored as nibble q + 8, even k in bits 0-3.
// Every step is a correctly rounded IEEE operation, so the result is
// bit-exact and independent of the launch shape.
#include "internal.cuh"

namespace w4a16 {

template <int G>
__global__ void __launch_bounds__(256) pack_kernel(const float* __restrict__ w, int64_t N, int64_t K,
                                                   uint8_t* __restrict__ qw, uint16_t* __restrict__ s) {
    constexpr int PER = G / 32;  // elements per lane
    const int lane = threadIdx.x & 31;
    const int64_t groups_per_row = K / G;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= N * groups_per_row) return;
    const int64_t n = warp / groups_per_row, j = warp % groups_per_row;
    const float* wr = w + n * K + j * G;

    float v[PER];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        v[i] = __ldg(wr + lane + 32 * i);
        amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

    const __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
    const float sf = __half2float(sh);
    if (lane == 0) s[n * groups_per_row + j] = __half_as_ushort(sh);

    uint8_t* out = qw + n * (K / 2) + (j * G) / 2;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        int q = 0;
        if (sf != 0.0f) {
            float r = rintf(__fdiv_rn(v[i], sf));
            q = (int)fminf(fmaxf(r, -8.0f), 7.0f);
        }
        const unsigned nib = (unsigned)(q + 8);
        const unsigned odd = __shfl_down_sync(0xffffffffu, nib, 1);  // k + 1 lives on lane + 1
        if ((lane & 1) == 0) out[(lane + 32 * i) / 2] = (uint8_t)(nib | (odd << 4));
    }
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ qw, int64_t bytes,
                                                     int8_t* __restrict__ q) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < bytes;
         i += (int64_t)gridDim.x * blockDim.x) {
        const unsigned b = qw[i];
        const int lo = (int)(b & 0xFu) - 8, hi = (int)(b >> 4) - 8;
        q[2 * i] = (int8_t)lo;
        q[2 * i + 1] = (int8_t)hi;
    }
}

w4a16_status pack_launch(const float* w, int64_t N, int64_t K, int group, uint8_t* qw, uint16_t* s,
                         cudaStream_t st) {
    const int64_t warps = N * (K / group);
    if (warps == 0) return W4A16_OK;
    const int64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    switch (group) {
        case 32: pack_kernel<32><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, qw, s); break;
        case 64: pack_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, qw, s); break;
        case 128: pack_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, qw, s); break;
        default: return W4A16_ERR_UNSUPPORTED;
    }
    return cuda_status(cudaGetLastError(), "pack: kernel launch");
}

w4a16_status unpack_launch(const uint8_t* qw, int64_t N, int64_t K, int8_t* q, cudaStream_t st) {
    const int64_t bytes = N * (K / 2);
    if (bytes == 0) return W4A16_OK;
    int64_t blocks = (bytes + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    unpack_kernel<<<(unsigned)blocks, 256, 0, st>>>(qw, bytes, q);
    return cuda_status(cudaGetLastError(), "unpack: kernel launch");
}

}  // namespace w4a16
