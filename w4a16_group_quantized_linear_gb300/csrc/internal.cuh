// Internal declarations shared by the translation units of libw4a16.so.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "w4a16.h"

namespace w4a16 {

constexpr int kMaxDevices = 64;  // device ordinals the library serves

// ----------------------------------------------------------------- device --

// Bit-select (a & b) | c in one instruction.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Eight packed nibbles (k0..k7 at bits 4i, value q+8) -> four fp16 pairs of
// the exact integers q, in the order (k0,k4), (k1,k5), (k2,k6), (k3,k7).
// A nibble placed in the low mantissa bits of the fp16 1024 (0x6400) reads as
// 1024 + nib; one at bits 4-7 reads as 1024 + 16 nib. Subtracting 1032, or
// scaling by 1/16 and subtracting 72, leaves nib - 8 exactly.
__device__ __forceinline__ void nibbles_to_half2(uint32_t v, uint32_t& h04, uint32_t& h15,
                                                 uint32_t& h26, uint32_t& h37) {
    const uint32_t lo_mask = 0x000F000Fu, hi_mask = 0x00F000F0u, magic = 0x64006400u;
    uint32_t t0 = lop3_and_or(v, lo_mask, magic);
    uint32_t t1 = lop3_and_or(v, hi_mask, magic);
    uint32_t v8 = v >> 8;
    uint32_t t2 = lop3_and_or(v8, lo_mask, magic);
    uint32_t t3 = lop3_and_or(v8, hi_mask, magic);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
    const __half2 bias16 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480)); // -72
    __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&t0), bias);
    __half2 r1 = __hfma2(*reinterpret_cast<__half2*>(&t1), sixteenth, bias16);
    __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&t2), bias);
    __half2 r3 = __hfma2(*reinterpret_cast<__half2*>(&t3), sixteenth, bias16);
    h04 = *reinterpret_cast<uint32_t*>(&r0);
    h15 = *reinterpret_cast<uint32_t*>(&r1);
    h26 = *reinterpret_cast<uint32_t*>(&r2);
    h37 = *reinterpret_cast<uint32_t*>(&r3);
}

// D = A * B + C, m16n8k16, fp16 inputs, fp32 accumulators (register operands;
// not volatile: a pure function of its operands, free to be scheduled).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B (zero accumulator input), m16n8k16, fp16 inputs, fp32 results.
__device__ __forceinline__ void mma_16816_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// Fused gate + up tiles of the tensor-core GEMMs: 128 weight rows per tile are
// 64 rows of Wg (shared-memory rows 0-63 of a packed stage) and the same 64 rows
// of Wu (rows 64-127). TMEM lane r holds output row gated_out_row(r) of the
// gate (bit 3 of r clear) or of the up projection (bit 3 set), read from
// shared-memory row gated_smem_row(r): g and u of one output sit in lanes r and
// r ^ 8 of one warp, and each run of 8 lanes reads 8 distinct swizzle rows.
__device__ __forceinline__ int gated_out_row(int r) { return ((r >> 4) << 3) | (r & 7); }
__device__ __forceinline__ int gated_smem_row(int r) { return ((r >> 3) & 1) * 64 + gated_out_row(r); }

// Sticky device error word (one per device, in api.cu's module).
__device__ __forceinline__ void raise_device_error(unsigned int* word, unsigned int code) {
    if (word) atomicCAS(word, 0u, code);
}

// ------------------------------------------------------------------- host --

struct DeviceInfo {
    int device;
    int sms;
    int cc_major, cc_minor;
    size_t smem_optin;                // largest dynamic shared memory a block may opt in to
    unsigned int* error_word;  // device address of the sticky error word
};

// Cached per-device properties of the current device (nullptr on failure).
const DeviceInfo* device_info();

// One-time set-up per device for one call site: kernel attributes such as the
// dynamic shared-memory limit belong to each device's context, so they are set
// once on every device that launches the kernel.
struct PerDeviceOnce {
    std::once_flag flag[kMaxDevices];
    cudaError_t err[kMaxDevices] = {};

    template <class F>
    cudaError_t run(int device, F&& setup) {
        std::call_once(flag[device], [&] { err[device] = setup(); });
        return err[device];
    }
};

// Host validation shared by w4a16_linear, w4a16_linear_ex and the
// allocation-free entry point: sizes, group, null pointers, 16-byte
// alignment and the device (sm_103). On W4A16_OK with M, N > 0, *dev is the
// current device's properties.
w4a16_status check_linear(const void* x, const void* qw, const void* s, const void* y, int64_t M, int64_t N,
                          int64_t K, int32_t group, const DeviceInfo** dev);

// Launch options of the decode GEMV (flags of the _ex entry points).
struct GemvOptions {
    bool static_weights = false;  // weights may be streamed before the previous kernel completes
};

// GEMV (decode, M <= 16).
size_t gemv_workspace_bytes(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K, bool gated = false);
// Offset of the arrival counters inside a GEMV workspace (they follow the partials).
size_t partial_region_bytes(const DeviceInfo& dev);
w4a16_status gemv_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw,
                         const uint16_t* s, uint16_t* y, int64_t M, int64_t N, int64_t K,
                         int group, void* workspace, size_t workspace_bytes, const GemvOptions& opt,
                         cudaStream_t st);
w4a16_status gemv_gated_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw_gate,
                               const uint16_t* s_gate, const uint8_t* qw_up, const uint16_t* s_up, uint16_t* y,
                               int64_t M, int64_t N, int64_t K, int group, void* workspace, size_t workspace_bytes,
                               const GemvOptions& opt, cudaStream_t st);

// Quantizer / unpack.
w4a16_status pack_launch(const float* w, int64_t N, int64_t K, int group, uint8_t* qw,
                         uint16_t* s, cudaStream_t st);
w4a16_status unpack_launch(const uint8_t* qw, int64_t N, int64_t K, int8_t* q, cudaStream_t st);

// Tensor-core GEMM (prefill and routed experts).
w4a16_status gemm_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw,
                         const uint16_t* s, uint16_t* y, int64_t M, int64_t N, int64_t K,
                         int group, const int32_t* expert_offsets, int E, cudaStream_t st);
// y = silu(x Wg^T) * (x Wu^T) for M > 16 on the tensor-core GEMM: each tile
// holds 64 rows of Wg and the same 64 rows of Wu.
w4a16_status gemm_gated_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qweight_gate,
                               const uint16_t* scales_gate, const uint8_t* qweight_up, const uint16_t* scales_up,
                               uint16_t* y, int64_t M, int64_t N, int64_t K, int group, cudaStream_t st);

// Tensor-core GEMM with the scale split exactly into the A operand (routed
// experts and dense layers): groups 32, 64 and 128, E <= 4096 experts.
bool split_supports(int group, int E);
// gather: token of each of the M rows (x is then [T, K], token-major); nullptr: x is [M, K].
w4a16_status split_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                          int64_t M, int64_t N, int64_t K, int group, const int32_t* expert_offsets, int E,
                          const int32_t* gather, int64_t T, cudaStream_t st);
// y = silu(x Wg^T) * (x Wu^T) on the split kernel (dense): each tile holds 64
// rows of Wg and the same 64 rows of Wu.
w4a16_status split_gated_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw_gate,
                                const uint16_t* s_gate, const uint8_t* qw_up, const uint16_t* s_up, uint16_t* y,
                                int64_t M, int64_t N, int64_t K, int group, cudaStream_t st);

// Routed-MoE router, dispatch (permutation + gather) and combine.
w4a16_status moe_route_launch(const float* logits, int64_t T, int E, int top_k, bool renormalize, int32_t* ids,
                              float* weights, cudaStream_t st);
size_t moe_dispatch_workspace_bytes(int64_t P, int E);
int moe_max_experts();
w4a16_status moe_dispatch_launch(const DeviceInfo& dev, const int32_t* ids, int64_t T, int k, int E,
                                 const uint16_t* x, int64_t K, int32_t* offsets, int32_t* row_of,
                                 int32_t* token_of_row, uint16_t* x_sorted, void* workspace, cudaStream_t st);
w4a16_status moe_combine_launch(const DeviceInfo& dev, const uint16_t* y_sorted, int64_t R, const int32_t* row_of,
                                const float* weights, int64_t T, int k, int64_t N, uint16_t* y, cudaStream_t st);

// GGUF block formats (Q4_K, Q5_1): decode GEMV and fp32 dequantizer.
int64_t blocks_row_bytes(int32_t format, int64_t K);
w4a16_status blocks_linear_launch(const DeviceInfo& dev, int32_t format, const uint16_t* x, const uint8_t* w,
                                  uint16_t* y, int64_t M, int64_t N, int64_t K, cudaStream_t st);
w4a16_status blocks_dequant_launch(int32_t format, const uint8_t* w, int64_t N, int64_t K, float* out,
                                   cudaStream_t st);

#ifdef W4A16_TEST_HOOKS
// Test-only build (compiled with -DW4A16_TEST_HOOKS into a separate library):
// the bounded waits give up after a limit the test chooses, and the TMA
// producers stop after a given number of copies, so a test can make a wait
// run out and check the error status and the unwind, with nothing faulting or
// hanging. The production library has none of this.
struct TestHooks {
    unsigned long long wait_limit_ns;  // limit of every bounded wait
    int issue_limit;                   // copies a producer may issue (per ring); < 0: no limit
};
// Counters the GEMM keeps in the test build: TMEM allocations and frees.
struct TestCounters {
    unsigned long long tmem_allocs, tmem_frees;
};
cudaError_t gemv_set_test_hooks(const TestHooks& h);
cudaError_t gemm_set_test_hooks(const TestHooks& h);
cudaError_t gemm_get_test_counters(TestCounters* c);
cudaError_t split_set_test_hooks(const TestHooks& h);
cudaError_t split_get_test_counters(TestCounters* c);
#endif

// Records a failed CUDA runtime call for w4a16_last_cuda_error (per host thread).
void note_cuda_error(cudaError_t e, const char* where);

inline w4a16_status cuda_status(cudaError_t e, const char* where = "CUDA call") {
    if (e == cudaSuccess) return W4A16_OK;
    note_cuda_error(e, where);
    return W4A16_ERR_CUDA;
}

}  // namespace w4a16
