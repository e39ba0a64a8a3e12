// C ABI of libw4a16.so: argument validation, per-device state and dispatch.
// The entry points and their contracts are documented in include/w4a16.h.
#include <mutex>

#include "internal.cuh"

#include <cstdio>

namespace w4a16 {

// Sticky device error word, one per device (module global).
__device__ unsigned int g_error_word;

namespace {
thread_local char t_last_error[256] = "no CUDA error recorded";
}

void note_cuda_error(cudaError_t e, const char* where) {
    snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

namespace {

constexpr int64_t kGemvMaxM = 16;

std::mutex g_info_mutex;
DeviceInfo g_info[kMaxDevices];
bool g_info_ready[kMaxDevices];

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

w4a16_status check_group(int64_t K, int32_t group) {
    if (group != 32 && group != 64 && group != 128) return W4A16_ERR_UNSUPPORTED;
    if (K < 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

}  // namespace

const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_info_mutex);
    if (!g_info_ready[dev]) {
        DeviceInfo d{};
        d.device = dev;
        int smem = 0;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return nullptr;
        d.smem_optin = (size_t)smem;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.error_word), g_error_word) != cudaSuccess)
            return nullptr;
        g_info[dev] = d;
        g_info_ready[dev] = true;
    }
    return &g_info[dev];
}

// Common validation of w4a16_linear / w4a16_grouped_linear / w4a16_linear_noalloc.
w4a16_status check_linear(const void* x, const void* qw, const void* s, const void* y, int64_t M, int64_t N,
                          int64_t K, int32_t group, const DeviceInfo** dev) {
    if (M < 0 || N < 0 || K < 0) return W4A16_ERR_INVALID_ARG;
    const w4a16_status g = check_group(K, group);
    if (g != W4A16_OK) return g;
    if (M == 0 || N == 0) return W4A16_OK;
    if (!y || (K > 0 && (!x || !qw || !s))) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(s) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
    *dev = device_info();
    if (!*dev) return W4A16_ERR_CUDA;
    if ((*dev)->cc_major != 10 || (*dev)->cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
    return W4A16_OK;
}

namespace {

constexpr uint32_t kKnownFlags = W4A16_STATIC_WEIGHTS;

GemvOptions gemv_options(uint32_t flags) {
    GemvOptions o;
    o.static_weights = (flags & W4A16_STATIC_WEIGHTS) != 0;
    return o;
}

w4a16_status linear_impl(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales, uint16_t* y, int64_t M,
                         int64_t N, int64_t K, int32_t group, uint32_t flags, void* workspace, size_t workspace_bytes,
                         void* stream) {
    if (flags & ~kKnownFlags) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    const w4a16_status v = check_linear(x, qweight, scales, y, M, N, K, group, &dev);
    if (v != W4A16_OK || M == 0 || N == 0) return v;
    cudaStream_t st = (cudaStream_t)stream;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(uint16_t), st));
    if (M <= kGemvMaxM)
        return gemv_launch(*dev, x, qweight, scales, y, M, N, K, group, workspace, workspace_bytes,
                           gemv_options(flags), st);
    return gemm_launch(*dev, x, qweight, scales, y, M, N, K, group, nullptr, 1, st);
}

w4a16_status linear_gated_impl(const uint16_t* x, const uint8_t* qweight_gate, const uint16_t* scales_gate,
                               const uint8_t* qweight_up, const uint16_t* scales_up, uint16_t* y, int64_t M,
                               int64_t N, int64_t K, int32_t group, uint32_t flags, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (flags & ~kKnownFlags) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    w4a16_status v = check_linear(x, qweight_gate, scales_gate, y, M, N, K, group, &dev);
    if (v != W4A16_OK || M == 0 || N == 0) return v;
    if (K > 0 && (!qweight_up || !scales_up)) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(qweight_up) || !aligned16(scales_up)) return W4A16_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(uint16_t), st));  // silu(0) * 0
    if (M > kGemvMaxM)
        return gemm_gated_launch(*dev, x, qweight_gate, scales_gate, qweight_up, scales_up, y, M, N, K, group, st);
    return gemv_gated_launch(*dev, x, qweight_gate, scales_gate, qweight_up, scales_up, y, M, N, K, group, workspace,
                             workspace_bytes, gemv_options(flags), st);
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" {

int32_t w4a16_version(void) { return 100; }

const char* w4a16_last_cuda_error(void) { return t_last_error; }

const char* w4a16_status_string(w4a16_status status) {
    switch (status) {
        case W4A16_OK: return "W4A16_OK";
        case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG: invalid argument";
        case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED: unsupported group, shape or device";
        case W4A16_ERR_MISALIGNED: return "W4A16_ERR_MISALIGNED: pointer not 16-byte aligned";
        case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA: CUDA runtime error";
        case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT: a device wait gave up";
        case W4A16_ERR_BAD_OFFSETS: return "W4A16_ERR_BAD_OFFSETS: expert offsets are not a partition of the rows";
        case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE: workspace missing or too small";
        case W4A16_ERR_BAD_ROUTING: return "W4A16_ERR_BAD_ROUTING: an expert id or a combine row is out of range";
    }
    return "W4A16: unknown status";
}

int64_t w4a16_blocks_row_bytes(int32_t format, int64_t K) { return blocks_row_bytes(format, K); }

w4a16_status w4a16_blocks_linear(int32_t format, const uint16_t* x, const uint8_t* blocks, uint16_t* y, int64_t M,
                                 int64_t N, int64_t K, void* stream) {
    if (format != W4A16_FORMAT_Q4_K && format != W4A16_FORMAT_Q5_1) return W4A16_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || blocks_row_bytes(format, K) < 0) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    if (!y || (K > 0 && (!x || !blocks))) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(blocks) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
    const DeviceInfo* dev = device_info();
    if (!dev) return W4A16_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, (size_t)(M * N) * sizeof(uint16_t), st));
    return blocks_linear_launch(*dev, format, x, blocks, y, M, N, K, st);
}

w4a16_status w4a16_blocks_dequant(int32_t format, const uint8_t* blocks, int64_t N, int64_t K, float* w,
                                  void* stream) {
    if (format != W4A16_FORMAT_Q4_K && format != W4A16_FORMAT_Q5_1) return W4A16_ERR_UNSUPPORTED;
    if (N < 0 || blocks_row_bytes(format, K) < 0) return W4A16_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return W4A16_OK;
    if (!blocks || !w) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(w)) return W4A16_ERR_MISALIGNED;
    const DeviceInfo* dev = device_info();
    if (!dev) return W4A16_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
    return blocks_dequant_launch(format, blocks, N, K, w, (cudaStream_t)stream);
}

w4a16_status w4a16_pack(const float* w, int64_t N, int64_t K, int32_t group, uint8_t* qweight, uint16_t* scales,
                        void* stream) {
    if (N < 0 || K < 0) return W4A16_ERR_INVALID_ARG;
    const w4a16_status g = check_group(K, group);
    if (g != W4A16_OK) return g;
    if (N == 0 || K == 0) return W4A16_OK;
    if (!w || !qweight || !scales) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = device_info();
    if (!dev) return W4A16_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
    return pack_launch(w, N, K, group, qweight, scales, (cudaStream_t)stream);
}

w4a16_status w4a16_unpack(const uint8_t* qweight, int64_t N, int64_t K, int8_t* q, void* stream) {
    if (N < 0 || K < 0 || (K & 1)) return W4A16_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return W4A16_OK;
    if (!qweight || !q) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = device_info();
    if (!dev) return W4A16_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
    return unpack_launch(qweight, N, K, q, (cudaStream_t)stream);
}

size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t group, int32_t E) {
    if (M <= 0 || N <= 0 || K <= 0 || E < 1 || check_group(K, group) != W4A16_OK) return 0;
    const DeviceInfo* dev = device_info();
    if (!dev) return 0;
    if (E == 1 && M <= kGemvMaxM) return gemv_workspace_bytes(*dev, M, N, K);
    return 0;
}

w4a16_status w4a16_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (workspace_bytes == 0) return W4A16_OK;
    if (!workspace) return W4A16_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream));
}

w4a16_status w4a16_linear(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales, uint16_t* y,
                          int64_t M, int64_t N, int64_t K, int32_t group, void* workspace, size_t workspace_bytes,
                          void* stream) {
    return linear_impl(x, qweight, scales, y, M, N, K, group, 0u, workspace, workspace_bytes, stream);
}

w4a16_status w4a16_linear_ex(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales, uint16_t* y,
                             int64_t M, int64_t N, int64_t K, int32_t group, uint32_t flags, void* workspace,
                             size_t workspace_bytes, void* stream) {
    return linear_impl(x, qweight, scales, y, M, N, K, group, flags, workspace, workspace_bytes, stream);
}

w4a16_status w4a16_linear_gated(const uint16_t* x, const uint8_t* qweight_gate, const uint16_t* scales_gate,
                                const uint8_t* qweight_up, const uint16_t* scales_up, uint16_t* y, int64_t M,
                                int64_t N, int64_t K, int32_t group, void* workspace, size_t workspace_bytes,
                                void* stream) {
    return linear_gated_impl(x, qweight_gate, scales_gate, qweight_up, scales_up, y, M, N, K, group, 0u, workspace,
                             workspace_bytes, stream);
}

w4a16_status w4a16_linear_gated_ex(const uint16_t* x, const uint8_t* qweight_gate, const uint16_t* scales_gate,
                                   const uint8_t* qweight_up, const uint16_t* scales_up, uint16_t* y, int64_t M,
                                   int64_t N, int64_t K, int32_t group, uint32_t flags, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    return linear_gated_impl(x, qweight_gate, scales_gate, qweight_up, scales_up, y, M, N, K, group, flags,
                             workspace, workspace_bytes, stream);
}

size_t w4a16_linear_gated_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t group) {
    if (M <= 0 || M > kGemvMaxM || N <= 0 || K <= 0 || check_group(K, group) != W4A16_OK) return 0;
    const DeviceInfo* dev = device_info();
    if (!dev) return 0;
    return gemv_workspace_bytes(*dev, M, N, K, true);
}

w4a16_status w4a16_grouped_linear(const uint16_t* x_sorted, const uint8_t* qweight, const uint16_t* scales,
                                  const int32_t* expert_offsets, uint16_t* y_sorted, int32_t E, int64_t R,
                                  int64_t N, int64_t K, int32_t group, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (E < 1 || !expert_offsets) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    const w4a16_status v = check_linear(x_sorted, qweight, scales, y_sorted, R, N, K, group, &dev);
    if (v != W4A16_OK || R == 0 || N == 0) return v;
    cudaStream_t st = (cudaStream_t)stream;
    if (K == 0) return cuda_status(cudaMemsetAsync(y_sorted, 0, (size_t)(R * N) * sizeof(uint16_t), st));
    return gemm_launch(*dev, x_sorted, qweight, scales, y_sorted, R, N, K, group, expert_offsets, E, st);
}

w4a16_status w4a16_grouped_linear_gather(const uint16_t* x, int64_t T, const int32_t* token_of_row,
                                         const uint8_t* qweight, const uint16_t* scales,
                                         const int32_t* expert_offsets, uint16_t* y_sorted, int32_t E, int64_t R,
                                         int64_t N, int64_t K, int32_t group, void* stream) {
    if (E < 1 || T < 0 || !expert_offsets) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    const w4a16_status v = check_linear(x, qweight, scales, y_sorted, R, N, K, group, &dev);
    if (v != W4A16_OK || R == 0 || N == 0) return v;
    if (group != 32 || !split_supports(group, E)) return W4A16_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    if (K == 0) return cuda_status(cudaMemsetAsync(y_sorted, 0, (size_t)(R * N) * sizeof(uint16_t), st));
    if (!token_of_row || T == 0) return W4A16_ERR_INVALID_ARG;
    return split_launch(*dev, x, qweight, scales, y_sorted, R, N, K, group, expert_offsets, E, token_of_row, T, st);
}

namespace {
// The current device, if it is the sm_103 part the kernels are built for.
w4a16_status current_device(const DeviceInfo** dev) {
    *dev = device_info();
    if (!*dev) return W4A16_ERR_CUDA;
    if ((*dev)->cc_major != 10 || (*dev)->cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
    return W4A16_OK;
}
}  // namespace

w4a16_status w4a16_moe_route(const float* logits, int64_t T, int32_t E, int32_t top_k, int32_t renormalize,
                             int32_t* topk_ids, float* topk_weights, void* stream) {
    if (T < 0 || E < 1 || top_k < 1 || top_k > E) return W4A16_ERR_INVALID_ARG;
    if (E > 1024 || top_k > 32) return W4A16_ERR_UNSUPPORTED;
    if (T == 0) return W4A16_OK;
    if (!logits || !topk_ids || !topk_weights) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    const w4a16_status d = current_device(&dev);
    if (d != W4A16_OK) return d;
    return moe_route_launch(logits, T, E, top_k, renormalize != 0, topk_ids, topk_weights, (cudaStream_t)stream);
}

size_t w4a16_moe_dispatch_workspace_bytes(int64_t T, int32_t top_k, int32_t E) {
    if (T < 0 || top_k < 1 || E < 1 || E > moe_max_experts() || T > 0x7fffffffLL / top_k) return 0;
    return moe_dispatch_workspace_bytes(T * top_k, E);
}

w4a16_status w4a16_moe_dispatch(const int32_t* topk_ids, int64_t T, int32_t top_k, int32_t E, const uint16_t* x,
                                int64_t K, int32_t* expert_offsets, int32_t* row_of, int32_t* token_of_row,
                                uint16_t* x_sorted, void* workspace, size_t workspace_bytes, void* stream) {
    if (T < 0 || top_k < 1 || E < 1 || K < 0 || !expert_offsets) return W4A16_ERR_INVALID_ARG;
    if (E > moe_max_experts() || T > 0x7fffffffLL / top_k) return W4A16_ERR_UNSUPPORTED;
    if (T > 0 && (!topk_ids || !row_of || !token_of_row)) return W4A16_ERR_INVALID_ARG;
    if (T > 0 && K > 0) {
        if (!x || !x_sorted) return W4A16_ERR_INVALID_ARG;
        if (K % 8 != 0) return W4A16_ERR_UNSUPPORTED;
        if (!aligned16(x) || !aligned16(x_sorted)) return W4A16_ERR_MISALIGNED;
    }
    const size_t need = moe_dispatch_workspace_bytes(T * top_k, E);
    if (need > 0 && (!workspace || workspace_bytes < need)) return W4A16_ERR_WORKSPACE;
    const DeviceInfo* dev = nullptr;
    const w4a16_status d = current_device(&dev);
    if (d != W4A16_OK) return d;
    return moe_dispatch_launch(*dev, topk_ids, T, top_k, E, x, T > 0 ? K : 0, expert_offsets, row_of, token_of_row,
                               x_sorted, workspace, (cudaStream_t)stream);
}

w4a16_status w4a16_moe_combine(const uint16_t* y_sorted, int64_t R, const int32_t* row_of, const float* topk_weights,
                               int64_t T, int32_t top_k, int64_t N, uint16_t* y, void* stream) {
    if (R < 0 || T < 0 || top_k < 1 || N < 0) return W4A16_ERR_INVALID_ARG;
    if (T == 0 || N == 0) return W4A16_OK;
    if (!row_of || !topk_weights || !y || (R > 0 && !y_sorted)) return W4A16_ERR_INVALID_ARG;
    const DeviceInfo* dev = nullptr;
    const w4a16_status d = current_device(&dev);
    if (d != W4A16_OK) return d;
    return moe_combine_launch(*dev, y_sorted, R, row_of, topk_weights, T, top_k, N, y, (cudaStream_t)stream);
}

#ifdef W4A16_TEST_HOOKS
// Test-only build: set the wait limit and the producers' issue limit of the
// GEMV and the GEMM (synchronous), and read the GEMM's TMEM counters.
W4A16_API w4a16_status w4a16_test_set_hooks(uint64_t wait_limit_ns, int32_t issue_limit) {
    const TestHooks h{(unsigned long long)wait_limit_ns, (int)issue_limit};
    w4a16_status a = cuda_status(gemv_set_test_hooks(h), "test hooks (gemv)");
    if (a == W4A16_OK) a = cuda_status(gemm_set_test_hooks(h), "test hooks (gemm)");
    if (a == W4A16_OK) a = cuda_status(split_set_test_hooks(h), "test hooks (gemm g32)");
    return a;
}

W4A16_API w4a16_status w4a16_test_tmem_counters(uint64_t* allocs, uint64_t* frees) {
    TestCounters c{}, d{};
    w4a16_status a = cuda_status(gemm_get_test_counters(&c), "test counters");
    if (a == W4A16_OK) a = cuda_status(split_get_test_counters(&d), "test counters (gemm g32)");
    if (a != W4A16_OK) return a;
    *allocs = c.tmem_allocs + d.tmem_allocs;
    *frees = c.tmem_frees + d.tmem_frees;
    return W4A16_OK;
}
#endif

w4a16_status w4a16_device_status(void* stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return W4A16_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    unsigned int word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return W4A16_ERR_CUDA;
    if (cudaMemcpyAsync(&word, dev->error_word, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(dev->error_word, 0, sizeof(word), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return W4A16_ERR_CUDA;
    return (w4a16_status)word;
}

}  // extern "C"
