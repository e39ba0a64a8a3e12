// w4a16_linear_noalloc: w4a16_linear for callers that cannot allocate device
// memory. The decode GEMV's scratch is a fixed array in this module instead of
// a caller-provided workspace; see include/w4a16.h for the contract.
#include <mutex>

#include "internal.cuh"

namespace w4a16 {
namespace {

constexpr size_t kScratchBytes = W4A16_NOALLOC_SCRATCH_BYTES;

// One copy per device, resident while the library is loaded.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device with that device current (nullptr on failure).
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch[dev] = p;
    }
    return g_scratch[dev];
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" w4a16_status w4a16_linear_noalloc(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales,
                                             uint16_t* y, int64_t M, int64_t N, int64_t K, int32_t group,
                                             void* stream) {
    // the same host checks as w4a16_linear, before the shared array is touched,
    // so an invalid call neither clears it nor reports anything but its own error
    const DeviceInfo* dev = nullptr;
    const w4a16_status v = check_linear(x, qweight, scales, y, M, N, K, group, &dev);
    if (v != W4A16_OK || M == 0 || N == 0 || K == 0)
        return v != W4A16_OK ? v : w4a16_linear(x, qweight, scales, y, M, N, K, group, nullptr, 0, stream);
    // 0 for the tensor-core path, which needs no scratch
    const size_t need = w4a16_workspace_bytes(M, N, K, group, 1);
    if (need > kScratchBytes) return W4A16_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_address();
        if (scratch == nullptr) return W4A16_ERR_CUDA;
        // the arrival counters must start at zero; the partial sums need no clearing
        const size_t counters = partial_region_bytes(*dev);
        if (cudaMemsetAsync(static_cast<char*>(scratch) + counters, 0, need - counters, (cudaStream_t)stream) !=
            cudaSuccess)
            return W4A16_ERR_CUDA;
    }
    return w4a16_linear(x, qweight, scales, y, M, N, K, group, scratch, scratch ? kScratchBytes : 0, stream);
}
