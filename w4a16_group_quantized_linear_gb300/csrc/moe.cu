// Routed-MoE dispatch around the grouped layer: the softmax top-k router, the
// expert-major permutation of the (token, slot) pairs with the gather of x into
// that order, and the router-weighted combine of the experts' outputs.
//
// The router is the one the infr README's model table names for the Qwen3 MoE
// ("softmax router, top-k experts"; the Gemma 4 MoE routes "8-of-128"); the
// LLM170 page runs such experts at group 32 ("MoE resident"). Every kernel here
// is deterministic: the permutation is a stable counting sort (integer counts
// only) and the sums run in a fixed order.
#include <cfloat>
#include <climits>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kChunk = 1024;  // pairs per counting-sort chunk
constexpr int kMaxE = 4096;   // experts (one int per expert in shared memory)
constexpr int kBlockRankMaxE = 256;  // experts up to which a whole block ranks a chunk at once

// Every kernel here may start while the kernel before it on the stream is still
// running (programmatic dependent launch): it reads nothing before the wait,
// which returns once that kernel has completed and its writes are visible.
__device__ __forceinline__ void after_previous_kernel() {
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
}

// ------------------------------------------------------------------ router --

// One warp per token. Lane l holds logits l, l+32, ... of its token (NPL per
// lane). The selection compares the fp32 logits themselves: the larger logit
// wins and equal logits go to the lower expert index, exactly as a stable sort
// by falling logit would order them.
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int64_t T, int E, int top_k,
                                                    int renormalize, int32_t* __restrict__ ids,
                                                    float* __restrict__ weights) {
    after_previous_kernel();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + t * E;
    float v[NPL];
    uint32_t avail = 0;  // bit i: logit i*32+lane exists and is not yet selected
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = i * 32 + lane;
        v[i] = e < E ? __ldg(row + e) : -FLT_MAX;
        if (e < E) avail |= 1u << i;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
        if (avail >> i & 1u) mx = fmaxf(mx, v[i]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
        if (avail >> i & 1u) sum += expf(v[i] - mx);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);

    float my_w = 0.0f;  // lane s keeps the weight of selection s
    int my_id = 0;
    for (int s = 0; s < top_k; ++s) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = i * 32 + lane;
            if ((avail >> i & 1u) && (bi == INT_MAX || v[i] > bv)) {  // first maximum of this lane
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
            if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
        if (lane == s) {
            my_id = bi;
            my_w = expf(bv - mx) / sum;
        }
    }
    if (renormalize) {
        float ws = lane < top_k ? my_w : 0.0f;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, d);
        my_w = my_w / ws;
    }
    if (lane < top_k) {
        ids[t * top_k + lane] = my_id;
        weights[t * top_k + lane] = my_w;
    }
}

// ---------------------------------------------------------------- dispatch --

// Pass 1: per-chunk expert counts. hist[c][e] = pairs of chunk c routed to e.
// Ids outside [0, E) are reported, left out of every count and given row -1.
__global__ void __launch_bounds__(256) count_kernel(const int32_t* __restrict__ ids, int64_t P, int E,
                                                    int32_t* __restrict__ hist, int32_t* __restrict__ row_of,
                                                    unsigned int* err) {
    extern __shared__ int32_t cnt[];
    after_previous_kernel();
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int64_t p0 = (int64_t)blockIdx.x * kChunk;
    for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
        const int64_t p = p0 + i;
        if (p >= P) break;
        const int e = __ldg(ids + p);
        if (e >= 0 && e < E) {
            atomicAdd(&cnt[e], 1);
        } else {
            row_of[p] = -1;
            raise_device_error(err, W4A16_ERR_BAD_ROUTING);
        }
    }
    __syncthreads();
    int32_t* h = hist + (int64_t)blockIdx.x * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = cnt[e];
}

// Pass 2 (one block of 1024 threads): expert_offsets from the column sums of
// hist, then hist[c][e] becomes the first row of chunk c's pairs of expert e.
// Threads own experts (coalesced over e) and read 8 chunks per batch, so the
// loads of a column overlap instead of waiting one by one.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ hist, int C, int E,
                                                    int32_t* __restrict__ offsets) {
    __shared__ int32_t first[kMaxE];  // column sums, then the first row of each expert
    __shared__ int32_t warp_sum[32];
    after_previous_kernel();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t sum = 0;
        int c = 0;
        for (; c + 8 <= C; c += 8) {
            int32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = hist[(int64_t)(c + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) sum += v[u];
        }
        for (; c < C; ++c) sum += hist[(int64_t)c * E + e];
        first[e] = sum;
    }
    __syncthreads();
    // exclusive scan over e: thread i owns experts [kPer i, kPer i + kPer)
    constexpr int kPer = kMaxE / 1024;
    const int e0 = threadIdx.x * kPer;
    int32_t mine = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (e0 + i < E) mine += first[e0 + i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int32_t w = warp_sum[lane];
        int32_t wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d) wi += o;
        }
        warp_sum[lane] = wi - w;
    }
    __syncthreads();
    int32_t base = warp_sum[warp] + incl - mine;
    if (threadIdx.x == 0) offsets[0] = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = e0 + i;
        if (e >= E) break;
        const int32_t n = first[e];
        first[e] = base;
        base += n;
        offsets[e + 1] = base;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = first[e];
        int c = 0;
        for (; c + 8 <= C; c += 8) {
            int32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = hist[(int64_t)(c + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                hist[(int64_t)(c + u) * E + e] = run;
                run += v[u];
            }
        }
        for (; c < C; ++c) {
            const int32_t n = hist[(int64_t)c * E + e];
            hist[(int64_t)c * E + e] = run;
            run += n;
        }
    }
}

// Pass 3: one warp per chunk walks its pairs in order, 32 at a time. Lanes that
// route to the same expert are ranked by lane (match_any), so the pairs of an
// expert keep their (token, slot) order.
__global__ void __launch_bounds__(32) scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int k, int E,
                                                     const int32_t* __restrict__ hist, int32_t* __restrict__ row_of,
                                                     int32_t* __restrict__ token_of_row) {
    extern __shared__ int32_t next[];
    after_previous_kernel();
    const int lane = threadIdx.x;
    const int64_t p0 = (int64_t)blockIdx.x * kChunk;
    int key[kChunk / 32];  // the chunk's expert ids, all loads in flight at once
#pragma unroll
    for (int i = 0; i < kChunk / 32; ++i) {
        const int64_t p = p0 + i * 32 + lane;
        key[i] = p < P ? __ldg(ids + p) : -2;  // -2: no pair
    }
    const int32_t* h = hist + (int64_t)blockIdx.x * E;
    for (int e = lane; e < E; e += 32) next[e] = h[e];
    __syncwarp();
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kChunk / 32; ++i) {
        const int64_t p = p0 + i * 32 + lane;
        int e = key[i];
        if (e != -2 && (e < 0 || e >= E)) e = -1;  // reported and marked by pass 1
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        int32_t pos = 0;
        if (e >= 0) pos = next[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && (peers & lt) == 0) next[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            row_of[p] = pos;
            token_of_row[pos] = (int32_t)(p / k);
        }
    }
}

// Pass 3 for E <= 256: a block of 32 warps ranks a whole chunk at once. Warp w
// takes pairs [32 w, 32 w + 32) of the chunk and ranks its lanes by expert
// (match_any); per-warp expert counts in shared memory, scanned over the warps,
// give each warp's first row per expert. The order is the pair order, as in
// scatter_kernel.
__global__ void __launch_bounds__(kChunk) scatter_block_kernel(const int32_t* __restrict__ ids, int64_t P, int k,
                                                               int E, const int32_t* __restrict__ hist,
                                                               int32_t* __restrict__ row_of,
                                                               int32_t* __restrict__ token_of_row) {
    extern __shared__ int32_t wcnt[];  // [32 warps][E]
    after_previous_kernel();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = lane; e < E; e += 32) wcnt[warp * E + e] = 0;
    const int64_t p = (int64_t)blockIdx.x * kChunk + threadIdx.x;
    int e = -2;  // no pair
    if (p < P) {
        e = __ldg(ids + p);
        if (e < 0 || e >= E) e = -1;  // reported and marked by pass 1
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t lt = (1u << lane) - 1u;
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    const int32_t* h = hist + (int64_t)blockIdx.x * E;
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int32_t run = h[x];
        for (int w = 0; w < kChunk / 32; ++w) {
            const int32_t n = wcnt[w * E + x];
            wcnt[w * E + x] = run;
            run += n;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int32_t pos = wcnt[warp * E + e] + __popc(peers & lt);
        row_of[p] = pos;
        token_of_row[pos] = (int32_t)(p / k);
    }
}

// x_sorted[r] = x[token_of_row[r]] for r < offsets[E]: one warp per row,
// 16-byte copies.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ x, int64_t K,
                                                     const int32_t* __restrict__ token_of_row,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     uint16_t* __restrict__ x_sorted) {
    after_previous_kernel();
    const int64_t rows = __ldg(offsets + E);
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t vec = K / 8;  // uint4 per row
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const int64_t t = __ldg(token_of_row + r);
        const uint4* src = reinterpret_cast<const uint4*>(x + t * K);
        uint4* dst = reinterpret_cast<uint4*>(x_sorted + r * K);
        int64_t i = lane;
        for (; i + 7 * 32 < vec; i += 8 * 32) {  // eight loads in flight per lane
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(src + i + u * 32);
#pragma unroll
            for (int u = 0; u < 8; ++u) dst[i + u * 32] = v[u];
        }
        for (; i < vec; i += 32) dst[i] = __ldg(src + i);
    }
}

// ----------------------------------------------------------------- combine --

// y[t, n] = sum_j w[t, j] * y_sorted[row_of[t, j], n]: fp32 FMAs in slot order,
// one rounding to fp16. Rows of -1 (dropped pairs) add nothing; a row outside
// [0, R) is reported and adds nothing. Each thread
// covers 8 consecutive n with 16-byte loads and stores.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y_sorted, int64_t R,
                                                      const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ weights, int k, int64_t N,
                                                      uint16_t* __restrict__ y, unsigned int* err) {
    after_previous_kernel();
    const int64_t t = blockIdx.x;
    const int64_t n0 = ((int64_t)blockIdx.y * blockDim.x + threadIdx.x) * 8;
    if (n0 >= N) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int32_t r = __ldg(row_of + t * k + j);
        if (r < 0) continue;
        if (r >= R) {
            raise_device_error(err, W4A16_ERR_BAD_ROUTING);
            continue;
        }
        const float w = __ldg(weights + t * k + j);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(y_sorted + (int64_t)r * N + n0));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
            acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(y + t * N + n0) = make_uint4(o[0], o[1], o[2], o[3]);
}

// The same for any N and alignment: one thread per element.
__global__ void __launch_bounds__(256) combine_scalar_kernel(const uint16_t* __restrict__ y_sorted, int64_t R,
                                                             const int32_t* __restrict__ row_of,
                                                             const float* __restrict__ weights, int k, int64_t N,
                                                             uint16_t* __restrict__ y, unsigned int* err) {
    after_previous_kernel();
    const int64_t t = blockIdx.x;
    const int64_t n = (int64_t)blockIdx.y * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int32_t r = __ldg(row_of + t * k + j);
        if (r < 0) continue;
        if (r >= R) {
            raise_device_error(err, W4A16_ERR_BAD_ROUTING);
            continue;
        }
        acc = fmaf(__ldg(weights + t * k + j), __half2float(__ushort_as_half(__ldg(y_sorted + (int64_t)r * N + n))),
                   acc);
    }
    y[t * N + n] = __half_as_ushort(__float2half_rn(acc));
}

}  // namespace

// ------------------------------------------------------------------- host --

template <typename... KArgs, typename... Args>
w4a16_status launch(const char* what, void (*kernel)(KArgs...), dim3 grid, unsigned block, size_t smem,
                    cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...), what);
}

w4a16_status moe_route_launch(const float* logits, int64_t T, int E, int top_k, bool renormalize, int32_t* ids,
                              float* weights, cudaStream_t st) {
    const int64_t blocks = (T + 7) / 8;
    if (blocks > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const int npl = (E + 31) / 32;
    const dim3 g((unsigned)blocks);
    const int rn = renormalize ? 1 : 0;
    if (npl <= 1) return launch("moe_route", route_kernel<1>, g, 256, 0, st, logits, T, E, top_k, rn, ids, weights);
    if (npl <= 2) return launch("moe_route", route_kernel<2>, g, 256, 0, st, logits, T, E, top_k, rn, ids, weights);
    if (npl <= 4) return launch("moe_route", route_kernel<4>, g, 256, 0, st, logits, T, E, top_k, rn, ids, weights);
    if (npl <= 8) return launch("moe_route", route_kernel<8>, g, 256, 0, st, logits, T, E, top_k, rn, ids, weights);
    if (npl <= 16) return launch("moe_route", route_kernel<16>, g, 256, 0, st, logits, T, E, top_k, rn, ids, weights);
    return launch("moe_route", route_kernel<32>, g, 256, 0, st, logits, T, E, top_k, rn, ids, weights);
}

size_t moe_dispatch_workspace_bytes(int64_t P, int E) {
    const int64_t C = (P + kChunk - 1) / kChunk;
    return (size_t)(C * E) * sizeof(int32_t);
}

int moe_max_experts() { return kMaxE; }

w4a16_status moe_dispatch_launch(const DeviceInfo& dev, const int32_t* ids, int64_t T, int k, int E,
                                 const uint16_t* x, int64_t K, int32_t* offsets, int32_t* row_of,
                                 int32_t* token_of_row, uint16_t* x_sorted, void* workspace, cudaStream_t st) {
    const int64_t P = T * k;
    const int64_t C = (P + kChunk - 1) / kChunk;
    if (C > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    int32_t* hist = static_cast<int32_t*>(workspace);
    const size_t smem = (size_t)E * sizeof(int32_t);
    w4a16_status s = W4A16_OK;
    if (C > 0) {
        s = launch("moe_dispatch: count", count_kernel, dim3((unsigned)C), 256, smem, st, ids, P, E, hist, row_of,
                   dev.error_word);
        if (s != W4A16_OK) return s;
    }
    s = launch("moe_dispatch: scan", scan_kernel, dim3(1), 1024, 0, st, hist, (int)C, E, offsets);
    if (s != W4A16_OK || C == 0) return s;
    if (E <= kBlockRankMaxE)
        s = launch("moe_dispatch: scatter", scatter_block_kernel, dim3((unsigned)C), kChunk,
                   (size_t)(kChunk / 32) * E * sizeof(int32_t), st, ids, P, k, E, (const int32_t*)hist, row_of,
                   token_of_row);
    else
        s = launch("moe_dispatch: scatter", scatter_kernel, dim3((unsigned)C), 32, smem, st, ids, P, k, E,
                   (const int32_t*)hist, row_of, token_of_row);
    if (s != W4A16_OK || K == 0) return s;
    const int64_t rows_per_block = 8;
    int64_t blocks = (P + rows_per_block - 1) / rows_per_block;
    const int64_t cap = (int64_t)dev.sms * 16;
    if (blocks > cap) blocks = cap;
    return launch("moe_dispatch: gather", gather_kernel, dim3((unsigned)blocks), 256, 0, st, x, K,
                  (const int32_t*)token_of_row, (const int32_t*)offsets, E, x_sorted);
}

w4a16_status moe_combine_launch(const DeviceInfo& dev, const uint16_t* y_sorted, int64_t R, const int32_t* row_of,
                                const float* weights, int64_t T, int k, int64_t N, uint16_t* y, cudaStream_t st) {
    if (T > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    const bool vec = N % 8 == 0 && ((uintptr_t)y_sorted & 15u) == 0 && ((uintptr_t)y & 15u) == 0;
    const int64_t per_block = vec ? 256 * 8 : 256;
    const int64_t gy = (N + per_block - 1) / per_block;
    if (gy > 65535) return W4A16_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)T, (unsigned)gy);
    if (vec)
        return launch("moe_combine", combine_kernel, grid, 256, 0, st, y_sorted, R, row_of, weights, k, N, y,
                      dev.error_word);
    return launch("moe_combine", combine_scalar_kernel, grid, 256, 0, st, y_sorted, R, row_of, weights, k, N, y,
                  dev.error_word);
}

}  // namespace w4a16
