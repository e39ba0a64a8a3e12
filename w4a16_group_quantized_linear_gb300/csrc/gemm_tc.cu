// Tensor-core GEMM of the W4A16 layer for prefill (M >= 17 rows) and for the
// routed-expert layer (LLM170 page: "pp512 / pp4096" prefill, "MoE resident"
// g32 models). sm_103a: TMA, tcgen05 MMA with TMEM accumulators.
//
// Formulation ("swap AB"): the MMA computes D[n, m] = sum_k W[n, k] x[m, k],
// so weight rows n sit in the 128 TMEM lanes and tokens m in the columns.
//
// Per CTA tile: 128 weight rows x 128 tokens, K in chunks of 64.
//   warp 0      TMA producer: x tile (fp16, 128-byte swizzle) and the packed
//               weight tile (128 rows x 32 bytes) into a 4-stage ring.
//   warps 2..5  dequant: thread i expands row i of the packed tile into the
//               exact fp16 integers q (no scale) in the swizzled K-major
//               layout the MMA reads.
//   warp 1      one lane issues tcgen05.mma (M=128, N=128, K=16) into TMEM.
//               Each scale group gets its own fp32 partial in one of two TMEM
//               buffers; a commit per group hands it to the epilogue.
//   warps 6..9  epilogue: per group, read the partial from TMEM, multiply by
//               that row's fp32 scale and add into fp32 registers
//               (acc += s[n, grp] * sum_{k in grp} x q); at the end round once
//               to fp16 and store y[m, n].
// So every product x*q is exact, each group sum is fp32 and the scale is
// applied in fp32, as in the decode GEMV: no fp16 rounding of s*q.
//
// Every mbarrier wait is bounded in time; a wait that gives up records
// W4A16_ERR_TIMEOUT in the device error word and the CTA unwinds (it drains
// its own TMA loads and MMAs first, then frees TMEM).
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kBM = 128;      // weight rows per tile (TMEM lanes)
constexpr int kBN = 128;      // tokens per tile (TMEM columns per partial buffer)
constexpr int kBK = 64;       // k per pipeline stage (one 128-byte swizzle row of fp16)
constexpr int kStages = 4;
constexpr int kThreads = 320;  // 10 warps
constexpr uint32_t kTmemCols = 2 * kBN;

constexpr int kABytes = kBM * kBK * 2;   // dequantized weights, fp16
constexpr int kXBytes = kBN * kBK * 2;   // activations, fp16
constexpr int kPBytes = kBM * kBK / 2;   // packed weights
constexpr int kSmemBytes = kStages * (kABytes + kXBytes + kPBytes) + 1024 /*align*/ + 256 /*barriers*/;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s

struct GemmArgs {
    const uint16_t* s;
    uint16_t* y;
    const int32_t* offsets;  // nullptr: dense layer
    int64_t M, N, K;         // M = rows of x (R for routed experts)
    int E;
    unsigned int* err;
};

struct Smem {
    uint64_t full[kStages];    // TMA bytes landed (x tile + packed tile)
    uint64_t empty[kStages];   // MMAs reading the stage finished
    uint64_t afull[kStages];   // dequantized A tile written
    uint64_t dfull[2];         // group partial ready in TMEM buffer b
    uint64_t dempty[2];        // epilogue done reading TMEM buffer b
    uint64_t mma_done;         // all MMAs of this CTA finished
    uint32_t tmem_base;
    int abort;
    int expert, row0, row_end, valid;
};

__device__ __forceinline__ void fail(const GemmArgs& a, Smem* sm, unsigned code) {
    raise_device_error(a.err, code);
    *reinterpret_cast<volatile int*>(&sm->abort) = 1;
}

// Routed experts: the CTA's token tile from the device offsets. One warp.
__device__ void find_tile(const GemmArgs& a, Smem* sm, int lane) {
    const int t = blockIdx.x;
    int base = 0;  // tiles of experts before the current chunk
    bool ok = true;
    int found = -1, f_row0 = 0, f_end = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0, hi = 0, tiles = 0;
        if (e < a.E) {
            lo = __ldg(a.offsets + e);
            hi = __ldg(a.offsets + e + 1);
            if (hi < lo || lo < 0 || (int64_t)hi > a.M) ok = false;
            tiles = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;
        }
        int incl = tiles;  // inclusive scan over the warp
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        const int start = base + incl - tiles;
        if (e < a.E && t >= start && t < start + tiles) {
            found = e;
            f_row0 = lo + (t - start) * kBN;
            f_end = hi;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    ok = __all_sync(0xffffffffu, ok);
    const bool ends_ok = __ldg(a.offsets) == 0 && (int64_t)__ldg(a.offsets + a.E) == a.M;
    if (lane == 0) {
        sm->valid = 0;
        if (!ok || !ends_ok) raise_device_error(a.err, W4A16_ERR_BAD_OFFSETS);
    }
    __syncwarp();
    if (ok && ends_ok && found >= 0) {  // tiles are disjoint: at most one lane
        sm->expert = found;
        sm->row0 = f_row0;
        sm->row_end = f_end;
        sm->valid = 1;
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                const GemmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = base;                                  // kStages x 16 KB
    uint8_t* sX = sA + kStages * kABytes;                // kStages x 16 KB
    uint8_t* sP = sX + kStages * kXBytes;                // kStages x 4 KB
    Smem* sm = reinterpret_cast<Smem*>(sP + kStages * kPBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = (int64_t)blockIdx.y * kBM;

    // ---- which tokens this CTA owns
    if (warp == 0) {
        if (a.offsets == nullptr) {
            if (lane == 0) {
                sm->expert = 0;
                sm->row0 = blockIdx.x * kBN;
                sm->row_end = (int)a.M;
                sm->valid = 1;
            }
        } else {
            find_tile(a, sm, lane);
        }
        if (lane == 0) {
            for (int i = 0; i < kStages; ++i) {
                ptx::mbar_init(&sm->full[i], 1);
                ptx::mbar_init(&sm->empty[i], 1);
                ptx::mbar_init(&sm->afull[i], 128);
            }
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(&sm->dfull[b], 1);
                ptx::mbar_init(&sm->dempty[b], 128);
            }
            ptx::mbar_init(&sm->mma_done, 1);
            sm->abort = 0;
            ptx::fence_mbar_init();
            ptx::prefetch_tensormap(&tmap_x);
            ptx::prefetch_tensormap(&tmap_w);
        }
    }
    __syncthreads();
    if (!sm->valid) return;  // tile past the last expert's rows, or bad offsets
    if (warp == 1) {
        ptx::tmem_alloc(&sm->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    const int expert = sm->expert, row0 = sm->row0, row_end = sm->row_end;
    const int nchunks = (int)((a.K + kBK - 1) / kBK);
    const int ngroups = (int)(a.K / G);
    volatile int* abort = &sm->abort;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kStages, round = c / kStages;
                if (round > 0 && !ptx::mbar_wait(&sm->empty[st], (round - 1) & 1, abort, kWaitLimitNs)) {
                    fail(a, sm, W4A16_ERR_TIMEOUT);
                    break;
                }
                ptx::mbar_arrive_expect_tx(&sm->full[st], kXBytes + kPBytes);
                ptx::tma_load_2d(sX + st * kXBytes, &tmap_x, &sm->full[st], c * kBK, row0);
                if (a.offsets == nullptr)
                    ptx::tma_load_2d(sP + st * kPBytes, &tmap_w, &sm->full[st], c * (kBK / 2), (int)n0);
                else
                    ptx::tma_load_3d(sP + st * kPBytes, &tmap_w, &sm->full[st], c * (kBK / 2), (int)n0, expert);
                ++issued;
            }
            if (*abort) {  // let our own loads land before the CTA exits
                volatile int never = 0;
                for (int c = issued - kStages < 0 ? 0 : issued - kStages; c < issued; ++c)
                    ptx::mbar_wait(&sm->full[c % kStages], (c / kStages) & 1, &never, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(kBM, kBN);
            for (int c = 0; c < nchunks && !*abort; ++c) {
                const int st = c % kStages, round = c / kStages;
                if (!ptx::mbar_wait(&sm->full[st], round & 1, abort, kWaitLimitNs) ||
                    !ptx::mbar_wait(&sm->afull[st], round & 1, abort, kWaitLimitNs)) {
                    fail(a, sm, W4A16_ERR_TIMEOUT);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a_addr = ptx::smem_u32(sA + st * kABytes);
                const uint32_t x_addr = ptx::smem_u32(sX + st * kXBytes);
                bool ok = true;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const int64_t k = (int64_t)c * kBK + kk * 16;
                    if (k >= a.K) break;
                    const int grp = (int)(k / G);
                    const bool first = (k % G) == 0;
                    const bool last = ((k + 16) % G) == 0;
                    const int b = grp & 1, use = grp >> 1;
                    if (first && use > 0) {
                        if (!ptx::mbar_wait(&sm->dempty[b], (use - 1) & 1, abort, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                    }
                    ptx::mma_f16_ss(tmem + (uint32_t)(b * kBN), ptx::smem_desc_sw128(a_addr + kk * 32),
                                    ptx::smem_desc_sw128(x_addr + kk * 32), idesc, first ? 0u : 1u);
                    if (last) ptx::mma_commit(&sm->dfull[b]);
                }
                if (!ok) {
                    fail(a, sm, W4A16_ERR_TIMEOUT);
                    break;
                }
                ptx::mma_commit(&sm->empty[st]);
            }
            // all of this thread's MMAs complete before TMEM is freed
            ptx::mma_commit(&sm->mma_done);
            volatile int never = 0;
            ptx::mbar_wait(&sm->mma_done, 0, &never, kDrainLimitNs);
        }
    } else if (warp < 6) {
        // -------------------------------------------------------------- dequant
        const int i = threadIdx.x - 64;  // weight row within the tile
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kStages, round = c / kStages;
            if (!ptx::mbar_wait(&sm->full[st], round & 1, abort, kWaitLimitNs)) {
                fail(a, sm, W4A16_ERR_TIMEOUT);
                break;
            }
            const uint4* src = reinterpret_cast<const uint4*>(sP + st * kPBytes + i * (kBK / 2));
            const uint4 p0 = src[0], p1 = src[1];
            const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            uint8_t* row = sA + st * kABytes + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16-byte chunk j holds k = 8j .. 8j+7
                uint32_t h04, h15, h26, h37;
                nibbles_to_half2(words[j], h04, h15, h26, h37);
                uint4 v;
                v.x = __byte_perm(h04, h15, 0x5410);  // (k0, k1)
                v.y = __byte_perm(h26, h37, 0x5410);  // (k2, k3)
                v.z = __byte_perm(h04, h15, 0x7632);  // (k4, k5)
                v.w = __byte_perm(h26, h37, 0x7632);  // (k6, k7)
                *reinterpret_cast<uint4*>(row + ((j ^ (i & 7)) << 4)) = v;
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&sm->afull[st]);
        }
    } else {
        // ------------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // TMEM lane = weight row in the tile
        const int64_t n = n0 + r;
        const bool n_ok = n < a.N;
        const uint16_t* srow = a.s + ((int64_t)expert * a.N + (n_ok ? n : 0)) * (a.K / G);
        float acc[kBN];
#pragma unroll
        for (int j = 0; j < kBN; ++j) acc[j] = 0.0f;
        bool ok = true;
        for (int grp = 0; grp < ngroups; ++grp) {
            const int b = grp & 1, use = grp >> 1;
            const float sv = n_ok ? __half2float(__ushort_as_half(__ldg(srow + grp))) : 0.0f;
            // warp-uniform: tcgen05.ld below is a warp-collective instruction
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm->dfull[b], use & 1, abort, kWaitLimitNs))) {
                fail(a, sm, W4A16_ERR_TIMEOUT);
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * kBN);
#pragma unroll
            for (int ch = 0; ch < kBN / 32; ++ch) {
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(taddr + ch * 32, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[ch * 32 + j] = fmaf(sv, __uint_as_float(v[j]), acc[ch * 32 + j]);
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm->dempty[b]);
        }
        if (ok && n_ok) {
#pragma unroll
            for (int j = 0; j < kBN; ++j) {
                const int64_t m = (int64_t)row0 + j;
                if (m < row_end) a.y[m * a.N + n] = __half_as_ushort(__float2half_rn(acc[j]));
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int G>
w4a16_status launch_g(const CUtensorMap& mx, const CUtensorMap& mw, const GemmArgs& a, dim3 grid, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gemm_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err != cudaSuccess) return W4A16_ERR_CUDA;
    gemm_kernel<G><<<grid, kThreads, kSmemBytes, st>>>(mx, mw, a);
    return cuda_status(cudaGetLastError());
}

}  // namespace

w4a16_status gemm_launch(const DeviceInfo& dev, const uint16_t* x, const uint8_t* qw, const uint16_t* s, uint16_t* y,
                         int64_t M, int64_t N, int64_t K, int group, const int32_t* expert_offsets, int E,
                         cudaStream_t st) {
    if ((size_t)kSmemBytes > dev.smem_optin) return W4A16_ERR_UNSUPPORTED;
    if (M > 0x7fffffffLL || N > 0x7fffffffLL) return W4A16_ERR_UNSUPPORTED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return W4A16_ERR_CUDA;
    CUtensorMap mx, mw;
    {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {kBK, kBN};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4A16_ERR_CUDA;
    }
    if (expert_offsets == nullptr) {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        cuuint32_t box[2] = {kBK / 2, kBM};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4A16_ERR_CUDA;
    } else {
        cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)(N * (K / 2))};
        cuuint32_t box[3] = {kBK / 2, kBM, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(qw), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4A16_ERR_CUDA;
    }
    GemmArgs a;
    a.s = s;
    a.y = y;
    a.offsets = expert_offsets;
    a.M = M;
    a.N = N;
    a.K = K;
    a.E = E;
    a.err = dev.error_word;
    const int64_t mt = expert_offsets ? (M + kBN - 1) / kBN + E : (M + kBN - 1) / kBN;
    const int64_t nt = (N + kBM - 1) / kBM;
    if (mt > 0x7fffffffLL || nt > 65535) return W4A16_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)mt, (unsigned)nt);
    switch (group) {
        case 32: return launch_g<32>(mx, mw, a, grid, st);
        case 64: return launch_g<64>(mx, mw, a, grid, st);
        case 128: return launch_g<128>(mx, mw, a, grid, st);
        default: return W4A16_ERR_UNSUPPORTED;
    }
}

}  // namespace w4a16
