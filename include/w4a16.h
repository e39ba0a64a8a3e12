/*
 * w4a16.h - C ABI of libw4a16.so, the GB300 (sm_103a) W4A16 group-quantized
 * linear layer.
 *
 * The operation (LLM170 page, introduction: "W4A16 (int4 sym g128, f16
 * activations)"; the MoE models of the same page use group 32):
 *
 *     y[m, n] = sum_k x[m, k] * s[n, k / g] * q[n, k]
 *
 * with x, y fp16, q a signed 4-bit integer in [-8, 7] and s one fp16 scale per
 * group of g consecutive input features k. This is y = x * W^T for the
 * dequantized weight W^[n, k] = s[n, k/g] * q[n, k]; per the same page's
 * Repository layout section the GPU result must match a CPU reference of that
 * definition.
 *
 * Data layout (all row-major, all in device memory unless stated):
 *   x        fp16 [M, K]           (uint16_t bit patterns)
 *   qweight  uint8 [N, K/2]        byte j of row n holds k = 2j in bits 0-3 and
 *                                  k = 2j+1 in bits 4-7; the stored nibble is q+8
 *                                  (byte-identical to little-endian int32
 *                                  [N, K/8] with nibble i = k mod 8)
 *   scales   fp16 [N, K/g]
 *   y        fp16 [M, N]
 *   routed experts: qweight [E, N, K/2], scales [E, N, K/g], expert_offsets
 *   int32 [E+1] (device memory), activations sorted by expert.
 *
 * Ownership and threading: the caller owns and allocates every buffer. The
 * library never allocates, frees or synchronizes (except w4a16_device_status,
 * which says so). Every call is asynchronous on `stream` (a cudaStream_t; NULL
 * is the legacy default stream). Calls on different streams must not share a
 * workspace. Results are deterministic: the same inputs give the same bits.
 *
 * Errors: every entry point validates its arguments on the host before any
 * launch and returns a status; it never aborts the process. A CUDA launch
 * error is returned as W4A16_ERR_CUDA. Problems only the device can see
 * (expert offsets that are not a valid partition, a bounded wait that ran
 * out) set a sticky device word read by w4a16_device_status.
 *
 * Numerics: products x * q are exact in fp32; each group's partial sum is
 * accumulated in fp32 and multiplied by its fp32 scale; the result is rounded
 * once to fp16 (round to nearest even). Element-wise it stays within
 * |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x[m,k] W^[n,k]| of the exact value.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,   /* null pointer, negative size, K % group != 0 ... */
    W4A16_ERR_UNSUPPORTED = 2,   /* group not in {32, 64, 128}, K not a multiple of 32,
                                    no sm_103 device */
    W4A16_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    W4A16_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    W4A16_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up (kernel returned early) */
    W4A16_ERR_BAD_OFFSETS = 6,   /* device: expert_offsets not 0 = o[0] <= ... <= o[E] = R */
    W4A16_ERR_WORKSPACE = 7,     /* workspace missing or smaller than w4a16_workspace_bytes */
    W4A16_ERR_BAD_ROUTING = 8    /* device: a top-k expert id outside [0, E), or a combine row
                                    outside [0, R) */
} w4a16_status;

/*
 * Symmetric int4 group quantizer (LLM170 page, introduction: "int4 sym").
 * For each row n and group j of `group` consecutive k:
 *   amax = max |w| over the group (fp32); s = fp16_rn(fp32(amax / 7));
 *   q = clamp(rint(w / s), -8, 7) computed in fp32 (rint: half to even);
 *   an all-zero group gives s = 0 and q = 0. Stored as described above.
 * w: fp32 [N, K] (device). qweight: uint8 [N, K/2]. scales: fp16 [N, K/group].
 * Bit-exact and deterministic. NaN weights are not supported; |w| must stay
 * below 7 * 65520 for the scale to be finite.
 * Requires N >= 0, K >= 0, K % group == 0, K even, group in {32, 64, 128}.
 */
W4A16_API w4a16_status w4a16_pack(const float* w, int64_t N, int64_t K, int32_t group,
                        uint8_t* qweight, uint16_t* scales, void* stream);

/*
 * Inverse of the storage step: q[n, k] = nibble - 8 as int8 [N, K] (device).
 * Bit-exact. Requires K even.
 */
W4A16_API w4a16_status w4a16_unpack(const uint8_t* qweight, int64_t N, int64_t K, int8_t* q,
                          void* stream);

/*
 * Dense layer y = x * W^T (see the definition at the top of this file).
 * M, N >= 0 (M = 0 or N = 0: nothing to do); K >= 0 with K % group == 0 and
 * K % 32 == 0 (K = 0 writes y = 0); group in {32, 64, 128}.
 * x, qweight, scales and y must be 16-byte aligned. y may also point to
 * page-locked host memory (cudaHostAlloc / cudaHostRegister) when K > 0: with
 * unified addressing the kernels store the result into it directly, so a
 * caller that wants the result on the host needs no separate copy.
 * Small M (decode, up to 16 rows) runs a split-K GEMV; larger M runs the
 * tensor-core GEMM. For group 128 and M <= 8 the GEMV sums its split
 * row-blocks inside thread-block clusters (distributed shared memory) and
 * leaves `workspace` untouched; for the other groups and M its cross-block
 * partial sums live in `workspace`.
 * workspace: device buffer of at least w4a16_workspace_bytes(M, N, K, group, 1)
 * bytes, zero-filled once before its first use (w4a16_workspace_init); every
 * call leaves it ready for the next (the counters it keeps there are back at
 * zero; the partial sums it parks there are always written before they are
 * read). One workspace may serve w4a16_linear and w4a16_linear_gated calls of
 * any shape in turn. May be NULL when that size is 0.
 */
W4A16_API w4a16_status w4a16_linear(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales,
                          uint16_t* y, int64_t M, int64_t N, int64_t K, int32_t group,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Routed-expert (MoE) layer over activations sorted by expert: for every
 * expert e and row r with expert_offsets[e] <= r < expert_offsets[e+1],
 *   y_sorted[r, n] = sum_k x_sorted[r, k] * W^_e[n, k],
 * W^_e from qweight[e] and scales[e] (LLM170 page: the routed-MoE models,
 * "g32"). E >= 1, R >= 0; the same K/group/alignment rules as w4a16_linear.
 * expert_offsets lives in device memory and is read only by the device, so
 * no host synchronization happens; an invalid partition sets
 * W4A16_ERR_BAD_OFFSETS in the device word and leaves y_sorted unspecified.
 * Empty experts are allowed. The grouped GEMM needs no scratch memory:
 * w4a16_workspace_bytes(R, N, K, group, E) is 0 and workspace /
 * workspace_bytes are ignored (NULL and 0 are fine).
 */
W4A16_API w4a16_status w4a16_grouped_linear(const uint16_t* x_sorted, const uint8_t* qweight,
                                  const uint16_t* scales, const int32_t* expert_offsets,
                                  uint16_t* y_sorted, int32_t E, int64_t R, int64_t N,
                                  int64_t K, int32_t group, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * w4a16_grouped_linear with the token gather fused into the activation loads:
 * row r of the expert-sorted activations is x[token_of_row[r]], read straight
 * from the token-major x fp16 [T, K] (device) as the GEMM needs it, so no
 * expert-sorted copy of x is written or read back. token_of_row int32 [R]
 * (device) is what w4a16_moe_dispatch returns (it may then skip its own
 * gather, K = 0). Otherwise the contract of w4a16_grouped_linear, with the
 * same results bit for bit. Group 32 only (the routed-expert group; else
 * W4A16_ERR_UNSUPPORTED), E <= 4096. A token id outside [0, T) sets
 * W4A16_ERR_BAD_ROUTING in the device word and that row reads zeros.
 * x must be 16-byte aligned; no workspace.
 */
W4A16_API w4a16_status w4a16_grouped_linear_gather(const uint16_t* x, int64_t T, const int32_t* token_of_row,
                                                   const uint8_t* qweight, const uint16_t* scales,
                                                   const int32_t* expert_offsets, uint16_t* y_sorted, int32_t E,
                                                   int64_t R, int64_t N, int64_t K, int32_t group, void* stream);

/*
 * Gate and up projections of a gated (SwiGLU) MLP fused into one pass:
 *   g = x * Wg^T,  u = x * Wu^T,  y[m, n] = silu(g[m, n]) * u[m, n],
 *   silu(v) = v / (1 + exp(-v)),
 * (rust-inference page, list of accuracy fixes, item 5: the SiLU-activated
 * gate projection multiplies the up projection). Wg and Wu have the same
 * shape [N, K] and group, in the format of w4a16_linear; g and u are formed
 * exactly as w4a16_linear forms y (fp32 group sums, scale in fp32) and stay
 * in fp32; silu and the product are fp32; y is rounded once to fp16.
 * M, N >= 0 and the K, group and alignment rules of w4a16_linear. Decode
 * (M <= 16) runs a split-K GEMV over both matrices; its workspace is
 * w4a16_linear_gated_workspace_bytes(M, N, K, group) bytes, zero-filled once
 * (w4a16_workspace_init), and every call leaves it ready for the next, as
 * for w4a16_linear (its fp32 g and u parking area is zero again when the
 * call ends). Larger M runs the tensor-core GEMM with tiles of 64 rows of Wg
 * and the same 64 rows of Wu, so one block holds g and u of the same outputs
 * in fp32; it needs no workspace (the size is 0; NULL is fine). Either way
 * one launch streams both weight matrices once and never writes g or u to
 * y's buffer.
 */
W4A16_API w4a16_status w4a16_linear_gated(const uint16_t* x, const uint8_t* qweight_gate,
                                          const uint16_t* scales_gate, const uint8_t* qweight_up,
                                          const uint16_t* scales_up, uint16_t* y, int64_t M, int64_t N,
                                          int64_t K, int32_t group, void* workspace, size_t workspace_bytes,
                                          void* stream);

/*
 * Flags of w4a16_linear_ex and w4a16_linear_gated_ex (0 gives exactly
 * w4a16_linear / w4a16_linear_gated; unknown bits return
 * W4A16_ERR_INVALID_ARG).
 *
 * W4A16_STATIC_WEIGHTS: the caller promises that the weights (qweight and
 * scales) were written by work that completed before this call was enqueued
 * (packed or copied in, then synchronized), and that nothing still pending
 * on `stream` writes them: the usual case for the weights of a decode loop.
 * The decode GEMV (M <= 16) may then start reading them while the kernel
 * before it on the stream is still running, and waits for that kernel only
 * before it reads x. Without the flag the GEMV reads nothing
 * before the previous kernel on the stream has completed. The flag changes
 * no result bit; if the promise is broken the results are undefined. The
 * tensor-core path (M > 16) ignores it.
 */
#define W4A16_STATIC_WEIGHTS 1u

/* w4a16_linear with flags (see above); otherwise the same contract. */
W4A16_API w4a16_status w4a16_linear_ex(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales,
                                       uint16_t* y, int64_t M, int64_t N, int64_t K, int32_t group, uint32_t flags,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* w4a16_linear_gated with flags (see above); otherwise the same contract. */
W4A16_API w4a16_status w4a16_linear_gated_ex(const uint16_t* x, const uint8_t* qweight_gate,
                                             const uint16_t* scales_gate, const uint8_t* qweight_up,
                                             const uint16_t* scales_up, uint16_t* y, int64_t M, int64_t N, int64_t K,
                                             int32_t group, uint32_t flags, void* workspace, size_t workspace_bytes,
                                             void* stream);

/* Bytes of workspace w4a16_linear_gated needs on the current device; 0 if the
 * problem is not one it runs. */
W4A16_API size_t w4a16_linear_gated_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t group);

/*
 * Allocation-free variant of w4a16_linear, for callers that cannot allocate
 * device memory: code that runs inside an allocator or memory-pool callback,
 * a plugin host that hands a kernel only its input and output buffers, or a
 * runtime that forbids allocation while it captures or replays work. The
 * pages this library follows have no counterpart to it.
 *
 * Same arguments and results as w4a16_linear, minus the workspace. The
 * scratch the decode GEMV needs (cross-block fp32 partial sums and per-row-
 * block arrival counters) lives in one fixed device array of
 * W4A16_NOALLOC_SCRATCH_BYTES that every GPU which loads the library keeps
 * until the process exits. A problem whose scratch would not fit is rejected
 * with W4A16_ERR_WORKSPACE before anything runs. The entry point calls no
 * cudaMalloc, cudaFree or other allocating routine. Its first call on a
 * device looks up the array's device address, so make that first call
 * before any stream capture. Each call clears the counters it uses
 * (cudaMemsetAsync on `stream`). All calls share the one array and it keeps
 * the last call's contents, so calls that overlap on the GPU (for example on
 * two streams) race with each other: serialize them.
 */
#define W4A16_NOALLOC_SCRATCH_BYTES (8u << 20)
W4A16_API w4a16_status w4a16_linear_noalloc(const uint16_t* x, const uint8_t* qweight, const uint16_t* scales,
                                            uint16_t* y, int64_t M, int64_t N, int64_t K, int32_t group,
                                            void* stream);

/*
 * Routed-MoE dispatch around w4a16_grouped_linear. The pages name the router
 * (infr README, model table: "softmax router, top-k experts" for the Qwen3 MoE,
 * "8-of-128 routed" for the Gemma 4 MoE) and run the routed experts at group 32
 * (LLM170 page, benchmark table: "g32, MoE resident"). A routed layer is
 *   route -> dispatch -> w4a16_grouped_linear (one or more) -> combine.
 * All three calls are deterministic and never synchronize.
 *
 * w4a16_moe_route: softmax router. For each token t of logits fp32 [T, E]
 * (device), the top_k experts with the largest logits, compared as fp32 values;
 * equal logits go to the lower expert index. topk_ids int32 [T, top_k] lists
 * them by falling logit; topk_weights fp32 [T, top_k] holds their softmax
 * probabilities exp(l - max l) / sum_e exp(l_e - max l) (fp32, expf), divided
 * by their sum when renormalize != 0. Requires 1 <= top_k <= min(E, 32) and
 * E <= 1024 (else UNSUPPORTED). NaN logits are not supported, and each token
 * needs at least one finite logit (-inf marks an expert that must get weight 0).
 */
W4A16_API w4a16_status w4a16_moe_route(const float* logits, int64_t T, int32_t E, int32_t top_k,
                                       int32_t renormalize, int32_t* topk_ids, float* topk_weights,
                                       void* stream);

/*
 * w4a16_moe_dispatch: expert-major order of the T * top_k (token, slot) pairs,
 * rows sorted by (expert, token, slot) (a stable counting sort):
 *   expert_offsets int32 [E+1]: rows of expert e are [offsets[e], offsets[e+1]);
 *   row_of int32 [T, top_k]:    the row of pair (t, j);
 *   token_of_row int32 [T*top_k]: the token of row r;
 *   x_sorted fp16 [T*top_k, K]:  x_sorted[r] = x[token_of_row[r]] (x fp16 [T, K]).
 * These are the inputs w4a16_grouped_linear takes (x_sorted, expert_offsets).
 * K = 0 skips the gather (x and x_sorted may then be NULL); otherwise K % 8 == 0
 * and x, x_sorted 16-byte aligned. E <= 4096, T * top_k < 2^31.
 * An id outside [0, E) sets W4A16_ERR_BAD_ROUTING in the device word; that pair
 * gets row -1 and no row, so offsets[E] < T * top_k.
 * workspace: w4a16_moe_dispatch_workspace_bytes(T, top_k, E) bytes (no
 * initialisation needed; NULL when that is 0).
 */
W4A16_API size_t w4a16_moe_dispatch_workspace_bytes(int64_t T, int32_t top_k, int32_t E);
W4A16_API w4a16_status w4a16_moe_dispatch(const int32_t* topk_ids, int64_t T, int32_t top_k, int32_t E,
                                          const uint16_t* x, int64_t K, int32_t* expert_offsets,
                                          int32_t* row_of, int32_t* token_of_row, uint16_t* x_sorted,
                                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * w4a16_moe_combine: y[t, n] = sum_j topk_weights[t, j] * y_sorted[row_of[t, j], n]
 * for y_sorted fp16 [R, N] (the grouped layer's output in dispatch order) and
 * y fp16 [T, N]: fp32 products and sum in slot order j = 0, 1, ..., rounded
 * once to fp16. A row of -1 adds nothing; a row outside [0, R) sets
 * W4A16_ERR_BAD_ROUTING and adds nothing.
 */
W4A16_API w4a16_status w4a16_moe_combine(const uint16_t* y_sorted, int64_t R, const int32_t* row_of,
                                         const float* topk_weights, int64_t T, int32_t top_k, int64_t N,
                                         uint16_t* y, void* stream);

/*
 * GGUF block formats. The infr README lists the block formats its GPU path
 * decodes byte-identically to the CPU dequant ("Also validated for
 * correctness", among them Q4_K_M) and stores routed expert banks as Q5_1
 * (footnote 3); the LLM170 README's status names q4_K and q5_1 MoE tiles. The
 * pages print no layout; these are ggml's block types as GGUF files carry
 * them (GGUF specification, ggml repository docs/gguf.md; Q4_K from the
 * k-quants change, llama.cpp pull request 1684), all fields little-endian:
 *
 *   W4A16_FORMAT_Q4_K  256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes
 *     of 6-bit sub-block scales sc[0..7] and minimums mn[0..7] (sc[j], mn[j]
 *     for j < 4 in the low 6 bits of bytes j and j + 4; for j >= 4 the low
 *     4 bits in the low and high nibble of byte j + 4 and the top 2 bits in
 *     the top bits of bytes j - 4 and j), then 128 bytes of nibbles: weight
 *     64c + l (l < 32) is the low nibble of byte 32c + l, weight 64c + 32 + l
 *     its high nibble. W^[i] = d * sc[i/32] * q - dmin * mn[i/32].
 *   W4A16_FORMAT_Q5_1  32 weights in 24 bytes: fp16 d, fp16 m, a 32-bit word
 *     qh, 16 bytes of nibbles: weight i < 16 is the low nibble of byte i,
 *     weight i >= 16 the high nibble of byte i - 16, and bit i of qh is its
 *     fifth bit. W^[i] = d * q + m.
 *
 * A matrix of N rows of K weights is uint8 [N, w4a16_blocks_row_bytes(format,
 * K)]: each row's blocks in k order, rows one after another (K a multiple of
 * 256 for Q4_K and of 32 for Q5_1).
 */
#define W4A16_FORMAT_Q4_K 1
#define W4A16_FORMAT_Q5_1 2

/* Bytes of one row of K weights, or -1 for an unknown format or a K that is
 * not a whole number of blocks. */
W4A16_API int64_t w4a16_blocks_row_bytes(int32_t format, int64_t K);

/*
 * y = x * W^T for block-format weights: y[m, n] = sum_k x[m, k] * W^[n, k]
 * with x fp16 [M, K], blocks as above (device) and y fp16 [M, N]. Products of
 * x and the integer q are exact; each 32-weight sub-block's sums of x q and
 * of x are accumulated in fp32 and scaled by the block's fp32 step and
 * offset; y is rounded once to fp16. Element-wise the result stays within
 * |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x[m, k]| (|a q| + |b|) of the
 * exact value, W^ = a q + b. A decode GEMV: each launch serves up to 8 rows
 * of x and reads the weights once; larger M runs one launch per 8 rows.
 * M, N >= 0 (M = 0 or N = 0: nothing to do); K >= 0, whole blocks (K = 0
 * writes y = 0). x, blocks and y must be 16-byte aligned. No workspace; the
 * result is deterministic. Unknown format: W4A16_ERR_UNSUPPORTED.
 */
W4A16_API w4a16_status w4a16_blocks_linear(int32_t format, const uint16_t* x, const uint8_t* blocks, uint16_t* y,
                                           int64_t M, int64_t N, int64_t K, void* stream);

/*
 * W^ as fp32 [N, K] (device, 16-byte aligned): the step and offset of each
 * sub-block in fp32 (exact), the step times q (exact), plus the offset,
 * rounded once; bit for bit what a CPU dequantizer forming the same values in
 * fp32 gets. Same sizes and rules as w4a16_blocks_linear.
 */
W4A16_API w4a16_status w4a16_blocks_dequant(int32_t format, const uint8_t* blocks, int64_t N, int64_t K, float* w,
                                            void* stream);

/* Bytes of workspace w4a16_linear (E = 1) or w4a16_grouped_linear (E experts,
 * M = R rows) needs for this problem on the current device; 0 if none. */
W4A16_API size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t group, int32_t E);

/* Zero-fills a workspace asynchronously on `stream` (cudaMemsetAsync; no
 * allocation). Needed once per workspace, and again after any call that
 * reported a device error. */
W4A16_API w4a16_status w4a16_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronizes `stream`, then reads and clears the current device's sticky
 * error word: W4A16_OK, W4A16_ERR_TIMEOUT (a bounded wait in the GEMV or the
 * GEMM gave up), W4A16_ERR_BAD_OFFSETS (w4a16_grouped_linear) or
 * W4A16_ERR_BAD_ROUTING (w4a16_moe_dispatch, w4a16_moe_combine). The word
 * keeps the first error raised since it was last cleared. */
W4A16_API w4a16_status w4a16_device_status(void* stream);

/* Static, human-readable name of a status code. */
W4A16_API const char* w4a16_status_string(w4a16_status status);

/* Text of the most recent CUDA runtime failure that made a call of this host
 * thread return W4A16_ERR_CUDA (which call, error name and message). The
 * string stays valid until this thread's next failing call. */
W4A16_API const char* w4a16_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
W4A16_API int32_t w4a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
