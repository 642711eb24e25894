/*
 * moe_gb300.h -- C ABI of the fused Mixture-of-Experts layer hot path on GB300 (sm_103a).
 *
 * The layer is the "modular kernel" path of three vLLM pull requests:
 *   [P1] vLLM PR #20903 "[Kernel] DeepGemm MoE : Integrate triton permute / unpermute
 *        kernels" -- Purpose items 1-2 (ep_scatter / ep_gather replace the old permute;
 *        workspaces sized from local_num_experts), Optimizations (FP8 e4m3 with
 *        128x128 block scales for the DeepGEMM experts).
 *   [P2] vLLM PR #20725 "[Misc] ModularKernel : Perform WeightAndReduce inside
 *        TritonExperts & DeepGemmExperts" -- Purpose and Changes (topk_weights and
 *        apply_router_weight_on_input passed to the experts, which apply the weights
 *        and reduce themselves; the output never aliases the workspace).
 *   [P3] vLLM PR #20392 "[Bugfix] Fused MoE Modular Kernel chunking loop" -- Purpose,
 *        Bug 1 (workspace shapes computed per chunk) and Bug 2 (count_expert_num_tokens
 *        recomputed per chunk from the chunk's topk_ids and expert_map).
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise, owned by the
 *    caller. The library never allocates, frees or synchronises: each call only
 *    enqueues kernels (and, where stated, a memset) on `stream` and returns. The one
 *    exception is moe_forward_host, which also enqueues copies on two streams of its
 *    own (created with a few events on its first call on a device, kept for the life of
 *    the process).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - Return value: MOE_OK, or an error code from the host-side checks (nothing is
 *    enqueued then), or MOE_ERR_CUDA if a launch failed.
 *  - Row-major layouts throughout. bf16 is IEEE bfloat16 (2 bytes); fp8 is OCP E4M3
 *    ("float8_e4m3fn", 1 byte); scales are fp32.
 *  - K (hidden) and N (intermediate) are multiples of 128; 1 <= topk <= 32;
 *    1 <= local_num_experts <= 1024; 1 <= E. Row indices (src2dst, expert_offsets,
 *    counts) are int32, so M * topk and the permuted row count rp_cap must not exceed
 *    2^31 - 1 (MOE_ERR_INVALID_ARG otherwise).
 *  - Local expert of a top-k slot: l = expert_map ? expert_map[id] : id. The slot is
 *    kept when 0 <= l < local_num_experts. An id of -1 is an empty slot and is dropped
 *    silently; any other id outside [0, E) is dropped and counted in *err_count (when
 *    err_count is not NULL). Dropped slots take no row and add nothing to the output.
 *  - topk_ids are int32. Every entry point that reads them has a twin with the suffix
 *    _i64 that takes int64 ids (the dtype torch.topk returns) and is otherwise the same
 *    call with the same results; an int64 id is range-checked at 64 bits, so an id such
 *    as 2^32 + 1 is a bad id, never expert 1. Outputs (src2dst, counts) stay int32.
 *  - Permuted ("expert-contiguous") row space: expert l owns rows
 *    [expert_offsets[l], expert_offsets[l+1]), each offset a multiple of 128, and the
 *    first expert_num_tokens[l] rows of its block hold its slots in ascending
 *    (token, k) order. The rest of the block is padding; its contents are unspecified
 *    and nothing reads them as data. rp_cap (moe_rp_cap) bounds expert_offsets[El]
 *    without a device-to-host read.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */
typedef struct CUevent_st* moe_event_t;   /* same type as cudaEvent_t */

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null pointer, bad size, K/N not multiple of 128 ... */
    MOE_ERR_WORKSPACE_TOO_SMALL = 2, /* workspace_bytes below the size query's answer */
    MOE_ERR_UNSUPPORTED_DEVICE = 3,  /* the current device is not compute capability 10.3 */
    MOE_ERR_CUDA = 4,                /* a CUDA call or launch failed */
    MOE_ERR_SCRATCH_LIMIT = 5,       /* moe_scatter_noalloc: problem too large for its fixed scratch */
};

enum moe_quant {
    MOE_QUANT_NONE = 0,      /* scatter copies bf16 rows */
    MOE_QUANT_FP8_1X128 = 1, /* scatter writes e4m3 codes + one fp32 scale per 1x128 group */
};

enum moe_epilogue {
    MOE_EPI_BF16 = 0,           /* out: bf16 [rp_cap, n_out] */
    MOE_EPI_F32 = 1,            /* out: fp32 [rp_cap, n_out] */
    MOE_EPI_SILU_MUL_QUANT = 2, /* out: e4m3 [rp_cap, n_out/2] h = silu(gate)*up,
                                   out_scale: fp32 [rp_cap, n_out/256] */
};

/* Text of a status code (static storage). */
MOE_API const char* moe_status_string(int status);

/* Number of kernels this library has launched in this process (all devices, all
 * streams), for accounting in benchmarks. */
MOE_API uint64_t moe_kernel_launch_count(void);

/* Device-side error word of this library's kernels on the current device: 0 when no
 * kernel has reported a problem, 1 when a grouped-GEMM pipeline wait gave up after its
 * time limit (the kernel then returned early and its output is not valid). Reading it
 * synchronises the device; clear != 0 resets it to 0. Returns -1 if the read failed. */
MOE_API int moe_device_error(int clear);

/* Row bound of the permuted buffers for a chunk of chunk_M tokens:
 * roundup128(chunk_M*topk + min(local_num_experts, chunk_M*topk) * 127). Every
 * non-empty expert pads its block by at most 127 rows, so expert_offsets[El] never
 * exceeds it (workspace sizing from local_num_experts, [P1] Purpose item 1, with a
 * device-side bound in place of the host-side counts). Returns -1 on bad arguments. */
MOE_API int64_t moe_rp_cap(int64_t chunk_M, int topk, int local_num_experts);

/* Scratch bytes moe_scatter needs for M tokens (its per-block expert histograms). */
MOE_API size_t moe_scatter_workspace_size(int64_t M, int topk, int local_num_experts);

/* Workspace bytes moe_forward_chunked needs when chunks hold at most chunk_M tokens
 * (pass min(chunk_size, M)). Returns 0 on bad arguments. */
MOE_API size_t moe_workspace_size(int64_t chunk_M, int K, int N, int topk, int local_num_experts);

/* count_expert_num_tokens ([P3] Purpose, Bug 2; review diff of utils.py): the number of
 * kept top-k slots routed to each local expert.
 *   topk_ids          int32 [M, topk]
 *   expert_map        int32 [E] or NULL (local = global id)
 *   expert_num_tokens int32 [local_num_experts], overwritten
 *   err_count         int32 [1] or NULL; bad ids are ADDED to it
 * May enqueue a memset of expert_num_tokens before the kernel. M = 0 writes zeros. */
MOE_API int moe_count_expert_tokens(const int32_t* topk_ids, int64_t M, int topk, const int32_t* expert_map,
                                    int E, int local_num_experts, int32_t* expert_num_tokens,
                                    int32_t* err_count, moe_stream_t stream);
/* The same with topk_ids int64 [M, topk]. */
MOE_API int moe_count_expert_tokens_i64(const int64_t* topk_ids, int64_t M, int topk, const int32_t* expert_map,
                                        int E, int local_num_experts, int32_t* expert_num_tokens,
                                        int32_t* err_count, moe_stream_t stream);

/* ep_scatter / deepgemm_moe_permute ([P1] Purpose item 2), with the per-token FP8
 * activation quantisation ([P1] Optimizations: e4m3, 128 blocks) done in the same pass.
 *   hidden_states     bf16 [M, K]
 *   topk_ids          int32 [M, topk];  topk_weights fp32 [M, topk] (read only when
 *                     apply_router_weight_on_input != 0: the copied row is then
 *                     bf16(x_t * w[t,k]), [P2] Changes)
 *   expert_num_tokens int32 [El]. count_here == 0: an input, as written by
 *                     moe_count_expert_tokens for the same ids. count_here != 0: an
 *                     output -- the scatter's own histogram pass counts the slots (the
 *                     count step fused into the scatter, as the chunk loop does) and
 *                     writes the same values moe_count_expert_tokens would; bad ids are
 *                     then added to *err_count (when not NULL)
 *   quant             MOE_QUANT_FP8_1X128: a_out e4m3 [rp_cap, K] and a_scale fp32
 *                     [rp_cap, K/128] with scale = amax/448 per 1x128 group (fp32 IEEE
 *                     division), code = e4m3(x/scale) rounded to nearest-even and
 *                     saturated; an all-zero group has scale 0 and codes 0.
 *                     MOE_QUANT_NONE: a_out bf16 [rp_cap, K]; a_scale unused (may be NULL).
 *   expert_offsets    int32 [El+1], written (block starts, multiples of 128)
 *   src2dst           int32 [M, topk], written: the permuted row of each slot, -1 if dropped
 *   rp_cap            rows of a_out / a_scale; must be >= moe_rp_cap(M, topk, El)
 *   workspace         device scratch of >= moe_scatter_workspace_size(M, topk, El) bytes
 * The permutation is the unique stable order: deterministic, independent of timing. */
MOE_API int moe_scatter(const void* hidden_states, int64_t M, int K, const int32_t* topk_ids,
                        const float* topk_weights, int topk, const int32_t* expert_map, int E,
                        int local_num_experts, int32_t* expert_num_tokens, int count_here, int32_t* err_count,
                        int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                        int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, void* workspace,
                        size_t workspace_bytes, moe_stream_t stream);
/* The same with topk_ids int64 [M, topk]. */
MOE_API int moe_scatter_i64(const void* hidden_states, int64_t M, int K, const int64_t* topk_ids,
                            const float* topk_weights, int topk, const int32_t* expert_map, int E,
                            int local_num_experts, int32_t* expert_num_tokens, int count_here, int32_t* err_count,
                            int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                            int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/* moe_scatter without a workspace argument, for callers that cannot allocate device
 * memory: for example an inference engine that plans every device buffer once at
 * start-up and allows no allocation on its request path (cudaMalloc may synchronise the
 * device and may fail when memory is fragmented), or a host runtime that only passes
 * input and output buffers. The vLLM pages have no counterpart: this is an interface
 * convenience of this library, not a step of the method.
 * Arguments and results are those of moe_scatter with count_here = 0 (expert_num_tokens
 * is an input), minus workspace/workspace_bytes.
 * The scratch it needs (per-block expert histograms) is a fixed array of 65536 int32
 * (256 KiB) in this library's own device memory, held by every GPU that loads the
 * library until the process exits. A problem needing more -- (number of scatter blocks)
 * x local_num_experts > 65536 when more than one block is used, e.g. beyond about
 * 131k top-k slots at 1024 local experts or about 16.7M slots at 128 -- is refused with
 * MOE_ERR_SCRATCH_LIMIT before anything is enqueued.
 * The first call on each device looks up the array's device address (with that device
 * current); make that first call before any stream capture. The address is kept for the
 * life of the process, so this entry point must not be called on a device after
 * cudaDeviceReset (or any other teardown of its primary context) in the same process:
 * the array then moves and the kept address is stale. Every call on a device
 * shares the one array and overwrites the entries it reads, so calls whose kernels
 * overlap on the GPU (different streams, no ordering between them) race and give wrong
 * results: order them on one stream or with events. Allocates nothing. */
MOE_API int moe_scatter_noalloc(const void* hidden_states, int64_t M, int K, const int32_t* topk_ids,
                                const float* topk_weights, int topk, const int32_t* expert_map, int E,
                                int local_num_experts, const int32_t* expert_num_tokens,
                                int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                                int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, moe_stream_t stream);
/* The same with topk_ids int64 [M, topk]. */
MOE_API int moe_scatter_noalloc_i64(const void* hidden_states, int64_t M, int K, const int64_t* topk_ids,
                                    const float* topk_weights, int topk, const int32_t* expert_map, int E,
                                    int local_num_experts, const int32_t* expert_num_tokens,
                                    int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                                    int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, moe_stream_t stream);

/* The DeepGEMM-style grouped ("m-grouped contiguous") GEMM with 128x128 block-scaled
 * FP8 weights ([P1] Optimizations, --block-shape 128 128), on tcgen05 tensor cores:
 *   out[r, j] = sum_kb a_scale[r, kb] * w_scale[l, j/128, kb] *
 *               sum_{k in block kb} A[r, k] * W[l, j, k]
 * for every row r in [expert_offsets[l], expert_offsets[l+1]) of every local expert l
 * (rows >= expert_offsets[El] are not touched).
 *   expert_num_tokens int32 [El] or NULL. When given, the rows of a block at or past
 *            expert_offsets[l] + expert_num_tokens[l] are padding, and for small batches
 *            (rp_cap below 256 rows per local expert, where most of each block is padding)
 *            an aligned group of 32 rows of a 128-row tile holding only padding is
 *            neither folded nor written: those output rows keep their old contents. In
 *            every other case all rows are computed, padding included.
 *            The batched ("masked") expert layout [El, max_tokens, K] that low-latency
 *            expert-parallel dispatch produces is the case expert_offsets[l] =
 *            l * max_tokens (max_tokens a multiple of 128) with expert_num_tokens = the
 *            per-expert token counts (the mask).
 *   a        e4m3 [rp_cap, k_in];  a_scale fp32 [rp_cap, k_in/128]
 *   w        e4m3 [El, n_out, k_in] (each expert's rows are K-contiguous)
 *   w_scale  fp32 [El, n_out/128, k_in/128]
 *   epilogue MOE_EPI_BF16 / MOE_EPI_F32: out as stated there, fp32 accumulation,
 *            rounded once at the end. MOE_EPI_SILU_MUL_QUANT (the w13 GEMM): n_out = 2N,
 *            columns [0, N) are the gate and [N, 2N) the up projection; out receives
 *            h = silu(gate) * up requantised 1x128 (e4m3 [rp_cap, N]) and out_scale its
 *            fp32 scales [rp_cap, N/128], computed from the fp32 accumulators.
 * n_out and k_in are multiples of 128 (n_out a multiple of 256 for SILU_MUL_QUANT). */
MOE_API int moe_grouped_gemm_fp8(const uint8_t* a, const float* a_scale, const uint8_t* w, const float* w_scale,
                                 const int32_t* expert_offsets, const int32_t* expert_num_tokens,
                                 int local_num_experts, int64_t rp_cap, int n_out, int k_in, int epilogue, void* out,
                                 float* out_scale, moe_stream_t stream);

/* SiLU-and-mul with 1x128 FP8 requantisation, standalone (the same arithmetic the
 * SILU_MUL_QUANT epilogue applies):
 *   c1      fp32 [rp_cap, 2N]: gate = columns [0, N), up = columns [N, 2N)
 *   h       e4m3 [rp_cap, N];  h_scale fp32 [rp_cap, N/128]
 * h = silu(g) * u with silu(g) = g / (1 + exp(-g)) in fp32; rows
 * >= expert_offsets[El] are not touched. */
MOE_API int moe_silu_mul_quant(const float* c1, const int32_t* expert_offsets, int local_num_experts,
                               int64_t rp_cap, int N, uint8_t* h, float* h_scale, moe_stream_t stream);

/* ep_gather / deepgemm_unpermute_and_reduce with the top-k weight-and-reduce folded in
 * ([P1] Purpose item 2; [P2] Purpose):
 *   out[t, c] = bf16( sum over k = 0..topk-1 with src2dst[t,k] >= 0, in ascending k,
 *                     of w'[t,k] * y[src2dst[t,k], c] ),
 * accumulated in fp32 with separately rounded multiply and add, w' = topk_weights, or 1
 * when apply_router_weight_on_input != 0. A token with no kept slot gets zeros.
 *   y      bf16 [rows, K] (rows >= every src2dst value + 1)
 *   out    bf16 [M, K]; must not overlap y ([P2]: the output never aliases scratch) */
MOE_API int moe_gather_weight_reduce(const void* y, const int32_t* src2dst, const float* topk_weights, int64_t M,
                                     int topk, int K, int apply_router_weight_on_input, void* out,
                                     moe_stream_t stream);

/* The whole layer under the chunking loop ([P3] Purpose, Bug 1 and Bug 2): tokens are
 * processed in chunks of chunk_size; each chunk recomputes its expert counts, offsets
 * and workspace carve-up from its own rows and runs
 *   count -> scatter (FP8 1x128) -> grouped GEMM w13 with the SiLU-and-mul requant
 *   epilogue -> grouped GEMM w2 (bf16) -> gather with weight-and-reduce
 * writing out[c0 : c0+Mc, :].
 *   hidden_states bf16 [M, K];  topk_ids int32 [M, topk];  topk_weights fp32 [M, topk]
 *   w13 e4m3 [El, 2N, K] (gate rows then up rows), w13_scale fp32 [El, 2N/128, K/128]
 *   w2  e4m3 [El, K, N],  w2_scale fp32 [El, K/128, N/128]
 *   out bf16 [M, K]; it may be hidden_states itself (in place) but must not otherwise
 *       overlap hidden_states, topk_ids, topk_weights or the workspace
 *   workspace >= moe_workspace_size(min(chunk_size, M), K, N, topk, El) bytes
 *   err_count int32 [1] or NULL (bad ids are added)
 * The result of every row depends only on its own chunk, and the GEMM tiling does not
 * depend on the chunk's size, so any chunk_size gives bit-identical output. */
MOE_API int moe_forward_chunked(const void* hidden_states, const int32_t* topk_ids, const float* topk_weights,
                                const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                const float* w2_scale, const int32_t* expert_map, int E, int local_num_experts,
                                int64_t M, int K, int N, int topk, int64_t chunk_size,
                                int apply_router_weight_on_input, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* err_count, moe_stream_t stream);
/* The same with topk_ids int64 [M, topk]. */
MOE_API int moe_forward_chunked_i64(const void* hidden_states, const int64_t* topk_ids, const float* topk_weights,
                                    const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, const int32_t* expert_map, int E, int local_num_experts,
                                    int64_t M, int K, int N, int topk, int64_t chunk_size,
                                    int apply_router_weight_on_input, void* out, void* workspace,
                                    size_t workspace_bytes, int32_t* err_count, moe_stream_t stream);

/* Expert-parallel combine (vLLM PR #20903 "[Kernel] DeepGemm MoE : Integrate triton
 * permute / unpermute kernels", Purpose: DeepEP high-throughput prepare/finalize with
 * expert parallelism). A rank that holds a subset of the experts runs the layer with an
 * expert_map and gets its share of every token's sum over its top-k experts (a zero row
 * for tokens whose experts are all elsewhere); the layer output is the sum of the shares.
 * After the caller has gathered the shares of all ranks on this GPU (an all-gather; the
 * exchange is not part of this library), this call adds them:
 *   out[t, c] = bf16( sum over r = 0..n_parts-1, in ascending r, of partials[r][t, c] ),
 * accumulated in fp32 with separately rounded adds.
 *   partials  HOST array of n_parts (1..64) DEVICE pointers, each bf16 [M, K], 16-byte aligned
 *   out       bf16 [M, K], 16-byte aligned, overlapping no part
 *   K         a multiple of 8
 * The sum of bf16 shares differs from a single-GPU run of the whole layer (one rounding
 * of the full top-k sum) by the rounding of each share. */
MOE_API int moe_ep_combine(const void* const* partials, int n_parts, int64_t M, int K, void* out,
                           moe_stream_t stream);

/* Workspace bytes moe_forward_host (or _i64) needs for batches of up to M tokens: the
 * layer's own workspace (moe_workspace_size for min(chunk_size, M)) followed by two
 * staging slots, each a device copy of a batch's hidden_states, topk_ids (room for int64
 * ids), topk_weights and output. Returns 0 on bad arguments. */
MOE_API size_t moe_host_workspace_size(int64_t M, int K, int N, int topk, int local_num_experts,
                                       int64_t chunk_size);

/* moe_forward_chunked with the batch in HOST memory: hidden_states_host bf16 [M, K],
 * topk_ids_host int32 [M, topk], topk_weights_host fp32 [M, topk] and out_host bf16
 * [M, K] are host pointers; they must be page-locked (cudaHostAlloc / pinned tensors)
 * for the copies to run asynchronously. Weights, expert_map, err_count and workspace
 * are device pointers as in moe_forward_chunked, and the result is the same, bit for
 * bit. The call is asynchronous:
 *   - the inputs are copied into one of the workspace's two staging slots on a copy
 *     stream of the library's own, once that slot's previous output has been copied
 *     out; successive calls alternate slots;
 *   - the layer runs on `stream` after the inputs have landed;
 *   - the output is copied to out_host on a second copy stream of the library's own.
 * So a call's input copy overlaps the previous call's layer, and its output copy the
 * next call's layer. out_host holds the result once `done` (a cudaEvent_t, or NULL) has
 * completed, or once `stream` has passed a later moe_host_wait. The host buffers must
 * stay untouched until then. `stream` itself is NOT ordered after the output copy.
 * Calls that share a workspace must use the same `stream`. Batches of different sizes may
 * share one workspace (sized for the largest): a call whose M, chunk_size or workspace
 * differs from the previous call's places its staging slots differently, so its input
 * copy first waits for every earlier call's layer and output copies; only calls of one
 * size overlap one another.
 * workspace >= moe_host_workspace_size(M, K, N, topk, El, chunk_size) bytes. */
MOE_API int moe_forward_host(const void* hidden_states_host, const int32_t* topk_ids_host,
                             const float* topk_weights_host, const uint8_t* w13, const float* w13_scale,
                             const uint8_t* w2, const float* w2_scale, const int32_t* expert_map, int E,
                             int local_num_experts, int64_t M, int K, int N, int topk, int64_t chunk_size,
                             int apply_router_weight_on_input, void* out_host, void* workspace,
                             size_t workspace_bytes, int32_t* err_count, moe_stream_t stream, moe_event_t done);
/* The same with topk_ids_host int64 [M, topk] (host, page-locked). */
MOE_API int moe_forward_host_i64(const void* hidden_states_host, const int64_t* topk_ids_host,
                                 const float* topk_weights_host, const uint8_t* w13, const float* w13_scale,
                                 const uint8_t* w2, const float* w2_scale, const int32_t* expert_map, int E,
                                 int local_num_experts, int64_t M, int K, int N, int topk, int64_t chunk_size,
                                 int apply_router_weight_on_input, void* out_host, void* workspace,
                                 size_t workspace_bytes, int32_t* err_count, moe_stream_t stream, moe_event_t done);

/* Makes `stream` wait until every output copy moe_forward_host has enqueued on the
 * current device so far has completed. */
MOE_API int moe_host_wait(moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
