// C ABI of the fused-MoE hot path: argument checks, workspace carve-up and the
// chunking loop. Every computation is enqueued as a kernel on the caller's stream;
// nothing here allocates, frees or synchronises.
#include <atomic>
#include <climits>

#include "common.cuh"
#include "route.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 sm_103, 2 other
std::atomic<int> g_dev_sms[kMaxDevices];

// MOE_OK when the current device is compute capability 10.3; fills the SM count.
int check_device(int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;
    int st = g_dev_state[dev].load(std::memory_order_acquire);
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        g_dev_sms[dev].store(sms, std::memory_order_relaxed);
        st = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_state[dev].store(st, std::memory_order_release);
    }
    if (num_sms) *num_sms = g_dev_sms[dev].load(std::memory_order_relaxed);
    return st == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

bool routing_args_ok(int64_t M, int topk, int E, int El) {
    // slots and permuted rows are indexed with int32 (src2dst, offsets, counts)
    return M >= 0 && topk >= 1 && topk <= 32 && E >= 1 && El >= 1 && El <= kMaxLocalExperts &&
           M <= INT32_MAX / topk && moe_rp_cap(M, topk, El) <= INT32_MAX;
}

// Byte layout of the chunk workspace (offsets from its base, each 256-aligned):
//   counts  int32 [El]        offsets int32 [El+1]     src2dst int32 [Mc*topk]
//   hist    scatter scratch   region1 = A e4m3 [cap,K] + A_scale fp32 [cap,K/128], later
//                                       reused by Y bf16 [cap,K] (A is dead after GEMM1)
//   H       e4m3 [cap, N]     H_scale fp32 [cap, N/128]  (written by GEMM1's SiLU epilogue)
struct Carve {
    size_t counts, offsets, src2dst, hist, a, a_scale, y, h, h_scale, total;
};

Carve carve(int64_t Mc, int K, int N, int topk, int El) {
    Carve c{};
    const int64_t cap = moe_rp_cap(Mc, topk, El);
    size_t p = 0;
    c.counts = p;   p += align256((size_t)El * 4);
    c.offsets = p;  p += align256((size_t)(El + 1) * 4);
    c.src2dst = p;  p += align256((size_t)Mc * topk * 4);
    c.hist = p;     p += align256(moe_scatter_workspace_size(Mc, topk, El));
    const size_t a_bytes = align256((size_t)cap * K) + align256((size_t)cap * (K / kGroup) * 4);
    const size_t y_bytes = align256((size_t)cap * K * 2);
    c.a = p;
    c.a_scale = p + align256((size_t)cap * K);
    c.y = p;
    p += a_bytes > y_bytes ? a_bytes : y_bytes;
    c.h = p;        p += align256((size_t)cap * N);
    c.h_scale = p;  p += align256((size_t)cap * (N / kGroup) * 4);
    c.total = p;
    return c;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

MOE_API const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3, sm_103a)";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_SCRATCH_LIMIT: return "problem too large for the fixed scratch of moe_scatter_noalloc";
        default: return "unknown status";
    }
}

MOE_API uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

MOE_API int moe_device_error(int clear) { return read_gemm_error(clear); }

MOE_API int64_t moe_rp_cap(int64_t chunk_M, int topk, int local_num_experts) {
    if (chunk_M < 0 || topk < 1 || local_num_experts < 1) return -1;
    const int64_t n = chunk_M * topk;
    const int64_t ne = local_num_experts < n ? local_num_experts : n;
    return (n + ne * (kGroup - 1) + kGroup - 1) / kGroup * kGroup;
}

MOE_API size_t moe_scatter_workspace_size(int64_t M, int topk, int local_num_experts) {
    if (M < 0 || topk < 1 || local_num_experts < 1) return 0;
    const int64_t n = M * topk;
    const int per = scatter_slots_per_cta(n);
    const int64_t grid = (n + per - 1) / per;
    const size_t b = (size_t)(grid > 1 ? grid : 0) * local_num_experts * sizeof(int32_t);
    return b < 256 ? 256 : b;
}

MOE_API size_t moe_workspace_size(int64_t chunk_M, int K, int N, int topk, int local_num_experts) {
    if (chunk_M < 0 || K <= 0 || N <= 0 || K % kGroup || N % kGroup || !routing_args_ok(chunk_M, topk, 1, local_num_experts))
        return 0;
    return carve(chunk_M, K, N, topk, local_num_experts).total;
}

}  // extern "C"

// The entry points that read top-k ids, for either id type (the _i64 exports take int64).
namespace moe {
namespace {

template <typename TId>
int count_impl(const TId* topk_ids, int64_t M, int topk, const int32_t* expert_map, int E, int local_num_experts,
               int32_t* expert_num_tokens, int32_t* err_count, moe_stream_t stream) {
    if (!routing_args_ok(M, topk, E, local_num_experts) || !expert_num_tokens || (M > 0 && !topk_ids))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return launch_count(topk_ids, M * topk, expert_map, E, local_num_experts, expert_num_tokens, err_count, sms,
                        (cudaStream_t)stream);
}

template <typename TId>
int scatter_impl(const void* hidden_states, int64_t M, int K, const TId* topk_ids, const float* topk_weights,
                 int topk, const int32_t* expert_map, int E, int local_num_experts, int32_t* expert_num_tokens,
                 int count_here, int32_t* err_count, int apply_router_weight_on_input, int quant, void* a_out,
                 float* a_scale, int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, void* workspace,
                 size_t workspace_bytes, moe_stream_t stream) {
    if (!routing_args_ok(M, topk, E, local_num_experts) || K <= 0 || K % kGroup || !expert_num_tokens ||
        !expert_offsets || (quant != MOE_QUANT_NONE && quant != MOE_QUANT_FP8_1X128))
        return MOE_ERR_INVALID_ARG;
    if (M > 0 && (!hidden_states || !topk_ids || !src2dst || !a_out ||
                  (quant == MOE_QUANT_FP8_1X128 && !a_scale) || (apply_router_weight_on_input && !topk_weights)))
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden_states) | reinterpret_cast<uintptr_t>(a_out)) & 15)
        return MOE_ERR_INVALID_ARG;
    if (rp_cap < moe_rp_cap(M, topk, local_num_experts) || rp_cap > INT32_MAX) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_scatter_workspace_size(M, topk, local_num_experts);
    const int64_t per = scatter_slots_per_cta(M * topk);
    const bool multi = (M * topk + per - 1) / per > 1;
    if (multi && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (int st = check_device(nullptr)) return st;
    return launch_scatter(static_cast<const uint16_t*>(hidden_states), M, K, topk_ids, topk_weights, topk, expert_map, E,
                          local_num_experts, count_here ? nullptr : expert_num_tokens,
                          count_here ? expert_num_tokens : nullptr, count_here ? err_count : nullptr,
                          apply_router_weight_on_input ? 1 : 0, quant, a_out, a_scale, expert_offsets, src2dst,
                          rp_cap, static_cast<int32_t*>(workspace), 0, (cudaStream_t)stream);
}

}  // namespace
}  // namespace moe

extern "C" {

MOE_API int moe_count_expert_tokens(const int32_t* topk_ids, int64_t M, int topk, const int32_t* expert_map, int E,
                                    int local_num_experts, int32_t* expert_num_tokens, int32_t* err_count,
                                    moe_stream_t stream) {
    return count_impl(topk_ids, M, topk, expert_map, E, local_num_experts, expert_num_tokens, err_count, stream);
}

MOE_API int moe_count_expert_tokens_i64(const int64_t* topk_ids, int64_t M, int topk, const int32_t* expert_map,
                                        int E, int local_num_experts, int32_t* expert_num_tokens, int32_t* err_count,
                                        moe_stream_t stream) {
    return count_impl(topk_ids, M, topk, expert_map, E, local_num_experts, expert_num_tokens, err_count, stream);
}

MOE_API int moe_scatter(const void* hidden_states, int64_t M, int K, const int32_t* topk_ids,
                        const float* topk_weights, int topk, const int32_t* expert_map, int E, int local_num_experts,
                        int32_t* expert_num_tokens, int count_here, int32_t* err_count,
                        int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                        int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, void* workspace,
                        size_t workspace_bytes, moe_stream_t stream) {
    return scatter_impl(hidden_states, M, K, topk_ids, topk_weights, topk, expert_map, E, local_num_experts,
                        expert_num_tokens, count_here, err_count, apply_router_weight_on_input, quant, a_out, a_scale,
                        expert_offsets, src2dst, rp_cap, workspace, workspace_bytes, stream);
}

MOE_API int moe_scatter_i64(const void* hidden_states, int64_t M, int K, const int64_t* topk_ids,
                            const float* topk_weights, int topk, const int32_t* expert_map, int E,
                            int local_num_experts, int32_t* expert_num_tokens, int count_here, int32_t* err_count,
                            int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                            int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
    return scatter_impl(hidden_states, M, K, topk_ids, topk_weights, topk, expert_map, E, local_num_experts,
                        expert_num_tokens, count_here, err_count, apply_router_weight_on_input, quant, a_out, a_scale,
                        expert_offsets, src2dst, rp_cap, workspace, workspace_bytes, stream);
}

MOE_API int moe_grouped_gemm_fp8(const uint8_t* a, const float* a_scale, const uint8_t* w, const float* w_scale,
                                 const int32_t* expert_offsets, const int32_t* expert_num_tokens,
                                 int local_num_experts, int64_t rp_cap, int n_out, int k_in, int epilogue, void* out,
                                 float* out_scale, moe_stream_t stream) {
    if (!a || !a_scale || !w || !w_scale || !expert_offsets || !out || local_num_experts < 1 ||
        local_num_experts > kMaxLocalExperts || rp_cap < 0 || rp_cap > INT32_MAX || rp_cap % kGroup || n_out <= 0 || k_in <= 0 ||
        n_out % kGroup || k_in % kGroup)
        return MOE_ERR_INVALID_ARG;
    if (epilogue != MOE_EPI_BF16 && epilogue != MOE_EPI_F32 && epilogue != MOE_EPI_SILU_MUL_QUANT)
        return MOE_ERR_INVALID_ARG;
    if (epilogue == MOE_EPI_SILU_MUL_QUANT && (n_out % 256 || !out_scale)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(out)) & 15)
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return launch_grouped_gemm(a, a_scale, w, w_scale, expert_offsets, expert_num_tokens, local_num_experts, rp_cap,
                               n_out, k_in, epilogue, out, out_scale, sms, (cudaStream_t)stream);
}

MOE_API int moe_silu_mul_quant(const float* c1, const int32_t* expert_offsets, int local_num_experts, int64_t rp_cap,
                               int N, uint8_t* h, float* h_scale, moe_stream_t stream) {
    if (!c1 || !expert_offsets || !h || !h_scale || local_num_experts < 1 || rp_cap < 0 || rp_cap > INT32_MAX ||
        N <= 0 || N % kGroup)
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(c1) | reinterpret_cast<uintptr_t>(h)) & 15) return MOE_ERR_INVALID_ARG;
    if (int st = check_device(nullptr)) return st;
    return launch_silu_mul_quant(c1, expert_offsets, local_num_experts, rp_cap, N, h, h_scale, (cudaStream_t)stream);
}

MOE_API int moe_gather_weight_reduce(const void* y, const int32_t* src2dst, const float* topk_weights, int64_t M,
                                     int topk, int K, int apply_router_weight_on_input, void* out,
                                     moe_stream_t stream) {
    if (M < 0 || topk < 1 || topk > 32 || M > INT32_MAX / topk || K <= 0 || K % kGroup) return MOE_ERR_INVALID_ARG;
    if (M > 0 && (!y || !src2dst || !out || (!apply_router_weight_on_input && !topk_weights)))
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(out)) & 15) return MOE_ERR_INVALID_ARG;
    if (int st = check_device(nullptr)) return st;
    return launch_gather(static_cast<const uint16_t*>(y), src2dst, topk_weights, M, topk, K,
                         apply_router_weight_on_input ? 1 : 0, static_cast<uint16_t*>(out), (cudaStream_t)stream);
}

MOE_API int moe_forward_chunked(const void* hidden_states, const int32_t* topk_ids, const float* topk_weights,
                                const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                const int32_t* expert_map, int E, int local_num_experts, int64_t M, int K, int N,
                                int topk, int64_t chunk_size, int apply_router_weight_on_input, void* out,
                                void* workspace, size_t workspace_bytes, int32_t* err_count, moe_stream_t stream) {
    return forward_chunked_impl(hidden_states, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, expert_map, E,
                                local_num_experts, M, K, N, topk, chunk_size, apply_router_weight_on_input, out,
                                workspace, workspace_bytes, err_count, stream);
}

MOE_API int moe_forward_chunked_i64(const void* hidden_states, const int64_t* topk_ids, const float* topk_weights,
                                    const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, const int32_t* expert_map, int E, int local_num_experts,
                                    int64_t M, int K, int N, int topk, int64_t chunk_size,
                                    int apply_router_weight_on_input, void* out, void* workspace,
                                    size_t workspace_bytes, int32_t* err_count, moe_stream_t stream) {
    return forward_chunked_impl(hidden_states, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, expert_map, E,
                                local_num_experts, M, K, N, topk, chunk_size, apply_router_weight_on_input, out,
                                workspace, workspace_bytes, err_count, stream);
}

}  // extern "C"

namespace moe {

// The chunking loop, for either top-k id type.
template <typename TId>
int forward_chunked_impl(const void* hidden_states, const TId* topk_ids, const float* topk_weights,
                         const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                         const int32_t* expert_map, int E, int local_num_experts, int64_t M, int K, int N, int topk,
                         int64_t chunk_size, int apply_router_weight_on_input, void* out, void* workspace,
                         size_t workspace_bytes, int32_t* err_count, moe_stream_t stream) {
    if (!routing_args_ok(M, topk, E, local_num_experts) || K <= 0 || N <= 0 || K % kGroup || N % kGroup ||
        chunk_size < 1)
        return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (!hidden_states || !topk_ids || !topk_weights || !w13 || !w13_scale || !w2 || !w2_scale || !out || !workspace)
        return MOE_ERR_INVALID_ARG;
    const int El = local_num_experts;
    const int64_t cmax = chunk_size < M ? chunk_size : M;
    if (workspace_bytes < moe_workspace_size(cmax, K, N, topk, El)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    // out must not overlap the workspace, nor the inputs, except hidden_states exactly
    // (in place: each chunk reads its own rows of hidden_states, and the next chunk's
    // scatter reads its rows while this chunk's gather still writes)
    {
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + (size_t)M * K * 2;
        auto hits = [&](const void* p, size_t bytes) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(p);
            return o0 < a + bytes && a < o1;
        };
        if (hits(workspace, workspace_bytes) || hits(topk_ids, (size_t)M * topk * sizeof(TId)) ||
            hits(topk_weights, (size_t)M * topk * sizeof(float)) ||
            (out != hidden_states && hits(hidden_states, (size_t)M * K * 2)))
            return MOE_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(hidden_states) | reinterpret_cast<uintptr_t>(out) |
         reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(w13) | reinterpret_cast<uintptr_t>(w2)) &
        15)
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint16_t* x = static_cast<const uint16_t*>(hidden_states);
    uint16_t* o = static_cast<uint16_t*>(out);
    for (int64_t c0 = 0; c0 < M; c0 += chunk_size) {
        const int64_t Mc = (M - c0) < chunk_size ? (M - c0) : chunk_size;
        // the workspace carve-up is derived from this chunk's own size
        const Carve cv = carve(Mc, K, N, topk, El);
        const int64_t cap = moe_rp_cap(Mc, topk, El);
        int32_t* counts = reinterpret_cast<int32_t*>(ws + cv.counts);
        int32_t* offs = reinterpret_cast<int32_t*>(ws + cv.offsets);
        int32_t* s2d = reinterpret_cast<int32_t*>(ws + cv.src2dst);
        int32_t* hist = reinterpret_cast<int32_t*>(ws + cv.hist);
        uint8_t* A = ws + cv.a;
        float* sa = reinterpret_cast<float*>(ws + cv.a_scale);
        uint16_t* Y = reinterpret_cast<uint16_t*>(ws + cv.y);
        uint8_t* H = ws + cv.h;
        float* sh = reinterpret_cast<float*>(ws + cv.h_scale);
        const TId* ids = topk_ids + c0 * topk;
        const float* tw = topk_weights + c0 * topk;
        // Several chunks, each expert's rows in a chunk mostly one 128-row block: GEMM1 reads
        // each W13 tile once per chunk, while W2 (a third of the weights) is read again by
        // every chunk. W13 is then streamed with the L2 evict-first policy, so that it does
        // not push W2 out of L2 between chunks.
        const bool w13_once = M > chunk_size && cap < (int64_t)El * 2 * kGroup;
        // the chunk's expert counts come out of the scatter's own histogram pass
        int st = launch_scatter(x + c0 * K, Mc, K, ids, tw, topk, expert_map, E, El, nullptr, counts, err_count,
                                apply_router_weight_on_input ? 1 : 0, MOE_QUANT_FP8_1X128, A, sa, offs, s2d, cap, hist, c0 > 0 ? 1 : 0, s);
        if (!st)
            st = launch_grouped_gemm(A, sa, w13, w13_scale, offs, counts, El, cap, 2 * N, K, MOE_EPI_SILU_MUL_QUANT, H, sh,
                                     sms, s, w13_once ? kOptWeightsEvictFirst : 0);
        if (!st)
            st = launch_grouped_gemm(H, sh, w2, w2_scale, offs, counts, El, cap, K, N, MOE_EPI_BF16, Y, nullptr, sms, s);
        // the next chunk's one-kernel scatter ranks its slots while this chunk's gather runs
        const int64_t next = M - c0 - Mc;
        const int early_next = next > 0 && scatter_is_one_kernel(next < chunk_size ? next : chunk_size, topk, El);
        if (!st)
            st = launch_gather(Y, s2d, tw, Mc, topk, K, apply_router_weight_on_input ? 1 : 0, o + c0 * K, s, early_next);
        if (st) return st;
    }
    return MOE_OK;
}

template int forward_chunked_impl<int32_t>(const void*, const int32_t*, const float*, const uint8_t*, const float*,
                                           const uint8_t*, const float*, const int32_t*, int, int, int64_t, int, int,
                                           int, int64_t, int, void*, void*, size_t, int32_t*, moe_stream_t);
template int forward_chunked_impl<int64_t>(const void*, const int64_t*, const float*, const uint8_t*, const float*,
                                           const uint8_t*, const float*, const int32_t*, int, int, int64_t, int, int,
                                           int, int64_t, int, void*, void*, size_t, int32_t*, moe_stream_t);

}  // namespace moe
