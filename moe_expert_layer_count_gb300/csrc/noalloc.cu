// moe_scatter_noalloc: moe_scatter for callers that cannot allocate device memory.
//
// moe_scatter needs a little device scratch (per-block expert histograms) and expects
// the caller to pass it. Some callers have no way to provide it: an inference engine
// that carves every device buffer out of a fixed pool at start-up and forbids any
// allocation on its request path (cudaMalloc can synchronise the device and can fail
// under fragmentation), or a host runtime that only hands over input and output
// buffers. For them this entry point keeps the scratch in a fixed-size array that lives
// in the library's own device memory, so the call itself allocates nothing.
#include <atomic>
#include <climits>

#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

// The scratch: room for kNoAllocScratchInts histogram entries (block count x local
// experts). Every GPU that loads this library holds these 256 KiB until the process exits.
constexpr int64_t kNoAllocScratchInts = 65536;
static __device__ __align__(256) int32_t g_scatter_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::atomic<int32_t*> g_scratch_ptr[kMaxDevices];

// Device address of g_scatter_scratch on the current device, looked up once per device
// (the first call on each device does it, with that device current) and kept for the
// life of the process: a device reset would reload the module elsewhere, which is why
// the header rules out calls after one.
int scratch_address(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;
    int32_t* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_scatter_scratch) != cudaSuccess || !q) return MOE_ERR_CUDA;
        p = static_cast<int32_t*>(q);
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return MOE_OK;
}

template <typename TId>
int scatter_noalloc_impl(const void* hidden_states, int64_t M, int K, const TId* topk_ids, const float* topk_weights,
                         int topk, const int32_t* expert_map, int E, int local_num_experts,
                         const int32_t* expert_num_tokens, int apply_router_weight_on_input, int quant, void* a_out,
                         float* a_scale, int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap,
                         moe_stream_t stream) {
    if (M < 0 || topk < 1 || topk > 32 || E < 1 || local_num_experts < 1 || local_num_experts > kMaxLocalExperts ||
        M > INT32_MAX / topk || K <= 0 || K % kGroup || !expert_num_tokens || !expert_offsets ||
        (quant != MOE_QUANT_NONE && quant != MOE_QUANT_FP8_1X128))
        return MOE_ERR_INVALID_ARG;
    if (M > 0 && (!hidden_states || !topk_ids || !src2dst || !a_out || (quant == MOE_QUANT_FP8_1X128 && !a_scale) ||
                  (apply_router_weight_on_input && !topk_weights)))
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden_states) | reinterpret_cast<uintptr_t>(a_out)) & 15)
        return MOE_ERR_INVALID_ARG;
    if (rp_cap < moe_rp_cap(M, topk, local_num_experts) || rp_cap > INT32_MAX) return MOE_ERR_INVALID_ARG;
    // the histograms of all blocks must fit the fixed scratch
    const int64_t n = M * topk;
    const int64_t per = scatter_slots_per_cta(n);
    const int64_t blocks = (n + per - 1) / per;
    if (blocks > 1 && blocks * local_num_experts > kNoAllocScratchInts) return MOE_ERR_SCRATCH_LIMIT;
    int32_t* scratch = nullptr;
    if (int st = scratch_address(&scratch)) return st;
    int major = 0, minor = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED_DEVICE;
    // the histogram kernel overwrites every entry the rank kernel then reads, so the
    // previous call's contents never leak into this one
    return launch_scatter(static_cast<const uint16_t*>(hidden_states), M, K, topk_ids, topk_weights, topk, expert_map,
                          E, local_num_experts, expert_num_tokens, nullptr, nullptr,
                          apply_router_weight_on_input ? 1 : 0, quant, a_out, a_scale, expert_offsets, src2dst, rp_cap,
                          scratch, 0, (cudaStream_t)stream);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

MOE_API int moe_scatter_noalloc(const void* hidden_states, int64_t M, int K, const int32_t* topk_ids,
                                const float* topk_weights, int topk, const int32_t* expert_map, int E,
                                int local_num_experts, const int32_t* expert_num_tokens,
                                int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                                int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, moe_stream_t stream) {
    return scatter_noalloc_impl(hidden_states, M, K, topk_ids, topk_weights, topk, expert_map, E, local_num_experts,
                                expert_num_tokens, apply_router_weight_on_input, quant, a_out, a_scale,
                                expert_offsets, src2dst, rp_cap, stream);
}

MOE_API int moe_scatter_noalloc_i64(const void* hidden_states, int64_t M, int K, const int64_t* topk_ids,
                                    const float* topk_weights, int topk, const int32_t* expert_map, int E,
                                    int local_num_experts, const int32_t* expert_num_tokens,
                                    int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                                    int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, moe_stream_t stream) {
    return scatter_noalloc_impl(hidden_states, M, K, topk_ids, topk_weights, topk, expert_map, E, local_num_experts,
                                expert_num_tokens, apply_router_weight_on_input, quant, a_out, a_scale,
                                expert_offsets, src2dst, rp_cap, stream);
}

}  // extern "C"
