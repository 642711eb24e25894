// moe_forward_host: the layer called with host buffers, its copies overlapped with
// compute.
//
// A serving loop hands the layer a batch in host memory and wants the output back in
// host memory. Run naively (copy in, compute, copy out, on one stream) the two copies
// add to every batch's time. On GB300 the host link has copy engines of its own, so a
// batch's copies can run while the previous and next batches compute. This entry point
// does exactly that:
//   * the caller's workspace holds, after the layer's own workspace, two staging slots
//     (device copies of a batch's inputs and output); successive calls alternate slots;
//   * the input copy of a call runs on a library-owned copy stream, the layer on the
//     caller's stream, the output copy on a second copy stream;
//   * events order the three: a slot is refilled only after the output copy of its
//     previous use, which itself follows that use's compute.
// So call n+1's input copy overlaps call n's compute, and call n's output copy overlaps
// call n+1's compute. The streams and events are created once per device, on the first
// call, and kept for the life of the process.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kMaxDevices = 64;

struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t in_done[2] = {}, compute_done[2] = {}, out_done[2] = {};
    unsigned calls = 0;
    int last = -1;  // slot of the most recent call
    bool ready = false;
    // Placement of the previous call's layer area and slots. A call of another size (or
    // on another workspace) places them differently, so its regions can overlap bytes
    // that earlier calls' kernels and copies are still using.
    const void* ws = nullptr;
    size_t layer_bytes = 0, slot_bytes = 0;
};

std::mutex g_pipe_mutex[kMaxDevices];
HostPipe g_pipe[kMaxDevices];

inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Byte layout of one staging slot for a batch of M tokens. The ids region has room for
// 8-byte ids, so one workspace size serves both id types.
struct Slot {
    size_t x, ids, w, out, total;
};
Slot slot_layout(int64_t M, int K, int topk) {
    Slot s{};
    size_t p = 0;
    s.x = p;   p += align256((size_t)M * K * 2);
    s.ids = p; p += align256((size_t)M * topk * 8);
    s.w = p;   p += align256((size_t)M * topk * 4);
    s.out = p; p += align256((size_t)M * K * 2);
    s.total = p;
    return s;
}

// Creates the device's copy streams and events on first use (the caller holds the
// device's mutex).
int pipe_init(HostPipe& p) {
    if (p.ready) return MOE_OK;
    if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess)
        return MOE_ERR_CUDA;
    for (int s = 0; s < 2; ++s)
        if (cudaEventCreateWithFlags(&p.in_done[s], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.compute_done[s], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.out_done[s], cudaEventDisableTiming) != cudaSuccess)
            return MOE_ERR_CUDA;
    p.ready = true;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API size_t moe_host_workspace_size(int64_t M, int K, int N, int topk, int local_num_experts,
                                                  int64_t chunk_size) {
    if (M < 1 || K <= 0 || N <= 0 || topk < 1 || local_num_experts < 1 || chunk_size < 1) return 0;
    const size_t layer = moe_workspace_size(chunk_size < M ? chunk_size : M, K, N, topk, local_num_experts);
    if (!layer) return 0;
    return align256(layer) + 2 * slot_layout(M, K, topk).total;
}

namespace moe {
namespace {

template <typename TId>
int forward_host_impl(const void* hidden_states_host, const TId* topk_ids_host, const float* topk_weights_host,
                      const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                      const int32_t* expert_map, int E, int local_num_experts, int64_t M, int K, int N, int topk,
                      int64_t chunk_size, int apply_router_weight_on_input, void* out_host, void* workspace,
                      size_t workspace_bytes, int32_t* err_count, moe_stream_t stream, moe_event_t done) {
    if (M < 0 || K <= 0 || N <= 0 || topk < 1 || topk > 32 || E < 1 || local_num_experts < 1 || chunk_size < 1)
        return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (!hidden_states_host || !topk_ids_host || !topk_weights_host || !out_host || !workspace)
        return MOE_ERR_INVALID_ARG;
    const size_t need = moe_host_workspace_size(M, K, N, topk, local_num_experts, chunk_size);
    if (!need) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;

    std::lock_guard<std::mutex> lock(g_pipe_mutex[dev]);
    HostPipe& p = g_pipe[dev];
    if (int st = pipe_init(p)) return st;
    const size_t layer_bytes = align256(moe_workspace_size(chunk_size < M ? chunk_size : M, K, N, topk,
                                                           local_num_experts));
    const Slot L = slot_layout(M, K, topk);
    const int s = (int)(p.calls & 1u);
    uint8_t* base = static_cast<uint8_t*>(workspace) + layer_bytes + (size_t)s * L.total;
    void* x = base + L.x;
    TId* ids = reinterpret_cast<TId*>(base + L.ids);
    float* w = reinterpret_cast<float*>(base + L.w);
    void* out = base + L.out;
    cudaStream_t cs = (cudaStream_t)stream;

    // A new placement drains the pipeline first: the input copy waits for every earlier
    // call's layer and both slots' output copies (an event never recorded is complete).
    // Calls of one size keep overlapping.
    if (p.calls && (p.ws != workspace || p.layer_bytes != layer_bytes || p.slot_bytes != L.total)) {
        if (cudaStreamWaitEvent(p.h2d, p.compute_done[p.last], 0) != cudaSuccess ||
            cudaStreamWaitEvent(p.h2d, p.out_done[0], 0) != cudaSuccess ||
            cudaStreamWaitEvent(p.h2d, p.out_done[1], 0) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    // inputs into the slot, once its previous use has been copied out
    if (cudaStreamWaitEvent(p.h2d, p.out_done[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(x, hidden_states_host, (size_t)M * K * 2, cudaMemcpyHostToDevice, p.h2d) != cudaSuccess ||
        cudaMemcpyAsync(ids, topk_ids_host, (size_t)M * topk * sizeof(TId), cudaMemcpyHostToDevice, p.h2d) != cudaSuccess ||
        cudaMemcpyAsync(w, topk_weights_host, (size_t)M * topk * 4, cudaMemcpyHostToDevice, p.h2d) != cudaSuccess ||
        cudaEventRecord(p.in_done[s], p.h2d) != cudaSuccess)
        return MOE_ERR_CUDA;
    // the layer on the caller's stream, after the inputs have landed
    if (cudaStreamWaitEvent(cs, p.in_done[s], 0) != cudaSuccess) return MOE_ERR_CUDA;
    int st = forward_chunked_impl(x, ids, w, w13, w13_scale, w2, w2_scale, expert_map, E, local_num_experts, M, K,
                                  N, topk, chunk_size, apply_router_weight_on_input, out, workspace, layer_bytes,
                                  err_count, cs);
    if (st) return st;
    // the output back to the host, after the layer
    if (cudaEventRecord(p.compute_done[s], cs) != cudaSuccess ||
        cudaStreamWaitEvent(p.d2h, p.compute_done[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(out_host, out, (size_t)M * K * 2, cudaMemcpyDeviceToHost, p.d2h) != cudaSuccess ||
        cudaEventRecord(p.out_done[s], p.d2h) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (done && cudaEventRecord((cudaEvent_t)done, p.d2h) != cudaSuccess) return MOE_ERR_CUDA;
    p.last = s;
    p.ws = workspace;
    p.layer_bytes = layer_bytes;
    p.slot_bytes = L.total;
    ++p.calls;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

MOE_API int moe_forward_host(const void* hidden_states_host, const int32_t* topk_ids_host,
                             const float* topk_weights_host, const uint8_t* w13, const float* w13_scale,
                             const uint8_t* w2, const float* w2_scale, const int32_t* expert_map, int E,
                             int local_num_experts, int64_t M, int K, int N, int topk, int64_t chunk_size,
                             int apply_router_weight_on_input, void* out_host, void* workspace,
                             size_t workspace_bytes, int32_t* err_count, moe_stream_t stream, moe_event_t done) {
    return forward_host_impl(hidden_states_host, topk_ids_host, topk_weights_host, w13, w13_scale, w2, w2_scale,
                             expert_map, E, local_num_experts, M, K, N, topk, chunk_size,
                             apply_router_weight_on_input, out_host, workspace, workspace_bytes, err_count, stream,
                             done);
}

MOE_API int moe_forward_host_i64(const void* hidden_states_host, const int64_t* topk_ids_host,
                                 const float* topk_weights_host, const uint8_t* w13, const float* w13_scale,
                                 const uint8_t* w2, const float* w2_scale, const int32_t* expert_map, int E,
                                 int local_num_experts, int64_t M, int K, int N, int topk, int64_t chunk_size,
                                 int apply_router_weight_on_input, void* out_host, void* workspace,
                                 size_t workspace_bytes, int32_t* err_count, moe_stream_t stream, moe_event_t done) {
    return forward_host_impl(hidden_states_host, topk_ids_host, topk_weights_host, w13, w13_scale, w2, w2_scale,
                             expert_map, E, local_num_experts, M, K, N, topk, chunk_size,
                             apply_router_weight_on_input, out_host, workspace, workspace_bytes, err_count, stream,
                             done);
}

MOE_API int moe_host_wait(moe_stream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_pipe_mutex[dev]);
    HostPipe& p = g_pipe[dev];
    if (!p.ready || p.last < 0) return MOE_OK;
    // output copies run in order on one stream: the latest one covers all earlier ones
    return cudaStreamWaitEvent((cudaStream_t)stream, p.out_done[p.last], 0) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
