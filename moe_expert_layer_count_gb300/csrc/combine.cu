// Expert-parallel combine: the sum of the partial layer outputs of the ranks that each
// hold a subset of the experts. With an expert_map, a rank's layer output is its share
// of the sum over a token's top-k experts (tokens whose experts are all elsewhere get a
// zero row); the full output is the sum of the shares. vLLM PR #20903 "[Kernel] DeepGemm
// MoE : Integrate triton permute / unpermute kernels" (Purpose: DeepEP high-throughput
// prepare/finalize with expert parallelism) runs the layer this way; the exchange of the
// shares between GPUs is the caller's (an all-gather); this kernel is the local sum.
#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kMaxParts = 64;
struct Parts {
    const uint16_t* p[kMaxParts];
};

// One thread per 8 consecutive bf16 of the output (16-byte loads and stores): the parts'
// values are added in fp32 in ascending part order (separately rounded adds), then
// rounded once to bf16.
__global__ void __launch_bounds__(256)
    ep_combine_kernel(Parts parts, int n_parts, int64_t n8, uint16_t* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= n8) return;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int r = 0; r < n_parts; ++r) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(parts.p[r]) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[2 * e] = __fadd_rn(acc[2 * e], __uint_as_float(w[e] << 16));
            acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __uint_as_float(w[e] & 0xffff0000u));
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = uint32_t(f32_to_bf16_bits(acc[2 * e])) | (uint32_t(f32_to_bf16_bits(acc[2 * e + 1])) << 16);
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API int moe_ep_combine(const void* const* partials, int n_parts, int64_t M, int K, void* out,
                                      moe_stream_t stream) {
    if (!partials || n_parts < 1 || n_parts > kMaxParts || M < 0 || K <= 0 || K % 8) return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (!out || (reinterpret_cast<uintptr_t>(out) & 15)) return MOE_ERR_INVALID_ARG;
    Parts parts{};
    const size_t bytes = (size_t)M * K * 2;
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + bytes;
    for (int r = 0; r < n_parts; ++r) {
        const uintptr_t p0 = reinterpret_cast<uintptr_t>(partials[r]);
        if (!p0 || (p0 & 15)) return MOE_ERR_INVALID_ARG;
        if (p0 < o1 && o0 < p0 + bytes) return MOE_ERR_INVALID_ARG;  // out must not overlap a part
        parts.p[r] = static_cast<const uint16_t*>(partials[r]);
    }
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED_DEVICE;
    const int64_t n8 = (int64_t)M * K / 8;
    launch_k(ep_combine_kernel, (unsigned)((n8 + 255) / 256), 256, 0, (cudaStream_t)stream, parts, n_parts, n8,
             static_cast<uint16_t*>(out));
    note_launches(1);
    return launch_status();
}
