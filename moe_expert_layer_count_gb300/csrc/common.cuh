// Device helpers shared by the kernels of the fused-MoE hot path (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_gb300.h"

namespace moe {

constexpr int kGroup = 128;  // 1x128 activation groups, 128x128 weight blocks

// Kernel launches made by this library (read by moe_kernel_launch_count()).
void note_launches(int n);

// Launch-status helper: returns MOE_ERR_CUDA if the last launch failed.
inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Programmatic dependent launch. Every kernel of this library is launched allowed to
// start while the previous kernel on the stream finishes; it waits for that kernel's
// completion (and memory) with pdl_wait() before its first global-memory access, and
// lets the next kernel launch with pdl_trigger(). Both are no-ops without the launch
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                            Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Round-to-nearest-even fp32 -> bf16 bits (the hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Two fp32 -> two e4m3 codes (low byte = a), round-to-nearest-even, saturating to
// +-448 (cvt.rn.satfinite.e4m3x2.f32).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Local expert of a top-k id (int32 or int64); -1 when dropped. Bad ids (outside
// [-1, E)) bump *bad; the range test is done at the id's own width, so a 64-bit id never
// aliases a small expert.
template <typename TId>
__device__ __forceinline__ int local_expert(TId id, const int32_t* __restrict__ expert_map, int E, int El, int& bad) {
    if (id == TId(-1)) return -1;
    if (id < 0 || id >= TId(E)) {
        ++bad;
        return -1;
    }
    int l = expert_map ? __ldg(expert_map + id) : (int)id;
    return (l >= 0 && l < El) ? l : -1;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// SiLU-and-mul of the w13 GEMM's gate g and up u: silu(g) * u with silu(g) = g/(1+e^-g),
// in fast fp32 (ex2.approx-based exponential, approximate division; a few ulp). The
// exponent is clamped so that 1 + e^-g stays finite. The fused GEMM epilogue and the
// standalone kernel both use this function, so their results are identical.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

// Correctly rounded quotient a / b (round-to-nearest-even) from r = RN(1/b): the
// product a*r is within an ulp of the quotient, and one fused correction with the exact
// remainder a - b*q gives RN(a/b) (Markstein's theorem for FMA division). Valid while
// 1/b does not overflow; callers keep b in the normal range.
__device__ __forceinline__ float div_rn_by(float a, float b, float r) {
    const float q = __fmul_rn(a, r);
    const float e = __fmaf_rn(-q, b, a);
    return __fmaf_rn(e, r, q);
}

// Quantise 16 consecutive fp32 values of one 1x128 group (8 lanes x 16 values, the 8
// lanes aligned on a multiple of 8 within the warp) to e4m3 with the group's fp32 scale
// amax/448. Returns the 16 codes packed in a uint4 and the scale.
__device__ __forceinline__ uint4 quant16_group8(const float (&v)[16], float& scale_out) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 448.0f);
    scale_out = s;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint16_t lo, hi;
        if (s == 0.f) {
            lo = hi = 0;
        } else {
            lo = f32x2_to_e4m3x2(__fdiv_rn(v[4 * i + 0], s), __fdiv_rn(v[4 * i + 1], s));
            hi = f32x2_to_e4m3x2(__fdiv_rn(v[4 * i + 2], s), __fdiv_rn(v[4 * i + 3], s));
        }
        w[i] = uint32_t(lo) | (uint32_t(hi) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace moe
