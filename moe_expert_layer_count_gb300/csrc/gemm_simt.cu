// Block-scaled FP8 grouped GEMM on CUDA cores: the plain tiled form of
//   out[r, j] = sum_kb a_scale[r, kb] * w_scale[l, j/128, kb] * sum_{k in kb} A[r,k] W[l,j,k]
// (the DeepGEMM grouped GEMM of vLLM PR #20903 "[Kernel] DeepGemm MoE : Integrate
// triton permute / unpermute kernels", section "Optimizations", --block-shape 128 128).
// 128x128 output tile per CTA, 8x8 per thread, fp32 partial sums per 128-wide K block
// promoted with the product of the two block scales.
#include "common.cuh"
#include "route.cuh"

namespace moe {

namespace {
constexpr int BM = 128, BN = 128, BK = 32;

__device__ __forceinline__ void decode16(uint4 q, float* out) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            __half2_raw p = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[i] >> (16 * h)) & 0xffffu), __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<__half2*>(&p));
            out[4 * i + 2 * h] = f.x;
            out[4 * i + 2 * h + 1] = f.y;
        }
    }
}

// Expert owning permuted row `row` (offsets[l] <= row < offsets[l+1]); -1 past the end.
__device__ __forceinline__ int expert_of_row(const int32_t* __restrict__ offsets, int El, int row) {
    if (row >= __ldg(offsets + El)) return -1;
    int lo = 0, hi = El - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offsets + mid) <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}
}  // namespace

__global__ void __launch_bounds__(256)
    gemm_simt_kernel(const uint8_t* __restrict__ A, const float* __restrict__ sa, const uint8_t* __restrict__ W,
                     const float* __restrict__ sw, const int32_t* __restrict__ offsets, int El, int n_out, int k_in,
                     int epilogue, void* __restrict__ out) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ int s_l;
    const int nt = blockIdx.x, row0 = blockIdx.y * BM;
    if (threadIdx.x == 0) s_l = expert_of_row(offsets, El, row0);
    __syncthreads();
    const int l = s_l;
    if (l < 0) return;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int KB = k_in / kGroup;
    const uint8_t* Wl = W + ((int64_t)l * n_out + (int64_t)nt * BN) * k_in;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    const int lr = threadIdx.x >> 1, lk = (threadIdx.x & 1) * 16;
    for (int kb = 0; kb < KB; ++kb) {
        float part[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) part[i][j] = 0.f;
        for (int k0 = kb * kGroup; k0 < (kb + 1) * kGroup; k0 += BK) {
            float fa[16], fb[16];
            decode16(__ldg(reinterpret_cast<const uint4*>(A + (int64_t)(row0 + lr) * k_in + k0 + lk)), fa);
            decode16(__ldg(reinterpret_cast<const uint4*>(Wl + (int64_t)lr * k_in + k0 + lk)), fb);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                As[lk + i][lr] = fa[i];
                Bs[lk + i][lr] = fb[i];
            }
            __syncthreads();
#pragma unroll 4
            for (int k = 0; k < BK; ++k) {
                float a[8], b[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = As[k][ty * 8 + i];
#pragma unroll
                for (int j = 0; j < 8; ++j) b[j] = Bs[k][tx * 8 + j];
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
            }
            __syncthreads();
        }
        const float sb = __ldg(sw + ((int64_t)l * (n_out / kGroup) + nt) * KB + kb);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float s = __ldg(sa + (int64_t)(row0 + ty * 8 + i) * KB + kb) * sb;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(s, part[i][j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row0 + ty * 8 + i;
        const int c = nt * BN + tx * 8;
        if (epilogue == MOE_EPI_F32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + r * n_out + c);
            o[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            o[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        } else {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = uint32_t(f32_to_bf16_bits(acc[i][2 * e])) | (uint32_t(f32_to_bf16_bits(acc[i][2 * e + 1])) << 16);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + r * n_out + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

int launch_grouped_gemm(const uint8_t* a, const float* a_scale, const uint8_t* w, const float* w_scale,
                        const int32_t* expert_offsets, int El, int64_t rp_cap, int n_out, int k_in, int epilogue,
                        void* out, float* out_scale, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    (void)out_scale;
    if (epilogue == MOE_EPI_SILU_MUL_QUANT) return MOE_ERR_INVALID_ARG;
    if (rp_cap == 0) return MOE_OK;
    dim3 grid(n_out / BN, (unsigned)(rp_cap / BM));
    gemm_simt_kernel<<<grid, 256, 0, stream>>>(a, a_scale, w, w_scale, expert_offsets, El, n_out, k_in, epilogue, out);
    note_launches(1);
    return launch_status();
}

}  // namespace moe
