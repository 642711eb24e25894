// HBM-bound kernels of the fused-MoE hot path: count_expert_num_tokens, the stable
// ep_scatter (histogram -> rank -> copy + 1x128 FP8 quant), ep_gather with the top-k
// weight-and-reduce, and the standalone SiLU-and-mul requantisation.
//
// Layer steps from vLLM PR #20392 "[Bugfix] Fused MoE Modular Kernel chunking loop"
// (Purpose, Bug 2: count_expert_num_tokens per chunk), vLLM PR #20903 "[Kernel]
// DeepGemm MoE : Integrate triton permute / unpermute kernels" (Purpose item 2:
// ep_scatter / ep_gather) and vLLM PR #20725 "[Misc] ModularKernel : Perform
// WeightAndReduce inside TritonExperts & DeepGemmExperts" (Purpose, Changes).
#include "common.cuh"
#include "route.cuh"

namespace moe {

// ------------------------------------------------------------------------ count
// One CTA builds a shared-memory histogram of its share of the top-k slots (16-byte
// id loads, warp-aggregated with __match_any_sync so that a popular expert costs one
// shared atomic per warp), then stores it (single CTA) or adds it to the zeroed
// global counts (one global atomic per CTA and expert).
template <int kThreads>
__global__ void __launch_bounds__(kThreads)
    count_kernel(const int32_t* __restrict__ ids, int64_t n, const int32_t* __restrict__ expert_map, int E, int El,
                 int32_t* __restrict__ counts, int32_t* __restrict__ err_count, int direct) {
    extern __shared__ int32_t hist[];
    for (int l = threadIdx.x; l < El; l += kThreads) hist[l] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    int bad = 0;
    auto add = [&](int l) {
        const unsigned m = __match_any_sync(0xffffffffu, l);
        if (l >= 0 && lane == __ffs(m) - 1) atomicAdd(&hist[l], __popc(m));
    };
    const bool vec = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    const int64_t n4 = vec ? n / 4 : 0;
    const int4* ids4 = reinterpret_cast<const int4*>(ids);
    for (int64_t i0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); i0 < n4; i0 += stride) {
        const int64_t i = i0 + lane;
        int4 v = make_int4(-1, -1, -1, -1);
        if (i < n4) v = __ldg(ids4 + i);
        add(local_expert(v.x, expert_map, E, El, bad));
        add(local_expert(v.y, expert_map, E, El, bad));
        add(local_expert(v.z, expert_map, E, El, bad));
        add(local_expert(v.w, expert_map, E, El, bad));
    }
    for (int64_t i0 = 4 * n4 + (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); i0 < n; i0 += stride) {
        const int64_t i = i0 + lane;
        add(i < n ? local_expert(__ldg(ids + i), expert_map, E, El, bad) : -1);
    }
    __syncthreads();
    for (int l = threadIdx.x; l < El; l += kThreads) {
        const int c = hist[l];
        if (direct)
            counts[l] = c;
        else if (c)
            atomicAdd(counts + l, c);
    }
    if (err_count) {
#pragma unroll
        for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if (lane == 0 && bad) atomicAdd(err_count, bad);
    }
}

int launch_count(const int32_t* ids, int64_t n, const int32_t* expert_map, int E, int El, int32_t* counts,
                 int32_t* err_count, int num_sms, cudaStream_t stream) {
    constexpr int kThreads = 1024;
    const size_t smem = (size_t)El * sizeof(int32_t);
    if (n <= 32768) {
        count_kernel<kThreads><<<1, kThreads, smem, stream>>>(ids, n, expert_map, E, El, counts, err_count, 1);
        note_launches(1);
        return launch_status();
    }
    if (cudaMemsetAsync(counts, 0, (size_t)El * sizeof(int32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    int64_t want = (n / 4 + kThreads - 1) / kThreads;
    int grid = (int)(want < 2 * num_sms ? want : 2 * num_sms);
    if (grid < 1) grid = 1;
    count_kernel<kThreads><<<grid, kThreads, smem, stream>>>(ids, n, expert_map, E, El, counts, err_count, 0);
    note_launches(1);
    return launch_status();
}

// ---------------------------------------------------------------------- scatter
// The stable permutation is a counting sort over the flat slot index i = t*topk + k:
//   dst(i) = offsets[l] + #{ i' < i : local(i') == l }.
// The slots are cut into contiguous per-CTA segments. Kernel 1 writes each segment's
// expert histogram; kernel 2 adds the histograms of the earlier segments to the
// expert offsets and ranks its own slots warp by warp (warp segments in order, 32
// slots at a time, rank within the 32 by __match_any_sync + popc). Kernel 3 copies
// and quantises the rows. Nothing depends on timing, so the order is unique.

int scatter_slots_per_cta(int64_t n) {
    int64_t per = (n + kMaxScatterCtas - 1) / kMaxScatterCtas;
    per = (per + kScatterThreads - 1) / kScatterThreads * kScatterThreads;
    return (int)(per < kScatterMinSlots ? kScatterMinSlots : per);
}

__global__ void __launch_bounds__(kScatterThreads)
    scatter_hist_kernel(const int32_t* __restrict__ ids, int64_t n, const int32_t* __restrict__ expert_map, int E,
                        int El, int per_cta, int32_t* __restrict__ hist) {
    extern __shared__ int32_t sh[];
    for (int l = threadIdx.x; l < El; l += kScatterThreads) sh[l] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t begin = (int64_t)blockIdx.x * per_cta;
    const int64_t end = min(n, begin + per_cta);
    int bad = 0;
    for (int64_t i0 = begin + (threadIdx.x & ~31); i0 < end; i0 += kScatterThreads) {
        const int64_t i = i0 + lane;
        const int l = i < end ? local_expert(__ldg(ids + i), expert_map, E, El, bad) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, l);
        if (l >= 0 && lane == __ffs(m) - 1) atomicAdd(&sh[l], __popc(m));
    }
    __syncthreads();
    for (int l = threadIdx.x; l < El; l += kScatterThreads) hist[(int64_t)blockIdx.x * El + l] = sh[l];
}

__global__ void __launch_bounds__(kScatterThreads)
    scatter_rank_kernel(const int32_t* __restrict__ ids, int64_t n, const int32_t* __restrict__ expert_map, int E,
                        int El, int per_cta, const int32_t* __restrict__ counts, const int32_t* __restrict__ hist,
                        int32_t* __restrict__ expert_offsets, int32_t* __restrict__ src2dst) {
    constexpr int kWarps = kScatterThreads / 32;
    extern __shared__ int32_t sm[];
    int32_t* off = sm;           // [El + 1]
    int32_t* wc = sm + El + 1;   // [kWarps][El]: per-warp counts, then per-warp cursors
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp == 0) {
        int run = 0;
        for (int l0 = 0; l0 < El; l0 += 32) {
            const int l = l0 + lane;
            const int c = l < El ? (__ldg(counts + l) + kGroup - 1) / kGroup * kGroup : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (l < El) off[l] = run + incl - c;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) off[El] = run;
    }
    for (int i = threadIdx.x; i < kWarps * El; i += kScatterThreads) wc[i] = 0;
    __syncthreads();
    if (blockIdx.x == 0)
        for (int l = threadIdx.x; l <= El; l += kScatterThreads) expert_offsets[l] = off[l];

    const int per_warp = per_cta / kWarps;
    const int64_t wbeg = (int64_t)blockIdx.x * per_cta + (int64_t)warp * per_warp;
    const int64_t wend = min(n, wbeg + per_warp);
    int bad = 0;
    int32_t* mine = wc + warp * El;
    for (int64_t i0 = wbeg; i0 < wend; i0 += 32) {
        const int64_t i = i0 + lane;
        const int l = i < wend ? local_expert(__ldg(ids + i), expert_map, E, El, bad) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, l);
        if (l >= 0 && lane == __ffs(m) - 1) mine[l] += __popc(m);
        __syncwarp();
    }
    __syncthreads();
    for (int l = threadIdx.x; l < El; l += kScatterThreads) {
        int run = off[l];
        for (int b = 0; b < (int)blockIdx.x; ++b) run += __ldg(hist + (int64_t)b * El + l);
        for (int w = 0; w < kWarps; ++w) {
            const int c = wc[w * El + l];
            wc[w * El + l] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int64_t i0 = wbeg; i0 < wend; i0 += 32) {
        const int64_t i = i0 + lane;
        const bool valid = i < wend;
        const int l = valid ? local_expert(__ldg(ids + i), expert_map, E, El, bad) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, l);
        const int rank = __popc(m & lanemask_lt());
        int dst = -1;
        if (l >= 0) {
            dst = mine[l] + rank;
            if (dst >= off[l + 1]) dst = -1;  // counts inconsistent with ids: drop, never overflow
        }
        __syncwarp();
        if (l >= 0 && rank == 0) mine[l] += __popc(m);
        __syncwarp();
        if (valid) src2dst[i] = dst;
    }
}

// One warp per (token, 512-column span): lane j holds 16 consecutive values, 8 lanes
// form one 1x128 group. The row is read once and written to each of its kept slots.
template <bool kQuant>
__global__ void __launch_bounds__(256)
    scatter_copy_kernel(const uint16_t* __restrict__ x, int64_t M, int K, const int32_t* __restrict__ src2dst,
                        const float* __restrict__ topk_weights, int topk, int apply_on_input,
                        void* __restrict__ a_out, float* __restrict__ a_scale) {
    const int lane = threadIdx.x & 31;
    const int spans = (K + 511) / 512;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= M * spans) return;
    const int64_t t = gw / spans;
    const int g = (int)(gw % spans) * 4 + (lane >> 3);
    const int G = K / kGroup;
    const bool active = g < G;
    const int col = g * kGroup + (lane & 7) * 16;
    const int my_dst = lane < topk ? __ldg(src2dst + t * topk + lane) : -1;
    const float my_w = (lane < topk && apply_on_input) ? __ldg(topk_weights + t * topk + lane) : 1.f;
    float v[16];
    uint4 raw0 = make_uint4(0, 0, 0, 0), raw1 = raw0;
    if (active) {
        const uint4* src = reinterpret_cast<const uint4*>(x + t * K + col);
        raw0 = __ldg(src);
        raw1 = __ldg(src + 1);
    }
    {
        const uint32_t w[8] = {raw0.x, raw0.y, raw0.z, raw0.w, raw1.x, raw1.y, raw1.z, raw1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    if (!apply_on_input) {
        float s = 0.f;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (kQuant) q = quant16_group8(v, s);
        for (int k = 0; k < topk; ++k) {
            const int d = __shfl_sync(0xffffffffu, my_dst, k);
            if (d < 0 || !active) continue;
            if (kQuant) {
                *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a_out) + (int64_t)d * K + col) = q;
                if ((lane & 7) == 0) a_scale[(int64_t)d * G + g] = s;
            } else {
                uint4* dstp = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a_out) + (int64_t)d * K + col);
                dstp[0] = raw0;
                dstp[1] = raw1;
            }
        }
    } else {
        for (int k = 0; k < topk; ++k) {
            const int d = __shfl_sync(0xffffffffu, my_dst, k);
            const float wk = __shfl_sync(0xffffffffu, my_w, k);
            if (d < 0) continue;  // warp-uniform
            float vk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) vk[i] = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(v[i], wk)));
            if (kQuant) {
                float s;
                const uint4 q = quant16_group8(vk, s);
                if (active) {
                    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a_out) + (int64_t)d * K + col) = q;
                    if ((lane & 7) == 0) a_scale[(int64_t)d * G + g] = s;
                }
            } else if (active) {
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = uint32_t(f32_to_bf16_bits(vk[2 * i])) | (uint32_t(f32_to_bf16_bits(vk[2 * i + 1])) << 16);
                uint4* dstp = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a_out) + (int64_t)d * K + col);
                dstp[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dstp[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    }
}

int launch_scatter(const uint16_t* x, int64_t M, int K, const int32_t* ids, const float* topk_weights, int topk,
                   const int32_t* expert_map, int E, int El, const int32_t* counts, int apply_on_input, int quant,
                   void* a_out, float* a_scale, int32_t* expert_offsets, int32_t* src2dst, int32_t* hist,
                   cudaStream_t stream) {
    const int64_t n = M * topk;
    const int per_cta = scatter_slots_per_cta(n);
    const int grid = (int)((n + per_cta - 1) / per_cta);
    const size_t smem_rank = (size_t)(El + 1 + (kScatterThreads / 32) * El) * sizeof(int32_t);
    int launches = 0;
    if (grid > 1) {
        scatter_hist_kernel<<<grid, kScatterThreads, (size_t)El * sizeof(int32_t), stream>>>(ids, n, expert_map, E, El,
                                                                                              per_cta, hist);
        ++launches;
    }
    scatter_rank_kernel<<<grid < 1 ? 1 : grid, kScatterThreads, smem_rank, stream>>>(
        ids, n, expert_map, E, El, per_cta, counts, hist, expert_offsets, src2dst);
    ++launches;
    if (M > 0) {
        const int64_t warps = M * ((K + 511) / 512);
        const unsigned cgrid = (unsigned)((warps + 7) / 8);
        if (quant == MOE_QUANT_FP8_1X128)
            scatter_copy_kernel<true><<<cgrid, 256, 0, stream>>>(x, M, K, src2dst, topk_weights, topk, apply_on_input,
                                                                  a_out, a_scale);
        else
            scatter_copy_kernel<false><<<cgrid, 256, 0, stream>>>(x, M, K, src2dst, topk_weights, topk,
                                                                   apply_on_input, a_out, a_scale);
        ++launches;
    }
    note_launches(launches);
    return launch_status();
}

// ----------------------------------------------------------------------- gather
// One warp per (token, 256-column span): lane j owns 8 bf16 columns (16 bytes). The
// kept rows of the token are loaded 8 at a time (independent 16-byte loads in flight),
// then accumulated in ascending k with separately rounded fp32 multiply and add.
__global__ void __launch_bounds__(256)
    gather_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ src2dst,
                  const float* __restrict__ topk_weights, int64_t M, int topk, int K, int apply_on_input,
                  uint16_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int spans = (K + 255) / 256;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= M * spans) return;
    const int64_t t = gw / spans;
    const int col = (int)(gw % spans) * 256 + lane * 8;
    const bool active = col < K;
    const int my_dst = lane < topk ? __ldg(src2dst + t * topk + lane) : -1;
    const float my_w = (lane < topk && !apply_on_input) ? __ldg(topk_weights + t * topk + lane) : 1.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int k0 = 0; k0 < topk; k0 += 8) {
        uint4 r[8];
        int d[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            d[j] = __shfl_sync(0xffffffffu, my_dst, (k0 + j) & 31);
            if (k0 + j >= topk) d[j] = -1;
            r[j] = make_uint4(0, 0, 0, 0);
            if (d[j] >= 0 && active) r[j] = __ldg(reinterpret_cast<const uint4*>(y + (int64_t)d[j] * K + col));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float wk = __shfl_sync(0xffffffffu, my_w, (k0 + j) & 31);
            if (d[j] < 0) continue;
            const uint32_t w[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wk, __uint_as_float(w[e] << 16)));
                acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wk, __uint_as_float(w[e] & 0xffff0000u)));
            }
        }
    }
    if (!active) return;
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = uint32_t(f32_to_bf16_bits(acc[2 * e])) | (uint32_t(f32_to_bf16_bits(acc[2 * e + 1])) << 16);
    *reinterpret_cast<uint4*>(out + t * K + col) = make_uint4(o[0], o[1], o[2], o[3]);
}

int launch_gather(const uint16_t* y, const int32_t* src2dst, const float* topk_weights, int64_t M, int topk, int K,
                  int apply_on_input, uint16_t* out, cudaStream_t stream) {
    if (M == 0) return MOE_OK;
    const int64_t warps = M * ((K + 255) / 256);
    gather_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(y, src2dst, topk_weights, M, topk, K,
                                                                     apply_on_input, out);
    note_launches(1);
    return launch_status();
}

// ------------------------------------------------------------- SiLU-and-mul quant
__device__ __forceinline__ float silu_mul(float g, float u) { return __fmul_rn(__fdiv_rn(g, 1.0f + expf(-g)), u); }

// One warp per (row, 512-column span of h).
__global__ void __launch_bounds__(256)
    silu_mul_quant_kernel(const float* __restrict__ c1, const int32_t* __restrict__ expert_offsets, int El,
                          int64_t rp_cap, int N, uint8_t* __restrict__ h, float* __restrict__ h_scale) {
    const int lane = threadIdx.x & 31;
    const int spans = (N + 511) / 512;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= rp_cap * spans) return;
    const int64_t r = gw / spans;
    if (r >= __ldg(expert_offsets + El)) return;
    const int g = (int)(gw % spans) * 4 + (lane >> 3);
    const int G = N / kGroup;
    const bool active = g < G;
    const int col = g * kGroup + (lane & 7) * 16;
    float v[16];
    if (active) {
        const float4* gp = reinterpret_cast<const float4*>(c1 + r * 2 * N + col);
        const float4* up = reinterpret_cast<const float4*>(c1 + r * 2 * N + N + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 a = __ldg(gp + i), b = __ldg(up + i);
            v[4 * i + 0] = silu_mul(a.x, b.x);
            v[4 * i + 1] = silu_mul(a.y, b.y);
            v[4 * i + 2] = silu_mul(a.z, b.z);
            v[4 * i + 3] = silu_mul(a.w, b.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
    }
    float s;
    const uint4 q = quant16_group8(v, s);
    if (!active) return;
    *reinterpret_cast<uint4*>(h + r * N + col) = q;
    if ((lane & 7) == 0) h_scale[r * G + g] = s;
}

int launch_silu_mul_quant(const float* c1, const int32_t* expert_offsets, int El, int64_t rp_cap, int N, uint8_t* h,
                          float* h_scale, cudaStream_t stream) {
    if (rp_cap == 0) return MOE_OK;
    const int64_t warps = rp_cap * ((N + 511) / 512);
    silu_mul_quant_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(c1, expert_offsets, El, rp_cap, N, h,
                                                                             h_scale);
    note_launches(1);
    return launch_status();
}

}  // namespace moe
