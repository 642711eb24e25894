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
// id loads: four int32 or two int64 ids each, four loads per thread issued back to
// back), one shared atomic per slot into one
// of kCountCopies sub-histograms (warp w uses copy w % kCountCopies, so that only lanes
// of one warp can collide on a popular expert), then sums the copies and stores the
// result (single CTA) or adds it to the zeroed global counts (one global atomic per CTA
// and expert). Aggregating equal experts with __match_any_sync first measured 2-4x
// slower: its cost per call exceeds the atomics it saves.
constexpr int kCountCopies = 8;
template <int kThreads, typename TId>
__global__ void __launch_bounds__(kThreads)
    count_kernel(const TId* __restrict__ ids, int64_t n, const int32_t* __restrict__ expert_map, int E, int El,
                 int32_t* __restrict__ counts, int32_t* __restrict__ err_count, int direct) {
    constexpr int kVec = 4;                      // 16-byte loads in flight per thread
    constexpr int kPer = 16 / (int)sizeof(TId);  // ids per 16-byte load
    extern __shared__ int32_t hist[];  // kCountCopies sub-histograms of El entries
    for (int l = threadIdx.x; l < kCountCopies * El; l += kThreads) hist[l] = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const int lane = threadIdx.x & 31;
    int32_t* mine = hist + ((threadIdx.x >> 5) % kCountCopies) * El;
    int bad = 0;
    auto add = [&](int l) {
        if (l >= 0) atomicAdd(&mine[l], 1);
    };
    // the ids of one 16-byte load (little-endian: an int64 id's low word comes first)
    auto add16 = [&](const uint4& v) {
        if constexpr (kPer == 4) {
            add(local_expert((int32_t)v.x, expert_map, E, El, bad));
            add(local_expert((int32_t)v.y, expert_map, E, El, bad));
            add(local_expert((int32_t)v.z, expert_map, E, El, bad));
            add(local_expert((int32_t)v.w, expert_map, E, El, bad));
        } else {
            add(local_expert((int64_t)(((uint64_t)v.y << 32) | v.x), expert_map, E, El, bad));
            add(local_expert((int64_t)(((uint64_t)v.w << 32) | v.z), expert_map, E, El, bad));
        }
    };
    const bool vec = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    const int64_t n4 = vec ? n / kPer : 0;
    const uint4* ids4 = reinterpret_cast<const uint4*>(ids);
    const int64_t step = (int64_t)gridDim.x * kThreads * kVec;
    for (int64_t b0 = (int64_t)blockIdx.x * kThreads * kVec + (threadIdx.x & ~31) * kVec; b0 < n4; b0 += step) {
        uint4 v[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i = b0 + j * 32 + lane;
            v[j] = i < n4 ? __ldg(ids4 + i) : make_uint4(~0u, ~0u, ~0u, ~0u);  // all ids -1
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) add16(v[j]);
    }
    for (int64_t i0 = kPer * n4 + (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); i0 < n;
         i0 += (int64_t)gridDim.x * kThreads) {
        const int64_t i = i0 + lane;
        add(i < n ? local_expert(__ldg(ids + i), expert_map, E, El, bad) : -1);
    }
    __syncthreads();
    for (int l = threadIdx.x; l < El; l += kThreads) {
        int c = 0;
#pragma unroll
        for (int k = 0; k < kCountCopies; ++k) c += hist[k * El + l];
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

template <typename TId>
int launch_count(const TId* ids, int64_t n, const int32_t* expert_map, int E, int El, int32_t* counts,
                 int32_t* err_count, int num_sms, cudaStream_t stream) {
    const size_t smem = (size_t)kCountCopies * El * sizeof(int32_t);
    if (n <= 16384) {  // one CTA, one (int32) or two (int64) batches of loads per thread: no memset needed
        launch_k(count_kernel<1024, TId>, 1, 1024, smem, stream, ids, n, expert_map, E, El, counts, err_count, 1);
        note_launches(1);
        return launch_status();
    }
    // 256-thread CTAs, 4096 slots each (16 ids per thread: one batch of int32 ids, two of
    // int64), adding into zeros
    if (cudaMemsetAsync(counts, 0, (size_t)El * sizeof(int32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t want = (n + 4095) / 4096;
    const int grid = (int)(want < 4 * num_sms ? want : 4 * num_sms);
    launch_k(count_kernel<256, TId>, grid, 256, smem, stream, ids, n, expert_map, E, El, counts, err_count, 0);
    note_launches(1);
    return launch_status();
}
template int launch_count<int32_t>(const int32_t*, int64_t, const int32_t*, int, int, int32_t*, int32_t*, int,
                                   cudaStream_t);
template int launch_count<int64_t>(const int64_t*, int64_t, const int32_t*, int, int, int32_t*, int32_t*, int,
                                   cudaStream_t);

// ---------------------------------------------------------------------- scatter
// The stable permutation is a counting sort over the flat slot index i = t*topk + k:
//   dst(i) = offsets[l] + #{ i' < i : local(i') == l }.
// The slots are cut into contiguous per-CTA segments, and each CTA's segment into 8
// contiguous warp segments walked 256 slots at a time (8 groups of 32, loaded back to
// back before any is used). Kernel 1 writes each segment's expert histogram; kernel 2
// adds the histograms of the earlier segments to the expert offsets and ranks its own
// slots (rank inside a group of 32 by __match_any_sync + popc, per-warp running
// cursors in shared memory). Kernel 3 copies and quantises the rows. Nothing depends
// on timing, so the order is unique.

constexpr int kRound = 8;  // groups of 32 slots loaded per warp per round

// A 16-byte load of data this kernel reads exactly once and that nothing writes while it
// runs: no L1 allocation, and 256-byte L2 fetches (a warp reads 512 contiguous bytes).
__device__ __forceinline__ uint4 ld_once_256(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

int scatter_slots_per_cta(int64_t n) {
    constexpr int64_t kUnit = (kScatterThreads / 32) * 32;  // 32 slots for each warp
    int64_t per = (n + kMaxScatterCtas - 1) / kMaxScatterCtas;
    per = (per + kUnit - 1) / kUnit * kUnit;
    return (int)(per < kScatterMinSlots ? kScatterMinSlots : per);
}

// Local experts of one round of a warp's segment: slot base + 32 j + lane, j < kRound.
template <typename TId>
__device__ __forceinline__ void load_round(const TId* __restrict__ ids, int64_t base, int64_t end,
                                           const int32_t* __restrict__ expert_map, int E, int El, int lane,
                                           int (&l)[kRound], int& bad) {
    TId id[kRound];
#pragma unroll
    for (int j = 0; j < kRound; ++j) {
        const int64_t i = base + j * 32 + lane;
        id[j] = i < end ? __ldg(ids + i) : TId(-1);
    }
#pragma unroll
    for (int j = 0; j < kRound; ++j) l[j] = local_expert(id[j], expert_map, E, El, bad);
}

template <typename TId>
__global__ void __launch_bounds__(kScatterThreads)
    scatter_hist_kernel(const TId* __restrict__ ids, int64_t n, const int32_t* __restrict__ expert_map, int E,
                        int El, int per_cta, int32_t* __restrict__ hist, int32_t* __restrict__ err_count) {
    extern __shared__ int32_t sh[];  // kCountCopies sub-histograms of El entries
    for (int l = threadIdx.x; l < kCountCopies * El; l += kScatterThreads) sh[l] = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t* mine = sh + (warp % kCountCopies) * El;
    const int per_warp = per_cta / (kScatterThreads / 32);
    const int64_t wbeg = (int64_t)blockIdx.x * per_cta + (int64_t)warp * per_warp;
    const int64_t wend = min(n, wbeg + per_warp);
    int bad = 0;
    for (int64_t r0 = wbeg; r0 < wend; r0 += 32 * kRound) {
        int l[kRound];
        load_round(ids, r0, wend, expert_map, E, El, lane, l, bad);
#pragma unroll
        for (int j = 0; j < kRound; ++j)
            if (l[j] >= 0) atomicAdd(&mine[l[j]], 1);
    }
    if (err_count) {
#pragma unroll
        for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if (lane == 0 && bad) atomicAdd(err_count, bad);
    }
    __syncthreads();
    for (int l = threadIdx.x; l < El; l += kScatterThreads) {
        int c = 0;
#pragma unroll
        for (int k = 0; k < kCountCopies; ++k) c += sh[k * El + l];
        hist[(int64_t)blockIdx.x * El + l] = c;
    }
}

// counts_in: the experts' slot counts (moe_scatter's input). When it is NULL the counts
// are derived here -- from all CTAs' histograms, or from this single CTA's own pass --
// and written to counts_out (the chunk loop's count step, fused into the scatter).
template <typename TId>
__global__ void __launch_bounds__(kScatterThreads)
    scatter_rank_kernel(const TId* __restrict__ ids, int64_t n, const int32_t* __restrict__ expert_map, int E,
                        int El, int per_cta, const int32_t* __restrict__ counts_in, const int32_t* __restrict__ hist,
                        int32_t* __restrict__ expert_offsets, int32_t* __restrict__ src2dst,
                        int32_t* __restrict__ counts_out, int32_t* __restrict__ err_count, int row_cap) {
    constexpr int kWarps = kScatterThreads / 32;
    extern __shared__ int32_t sm[];
    int32_t* off = sm;               // [El + 1]
    int32_t* base = sm + El + 1;     // [El]: slots of the earlier CTAs
    int32_t* tot = base + El;        // [El]: slots of all CTAs (counts derived here)
    int32_t* wc = tot + El;          // [kWarps][El]: per-warp counts, then per-warp cursors
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int per_warp = per_cta / kWarps;
    const int64_t wbeg = (int64_t)blockIdx.x * per_cta + (int64_t)warp * per_warp;
    const int64_t wend = min(n, wbeg + per_warp);
    int bad = 0;
    // With more than one CTA the histogram kernel ran just before this one and waited for
    // the kernel before it before letting this one launch, so the caller's inputs are
    // final: the ids are loaded and counted per warp (shared memory only) while the
    // histogram kernel is still running, and this kernel waits only before its first
    // read of the histograms. A single CTA is the scatter's first kernel and waits first.
    const bool early = G > 1;
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
    int l0[kRound];
    load_round(ids, wbeg, wend, expert_map, E, El, lane, l0, bad);
    for (int l = threadIdx.x; l < El; l += kScatterThreads) base[l] = tot[l] = 0;
    for (int i = threadIdx.x; i < kWarps * El; i += kScatterThreads) wc[i] = 0;
    __syncthreads();
    int32_t* mine = wc + warp * El;
    for (int64_t r0 = wbeg; r0 < wend; r0 += 32 * kRound) {
        int l[kRound];
        if (r0 == wbeg) {
#pragma unroll
            for (int j = 0; j < kRound; ++j) l[j] = l0[j];
        } else {
            load_round(ids, r0, wend, expert_map, E, El, lane, l, bad);
        }
        // per-warp counts: equal experts of a round are aggregated first (this pass sees
        // few slots per warp, where a hot expert would serialise per-lane atomics)
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            const unsigned m = __match_any_sync(0xffffffffu, l[j]);
            if (l[j] >= 0 && lane == __ffs(m) - 1) mine[l[j]] += __popc(m);
            __syncwarp();
        }
    }
    if (early) {
        pdl_wait();
        pdl_trigger();
    }
    const bool derive = counts_in == nullptr;
    if (G > 1) {
        // per expert: sum of the earlier CTAs' histograms (and of all, when deriving the
        // counts); several threads per expert, loads issued 8 at a time
        const int rows = derive ? G : (int)blockIdx.x;
        const int tpl = El >= kScatterThreads ? 1 : kScatterThreads / El;
        for (int t = threadIdx.x; t < tpl * El; t += kScatterThreads) {
            const int l = t % El, part = t / El;
            int pre = 0, all = 0;
            for (int b0 = part; b0 < rows; b0 += 8 * tpl) {
                int v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int b = b0 + j * tpl;
                    v[j] = b < rows ? __ldg(hist + (int64_t)b * El + l) : 0;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int b = b0 + j * tpl;
                    all += v[j];
                    if (b < (int)blockIdx.x) pre += v[j];
                }
            }
            if (pre) atomicAdd(&base[l], pre);
            if (all) atomicAdd(&tot[l], all);
        }
    }
    if (derive && G == 1 && err_count) {
#pragma unroll
        for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if (lane == 0 && bad) atomicAdd(err_count, bad);
    }
    __syncthreads();
    for (int l = threadIdx.x; l < El; l += kScatterThreads) {
        int c;
        if (!derive) {
            c = __ldg(counts_in + l);
        } else if (G > 1) {
            c = tot[l];
        } else {
            c = 0;
            for (int w = 0; w < kWarps; ++w) c += wc[w * El + l];
        }
        if (derive && blockIdx.x == 0) counts_out[l] = c;
        off[l] = (c + kGroup - 1) / kGroup * kGroup;  // padded block sizes, scanned below
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of the padded block sizes
        // Offsets never pass the caller's row bound (a multiple of 128): counts given by
        // the caller that disagree with the ids cannot place rows outside a_out. With
        // consistent counts the bound is never reached.
        int run = 0;
        for (int lb = 0; lb < El; lb += 32) {
            const int l = lb + lane;
            const int c = l < El ? off[l] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (l < El) off[l] = min(run + incl - c, row_cap);
            run = min(run + __shfl_sync(0xffffffffu, incl, 31), row_cap);
        }
        if (lane == 0) off[El] = run;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int l = threadIdx.x; l <= El; l += kScatterThreads) expert_offsets[l] = off[l];
    for (int l = threadIdx.x; l < El; l += kScatterThreads) {
        int run = off[l] + base[l];
        for (int w = 0; w < kWarps; ++w) {
            const int c = wc[w * El + l];
            wc[w * El + l] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int64_t r0 = wbeg; r0 < wend; r0 += 32 * kRound) {
        int l[kRound];
        if (r0 == wbeg) {
#pragma unroll
            for (int j = 0; j < kRound; ++j) l[j] = l0[j];
        } else {
            load_round(ids, r0, wend, expert_map, E, El, lane, l, bad);
        }
        int dst[kRound];
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            const unsigned m = __match_any_sync(0xffffffffu, l[j]);
            const int rank = __popc(m & lanemask_lt());
            dst[j] = -1;
            if (l[j] >= 0) {
                dst[j] = mine[l[j]] + rank;
                // counts inconsistent with the ids: the slot is dropped, never written past
                // its expert's block (whose end is at most the row bound)
                if (dst[j] >= off[l[j] + 1]) dst[j] = -1;
            }
            __syncwarp();
            if (l[j] >= 0 && rank == 0) mine[l[j]] += __popc(m);
            __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            const int64_t i = r0 + j * 32 + lane;
            if (i < wend) src2dst[i] = dst[j];
        }
    }
}

// One (token, 512-column span) unit of the row copy: lane j holds 16 consecutive values of
// the span (raw0, raw1: its bf16 bits), 8 lanes form one 1x128 group; my_dst / my_w are
// the token's slot destinations and weights, lane k holding slot k. The row was read
// once and is written to each kept slot.
// the 16 bf16 values of raw0, raw1 as fp32
__device__ __forceinline__ void unpack16(uint4 raw0, uint4 raw1, float (&v)[16]) {
    const uint32_t w[8] = {raw0.x, raw0.y, raw0.z, raw0.w, raw1.x, raw1.y, raw1.z, raw1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// have_q: the weights are not applied on the input and the caller has already quantised
// the span (codes q0, scale s0); otherwise it is quantised here.
template <bool kQuant>
__device__ __forceinline__ void copy_unit(int lane, int K, int g, int col, bool active, int topk, int apply_on_input,
                                          int my_dst, float my_w, uint4 raw0, uint4 raw1, void* __restrict__ a_out,
                                          float* __restrict__ a_scale, bool have_q = false,
                                          uint4 q0 = make_uint4(0, 0, 0, 0), float s0 = 0.f) {
    const int G = K / kGroup;
    float v[16];
    unpack16(raw0, raw1, v);
    if (!apply_on_input) {
        float s = s0;
        uint4 q = q0;
        if (kQuant && !have_q) q = quant16_group8(v, s);
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

// One warp per (token, 512-column span). The kernel before this one is always the rank
// kernel, which waited for everything before it before letting this one launch: the
// caller's inputs (x, the weights) are final, so the span is read (and, without the
// weights on the input, quantised) before the wait; the destinations and every write come
// after it.
template <bool kQuant>
__global__ void __launch_bounds__(256)
    scatter_copy_kernel(const uint16_t* __restrict__ x, int64_t M, int K, const int32_t* __restrict__ src2dst,
                        const float* __restrict__ topk_weights, int topk, int apply_on_input,
                        void* __restrict__ a_out, float* __restrict__ a_scale) {
    const int lane = threadIdx.x & 31;
    const int spans = (K + 511) / 512;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const bool unit = gw < M * spans;
    const int64_t t = unit ? gw / spans : 0;
    const int g = (int)(gw % spans) * 4 + (lane >> 3);
    const bool active = unit && g < K / kGroup;
    const int col = g * kGroup + (lane & 7) * 16;
    const float my_w = (unit && lane < topk && apply_on_input) ? __ldg(topk_weights + t * topk + lane) : 1.f;
    uint4 raw0 = make_uint4(0, 0, 0, 0), raw1 = raw0;
    if (active) {
        const uint4* src = reinterpret_cast<const uint4*>(x + t * K + col);
        raw0 = __ldg(src);
        raw1 = __ldg(src + 1);
    }
    uint4 q = make_uint4(0, 0, 0, 0);
    float s = 0.f;
    if (kQuant && !apply_on_input) {
        float v[16];
        unpack16(raw0, raw1, v);
        q = quant16_group8(v, s);
    }
    pdl_wait();
    pdl_trigger();
    if (!unit) return;
    const int my_dst = lane < topk ? __ldg(src2dst + t * topk + lane) : -1;
    copy_unit<kQuant>(lane, K, g, col, active, topk, apply_on_input, my_dst, my_w, raw0, raw1, a_out, a_scale,
                      !apply_on_input, q, s);
}

// ------------------------------------------------------- scatter, small batches
// For at most kSmallSlots top-k slots the whole scatter is one kernel: every CTA ranks all
// the slots itself in shared memory (the same stable counting sort as the rank kernel: 8
// contiguous warp segments, per-warp counts, expert offsets, per-warp cursors, ranks by
// __match_any_sync), then copies and quantises its own (token, span) units. Ranking a few
// thousand slots costs each CTA far less than the launch and the global round trip of a
// separate index kernel. CTA 0 writes the offsets, counts and src2dst.
// early != 0 (only for chunks after the first inside the chunk loop, where the kernels
// still running before this one are the previous chunk's GEMMs and gather, none of which
// writes these inputs): the ids, expert map, weights and the unit's row are read and
// ranked before waiting for them; every write still comes after the wait.
constexpr int kSmallSlots = 4096;
constexpr int kSmallGroups = kSmallSlots / (kScatterThreads / 32) / 32;  // groups of 32 per warp at most

template <typename TId, bool kQuant>
__global__ void __launch_bounds__(kScatterThreads)
    scatter_small_kernel(const uint16_t* __restrict__ x, int64_t M, int K, const TId* __restrict__ ids,
                         const float* __restrict__ topk_weights, int topk, const int32_t* __restrict__ expert_map,
                         int E, int El, const int32_t* __restrict__ counts_in, int32_t* __restrict__ counts_out,
                         int32_t* __restrict__ err_count, int apply_on_input, void* __restrict__ a_out,
                         float* __restrict__ a_scale, int32_t* __restrict__ expert_offsets,
                         int32_t* __restrict__ src2dst, int row_cap, int early) {
    constexpr int kWarps = kScatterThreads / 32;
    extern __shared__ int32_t sm[];
    int32_t* off = sm;               // [El + 1]
    int32_t* wc = off + El + 1;      // [kWarps][El]: per-warp counts, then per-warp cursors
    int32_t* s_dst = wc + kWarps * El;  // [n]: permuted row of every slot, -1 if dropped
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = (int)(M * topk);
    if (!early) pdl_wait();
    // this warp's copy unit: its row span is loaded first, so that the loads are in flight
    // while the slots are ranked
    const int spans = (K + 511) / 512;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
    const bool unit = gw < M * spans;
    const int64_t t = unit ? gw / spans : 0;
    const int g = (int)(gw % spans) * 4 + (lane >> 3);
    const bool active = unit && g < K / kGroup;
    const int col = g * kGroup + (lane & 7) * 16;
    uint4 raw0 = make_uint4(0, 0, 0, 0), raw1 = raw0;
    if (active) {
        const uint4* src = reinterpret_cast<const uint4*>(x + t * K + col);
        raw0 = __ldg(src);
        raw1 = __ldg(src + 1);
    }
    const float my_w = (unit && lane < topk && apply_on_input) ? __ldg(topk_weights + t * topk + lane) : 1.f;
    // the warp's segment of the slots, in groups of 32
    const int pw = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
    const int wbeg = warp * pw, wend = min(n, wbeg + pw);
    int lv[kSmallGroups];
    int bad = 0;
#pragma unroll
    for (int j = 0; j < kSmallGroups; ++j) {
        const int i = wbeg + j * 32 + lane;
        lv[j] = (i < wend) ? local_expert(__ldg(ids + i), expert_map, E, El, bad) : -1;
    }
    for (int i = threadIdx.x; i < kWarps * El; i += kScatterThreads) wc[i] = 0;
    __syncthreads();
    int32_t* mine = wc + warp * El;
#pragma unroll
    for (int j = 0; j < kSmallGroups; ++j) {
        if (wbeg + j * 32 >= wend) break;  // warp-uniform
        const unsigned m = __match_any_sync(0xffffffffu, lv[j]);
        if (lv[j] >= 0 && lane == __ffs(m) - 1) mine[lv[j]] += __popc(m);
        __syncwarp();
    }
    __syncthreads();
    const bool derive = counts_in == nullptr;
    for (int l = threadIdx.x; l < El; l += kScatterThreads) {
        int c = 0;
        if (derive) {
            for (int w = 0; w < kWarps; ++w) c += wc[w * El + l];
        } else {
            c = __ldg(counts_in + l);
        }
        off[l] = (c + kGroup - 1) / kGroup * kGroup;
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of the padded block sizes, clamped to the row bound
        int run = 0;
        for (int lb = 0; lb < El; lb += 32) {
            const int l = lb + lane;
            const int c = l < El ? off[l] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tt = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += tt;
            }
            if (l < El) off[l] = min(run + incl - c, row_cap);
            run = min(run + __shfl_sync(0xffffffffu, incl, 31), row_cap);
        }
        if (lane == 0) off[El] = run;
    }
    __syncthreads();
    // per-warp cursors; the counts derived here are read back before they are overwritten
    int cnt_l[4];  // at most El / kScatterThreads + 1 = 4 experts per thread for El <= 1024
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int l = threadIdx.x + q * kScatterThreads;
        cnt_l[q] = 0;
        if (l < El) {
            int run = off[l];
            for (int w = 0; w < kWarps; ++w) {
                const int c = wc[w * El + l];
                cnt_l[q] += c;
                wc[w * El + l] = run;
                run += c;
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kSmallGroups; ++j) {
        if (wbeg + j * 32 >= wend) break;  // warp-uniform
        const unsigned m = __match_any_sync(0xffffffffu, lv[j]);
        const int rank = __popc(m & lanemask_lt());
        int dst = -1;
        if (lv[j] >= 0) {
            dst = mine[lv[j]] + rank;
            // counts given by the caller that disagree with the ids: the slot is dropped
            if (dst >= off[lv[j] + 1]) dst = -1;
        }
        __syncwarp();
        if (lv[j] >= 0 && rank == 0) mine[lv[j]] += __popc(m);
        __syncwarp();
        const int i = wbeg + j * 32 + lane;
        if (i < wend) s_dst[i] = dst;
    }
    __syncthreads();
    if (early) pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0) {
        for (int l = threadIdx.x; l <= El; l += kScatterThreads) expert_offsets[l] = off[l];
        if (derive) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int l = threadIdx.x + q * kScatterThreads;
                if (l < El) counts_out[l] = cnt_l[q];
            }
            if (err_count) {
#pragma unroll
                for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
                if (lane == 0 && bad) atomicAdd(err_count, bad);
            }
        }
        for (int i = threadIdx.x; i < n; i += kScatterThreads) src2dst[i] = s_dst[i];
    }
    if (!unit) return;
    const int my_dst = lane < topk ? s_dst[t * topk + lane] : -1;
    copy_unit<kQuant>(lane, K, g, col, active, topk, apply_on_input, my_dst, my_w, raw0, raw1, a_out, a_scale);
}

bool scatter_is_one_kernel(int64_t M, int topk, int El) {
    const int64_t n = M * topk;
    return n <= kSmallSlots && (size_t)(El + 1 + (kScatterThreads / 32) * El + n) * sizeof(int32_t) <= 48 * 1024;
}

template <typename TId>
int launch_scatter(const uint16_t* x, int64_t M, int K, const TId* ids, const float* topk_weights, int topk,
                   const int32_t* expert_map, int E, int El, const int32_t* counts_in, int32_t* counts_out,
                   int32_t* err_count, int apply_on_input, int quant, void* a_out, float* a_scale,
                   int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, int32_t* hist, int early,
                   cudaStream_t stream) {
    const int64_t n = M * topk;
    const int row_cap = (int)(rp_cap / kGroup * kGroup);
    if (scatter_is_one_kernel(M, topk, El)) {
        const size_t small_smem = (size_t)(El + 1 + (kScatterThreads / 32) * El + n) * sizeof(int32_t);
        const int64_t units = M * ((K + 511) / 512);
        const unsigned sgrid = (unsigned)(units > 0 ? (units + 7) / 8 : 1);
        const size_t smem = small_smem;
        const int e = (early && !counts_in) ? 1 : 0;  // caller-given counts may come from the kernel before
        if (quant == MOE_QUANT_FP8_1X128)
            launch_k(scatter_small_kernel<TId, true>, sgrid, kScatterThreads, smem, stream, x, M, K, ids, topk_weights,
                     topk, expert_map, E, El, counts_in, counts_out, err_count, apply_on_input, a_out, a_scale,
                     expert_offsets, src2dst, row_cap, e);
        else
            launch_k(scatter_small_kernel<TId, false>, sgrid, kScatterThreads, smem, stream, x, M, K, ids, topk_weights,
                     topk, expert_map, E, El, counts_in, counts_out, err_count, apply_on_input, a_out, a_scale,
                     expert_offsets, src2dst, row_cap, e);
        note_launches(1);
        return launch_status();
    }
    const int per_cta = scatter_slots_per_cta(n);
    const int grid = (int)((n + per_cta - 1) / per_cta);
    const size_t smem_rank = (size_t)(3 * El + 1 + (kScatterThreads / 32) * El) * sizeof(int32_t);
    int launches = 0;
    if (grid > 1) {
        launch_k(scatter_hist_kernel<TId>, grid, kScatterThreads, (size_t)kCountCopies * El * sizeof(int32_t), stream, ids, n, expert_map, E, El, per_cta, hist, counts_in ? nullptr : err_count);
        ++launches;
    }
    launch_k(scatter_rank_kernel<TId>, grid < 1 ? 1 : grid, kScatterThreads, smem_rank, stream, ids, n, expert_map, E, El, per_cta, counts_in, hist, expert_offsets, src2dst, counts_out, counts_in ? nullptr : err_count, row_cap);
    ++launches;
    if (M > 0) {
        const int64_t warps = M * ((K + 511) / 512);
        const unsigned cgrid = (unsigned)((warps + 7) / 8);
        if (quant == MOE_QUANT_FP8_1X128)
            launch_k(scatter_copy_kernel<true>, cgrid, 256, 0, stream, x, M, K, src2dst, topk_weights, topk, apply_on_input, a_out, a_scale);
        else
            launch_k(scatter_copy_kernel<false>, cgrid, 256, 0, stream, x, M, K, src2dst, topk_weights, topk, apply_on_input, a_out, a_scale);
        ++launches;
    }
    note_launches(launches);
    return launch_status();
}
#define MOE_INSTANTIATE_SCATTER(TId)                                                                              \
    template int launch_scatter<TId>(const uint16_t*, int64_t, int, const TId*, const float*, int, const int32_t*, \
                                     int, int, const int32_t*, int32_t*, int32_t*, int, int, void*, float*,         \
                                     int32_t*, int32_t*, int64_t, int32_t*, int, cudaStream_t);
MOE_INSTANTIATE_SCATTER(int32_t)
MOE_INSTANTIATE_SCATTER(int64_t)
#undef MOE_INSTANTIATE_SCATTER

// ----------------------------------------------------------------------- gather
// One warp per (token, 256-column span): lane j owns 8 bf16 columns (16 bytes). The
// kept rows of the token are loaded 8 at a time (independent 16-byte loads in flight),
// then accumulated in ascending k with separately rounded fp32 multiply and add.
// Y is read exactly once (ld_once_256).

__global__ void __launch_bounds__(256)
    gather_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ src2dst,
                  const float* __restrict__ topk_weights, int64_t M, int topk, int K, int apply_on_input,
                  uint16_t* __restrict__ out, int early_trigger) {
    const int lane = threadIdx.x & 31;
    // early_trigger (inside a chunk loop, when the next chunk's one-kernel scatter follows,
    // which reads only the call's own inputs before its own wait): the next kernel may
    // launch at once, and ranks its slots while this one runs.
    if (early_trigger) pdl_trigger();
    pdl_wait();
    if (!early_trigger) pdl_trigger();
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
            if (d[j] >= 0 && active) r[j] = ld_once_256(y + (int64_t)d[j] * K + col);
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
                  int apply_on_input, uint16_t* out, cudaStream_t stream, int early_trigger) {
    if (M == 0) return MOE_OK;
    const int64_t warps = M * ((K + 255) / 256);
    launch_k(gather_kernel, (unsigned)((warps + 7) / 8), 256, 0, stream, y, src2dst, topk_weights, M, topk, K, apply_on_input,
             out, early_trigger);
    note_launches(1);
    return launch_status();
}

// ------------------------------------------------------------- SiLU-and-mul quant
// Requantisation of 16 h values of one 1x128 group (8 lanes x 16): scale = amax/448,
// code = e4m3(h/scale) with the correctly rounded quotient (same rule as the scatter).
__device__ __forceinline__ uint4 requant16_group8(const float (&v)[16], float& scale_out) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 448.0f);
    scale_out = s;
    float q[16];
    if (s == 0.f) {
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = 0.f;
    } else if (s >= 1e-30f) {  // 1/s finite and normal
        const float r = __frcp_rn(s);
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = div_rn_by(v[j], s, r);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = __fdiv_rn(v[j], s);
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = uint32_t(f32x2_to_e4m3x2(q[4 * i], q[4 * i + 1])) | (uint32_t(f32x2_to_e4m3x2(q[4 * i + 2], q[4 * i + 3])) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// One warp per (row, 512-column span of h).
__global__ void __launch_bounds__(256)
    silu_mul_quant_kernel(const float* __restrict__ c1, const int32_t* __restrict__ expert_offsets, int El,
                          int64_t rp_cap, int N, uint8_t* __restrict__ h, float* __restrict__ h_scale) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
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
    const uint4 q = requant16_group8(v, s);
    if (!active) return;
    *reinterpret_cast<uint4*>(h + r * N + col) = q;
    if ((lane & 7) == 0) h_scale[r * G + g] = s;
}

int launch_silu_mul_quant(const float* c1, const int32_t* expert_offsets, int El, int64_t rp_cap, int N, uint8_t* h,
                          float* h_scale, cudaStream_t stream) {
    if (rp_cap == 0) return MOE_OK;
    const int64_t warps = rp_cap * ((N + 511) / 512);
    launch_k(silu_mul_quant_kernel, (unsigned)((warps + 7) / 8), 256, 0, stream, c1, expert_offsets, El, rp_cap, N, h, h_scale);
    note_launches(1);
    return launch_status();
}

}  // namespace moe
