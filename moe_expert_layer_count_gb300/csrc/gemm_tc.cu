// Block-scaled FP8 grouped GEMM on the 5th-generation tensor cores (tcgen05, sm_103a):
//   out[r, j] = sum_kb a_scale[r, kb] * w_scale[l, j/128, kb] * sum_{k in kb} A[r,k] W[l,j,k]
// for the rows r of every local expert l's 128-aligned block -- the DeepGEMM "m-grouped
// contiguous" GEMM of vLLM PR #20903 "[Kernel] DeepGemm MoE : Integrate triton permute
// / unpermute kernels", section "Optimizations" (float8_e4m3fn, --block-shape 128 128).
//
// Design (one persistent CTA per SM, warp-specialised):
//  * warp 8 (one thread) streams 128x128 A tiles and BNx128 W tiles into a ring of
//    shared-memory stages with TMA (128-byte swizzle), one stage per 128-wide K block;
//  * bf16/fp32 epilogues: warp 10 copies each K block's block scales (the 128 row
//    scales of A, two W scales) into a ring of shared-memory slots with cp.async,
//    running up to 8 K blocks ahead of the epilogue. The SiLU epilogue has no warp 10:
//    each epilogue thread loads its row's scales itself, one K block ahead (measured
//    faster for that GEMM, whose 16 K blocks per tile leave the loads time to land);
//  * warp 9 (one thread) issues tcgen05.mma kind::f8f6f4 (M=128, N=BN, K=32, four per
//    K block) into one of the 512/BN TMEM accumulators (two for 256-wide tiles),
//    starting each K block from zero;
//  * warps 0-7 (two warpgroups, each one TMEM lane = one row per thread, half of the
//    tile's columns each) read the K block's partial sums from TMEM, release the buffer
//    and fold them into fp32 registers with the product of the two block scales. The
//    scales are fp32 amax/448 values, not powers of two, so they are applied here in
//    software rather than by the block-scaled MMA kinds. Double-buffering TMEM lets the
//    MMA of block kb+1 run while block kb is promoted.
//  * Epilogues: bf16 or fp32 rows, or SiLU-and-mul with 1x128 FP8 requantisation. For
//    the latter the W tile is gate rows [j, j+64) | up rows [j, j+64) | gate [j+64, j+128)
//    | up [j+64, j+128), so each warpgroup holds matching gate/up columns of 64 outputs
//    and one amax exchange per row (shared memory and a hardware named barrier over the
//    8 epilogue warps) completes the 128-wide group.
// Small batches (given the experts' valid row counts) run a variant in which an epilogue
// warp whose 32 rows are all padding skips the TMEM reads, folding and stores, and in
// which a tile whose kept rows all lie in its first 32 (or 64) loads only those rows of A.
// With kOptWeightsEvictFirst the weight tiles are loaded under the L2 evict-first policy
// (the chunk loop sets it for W13 when every chunk reads each W13 tile once).
// Every wait on a pipeline barrier gives up after 2 s, sets a device error word and an
// abort flag seen by all roles, waits (bounded) for its own copies and MMAs in flight,
// and the CTA frees its TMEM and returns. An epilogue warp that gives up arrives on the
// named barrier of the tile it leaves, so the exchange never waits for it.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "route.cuh"
#include "sm100_ptx.cuh"

namespace moe {

__device__ int g_gemm_error;  // set to 1 when a pipeline wait ran out of time

namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;  // one K block: 128 fp8 = one 128-byte swizzled row
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kScaleWarp = 10;
constexpr int kMaxDevices = 64;

// Whether an epilogue gets its block scales from the scale warp's ring, and the block
// size that follows (at most 3 warps per SM sub-partition either way).
template <int EPI>
__host__ __device__ constexpr bool staged_scales() { return EPI != MOE_EPI_SILU_MUL_QUANT; }
template <int EPI>
__host__ __device__ constexpr int threads_of() { return (kEpiWarps + (staged_scales<EPI>() ? 3 : 2)) * 32; }
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kBoxRows = 64;  // W is loaded in 64-row TMA boxes

template <int BN, int EPI>
struct Cfg {
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemBufs = 512 / BN;  // K-block partials TMEM holds at once
    static constexpr int kTmemCols = kTmemBufs * BN;
    static constexpr int kCols = BN / 2;  // accumulator columns per epilogue thread
    // bf16 output leaves in 128-byte-wide boxes from a staging buffer that holds the
    // warp's whole 32-row slab (all its stores of a tile go out without waiting); the
    // other epilogues stage one 32 x 64-byte box per warp. The pipeline gets what
    // shared memory is left.
    static constexpr bool kWide = EPI == MOE_EPI_BF16;
    static constexpr int kStageWarpBytes = kWide ? 32 * kCols * 2 : 32 * 64;
    static constexpr int kStages = BN == 256 ? (kWide ? 3 : 4) : (kWide ? 5 : 6);
};

// Block scales of one K block of one tile: a_scale of the tile's 128 rows and the two
// W scales its columns need (the two 128-column halves for BN = 256, the same value
// twice for BN = 128).
struct __align__(16) ScaleSlot {
    float sa[kBM];
    float sw[4];
};
// The scale warp fills it up to kScaleRing K blocks ahead of the epilogue.
constexpr int kScaleRing = 8;

struct __align__(8) Tail {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[4];
    uint64_t tempty[4];
    uint64_t sfull[kScaleRing];
    uint64_t sempty[kScaleRing];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

constexpr int kStageRowBytes = 64;  // rows of the 64-byte-wide output boxes

template <int BN, int EPI>
constexpr size_t smem_bytes(int El) {
    using C = Cfg<BN, EPI>;
    return 1024 + (size_t)C::kStages * C::kStageBytes + sizeof(Tail) + 16 + kScaleRing * sizeof(ScaleSlot) +
           2 * 2 * 128 * sizeof(float) + (size_t)(2 * El + 1) * sizeof(int32_t) + 1024 +
           (size_t)kEpiWarps * C::kStageWarpBytes;
}

// Byte offset of 16-byte chunk c (0..3) of row r (0..31) in a warp's 32 x 64-byte
// staging buffer. The XOR spreads the 8 rows of every 512-byte group over all 32 banks,
// so both the row-per-lane writes and the 8-rows-per-instruction reads are conflict-free.
__device__ __forceinline__ uint32_t stage_off(int r, int c) {
    return (uint32_t)(r * kStageRowBytes + ((c ^ ((r >> 1) & 3)) << 4));
}

// Stores a 32-row x 64-byte box of the output (lane = row of the warp's 32-row slab,
// 64 bytes per lane) with one TMA store: the lanes write the swizzled staging buffer
// (the layout above is exactly TMA's 64-byte swizzle), then lane 0 issues the bulk
// store at tensor coordinates (x, y). The buffer is reused only after the previous
// store has read it.
__device__ __forceinline__ void store_box64(uint8_t* stage, int lane, const uint4 (&v)[4], const CUtensorMap* tm,
                                            int32_t x, int32_t y) {
    if (lane == 0) ptx::bulk_wait_read0();
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(stage + stage_off(lane, c)) = v[c];
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        ptx::tma_store_2d(tm, ptx::smem_addr(stage), x, y);
        ptx::bulk_commit();
    }
}

// Bounded wait on an mbarrier phase. With check_abort, returns false as soon as another
// role has aborted; otherwise waits for the phase or the time limit only.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort, bool check_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 31) == 0) {
            if (check_abort && *abort) return false;
            if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
                *abort = 1;
                atomicExch(&g_gemm_error, 1);
                return false;
            }
        }
    }
}

__device__ __forceinline__ int expert_of(const int32_t* s_off, int El, int row0) {
    int lo = 0, hi = El - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= row0) lo = mid; else hi = mid - 1;
    }
    return lo;
}


template <int BN, int EPI, bool kSkip>
__global__ void __launch_bounds__(threads_of<EPI>(), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA32,
                   const __grid_constant__ CUtensorMap tmA64, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, const float* __restrict__ sa, const float* __restrict__ sw,
                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts,
                   int El, int row_cap, int n_out, int k_in, void* __restrict__ out, float* __restrict__ out_scale,
                   int opts) {
    using C = Cfg<BN, EPI>;
    constexpr bool kSilu = EPI == MOE_EPI_SILU_MUL_QUANT;
    constexpr bool kStaged = staged_scales<EPI>();
    static_assert(!kSilu || BN == 256, "the SiLU epilogue pairs 128 gate with 128 up columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Tail* st = reinterpret_cast<Tail*>(smem + C::kStages * C::kStageBytes);
    ScaleSlot* s_scale = reinterpret_cast<ScaleSlot*>((reinterpret_cast<uintptr_t>(st + 1) + 15) & ~uintptr_t(15));
    float* s_amax = reinterpret_cast<float*>(s_scale + kScaleRing);  // [2 parities][2 warpgroups][128 rows]
    int32_t* s_off = reinterpret_cast<int32_t*>(s_amax + 2 * 2 * 128);
    int32_t* s_cnt = s_off + El + 1;  // valid rows of each expert's block (kSkip only)
    uint8_t* s_stage = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(s_cnt + (kSkip ? El : 0)) + 1023) & ~uintptr_t(1023));
    volatile int* abort = &st->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&st->full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&st->empty[s]), 1);
        }
        for (int b = 0; b < C::kTmemBufs; ++b) {
            ptx::mbar_init(ptx::smem_addr(&st->tfull[b]), 1);
            ptx::mbar_init(ptx::smem_addr(&st->tempty[b]), kEpiWarps);
        }
        for (int j = 0; j < kScaleRing; ++j) {
            ptx::mbar_init(ptx::smem_addr(&st->sfull[j]), 32);  // one cp.async arrival per producer lane
            ptx::mbar_init(ptx::smem_addr(&st->sempty[j]), kEpiWarps);
        }
        ptx::mbar_init(ptx::smem_addr(&st->mma_done), 1);
        st->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&st->tmem_base), C::kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
    }
    if (warp == kProducerWarp && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        if (kSkip) {
            ptx::prefetch_tmap(&tmA32);
            ptx::prefetch_tmap(&tmA64);
        }
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmO);
    }
    // the prologue above overlaps the previous kernel's end; global memory only after this
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= El; i += threads_of<EPI>()) {
        s_off[i] = __ldg(offsets + i);
        if (kSkip && i < El) s_cnt[i] = __ldg(counts + i);
    }
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = st->tmem_base;

    // rows past the buffers' row count are never touched, whatever the offsets say
    const int m_tiles = min(s_off[El], row_cap) / kBM;
    const int n_tiles = kSilu ? n_out / 256 : n_out / BN;
    const int tiles = m_tiles * n_tiles;
    const int KB = k_in / kBK;
    const int NB = n_out / 128;  // weight-scale blocks along n_out

    if (warp == kProducerWarp) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            // weight tiles take the cache-hinted load only under kOptWeightsEvictFirst (the
            // plain load measured faster than a hinted one at the normal priority)
            const bool w_evict_first = (opts & kOptWeightsEvictFirst) != 0;
            const uint64_t w_policy = ptx::policy_evict_first();
            for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
                const int mt = tile / n_tiles, nt = tile % n_tiles;
                const int row0 = mt * kBM;
                const int l = expert_of(s_off, El, row0);
                // small batches: when all of the tile's kept rows lie in its first 32 (64),
                // only those rows of A are loaded (the rest of the tile's A stays whatever
                // the stage held before: those rows are padding, whose warps neither fold
                // nor store anything)
                int a_rows = kBM;
                if constexpr (kSkip) {
                    const int kept = s_off[l] + s_cnt[l] - row0;
                    a_rows = kept <= 32 ? 32 : kept <= 64 ? 64 : kBM;
                }
                const CUtensorMap* tma = a_rows == 32 ? &tmA32 : a_rows == 64 ? &tmA64 : &tmA;
                const uint32_t stage_bytes = C::kStageBytes - (uint32_t)(kBM - a_rows) * kBK;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t ph = (it / C::kStages) & 1;
                    if (!wait_phase(ptx::smem_addr(&st->empty[s]), ph ^ 1, abort)) { ok = false; break; }
                    const uint32_t full = ptx::smem_addr(&st->full[s]);
                    ptx::mbar_arrive_expect_tx(full, stage_bytes);
                    const uint32_t a_dst = ptx::smem_addr(smem + s * C::kStageBytes);
                    const uint32_t b_dst = a_dst + C::kABytes;
                    ptx::tma_load_2d(a_dst, tma, kb * kBK, row0, full);
#pragma unroll
                    for (int p = 0; p < BN / kBoxRows; ++p) {
                        int brow;
                        if (kSilu)  // gate | up | gate | up, 64 rows each
                            brow = l * n_out + (p & 1) * (n_out / 2) + nt * 128 + (p >> 1) * kBoxRows;
                        else
                            brow = l * n_out + nt * BN + p * kBoxRows;
                        if (w_evict_first)
                            ptx::tma_load_2d_hint(b_dst + p * kBoxRows * kBK, &tmB, kb * kBK, brow, full, w_policy);
                        else
                            ptx::tma_load_2d(b_dst + p * kBoxRows * kBK, &tmB, kb * kBK, brow, full);
                    }
                }
            }
            // never leave with copies in flight: the last stages' loads must have landed
            const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0;
            for (uint32_t j = first; j < it; ++j)
                wait_phase(ptx::smem_addr(&st->full[j % C::kStages]), (j / C::kStages) & 1, abort, false);
        }
    } else if (kStaged && warp == kScaleWarp) {
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
            const int mt = tile / n_tiles, nt = tile % n_tiles;
            const int row0 = mt * kBM;
            const int l = expert_of(s_off, El, row0);
            // this lane's four rows of a_scale, and the tile's two W-scale rows
            const float* sa_lane = sa + (int64_t)(row0 + lane) * KB;
            const int nb0 = BN == 256 ? 2 * nt : nt;
            const int nb1 = BN == 256 ? 2 * nt + 1 : nt;
            const float* swa = sw + ((int64_t)l * NB + nb0) * KB;
            const float* swb = sw + ((int64_t)l * NB + nb1) * KB;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int j = it % kScaleRing;
                bool go = true;
                if (lane == 0) go = wait_phase(ptx::smem_addr(&st->sempty[j]), ((it / kScaleRing) & 1) ^ 1, abort);
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) { ok = false; break; }
                const uint32_t slot = ptx::smem_addr(&s_scale[j]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    ptx::cp_async4(slot + 4u * (uint32_t)(lane + 32 * q), sa_lane + (int64_t)32 * q * KB + kb);
                if (lane == 0) {
                    ptx::cp_async4(slot + 4u * kBM, swa + kb);
                    ptx::cp_async4(slot + 4u * (kBM + 1), swb + kb);
                }
                ptx::cp_async_mbar_arrive_noinc(ptx::smem_addr(&st->sfull[j]));
            }
        }
        // never leave with copies in flight
        ptx::cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_e4m3_f32(kBM, BN);
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t ph = (it / C::kStages) & 1;
                    const int b = it % C::kTmemBufs;
                    const uint32_t tph = (it / C::kTmemBufs) & 1;
                    if (!wait_phase(ptx::smem_addr(&st->tempty[b]), tph ^ 1, abort)) { ok = false; break; }
                    if (!wait_phase(ptx::smem_addr(&st->full[s]), ph, abort)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a_base = ptx::smem_addr(smem + s * C::kStageBytes);
                    const uint32_t b_base = a_base + C::kABytes;
                    const uint32_t d = tmem + (uint32_t)(b * BN);
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        ptx::mma_f8f6f4(d, ptx::smem_desc_sw128(a_base + 32 * k, 1024),
                                        ptx::smem_desc_sw128(b_base + 32 * k, 1024), idesc, k > 0 ? 1u : 0u);
                    ptx::mma_commit(ptx::smem_addr(&st->empty[s]));
                    ptx::mma_commit(ptx::smem_addr(&st->tfull[b]));
                }
            }
            // never leave with MMAs in flight
            ptx::mma_commit(ptx::smem_addr(&st->mma_done));
            wait_phase(ptx::smem_addr(&st->mma_done), 0, abort, false);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int wg = warp >> 2;
        const int row_in_tile = (warp & 3) * 32 + lane;
        const uint32_t lane_field = (uint32_t)((warp & 3) * 32) << 16;
        uint32_t it = 0;
        int tcount = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x, ++tcount) {
            const int mt = tile / n_tiles, nt = tile % n_tiles;
            const int row0 = mt * kBM;
            const int64_t r = row0 + row_in_tile;
            if constexpr (kSkip) {
                // a warp whose 32 rows are all padding of the expert's block (small
                // batches leave most of a block empty) reads no partial sums and stores
                // nothing: it only keeps step with the pipeline barriers
                const int le = expert_of(s_off, El, row0);
                if ((warp & 3) * 32 >= s_off[le] + s_cnt[le] - row0) {
                    for (int kb = 0; kb < KB; ++kb, ++it) {
                        const int b = it % C::kTmemBufs;
                        bool got;
                        if constexpr (kStaged) {
                            const int j = it % kScaleRing;
                            got = wait_phase(ptx::smem_addr(&st->sfull[j]), (it / kScaleRing) & 1, abort) &&
                                  wait_phase(ptx::smem_addr(&st->tfull[b]), (it / C::kTmemBufs) & 1, abort);
                        } else {
                            got = wait_phase(ptx::smem_addr(&st->tfull[b]), (it / C::kTmemBufs) & 1, abort);
                        }
                        got = __all_sync(0xffffffffu, got);
                        if (!got) { ok = false; break; }
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (kStaged) ptx::mbar_arrive(ptx::smem_addr(&st->sempty[it % kScaleRing]));
                            ptx::mbar_arrive(ptx::smem_addr(&st->tempty[b]));
                        }
                    }
                    if (kSilu) {
                        if (!ok) {
                            asm volatile("bar.arrive 1, 256;" ::: "memory");
                            break;
                        }
                        // the partner warp (same rows) is idle too; the exchange still
                        // needs every epilogue warp once per tile
                        asm volatile("bar.sync 1, 256;" ::: "memory");
                    }
                    continue;
                }
            }
            // fp32 accumulators as pairs, updated with packed fp32 FMAs (two per
            // instruction, each rounded exactly like fmaf)
            float2 acc2[C::kCols / 2];
#pragma unroll
            for (int c = 0; c < C::kCols / 2; ++c) acc2[c] = make_float2(0.f, 0.f);
            const uint32_t tcol = lane_field + (uint32_t)(wg * C::kCols);
            // SiLU: this row's a_scale and the gate/up W scales, loaded one K block ahead
            const float* sa_row = nullptr;
            const float* sw0 = nullptr;
            const float* sw1 = nullptr;
            float sr_n = 0.f, s0_n = 0.f, s1_n = 0.f;
            if constexpr (!kStaged) {
                const int l = expert_of(s_off, El, row0);
                sa_row = sa + r * KB;
                sw0 = sw + ((int64_t)l * NB + nt) * KB;
                sw1 = sw + ((int64_t)l * NB + NB / 2 + nt) * KB;
                sr_n = __ldg(sa_row);
                s0_n = __ldg(sw0);
                s1_n = __ldg(sw1);
            }
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int b = it % C::kTmemBufs;
                float s0, s1;  // scale products for the two halves of this thread's columns
                if constexpr (kStaged) {
                    // the K block's scales, staged by the scale warp well ahead
                    const int j = it % kScaleRing;
                    bool got = wait_phase(ptx::smem_addr(&st->sfull[j]), (it / kScaleRing) & 1, abort) &&
                               wait_phase(ptx::smem_addr(&st->tfull[b]), (it / C::kTmemBufs) & 1, abort);
                    got = __all_sync(0xffffffffu, got);
                    if (!got) { ok = false; break; }
                    ptx::tc_fence_after();
                    s0 = s1 = s_scale[j].sa[row_in_tile] * s_scale[j].sw[BN == 256 ? wg : 0];
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&st->sempty[j]));
                } else {
                    const float sr = sr_n, sb0 = s0_n, sb1 = s1_n;
                    if (kb + 1 < KB) {
                        sr_n = __ldg(sa_row + kb + 1);
                        s0_n = __ldg(sw0 + kb + 1);
                        s1_n = __ldg(sw1 + kb + 1);
                    }
                    bool got = wait_phase(ptx::smem_addr(&st->tfull[b]), (it / C::kTmemBufs) & 1, abort);
                    got = __all_sync(0xffffffffu, got);
                    if (!got) { ok = false; break; }
                    ptx::tc_fence_after();
                    s0 = sr * sb0;
                    s1 = sr * sb1;
                }
                const uint32_t tbase = tmem + tcol + (uint32_t)(b * BN);
                // 16-column TMEM loads, double-buffered: the load of the next 16 columns
                // is in flight while the current 16 are folded in
                uint32_t va[16], vb[16];
                ptx::tmem_ld_32x32b_x16(tbase, va);
#pragma unroll
                for (int c = 0; c < C::kCols; c += 32) {
                    ptx::tmem_wait_ld_regs(va);
                    ptx::tmem_ld_32x32b_x16(tbase + c + 16, vb);
                    const float sa_ = (c < C::kCols / 2) ? s0 : s1;
                    const float2 sa2 = make_float2(sa_, sa_);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc2[c / 2 + i] = __ffma2_rn(
                            sa2, make_float2(__uint_as_float(va[2 * i]), __uint_as_float(va[2 * i + 1])),
                            acc2[c / 2 + i]);
                    ptx::tmem_wait_ld_regs(vb);
                    if (c + 32 < C::kCols) ptx::tmem_ld_32x32b_x16(tbase + c + 32, va);
                    const float sb_ = (c + 16 < C::kCols / 2) ? s0 : s1;
                    const float2 sb2 = make_float2(sb_, sb_);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc2[c / 2 + 8 + i] = __ffma2_rn(
                            sb2, make_float2(__uint_as_float(vb[2 * i]), __uint_as_float(vb[2 * i + 1])),
                            acc2[c / 2 + 8 + i]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&st->tempty[b]));
            }
            if (!ok) {
                // a warp leaving mid-tile still counts in that tile's amax exchange, so
                // that no other epilogue warp can be left waiting at its barrier
                if constexpr (kSilu) asm volatile("bar.arrive 1, 256;" ::: "memory");
                break;
            }
            float* acc = reinterpret_cast<float*>(acc2);
            if (kSilu) {
                // acc[0:64) gate, acc[64:128) up of h columns nt*128 + wg*64 + [0, 64)
                const int N = n_out / 2;
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    acc[j] = silu_mul(acc[j], acc[64 + j]);
                    amax = fmaxf(amax, fabsf(acc[j]));
                }
                float* xa = s_amax + (tcount & 1) * 256;
                xa[wg * 128 + row_in_tile] = amax;
                // both warpgroups' row maxima: hardware barrier 1 over the 8 epilogue warps
                // (threads 0-255). Every epilogue warp reaches it once per tile, or has
                // arrived on it when it left the tile early.
                asm volatile("bar.sync 1, 256;" ::: "memory");
                amax = fmaxf(xa[row_in_tile], xa[128 + row_in_tile]);
                const float s = __fdiv_rn(amax, 448.0f);
                // code = e4m3(h / s) with the correctly rounded quotient; the branch is per
                // row (uniform over the loop), so only one division path is executed
                if (s == 0.f) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
                } else if (s >= 1e-30f) {
                    const float rs = __frcp_rn(s);
#pragma unroll
                    for (int j = 0; j < 64; ++j) acc[j] = div_rn_by(acc[j], s, rs);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) acc[j] = __fdiv_rn(acc[j], s);
                }
                uint32_t w[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    w[q] = uint32_t(f32x2_to_e4m3x2(acc[4 * q], acc[4 * q + 1])) |
                           (uint32_t(f32x2_to_e4m3x2(acc[4 * q + 2], acc[4 * q + 3])) << 16);
                const uint4 v4[4] = {make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]),
                                     make_uint4(w[8], w[9], w[10], w[11]), make_uint4(w[12], w[13], w[14], w[15])};
                store_box64(s_stage + warp * C::kStageWarpBytes, lane, v4, &tmO, nt * 128 + wg * 64, (int)(r - lane));
                if (wg == 0) out_scale[r * (N / 128) + nt] = s;
            } else if (EPI == MOE_EPI_F32) {
                // 16 fp32 columns (64 bytes) per round
#pragma unroll
                for (int q = 0; q < C::kCols / 16; ++q) {
                    uint4 v4[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        v4[c] = make_uint4(__float_as_uint(acc[16 * q + 4 * c]), __float_as_uint(acc[16 * q + 4 * c + 1]),
                                           __float_as_uint(acc[16 * q + 4 * c + 2]),
                                           __float_as_uint(acc[16 * q + 4 * c + 3]));
                    store_box64(s_stage + warp * C::kStageWarpBytes, lane, v4, &tmO, nt * BN + wg * C::kCols + q * 16,
                                (int)(r - lane));
                }
            } else {
                // the warp's 32 rows x kCols bf16 columns as 128-byte-wide boxes (64
                // columns each), written in TMA's 128-byte swizzle: 16-byte chunk c of row
                // r sits at r * 128 + ((c ^ (r % 8)) * 16), so every 8 lanes of a store
                // cover all 32 banks
                uint8_t* stg = s_stage + warp * C::kStageWarpBytes;
                if (lane == 0) ptx::bulk_wait_read0();  // the previous tile's stores have read it
                __syncwarp();
#pragma unroll
                for (int q = 0; q < C::kCols / 64; ++q) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {  // two round-to-nearest-even conversions per instruction
                            __nv_bfloat162 h2 =
                                __floats2bfloat162_rn(acc[64 * q + 8 * c + 2 * e], acc[64 * q + 8 * c + 2 * e + 1]);
                            w[e] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        *reinterpret_cast<uint4*>(stg + q * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int q = 0; q < C::kCols / 64; ++q)
                        ptx::tma_store_2d(&tmO, ptx::smem_addr(stg + q * 4096), nt * BN + wg * C::kCols + q * 64,
                                          (int)(r - lane));
                    ptx::bulk_commit();
                }
            }
        }
    }
    if (warp < kEpiWarps && lane == 0) ptx::bulk_wait0();  // this warp's output stores have completed
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D uint8 tensor [rows, inner] (row-major), boxes of box_rows x 128 bytes, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tensor [rows, cols] of `esize`-byte elements. Output map: bf16 in 32-row x 128-byte boxes with the 128-byte swizzle, fp8 and fp32
// in 32-row x 64-byte boxes with the 64-byte swizzle (the staging layouts above).
bool make_out_tmap(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, int esize) {
    auto fn = encode_fn();
    if (!fn) return false;
    const CUtensorMapDataType dt = esize == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (uint64_t)esize};
    const bool wide = esize == 2;
    const cuuint32_t box[2] = {(cuuint32_t)((wide ? 128 : kStageRowBytes) / esize), 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EPI, bool kSkip>
int launch_tc_k(const CUtensorMap& ta, const CUtensorMap& ta32, const CUtensorMap& ta64, const CUtensorMap& tb, const CUtensorMap& to,
                const float* a_scale,
                const float* w_scale, const int32_t* offsets, const int32_t* counts, int El, int64_t rp_cap,
                int n_out, int k_in, void* out, float* out_scale, int num_sms, cudaStream_t stream, int opts) {
    const size_t smem = smem_bytes<BN, EPI>(El);
    // the shared-memory opt-in is a property of the kernel in each device's context: set
    // it once per device (racing first calls only set the same value twice)
    static std::atomic<bool> attr_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI, kSkip>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes<BN, EPI>(kMaxLocalExperts)) != cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int n_tiles = EPI == MOE_EPI_SILU_MUL_QUANT ? n_out / 256 : n_out / BN;
    const int64_t max_tiles = rp_cap / kBM * n_tiles;
    const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
    if (grid < 1) return MOE_OK;
    launch_k(gemm_tc_kernel<BN, EPI, kSkip>, grid, threads_of<EPI>(), smem, stream, ta, ta32, ta64, tb, to, a_scale, w_scale,
             offsets, counts, El, (int)rp_cap, n_out, k_in, out, out_scale, opts);
    note_launches(1);
    return launch_status();
}

// Small batches (fewer than two 128-row blocks per local expert on average, so that most
// of each block is padding) run the kernel that skips all-padding row groups; large ones
// the kernel without that path, which leaves its registers to the full tiles.
template <int BN, int EPI>
int launch_tc(const CUtensorMap& ta, const CUtensorMap& ta32, const CUtensorMap& ta64, const CUtensorMap& tb, const CUtensorMap& to,
              const float* a_scale,
              const float* w_scale, const int32_t* offsets, const int32_t* counts, int El, int64_t rp_cap, int n_out,
              int k_in, void* out, float* out_scale, int num_sms, cudaStream_t stream, int opts) {
    if (counts && rp_cap < (int64_t)El * 2 * kBM)
        return launch_tc_k<BN, EPI, true>(ta, ta32, ta64, tb, to, a_scale, w_scale, offsets, counts, El, rp_cap, n_out, k_in, out,
                                          out_scale, num_sms, stream, opts);
    return launch_tc_k<BN, EPI, false>(ta, ta32, ta64, tb, to, a_scale, w_scale, offsets, counts, El, rp_cap, n_out, k_in, out,
                                       out_scale, num_sms, stream, opts);
}

}  // namespace

int launch_grouped_gemm(const uint8_t* a, const float* a_scale, const uint8_t* w, const float* w_scale,
                        const int32_t* expert_offsets, const int32_t* expert_counts, int El, int64_t rp_cap, int n_out,
                        int k_in, int epilogue,
                        void* out, float* out_scale, int num_sms, cudaStream_t stream, int opts) {
    if (rp_cap == 0) return MOE_OK;
    // 256-wide tiles, except for a bf16/fp32 output of a small batch whose 256-wide tiles
    // would fill fewer than four waves of the SMs (a 128-token chunk: ~3 waves, the last
    // mostly idle): twice as many 128-wide tiles balance the SMs better there
    const bool small = expert_counts && rp_cap < (int64_t)El * 2 * kBM;
    const bool few_tiles = rp_cap / kBM * (n_out / 256) < 4 * (int64_t)num_sms;
    const bool bn256 = n_out % 256 == 0 && !(small && few_tiles && epilogue != MOE_EPI_SILU_MUL_QUANT);
    CUtensorMap ta, ta32, ta64, tb, to;
    const int o_cols = epilogue == MOE_EPI_SILU_MUL_QUANT ? n_out / 2 : n_out;
    const int o_esize = epilogue == MOE_EPI_SILU_MUL_QUANT ? 1 : epilogue == MOE_EPI_F32 ? 4 : 2;
    if (!make_tmap(&ta, a, (uint64_t)k_in, (uint64_t)rp_cap, kBM) ||
        !make_tmap(&ta32, a, (uint64_t)k_in, (uint64_t)rp_cap, 32) ||
        !make_tmap(&ta64, a, (uint64_t)k_in, (uint64_t)rp_cap, 64) ||
        !make_tmap(&tb, w, (uint64_t)k_in, (uint64_t)El * n_out, kBoxRows) ||
        !make_out_tmap(&to, out, (uint64_t)o_cols, (uint64_t)rp_cap, o_esize))
        return MOE_ERR_CUDA;
    switch (epilogue) {
        case MOE_EPI_SILU_MUL_QUANT:
            return launch_tc<256, MOE_EPI_SILU_MUL_QUANT>(ta, ta32, ta64, tb, to, a_scale, w_scale, expert_offsets, expert_counts, El, rp_cap, n_out,
                                                          k_in, out, out_scale, num_sms, stream, opts);
        case MOE_EPI_F32:
            return bn256 ? launch_tc<256, MOE_EPI_F32>(ta, ta32, ta64, tb, to, a_scale, w_scale, expert_offsets, expert_counts, El, rp_cap, n_out,
                                                       k_in, out, out_scale, num_sms, stream, opts)
                         : launch_tc<128, MOE_EPI_F32>(ta, ta32, ta64, tb, to, a_scale, w_scale, expert_offsets, expert_counts, El, rp_cap, n_out,
                                                       k_in, out, out_scale, num_sms, stream, opts);
        default:
            return bn256 ? launch_tc<256, MOE_EPI_BF16>(ta, ta32, ta64, tb, to, a_scale, w_scale, expert_offsets, expert_counts, El, rp_cap, n_out,
                                                        k_in, out, out_scale, num_sms, stream, opts)
                         : launch_tc<128, MOE_EPI_BF16>(ta, ta32, ta64, tb, to, a_scale, w_scale, expert_offsets, expert_counts, El, rp_cap, n_out,
                                                        k_in, out, out_scale, num_sms, stream, opts);
    }
}

int read_gemm_error(int clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int z = 0;
        cudaMemcpyToSymbol(g_gemm_error, &z, sizeof(int));
    }
    return v;
}

}  // namespace moe
