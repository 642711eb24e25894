// Host-side launchers of the HBM-bound kernels (route.cu) and the grouped GEMM.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kScatterThreads = 256;   // 8 warps per CTA in the scatter index kernels
constexpr int kScatterMinSlots = 1024; // top-k slots per CTA at least (measured: 2048 and 512 were slower)
constexpr int kMaxScatterCtas = 256;   // at most this many CTAs rank the slots
constexpr int kMaxLocalExperts = 1024;

int scatter_slots_per_cta(int64_t n);

// TId: the top-k id type, int32_t or int64_t (both instantiated in route.cu).
template <typename TId>
int launch_count(const TId* ids, int64_t n, const int32_t* expert_map, int E, int El, int32_t* counts,
                 int32_t* err_count, int num_sms, cudaStream_t stream);

// counts_in NULL: the experts' slot counts are derived by the scatter's own histogram
// pass and written to counts_out (bad ids then added to err_count, if not NULL).
// rp_cap: rows of a_out / a_scale; expert_offsets never exceed it (rounded down to 128).
// early != 0: the kernels that can still be running before this call's first kernel are
// this library's kernels of an earlier chunk of the same call (its GEMMs and gather), none
// of which writes the call's inputs, so inputs may be read before waiting for them (small
// batches only; every write still waits).
template <typename TId>
int launch_scatter(const uint16_t* x, int64_t M, int K, const TId* ids, const float* topk_weights, int topk,
                   const int32_t* expert_map, int E, int El, const int32_t* counts_in, int32_t* counts_out,
                   int32_t* err_count, int apply_on_input, int quant, void* a_out, float* a_scale,
                   int32_t* expert_offsets, int32_t* src2dst, int64_t rp_cap, int32_t* hist, int early,
                   cudaStream_t stream);

// Whether launch_scatter runs as the single small-batch kernel for these sizes.
bool scatter_is_one_kernel(int64_t M, int topk, int El);

// early_trigger != 0: the next kernel may launch as soon as this one starts (the caller
// guarantees that it is a one-kernel scatter of the same call launched with early != 0).
int launch_gather(const uint16_t* y, const int32_t* src2dst, const float* topk_weights, int64_t M, int topk, int K,
                  int apply_on_input, uint16_t* out, cudaStream_t stream, int early_trigger = 0);

int launch_silu_mul_quant(const float* c1, const int32_t* expert_offsets, int El, int64_t rp_cap, int N, uint8_t* h,
                          float* h_scale, cudaStream_t stream);

// Options of launch_grouped_gemm (bits of opts):
//  kOptWeightsEvictFirst: the weight tiles are loaded with the L2 evict-first policy.
constexpr int kOptWeightsEvictFirst = 1;

// expert_counts (nullable): valid rows of each expert's block; rows past them are
// padding, and 32-row groups made only of padding are neither computed nor stored.
int launch_grouped_gemm(const uint8_t* a, const float* a_scale, const uint8_t* w, const float* w_scale,
                        const int32_t* expert_offsets, const int32_t* expert_counts, int El, int64_t rp_cap,
                        int n_out, int k_in, int epilogue, void* out, float* out_scale, int num_sms,
                        cudaStream_t stream, int opts = 0);

// moe_forward_chunked for either top-k id type (the argument checks included).
template <typename TId>
int forward_chunked_impl(const void* hidden_states, const TId* topk_ids, const float* topk_weights,
                         const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                         const int32_t* expert_map, int E, int local_num_experts, int64_t M, int K, int N, int topk,
                         int64_t chunk_size, int apply_router_weight_on_input, void* out, void* workspace,
                         size_t workspace_bytes, int32_t* err_count, cudaStream_t stream);

// Device error word of the grouped GEMM (1: a pipeline wait ran out of time). Reading
// it synchronises the device; `clear` resets it.
int read_gemm_error(int clear);

}  // namespace moe
