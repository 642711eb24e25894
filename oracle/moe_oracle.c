/*
 * moe_oracle.c -- plain, slow CPU oracle of the fused-MoE layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg and reference arm may load this file's library. It shares no code, header,
 * table or constant with the CUDA path, and the CUDA path never calls it.
 *
 * What is computed follows three vLLM pull-request pages:
 *   P1  vLLM PR #20903 "[Kernel] DeepGemm MoE : Integrate triton permute / unpermute
 *       kernels" (Purpose items 1-2; Optimizations: FP8 e4m3 with 128x128 blocks)
 *   P2  vLLM PR #20725 "[Misc] ModularKernel : Perform WeightAndReduce inside
 *       TritonExperts & DeepGemmExperts" (Purpose; Changes)
 *   P3  vLLM PR #20392 "[Bugfix] Fused MoE Modular Kernel chunking loop"
 *       (Purpose, Bug 1 and Bug 2; review diff of modular_kernel.py / utils.py)
 * The pages name the steps but print no arithmetic; where they are silent the reading
 * taken is written beside the step. Every function is a direct transcription of the
 * step's definition: no blocking, fusion or reordering beyond what is stated.
 *
 * Precision: fp32 wherever the method keeps fp32 (scales, C1, h, the top-k sum), fp64
 * for the GEMM dot products (the per-128 partial sums of fp8 x fp8 products are exact
 * in fp64), bf16 round-to-nearest-even where the layer stores bf16.
 * Build with -ffp-contract=off so that no multiply-add is fused.
 *
 * Built twice: single-threaded (the checker the tests use) and with -fopenmp (the CPU
 * baseline timed over all host cores). The OpenMP build only spreads the independent
 * permuted rows of the chunking loop over threads, each with its own scratch; every
 * row's arithmetic is the same code in the same order, so both builds give identical
 * results.
 */
#ifdef _OPENMP
#include <omp.h>
#endif
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GROUP 128 /* 1x128 activation groups, 128x128 weight blocks */

/* ---------------------------------------------------------------- number formats */

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even. */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* FP8 E4M3 ("fn") decode, from the format definition: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (2^-6 * m/8); S.1111.111 is
 * NaN; there is no infinity. Largest finite value 448 = 2^8 * 1.75. */
float oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* FP8 E4M3 encode: round to nearest, ties to even, saturating to +-448; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(float f) {
    if (isnan(f)) return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid: multiples of 2^-9; m == 8 is the smallest normal, code 0x08 */
        double m = rint(a * 512.0);
        return sign | (uint8_t)m;
    }
    int e;
    double fr = frexp(a, &e);         /* a = fr * 2^e, fr in [0.5, 1) */
    int ue = e - 1;                   /* a = (2 fr) * 2^ue, significand in [1, 2) */
    double m = rint((2.0 * fr - 1.0) * 8.0);
    if (m == 8.0) {
        m = 0.0;
        ue += 1;
    }
    int code = ((ue + 7) << 3) | (int)m;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

static float g_dec[256];
static int g_dec_ready = 0;
static float dec(uint8_t c) {
    if (!g_dec_ready) {
        for (int i = 0; i < 256; ++i) g_dec[i] = oracle_e4m3_decode((uint8_t)i);
        g_dec_ready = 1;
    }
    return g_dec[c];
}

/* One 1x128 group of activation quantisation: amax over the group in fp32,
 * scale = amax / 448 (fp32 IEEE division), code = e4m3(x / scale) with fp32 IEEE
 * division; a zero group gets scale 0 and codes +0. P1 "Optimizations" names
 * float8_e4m3fn with block shape 128; the amax/448 rule is the reading taken. */
void oracle_quant_group(const float* x, int n, uint8_t* q, float* scale) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) q[i] = (s == 0.0f) ? 0x00 : oracle_e4m3_encode(x[i] / s);
}

/* A row of K values (K a multiple of 128) -> K codes + K/128 scales. */
void oracle_quant_row(const float* x, int K, uint8_t* q, float* scales) {
    for (int g = 0; g < K / GROUP; ++g) oracle_quant_group(x + g * GROUP, GROUP, q + g * GROUP, scales + g);
}

/* ------------------------------------------------------------------ routing plumbing */

/* Local expert of one top-k slot (P3, review diff of modular_kernel.py:
 * slice_expert_num_tokens(c_topk_ids, local_num_experts, expert_map)). expert_map maps
 * a global id to a local id or -1 (expert not on this GPU); with no map, local = global.
 * A slot is kept when its local id is in [0, El). Id -1 marks an empty slot and is
 * dropped silently; any other id outside [0, E) is dropped and counted as bad. Ids are
 * taken as 64-bit integers (int32 ids widen exactly), so an int64 id beyond the int32
 * range is out of [0, E) like any other, never an alias of a small id. */
static int local_of(int64_t id, const int32_t* map, int E, int El, int64_t* bad) {
    if (id == -1) return -1;
    if (id < 0 || id >= E) {
        ++*bad;
        return -1;
    }
    int l = map ? map[id] : id;
    return (l >= 0 && l < El) ? l : -1;
}

/* Step a1, count_expert_num_tokens (P3 Purpose, Bug 2): the number of (token, k) slots
 * routed to each local expert. Returns the number of bad ids. */
int64_t oracle_count(const int64_t* topk_ids, int64_t M, int topk, const int32_t* expert_map, int E,
                     int El, int32_t* counts) {
    int64_t bad = 0;
    for (int l = 0; l < El; ++l) counts[l] = 0;
    for (int64_t i = 0; i < M * topk; ++i) {
        int l = local_of(topk_ids[i], expert_map, E, El, &bad);
        if (l >= 0) counts[l] += 1;
    }
    return bad;
}

/* Expert blocks start on 128-row boundaries: offsets[l] = sum over l' < l of
 * ceil128(counts[l']); offsets[El] is the padded row total Rp. */
void oracle_offsets(const int32_t* counts, int El, int32_t* offsets) {
    offsets[0] = 0;
    for (int l = 0; l < El; ++l) offsets[l + 1] = offsets[l] + (counts[l] + GROUP - 1) / GROUP * GROUP;
}

/* Workspace row bound with no device->host read: every non-empty expert pads at most
 * 127 rows, and at most min(El, Mc*topk) experts are non-empty. */
int64_t oracle_rp_cap(int64_t Mc, int topk, int El) {
    int64_t n = Mc * topk;
    int64_t ne = El < n ? El : n;
    return (n + ne * (GROUP - 1) + GROUP - 1) / GROUP * GROUP;
}

/* Step a2, ep_scatter / deepgemm_moe_permute (P1 Purpose item 2): every kept (t, k)
 * slot gets a row of the expert-contiguous buffer. Within expert l the rows are taken
 * in ascending flat index t*topk + k (a stable counting sort); the dropped slots get
 * src2dst = -1. The row is x_t, or bf16(x_t * w[t,k]) when the router weight is applied
 * on the input (P2 Changes, apply_router_weight_on_input). quant = 1: 1x128 FP8
 * codes + fp32 scales ([rows, K/128] row-major); quant = 0: a bf16 copy.
 * Padding rows are not written. Returns the number of bad ids. */
int64_t oracle_scatter(const uint16_t* x, int64_t M, int K, const int64_t* topk_ids,
                       const float* topk_weights, int topk, const int32_t* expert_map, int E, int El,
                       int apply_router_weight_on_input, int quant, void* a_out, float* a_scale,
                       int32_t* offsets, int32_t* src2dst) {
    int32_t* counts = (int32_t*)calloc((size_t)El, sizeof(int32_t));
    int64_t* cursor = (int64_t*)calloc((size_t)El, sizeof(int64_t));
    float* row = (float*)malloc((size_t)K * sizeof(float));
    int64_t bad = oracle_count(topk_ids, M, topk, expert_map, E, El, counts);
    oracle_offsets(counts, El, offsets);
    for (int l = 0; l < El; ++l) cursor[l] = offsets[l];
    int64_t dummy = 0;
    for (int64_t i = 0; i < M * topk; ++i) {
        int64_t t = i / topk;
        int l = local_of(topk_ids[i], expert_map, E, El, &dummy);
        if (l < 0) {
            src2dst[i] = -1;
            continue;
        }
        int64_t dst = cursor[l]++;
        src2dst[i] = (int32_t)dst;
        for (int c = 0; c < K; ++c) {
            float v = bf16_to_f32(x[t * K + c]);
            if (apply_router_weight_on_input) v = bf16_to_f32(f32_to_bf16(v * topk_weights[i]));
            row[c] = v;
        }
        if (quant) {
            oracle_quant_row(row, K, (uint8_t*)a_out + dst * K, a_scale + dst * (K / GROUP));
        } else {
            for (int c = 0; c < K; ++c) ((uint16_t*)a_out)[dst * K + c] = f32_to_bf16(row[c]);
        }
    }
    free(row);
    free(cursor);
    free(counts);
    return bad;
}

/* One output element of the block-scaled FP8 GEMM (steps a3/a5, the DeepGEMM grouped
 * GEMM of P1 "Optimizations", --block-shape 128 128):
 *   C[r, j] = sum_kb a_scale[r, kb] * w_scale[j/128, kb] * sum_{k in kb} A[r,k] W[j,k]
 * a: Kin codes of row r, sa: its Kin/128 scales; w: Kin codes of weight row j,
 * sw: the Kin/128 scales of weight block row j/128. */
static double block_dot(const uint8_t* a, const float* sa, const uint8_t* w, const float* sw, int Kin) {
    double acc = 0.0;
    for (int kb = 0; kb < Kin / GROUP; ++kb) {
        double part = 0.0;
        for (int k = kb * GROUP; k < (kb + 1) * GROUP; ++k) part += (double)dec(a[k]) * (double)dec(w[k]);
        acc += (double)sa[kb] * (double)sw[kb] * part;
    }
    return acc;
}

/* Steps a3/a5 over all kept rows: rows [offsets[l], offsets[l] + counts[l]) use
 * expert l's weights W [El, Nout, Kin] and scales [El, Nout/128, Kin/128].
 * C is [rows, Nout] fp64; padding rows are left as they are. */
void oracle_grouped_gemm(const uint8_t* A, const float* a_scale, const uint8_t* W, const float* w_scale,
                         const int32_t* offsets, const int32_t* counts, int El, int Nout, int Kin,
                         double* C) {
    int kb = Kin / GROUP;
    for (int l = 0; l < El; ++l)
        for (int64_t r = offsets[l]; r < (int64_t)offsets[l] + counts[l]; ++r)
            for (int j = 0; j < Nout; ++j) {
                const uint8_t* w = W + ((int64_t)l * Nout + j) * Kin;
                const float* sw = w_scale + ((int64_t)l * (Nout / GROUP) + j / GROUP) * kb;
                C[r * Nout + j] = block_dot(A + r * Kin, a_scale + r * kb, w, sw, Kin);
            }
}

/* SiLU-and-mul of one row of C1 (fp32 [2N]): the gate is C1[0:N), the up projection
 * C1[N:2N); h = silu(gate) * up with silu(g) = g / (1 + e^-g), evaluated in fp64 and
 * rounded to fp32. */
static void silu_mul_row(const float* c1, int N, float* h) {
    for (int j = 0; j < N; ++j) {
        double g = c1[j], u = c1[N + j];
        h[j] = (float)(g / (1.0 + exp(-g)) * u);
    }
}

/* Step a4 over all kept rows: C1 fp32 [rows, 2N] -> H codes [rows, N] + fp32 scales
 * [rows, N/128] by the 1x128 rule. */
void oracle_silu_mul_quant(const float* C1, const int32_t* offsets, const int32_t* counts, int El, int N,
                           uint8_t* H, float* h_scale) {
    float* h = (float*)malloc((size_t)N * sizeof(float));
    for (int l = 0; l < El; ++l)
        for (int64_t r = offsets[l]; r < (int64_t)offsets[l] + counts[l]; ++r) {
            silu_mul_row(C1 + r * 2 * N, N, h);
            oracle_quant_row(h, N, H + r * N, h_scale + r * (N / GROUP));
        }
    free(h);
}

/* Step a6, ep_gather / deepgemm_unpermute_and_reduce with the top-k weight-and-reduce
 * folded in (P1 Purpose item 2; P2 Purpose): out[t, c] = bf16(sum over kept k, in
 * ascending k, of w'[t,k] * Y[src2dst[t,k], c]) with an fp32 accumulator, w' = the
 * router weight, or 1 when it was applied on the input. A token with no kept slot gets
 * a zero row (this GPU's share of an expert-parallel sum). */
void oracle_gather(const uint16_t* Y, const int32_t* src2dst, const float* topk_weights, int64_t M, int topk,
                   int K, int apply_router_weight_on_input, uint16_t* out) {
    for (int64_t t = 0; t < M; ++t)
        for (int c = 0; c < K; ++c) {
            float acc = 0.0f;
            for (int k = 0; k < topk; ++k) {
                int32_t d = src2dst[t * topk + k];
                if (d < 0) continue;
                float w = apply_router_weight_on_input ? 1.0f : topk_weights[t * topk + k];
                float p = w * bf16_to_f32(Y[(int64_t)d * K + c]);
                acc = acc + p;
            }
            out[t * K + c] = f32_to_bf16(acc);
        }
}

/* Steps a3 -> a4 -> a5 for one permuted row r of expert l: GEMM1 (C1 rounded to
 * fp32), SiLU-and-mul, 1x128 requantisation, GEMM2, Y rounded to bf16. */
static void expert_row(const uint8_t* a, const float* sa, int l, const uint8_t* w13, const float* w13_scale,
                       const uint8_t* w2, const float* w2_scale, int K, int N, float* c1, float* h,
                       uint8_t* hq, float* hs, uint16_t* y) {
    int kbK = K / GROUP, kbN = N / GROUP;
    for (int j = 0; j < 2 * N; ++j) {
        const uint8_t* w = w13 + ((int64_t)l * 2 * N + j) * K;
        const float* sw = w13_scale + ((int64_t)l * (2 * N / GROUP) + j / GROUP) * kbK;
        c1[j] = (float)block_dot(a, sa, w, sw, K);
    }
    silu_mul_row(c1, N, h);
    oracle_quant_row(h, N, hq, hs);
    for (int c = 0; c < K; ++c) {
        const uint8_t* w = w2 + ((int64_t)l * K + c) * N;
        const float* sw = w2_scale + ((int64_t)l * (K / GROUP) + c / GROUP) * kbN;
        y[c] = f32_to_bf16((float)block_dot(hq, hs, w, sw, N));
    }
}

/* Step a7, the chunking loop (P3 Purpose, Bug 1 and Bug 2): tokens are taken in chunks
 * of chunk_size; for each chunk the expert counts, offsets and workspace are derived
 * from that chunk's own topk_ids and the chunk runs a1..a6 on its own rows. out is
 * bf16 [M, K]. Returns the number of bad ids, or -1 on bad arguments. */
int64_t oracle_forward_chunked(const uint16_t* x, const int64_t* topk_ids, const float* topk_weights,
                               const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                               const float* w2_scale, const int32_t* expert_map, int E, int El, int64_t M,
                               int K, int N, int topk, int64_t chunk_size, int apply_router_weight_on_input,
                               uint16_t* out) {
    if (chunk_size < 1 || K % GROUP || N % GROUP || topk < 1) return -1;
    int64_t bad = 0;
    int64_t cmax = chunk_size < M ? chunk_size : M;
    int64_t rp_cap = oracle_rp_cap(cmax, topk, El);
    uint8_t* A = (uint8_t*)malloc((size_t)rp_cap * K);
    float* sa = (float*)malloc((size_t)rp_cap * (K / GROUP) * sizeof(float));
    uint16_t* Y = (uint16_t*)malloc((size_t)rp_cap * K * sizeof(uint16_t));
    int32_t* offsets = (int32_t*)malloc((size_t)(El + 1) * sizeof(int32_t));
    int32_t* counts = (int32_t*)malloc((size_t)El * sizeof(int32_t));
    int32_t* src2dst = (int32_t*)malloc((size_t)cmax * topk * sizeof(int32_t));
    int64_t* kept_row = (int64_t*)malloc((size_t)cmax * topk * sizeof(int64_t));
    int* kept_expert = (int*)malloc((size_t)cmax * topk * sizeof(int));
    for (int64_t c0 = 0; c0 < M; c0 += chunk_size) {
        int64_t Mc = (M - c0) < chunk_size ? (M - c0) : chunk_size;
        bad += oracle_scatter(x + c0 * K, Mc, K, topk_ids + c0 * topk, topk_weights + c0 * topk, topk,
                              expert_map, E, El, apply_router_weight_on_input, 1, A, sa, offsets, src2dst);
        oracle_count(topk_ids + c0 * topk, Mc, topk, expert_map, E, El, counts);
        /* the kept rows; rows [offsets[l] + counts[l], offsets[l + 1]) are padding and never read */
        int64_t nk = 0;
        for (int l = 0; l < El; ++l)
            for (int64_t r = offsets[l]; r < (int64_t)offsets[l] + counts[l]; ++r) {
                kept_row[nk] = r;
                kept_expert[nk++] = l;
            }
#ifdef _OPENMP
#pragma omp parallel
#endif
        {
            float* c1 = (float*)malloc((size_t)2 * N * sizeof(float));
            float* h = (float*)malloc((size_t)N * sizeof(float));
            uint8_t* hq = (uint8_t*)malloc((size_t)N);
            float* hs = (float*)malloc((size_t)(N / GROUP) * sizeof(float));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t i = 0; i < nk; ++i) {
                const int64_t r = kept_row[i];
                expert_row(A + r * K, sa + r * (K / GROUP), kept_expert[i], w13, w13_scale, w2, w2_scale, K, N, c1,
                           h, hq, hs, Y + r * K);
            }
            free(hs);
            free(hq);
            free(h);
            free(c1);
        }
        oracle_gather(Y, src2dst, topk_weights + c0 * topk, Mc, topk, K, apply_router_weight_on_input,
                      out + c0 * K);
    }
    free(kept_expert);
    free(kept_row);
    free(src2dst);
    free(counts);
    free(offsets);
    free(Y);
    free(sa);
    free(A);
    return bad;
}

/* The same layer output for one token t, evaluated directly from the definition with no
 * permutation at all: for each kept slot k, quantise the (weighted) input row, run the
 * expert, and accumulate w' * y in ascending k. out_row is bf16 [K]. */
void oracle_forward_token(int64_t t, const uint16_t* x, const int64_t* topk_ids, const float* topk_weights,
                          const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                          const int32_t* expert_map, int E, int El, int K, int N, int topk,
                          int apply_router_weight_on_input, uint16_t* out_row) {
    float* row = (float*)malloc((size_t)K * sizeof(float));
    uint8_t* a = (uint8_t*)malloc((size_t)K);
    float* sa = (float*)malloc((size_t)(K / GROUP) * sizeof(float));
    float* c1 = (float*)malloc((size_t)2 * N * sizeof(float));
    float* h = (float*)malloc((size_t)N * sizeof(float));
    uint8_t* hq = (uint8_t*)malloc((size_t)N);
    float* hs = (float*)malloc((size_t)(N / GROUP) * sizeof(float));
    uint16_t* y = (uint16_t*)malloc((size_t)K * sizeof(uint16_t));
    float* acc = (float*)calloc((size_t)K, sizeof(float));
    int64_t bad = 0;
    for (int k = 0; k < topk; ++k) {
        int l = local_of(topk_ids[t * topk + k], expert_map, E, El, &bad);
        if (l < 0) continue;
        float w = topk_weights[t * topk + k];
        for (int c = 0; c < K; ++c) {
            float v = bf16_to_f32(x[t * K + c]);
            row[c] = apply_router_weight_on_input ? bf16_to_f32(f32_to_bf16(v * w)) : v;
        }
        oracle_quant_row(row, K, a, sa);
        expert_row(a, sa, l, w13, w13_scale, w2, w2_scale, K, N, c1, h, hq, hs, y);
        float wk = apply_router_weight_on_input ? 1.0f : w;
        for (int c = 0; c < K; ++c) {
            float p = wk * bf16_to_f32(y[c]);
            acc[c] = acc[c] + p;
        }
    }
    for (int c = 0; c < K; ++c) out_row[c] = f32_to_bf16(acc[c]);
    free(acc);
    free(y);
    free(hs);
    free(hq);
    free(h);
    free(c1);
    free(sa);
    free(a);
    free(row);
}

/* Threads the OpenMP build runs the row loop on (1 in the single-threaded build). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Expert-parallel combine (P1 Purpose: DeepEP high-throughput prepare/finalize with
 * expert parallelism; reading C10: a rank's layer output is its share of each token's
 * top-k sum). The full output is the sum of the n_parts shares (bf16 [M, K] each):
 * fp32 accumulation in ascending part order, one rounding to bf16. */
void oracle_ep_combine(const uint16_t* const* parts, int n_parts, int64_t M, int K, uint16_t* out) {
    for (int64_t i = 0; i < M * K; ++i) {
        float acc = 0.0f;
        for (int r = 0; r < n_parts; ++r) acc = acc + bf16_to_f32(parts[r][i]);
        out[i] = f32_to_bf16(acc);
    }
}
