"""GPU parity of the grouped FP8 GEMM and of the whole chunked layer against the CPU
oracle, through the C ABI, from tiny cases to the full-size workloads the benchmark
times (sampled tokens there)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
import oracle
from helpers import dev, host, host_bits, layer_tolerance, e4m3_ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def permuted_inputs(counts, K, seed):
    """Random FP8 activations laid out in 128-aligned expert blocks (padding rows hold
    random codes too: they must not disturb the kept rows)."""
    rng = np.random.default_rng(seed)
    counts = np.array(counts, np.int32)
    offs = oracle.offsets(counts)
    R = int(offs[-1])
    x = (rng.standard_normal((max(R, 1), K)) * rng.uniform(0.05, 8, (max(R, 1), 1))).astype(np.float32)
    A, SA = oracle.quant_rows(x)
    return counts, offs, A[:R], SA[:R]


def kept_rows(offs, counts):
    return np.concatenate([np.arange(offs[l], offs[l] + counts[l]) for l in range(len(counts))] + [np.zeros(0, int)])


@pytest.mark.parametrize("counts,n_out,k_in", [([5, 0, 130], 256, 384), ([128], 128, 128),
                                               ([1, 300, 17, 0, 0, 64], 512, 768), ([200] * 3, 2048, 768)])
@pytest.mark.parametrize("epi", [moe.MOE_EPI_F32, moe.MOE_EPI_BF16])
def test_grouped_gemm_matches_oracle(counts, n_out, k_in, epi):
    counts, offs, A, SA = permuted_inputs(counts, k_in, seed=n_out + k_in)
    El = len(counts)
    W, S = mi.expert_weights(El, n_out, k_in, seed=7, stream=1)
    S = S * np.random.default_rng(3).uniform(0.5, 2.0, S.shape).astype(np.float32)
    out = moe.moe_grouped_gemm_fp8(dev(A), dev(SA), dev(W), dev(S), dev(offs), epi)
    torch.cuda.synchronize()
    C = oracle.grouped_gemm(A, SA, W, S, offs, counts)
    rows = kept_rows(offs, counts)
    ref = C[rows]
    got = host(out)[rows] if epi == moe.MOE_EPI_F32 else mi.bf16_to_f32(host_bits(out)[rows]).astype(np.float64)
    tol = 1e-5 if epi == moe.MOE_EPI_F32 else 8e-3
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= tol * np.abs(ref).max(), err.max() / np.abs(ref).max()


@pytest.mark.parametrize("counts,N,K", [([5, 0, 130], 256, 384), ([1, 300, 17, 0, 64], 768, 2048)])
def test_grouped_gemm_silu_epilogue(counts, N, K):
    """GEMM1 with the fused SiLU-and-mul + FP8 requant epilogue: equal, bit for bit, to the
    fp32-output GEMM followed by the standalone SiLU-mul-quant kernel, and within one e4m3
    step of the oracle (fp64 GEMM, fp64 SiLU)."""
    counts, offs, A, SA = permuted_inputs(counts, K, seed=N)
    El = len(counts)
    W, S = mi.expert_weights(El, 2 * N, K, seed=11, stream=1)
    h, hs = moe.moe_grouped_gemm_fp8(dev(A), dev(SA), dev(W), dev(S), dev(offs), moe.MOE_EPI_SILU_MUL_QUANT)
    c1 = moe.moe_grouped_gemm_fp8(dev(A), dev(SA), dev(W), dev(S), dev(offs), moe.MOE_EPI_F32)
    h2, hs2 = moe.moe_silu_mul_quant(c1, dev(offs))
    torch.cuda.synchronize()
    rows = kept_rows(offs, counts)
    assert (host(h)[rows] == host(h2)[rows]).all()
    assert (host(hs)[rows].view(np.uint32) == host(hs2)[rows].view(np.uint32)).all()
    C1 = oracle.grouped_gemm(A, SA, W, S, offs, counts).astype(np.float32)
    Href, hsref = oracle.silu_mul_quant(C1, offs, counts)
    np.testing.assert_allclose(host(hs)[rows], hsref[rows], rtol=2e-5, atol=0)
    d = e4m3_ulp_diff(host(h)[rows], Href[rows])
    assert d.max() <= 1 and (d == 0).mean() >= 0.99


@pytest.mark.parametrize("epi", [moe.MOE_EPI_SILU_MUL_QUANT, moe.MOE_EPI_BF16, moe.MOE_EPI_F32])
def test_grouped_gemm_with_counts_skips_padding(epi):
    """With expert_num_tokens the kept rows are bit-identical to the run without it, and
    aligned 32-row groups of pure padding are left untouched (their sentinel survives)."""
    counts = [1, 33, 0, 64, 100, 130]
    K, n_out = 384, 512
    counts, offs, A, SA = permuted_inputs(counts, K, seed=5)
    El = len(counts)
    W, S = mi.expert_weights(El, n_out, K, seed=8, stream=1)
    a, sa, w, s, o = dev(A), dev(SA), dev(W), dev(S), dev(offs)
    full = moe.moe_grouped_gemm_fp8(a, sa, w, s, o, epi)
    torch.cuda.synchronize()
    R = A.shape[0]
    cols = n_out // 2 if epi == moe.MOE_EPI_SILU_MUL_QUANT else n_out
    dt = {moe.MOE_EPI_SILU_MUL_QUANT: torch.uint8, moe.MOE_EPI_BF16: torch.bfloat16, moe.MOE_EPI_F32: torch.float32}
    out = torch.full((R, cols), 7, dtype=dt[epi], device="cuda")
    osc = torch.full((R, n_out // 256), -1.0, device="cuda") if epi == moe.MOE_EPI_SILU_MUL_QUANT else None
    got = moe.moe_grouped_gemm_fp8(a, sa, w, s, o, epi, out=out, out_scale=osc, expert_num_tokens=dev(counts))
    torch.cuda.synchronize()
    rows = kept_rows(offs, counts)
    g, f = (got[0], full[0]) if epi == moe.MOE_EPI_SILU_MUL_QUANT else (got, full)
    assert torch.equal(g[rows].view(torch.uint8), f[rows].view(torch.uint8))
    if epi == moe.MOE_EPI_SILU_MUL_QUANT:
        assert torch.equal(got[1][rows], full[1][rows])
    # rows of 32-row groups that hold no kept row keep the sentinel
    idle = [r for l in range(El) for r in range(int(offs[l]), int(offs[l + 1]))
            if (r - int(offs[l])) // 32 * 32 >= counts[l]]
    assert idle, "the case must have idle groups"
    assert bool((g[idle] == 7).all())
    if epi == moe.MOE_EPI_SILU_MUL_QUANT:
        assert bool((got[1][idle] == -1).all())


@pytest.mark.parametrize("epi", [moe.MOE_EPI_BF16, moe.MOE_EPI_SILU_MUL_QUANT])
def test_grouped_gemm_masked_batched_layout(epi):
    """The batched ("masked") expert layout [El, max_tokens, K] that low-latency
    expert-parallel dispatch produces: expert l owns rows [l * max_tokens, (l+1) *
    max_tokens) and only its first mask[l] rows hold tokens. It is the grouped GEMM with
    expert_offsets = l * max_tokens and expert_num_tokens = mask."""
    El, max_tokens, K = 8, 256, 384
    n_out = 512
    rng = np.random.default_rng(11)
    mask = rng.integers(0, max_tokens + 1, El).astype(np.int32)
    mask[2], mask[5] = 0, max_tokens
    offs = (np.arange(El + 1) * max_tokens).astype(np.int32)
    x = (rng.standard_normal((El * max_tokens, K)) * rng.uniform(0.05, 8, (El * max_tokens, 1))).astype(np.float32)
    A, SA = oracle.quant_rows(x)
    W, S = mi.expert_weights(El, n_out, K, seed=12, stream=1)
    out = moe.moe_grouped_gemm_fp8(dev(A), dev(SA), dev(W), dev(S), dev(offs), epi, expert_num_tokens=dev(mask))
    torch.cuda.synchronize()
    rows = kept_rows(offs, mask)
    C = oracle.grouped_gemm(A, SA, W, S, offs, mask)
    if epi == moe.MOE_EPI_BF16:
        got = mi.bf16_to_f32(host_bits(out)[rows]).astype(np.float64)
        ref = C[rows]
        assert np.abs(got - ref).max() <= 8e-3 * np.abs(ref).max()
    else:
        counts = mask
        Href, hsref = oracle.silu_mul_quant(C.astype(np.float32), offs, counts)
        hs = host(out[1])[rows]
        np.testing.assert_allclose(hs, hsref[rows], rtol=2e-5, atol=0)
        d = e4m3_ulp_diff(host(out[0])[rows], Href[rows])
        assert d.max() <= 1 and (d == 0).mean() >= 0.99


def test_device_error_word_is_clear():
    assert moe.moe_device_error() == 0


def test_grouped_gemm_identity_weights_bit_exact():
    """W = block-diagonal 1.0, scale 1: each output is a single product, no summation
    order freedom, so the fp32 results equal the oracle's exactly."""
    K = 256
    counts, offs, A, SA = permuted_inputs([5, 0, 130], K, seed=1)
    El = 3
    W = np.zeros((El, K, K), np.uint8)
    for l in range(El):
        np.fill_diagonal(W[l], 0x38)
    S = np.ones((El, 2, 2), np.float32)
    out = moe.moe_grouped_gemm_fp8(dev(A), dev(SA), dev(W), dev(S), dev(offs), moe.MOE_EPI_F32)
    torch.cuda.synchronize()
    C = oracle.grouped_gemm(A, SA, W, S, offs, counts).astype(np.float32)
    rows = kept_rows(offs, counts)
    assert (host(out)[rows].view(np.uint32) == C[rows].view(np.uint32)).all()


def to_dev_layer(li):
    return dict(x=dev(li.x), ids=dev(li.topk_ids), w=dev(li.topk_weights), w13=dev(li.w13),
                s13=dev(li.w13_scale), w2=dev(li.w2), s2=dev(li.w2_scale),
                m=None if li.expert_map is None else dev(li.expert_map))


def gpu_forward(d, E, chunk=None, apply_on_input=False):
    out = moe.moe_forward_chunked(d["x"], d["ids"], d["w"], d["w13"], d["s13"], d["w2"], d["s2"], E,
                                  expert_map=d["m"], chunk_size=chunk, apply_router_weight_on_input=apply_on_input)
    torch.cuda.synchronize()
    return host_bits(out)


def oracle_forward(li, chunk=None, apply_on_input=False):
    return oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2, li.w2_scale,
                                  li.wl.E, expert_map=li.expert_map, chunk_size=chunk,
                                  apply_router_weight_on_input=apply_on_input)


@pytest.fixture(scope="module")
def tiny():
    li = mi.make_layer_inputs(mi.TINY)
    return li, to_dev_layer(li)


@pytest.mark.parametrize("apply_on_input", [False, True])
def test_tiny_layer(tiny, apply_on_input):
    li, d = tiny
    got = gpu_forward(d, li.wl.E, apply_on_input=apply_on_input)
    ref = oracle_forward(li, apply_on_input=apply_on_input)
    layer_tolerance(got, ref)


def test_tiny_layer_chunk_sizes_bit_identical(tiny):
    li, d = tiny
    full = gpu_forward(d, li.wl.E)
    for chunk in (1, 7, 63, 64, 1000):
        assert (gpu_forward(d, li.wl.E, chunk=chunk) == full).all(), chunk


def test_layer_in_place_equals_separate_output():
    """out may be hidden_states itself: every chunk reads only its own rows before its
    gather writes them, also while the next chunk's scatter reads ahead. Several chunks of
    the one-kernel scatter (128-token chunks) and of the three-kernel one (1024)."""
    wl = mi.QWEN3_DECODE
    for M, chunk in ((1000, 128), (3000, 1024)):
        ids, tw = mi.route(M, wl.E, wl.topk, 41, 1.2)
        x = mi.hidden_states(M, wl.K, 41)
        li = mi.make_layer_inputs(wl)
        w = (dev(li.w13), dev(li.w13_scale), dev(li.w2), dev(li.w2_scale))
        d_ids, d_tw = dev(ids), dev(tw)
        ref = moe.moe_forward_chunked(dev(x), d_ids, d_tw, *w, wl.E, chunk_size=chunk)
        xin = dev(x)
        got = moe.moe_forward_chunked(xin, d_ids, d_tw, *w, wl.E, chunk_size=chunk, out=xin)
        torch.cuda.synchronize()
        assert got.data_ptr() == xin.data_ptr()
        assert (host_bits(got) == host_bits(ref)).all(), (M, chunk)


def test_layer_chunk_sizes_mix_scatter_forms_bit_identical():
    """Chunk sizes whose chunks take different scatter forms give the same output bit for
    bit: one chunk of 8800 slots (three-kernel scatter), chunks of 600 tokens (three-kernel,
    then a last chunk of 500 tokens = 4000 slots in the one-kernel form), chunks of 512
    (4096 slots, the one-kernel form's limit) and of 100 (one-kernel, the gather of each
    chunk launching the next chunk's scatter early)."""
    wl = mi.QWEN3_DECODE
    M = 1100
    ids, tw = mi.route(M, wl.E, wl.topk, 77, 1.2)
    x = dev(mi.hidden_states(M, wl.K, 77))
    li = mi.make_layer_inputs(wl)
    w = (dev(li.w13), dev(li.w13_scale), dev(li.w2), dev(li.w2_scale))
    d_ids, d_tw = dev(ids), dev(tw)
    outs = {}
    for chunk in (None, 600, 512, 100):
        out = moe.moe_forward_chunked(x, d_ids, d_tw, *w, wl.E, chunk_size=chunk)
        torch.cuda.synchronize()
        outs[chunk] = host_bits(out)
    for chunk in (600, 512, 100):
        assert (outs[chunk] == outs[None]).all(), chunk
    toks = np.array([0, 1, 599, 600, 1023, 1099])
    ref = oracle.forward_tokens(toks, mi.hidden_states(M, wl.K, 77), ids, tw, li.w13, li.w13_scale, li.w2,
                                li.w2_scale, wl.E)
    layer_tolerance(outs[None][toks], ref)


def test_tiny_layer_local_experts(tiny):
    li, d = tiny
    E = li.wl.E
    m = mi.random_expert_map(E, 3, seed=5)
    sel = np.nonzero(m >= 0)[0]
    d2 = dict(d, m=dev(m), w13=dev(li.w13[sel]), s13=dev(li.w13_scale[sel]), w2=dev(li.w2[sel]),
              s2=dev(li.w2_scale[sel]))
    got = gpu_forward(d2, E, chunk=10)
    ref = oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13[sel], li.w13_scale[sel], li.w2[sel],
                                 li.w2_scale[sel], E, expert_map=m, chunk_size=10)
    layer_tolerance(got, ref)
    # tokens with no local expert give zero rows
    none_local = ~(m[li.topk_ids] >= 0).any(axis=1)
    assert (mi.bf16_to_f32(got[none_local]) == 0).all()


def test_layer_no_local_expert_is_zero(tiny):
    li, d = tiny
    E = li.wl.E
    m = np.full(E, -1, np.int32)
    d2 = dict(d, m=dev(m))
    got = gpu_forward(d2, E)
    assert (mi.bf16_to_f32(got) == 0).all()


@pytest.mark.parametrize("E,topk,local,chunk", [(1024, 8, None, None),   # the most local experts the ABI takes
                                               (64, 1, None, 77),       # top-1, ragged chunks
                                               (64, 32, 48, None),      # the widest top-k, a local subset
                                               (1, 1, None, None)])     # a single expert
def test_layer_interface_extremes(E, topk, local, chunk):
    """The layer at the ends of its argument ranges, against the oracle."""
    wl = mi.Workload(f"extreme_e{E}_top{topk}", M=300, K=256, N=256, E=E, topk=topk, seed=E + topk,
                     zipf_s=1.2, local_experts=local, chunk_size=chunk)
    li = mi.make_layer_inputs(wl)
    got = gpu_forward(to_dev_layer(li), E, chunk=chunk)
    ref = oracle_forward(li, chunk=chunk)
    layer_tolerance(got, ref)


@pytest.mark.parametrize("K,N,E,topk,M", [(7168, 256, 8, 2, 40),    # a wide hidden size: 56 K blocks in GEMM1
                                           (512, 2048, 4, 2, 40),     # a wide expert: 16 K blocks in GEMM2
                                           (4096, 1408, 6, 2, 30)])   # 2N = 2816: an odd count of 256-wide tiles
def test_layer_other_model_shapes(K, N, E, topk, M):
    """Hidden and expert sizes of other MoE models (long K loops wrap the pipeline's
    stage and TMEM-buffer phases many times per tile), against the oracle."""
    wl = mi.Workload(f"shape_k{K}_n{N}", M=M, K=K, N=N, E=E, topk=topk, seed=K + N, zipf_s=1.2)
    li = mi.make_layer_inputs(wl)
    got = gpu_forward(to_dev_layer(li), E)
    ref = oracle_forward(li)
    layer_tolerance(got, ref)


def random_layer_case(seed):
    """A seeded random layer configuration: sizes, expert count, top-k, a random local
    expert map (or none), chunking, routing skew and where the router weight applies."""
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([1, 3, 16, 64, 200]))
    topk = int(rng.integers(1, min(E, 8) + 1))
    wl = mi.Workload(f"random_{seed}", M=int(rng.integers(1, 700)), K=int(rng.choice([128, 256, 384])),
                     N=int(rng.choice([128, 256, 384])), E=E, topk=topk, seed=2000 + seed,
                     zipf_s=float(rng.choice([0.0, 1.2])),
                     chunk_size=int(rng.choice([0, 1, 33, 128, 256])) or None,
                     apply_router_weight_on_input=bool(rng.integers(0, 2)) and topk == 1)
    li = mi.make_layer_inputs(wl)
    if E > 1 and rng.integers(0, 2):
        local = int(rng.integers(1, E + 1))
        li.expert_map = mi.random_expert_map(E, local, seed=3000 + seed)
        li.w13, li.w13_scale = mi.expert_weights(local, 2 * wl.N, wl.K, wl.seed, 13)
        li.w2, li.w2_scale = mi.expert_weights(local, wl.K, wl.N, wl.seed, 2)
    return li


@pytest.mark.parametrize("seed", range(12))
def test_layer_random_configurations(seed):
    li = random_layer_case(seed)
    wl = li.wl
    apply = wl.apply_router_weight_on_input
    got = gpu_forward(to_dev_layer(li), wl.E, chunk=wl.chunk_size, apply_on_input=apply)
    ref = oracle_forward(li, chunk=wl.chunk_size, apply_on_input=apply)
    layer_tolerance(got, ref)


@pytest.fixture(scope="module")
def decode():
    li = mi.make_layer_inputs(mi.QWEN3_DECODE)
    return li, to_dev_layer(li)


def test_qwen3_decode_layer(decode):
    li, d = decode
    got = gpu_forward(d, li.wl.E)
    ref = oracle_forward(li)
    layer_tolerance(got, ref)


def sampled_tokens(M, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, n, replace=False)]))


def check_full_size(li, chunk, n_samples):
    """The benchmark's launch configuration at full size: routing/permutation/FP8
    activations bit-exact over the first chunk, layer output on sampled tokens."""
    wl = li.wl
    d = to_dev_layer(li)
    got = gpu_forward(d, wl.E, chunk=chunk)
    assert np.isfinite(mi.bf16_to_f32(got)).all()
    toks = sampled_tokens(wl.M, n_samples, wl.seed)
    ref = oracle.forward_tokens(toks, li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2,
                                li.w2_scale, wl.E, expert_map=li.expert_map)
    layer_tolerance(got[toks], ref)
    # first chunk: counts, offsets, src2dst and FP8 activations vs the oracle
    Mc = min(chunk or wl.M, wl.M)
    El = wl.El
    ids = d["ids"][:Mc].contiguous()
    counts = moe.moe_count_expert_tokens(ids, wl.E, El, d["m"])
    a, sa, offs, s2d = moe.moe_scatter(d["x"][:Mc].contiguous(), ids, d["w"][:Mc].contiguous(), wl.E, El, counts,
                                       d["m"])
    torch.cuda.synchronize()
    r = oracle.scatter(li.x[:Mc], li.topk_ids[:Mc], li.topk_weights[:Mc], wl.E, El, li.expert_map)
    assert (host(counts) == r["counts"]).all()
    assert (host(offs) == r["offsets"]).all()
    assert (host(s2d) == r["src2dst"]).all()
    rows = r["src2dst"].reshape(-1)
    rows = rows[rows >= 0]
    assert (host(a)[rows] == r["a"][rows]).all()
    assert (host(sa)[rows].view(np.uint32) == r["a_scale"][rows].view(np.uint32)).all()
    # the last chunk (possibly a single token) through the chunk loop equals a standalone call
    c0 = (wl.M - 1) // chunk * chunk if chunk else 0
    tail = dict(d, x=d["x"][c0:].contiguous(), ids=d["ids"][c0:].contiguous(), w=d["w"][c0:].contiguous())
    assert (gpu_forward(tail, wl.E, chunk=chunk) == got[c0:]).all()


@pytest.mark.slow
def test_qwen3_prefill_full_size():
    check_full_size(mi.make_layer_inputs(mi.QWEN3_PREFILL), None, 24)


@pytest.mark.slow
def test_qwen3_chunked_local_full_size():
    check_full_size(mi.make_layer_inputs(mi.QWEN3_CHUNKED), 128, 24)
