"""Parity at the prefill workload's full size (8192 tokens, hidden 2048, moe intermediate
768, 128 experts, top-8, Zipf-1.2 routing), in the launch configuration the benchmark
times:

* both grouped GEMMs against the fp64 oracle on every column of a row sample that holds
  the first and the last kept row of every expert block and one kept row of every
  128-row tile (so every tile of every persistent CTA's loop, its last one included, is
  checked). The activations come from the oracle's own scatter, the GEMM2 input from
  the oracle's quantiser: nothing the oracle reads comes from the CUDA path;
* the fused SiLU-and-mul epilogue equals the fp32 GEMM followed by the standalone
  SiLU-and-mul kernel, bit for bit, over every kept row;
* the layer with the router weight applied on the input (vLLM PR #20725, "Changes")
  on sampled tokens against the per-token oracle.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
import oracle
from helpers import dev, e4m3_ulp_diff, host, host_bits, layer_tolerance

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WL = mi.QWEN3_PREFILL


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def prefill():
    li = mi.make_layer_inputs(WL)
    r = oracle.scatter(li.x, li.topk_ids, li.topk_weights, WL.E, WL.El)
    return li, r


def sample_rows(offs, counts, seed):
    """First and last kept row of every expert, and one random kept row of every 128-row
    tile that holds any."""
    rng = np.random.default_rng(seed)
    rows = set()
    for l in range(len(counts)):
        if counts[l]:
            rows.update((int(offs[l]), int(offs[l] + counts[l] - 1)))
    for mt in range(int(offs[-1]) // 128):
        r0 = mt * 128
        l = int(np.searchsorted(offs, r0, side="right") - 1)
        end = min(r0 + 128, int(offs[l] + counts[l]))
        if end > r0:
            rows.add(int(rng.integers(r0, end)))
    return np.array(sorted(rows), np.int64)


def oracle_rows(A, SA, W, S, offs, counts, rows):
    """The oracle's grouped GEMM on the given rows only (fp64 [len(rows), n_out])."""
    out = np.zeros((len(rows), W.shape[1]), np.float64)
    le = np.searchsorted(offs, rows, side="right") - 1
    for l in np.unique(le):
        sel = np.nonzero(le == l)[0]
        rr = rows[sel]
        n = len(rr)
        out[sel] = oracle.grouped_gemm(A[rr], SA[rr], W[l:l + 1], S[l:l + 1], np.array([0, n], np.int32),
                                       np.array([n], np.int32))
    return out


def padded(a, cap, fill_seed):
    """a [R, C] placed in a [cap, C] buffer whose padding rows hold random bytes."""
    buf = np.random.default_rng(fill_seed).integers(0, 256, (cap,) + a.shape[1:], dtype=np.uint8)
    if a.dtype != np.uint8:
        buf = np.random.default_rng(fill_seed).uniform(0.5, 2.0, (cap,) + a.shape[1:]).astype(a.dtype)
    buf[:a.shape[0]] = a
    return buf


def test_gemm1_full_size_every_tile(prefill):
    li, r = prefill
    counts, offs = r["counts"], r["offsets"]
    cap = moe.moe_rp_cap(WL.M, WL.topk, WL.El)
    A = dev(padded(r["a"], cap, 1))
    SA = dev(padded(r["a_scale"], cap, 2))
    W, S = dev(li.w13), dev(li.w13_scale)
    d_offs, d_cnt = dev(offs), dev(counts)
    c1 = moe.moe_grouped_gemm_fp8(A, SA, W, S, d_offs, moe.MOE_EPI_F32, expert_num_tokens=d_cnt)
    H, HS = moe.moe_grouped_gemm_fp8(A, SA, W, S, d_offs, moe.MOE_EPI_SILU_MUL_QUANT, expert_num_tokens=d_cnt)
    h2, hs2 = moe.moe_silu_mul_quant(c1, d_offs)
    torch.cuda.synchronize()
    rows = sample_rows(offs, counts, seed=11)
    assert len(rows) > 500
    ref = oracle_rows(r["a"], r["a_scale"], li.w13, li.w13_scale, offs, counts, rows)
    got = host(c1)[rows].astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= 1e-5 * np.abs(ref).max(), err.max() / np.abs(ref).max()
    # per row too: no row may be far off relative to its own magnitude
    row_err = err.max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)
    assert row_err.max() <= 1e-4, (rows[row_err.argmax()], row_err.max())
    # the fused epilogue is the fp32 GEMM + standalone SiLU-and-mul, bit for bit, on every kept row
    kept = np.concatenate([np.arange(offs[l], offs[l] + counts[l]) for l in range(WL.El)])
    assert (host(H)[kept] == host(h2)[kept]).all()
    assert (host(HS)[kept].view(np.uint32) == host(hs2)[kept].view(np.uint32)).all()
    # and against the oracle's SiLU-and-mul requant of the GPU-independent fp32 sums
    one = np.array([0, len(rows)], np.int32)
    Hr, HSr = oracle.silu_mul_quant(ref.astype(np.float32), one, np.array([len(rows)], np.int32))
    d = e4m3_ulp_diff(host(H)[rows], Hr)
    assert d.max() <= 1 and (d == 0).mean() >= 0.99, ((d == 0).mean(), d.max())
    np.testing.assert_allclose(host(HS)[rows], HSr, rtol=2e-5)


def test_gemm2_full_size_every_tile(prefill):
    li, r = prefill
    counts, offs = r["counts"], r["offsets"]
    cap = moe.moe_rp_cap(WL.M, WL.topk, WL.El)
    R = int(offs[-1])
    rng = np.random.default_rng(5)
    h = (rng.standard_normal((R, WL.N)) * rng.uniform(0.01, 4, (R, 1))).astype(np.float32)
    Hq, HSq = oracle.quant_rows(h)
    H = dev(padded(Hq, cap, 3))
    HS = dev(padded(HSq, cap, 4))
    y = moe.moe_grouped_gemm_fp8(H, HS, dev(li.w2), dev(li.w2_scale), dev(offs), moe.MOE_EPI_BF16,
                                 expert_num_tokens=dev(counts))
    torch.cuda.synchronize()
    rows = sample_rows(offs, counts, seed=12)
    ref = oracle_rows(Hq, HSq, li.w2, li.w2_scale, offs, counts, rows)
    got = mi.bf16_to_f32(host_bits(y)[rows]).astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= 8e-3 * np.abs(ref).max(), err.max() / np.abs(ref).max()
    # per row: one bf16 rounding (half an ulp, 2^-9 relative) plus fp32 accumulation noise
    row_max = np.abs(ref).max(axis=1, keepdims=True)
    assert (err <= np.abs(ref) * 2.0 ** -8 + 1e-5 * row_max).all(), (err / row_max).max()


def test_layer_router_weight_on_input_full_size(prefill):
    li, _ = prefill
    d = dict(x=dev(li.x), ids=dev(li.topk_ids), w=dev(li.topk_weights))
    out = moe.moe_forward_chunked(d["x"], d["ids"], d["w"], dev(li.w13), dev(li.w13_scale), dev(li.w2),
                                  dev(li.w2_scale), WL.E, apply_router_weight_on_input=True)
    torch.cuda.synchronize()
    got = host_bits(out)
    assert np.isfinite(mi.bf16_to_f32(got)).all()
    rng = np.random.default_rng(WL.seed)
    toks = np.unique(np.concatenate([[0, WL.M - 1], rng.choice(WL.M, 24, replace=False)]))
    ref = oracle.forward_tokens(toks, li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2,
                                li.w2_scale, WL.E, apply_router_weight_on_input=True)
    layer_tolerance(got[toks], ref)
    # weights applied on the input change the result (SiLU is not linear)
    out0 = moe.moe_forward_chunked(d["x"], d["ids"], d["w"], dev(li.w13), dev(li.w13_scale), dev(li.w2),
                                   dev(li.w2_scale), WL.E)
    torch.cuda.synchronize()
    assert (host_bits(out0)[toks] != got[toks]).any()
