"""Guard bands: every entry point writes only inside the rows it is given. Each output
buffer is allocated with extra rows (or bytes) past what the call is told, filled with a
sentinel, and checked afterwards -- for the count, the scatter (also when the caller's
counts disagree with the ids), both GEMM epilogues (also when the caller's offsets run
past the row bound), the gather and the whole layer with its workspace."""
import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
import oracle
from helpers import dev, host

pytestmark = pytest.mark.gpu

G = 64          # guard rows
SENT = 0xA5     # sentinel byte


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def guarded(rows, cols, dtype):
    """A [rows + G, cols] tensor filled with the sentinel byte; returns (full, view of rows)."""
    t = torch.empty(rows + G, cols, dtype=dtype, device="cuda")
    t.view(torch.uint8).fill_(SENT)
    return t, t[:rows]


def untouched(full, rows):
    g = full[rows:].contiguous().view(torch.uint8)
    return bool((g == SENT).all())


def test_count_writes_only_its_experts():
    ids, _ = mi.route(5000, 128, 8, 1, 1.2)
    full, cnt = guarded(1, 64, torch.int32)
    moe.moe_count_expert_tokens(dev(ids), 128, 64, dev(mi.expert_map(128, 64)), expert_num_tokens=cnt[0])
    torch.cuda.synchronize()
    assert untouched(full, 1)
    assert (host(cnt[0]) == oracle.count(ids, 128, 64, mi.expert_map(128, 64))[0]).all()


@pytest.mark.parametrize("M,inflate", [(300, 0), (5000, 0), (300, 700), (5000, 40)])
def test_scatter_stays_inside_rp_cap(M, inflate):
    """With counts that disagree with the ids (inflated by `inflate` per expert) the
    result is unspecified, but no offset passes rp_cap and nothing is written past it."""
    E, El, topk, K = 128, 128, 8, 512
    x = mi.hidden_states(M, K, 7)
    ids, tw = mi.route(M, E, topk, 7, 1.2)
    cap = moe.moe_rp_cap(M, topk, El)
    cnt = oracle.count(ids, E, El)[0] + inflate
    a_full, a = guarded(cap, K, torch.uint8)
    s_full, s = guarded(cap, K // 128, torch.float32)
    o_full, o = guarded(1, El + 1, torch.int32)
    d_full, d = guarded(M, topk, torch.int32)
    moe.moe_scatter(dev(x), dev(ids), dev(tw), E, El, dev(cnt.astype(np.int32)), rp_cap=cap, a_out=a, a_scale=s,
                    expert_offsets=o[0], src2dst=d)
    torch.cuda.synchronize()
    for full, rows in ((a_full, cap), (s_full, cap), (o_full, 1), (d_full, M)):
        assert untouched(full, rows)
    offs = host(o[0])
    s2d = host(d)
    assert (offs <= cap).all() and (offs % 128 == 0).all() and (np.diff(offs) >= 0).all()
    assert s2d.max() < cap
    if inflate == 0:
        ref = oracle.scatter(x, ids, tw, E, El)
        assert (offs == ref["offsets"]).all() and (s2d == ref["src2dst"]).all()


@pytest.mark.parametrize("epi", [moe.MOE_EPI_SILU_MUL_QUANT, moe.MOE_EPI_BF16, moe.MOE_EPI_F32])
@pytest.mark.parametrize("overrun", [False, True])
def test_gemm_stays_inside_rp_cap(epi, overrun):
    """The GEMM writes rows below min(expert_offsets[El], rp_cap) only: offsets that run
    past the row bound (a caller's mistake) are cut at it."""
    counts = np.array([130, 0, 77, 300], np.int32)
    offs = oracle.offsets(counts)
    cap = int(offs[-1])
    K, n_out = 256, 512
    rng = np.random.default_rng(3)
    A, SA = oracle.quant_rows(rng.standard_normal((cap, K)).astype(np.float32))
    W, S = mi.expert_weights(4, n_out, K, seed=9, stream=1)
    d_offs = offs.copy()
    if overrun:
        d_offs[-2:] += 256   # the last expert's block claims 256 rows past the bound
    ocols = n_out // 2 if epi == moe.MOE_EPI_SILU_MUL_QUANT else n_out
    odt = {moe.MOE_EPI_SILU_MUL_QUANT: torch.uint8, moe.MOE_EPI_BF16: torch.bfloat16,
           moe.MOE_EPI_F32: torch.float32}[epi]
    o_full, o = guarded(cap, ocols, odt)
    s_full, s = guarded(cap, n_out // 256, torch.float32)
    moe.moe_grouped_gemm_fp8(dev(A), dev(SA), dev(W), dev(S), dev(d_offs), epi, out=o,
                             out_scale=s if epi == moe.MOE_EPI_SILU_MUL_QUANT else None)
    torch.cuda.synchronize()
    assert untouched(o_full, cap)
    assert untouched(s_full, cap)


def test_gather_writes_only_its_tokens():
    M, topk, K = 333, 8, 384
    rng = np.random.default_rng(4)
    Y = mi.bf16_bits(rng.standard_normal((2048, K)).astype(np.float32))
    s2d = rng.integers(-1, 2048, (M, topk)).astype(np.int32)
    tw = rng.uniform(0, 1, (M, topk)).astype(np.float32)
    o_full, o = guarded(M, K, torch.bfloat16)
    moe.moe_gather_weight_reduce(dev(Y), dev(s2d), dev(tw), out=o)
    torch.cuda.synchronize()
    assert untouched(o_full, M)


@pytest.mark.parametrize("wl,chunk", [(mi.TINY, None), (mi.TINY, 24), (mi.QWEN3_DECODE, 40)])
def test_layer_writes_only_its_rows_and_workspace(wl, chunk):
    li = mi.make_layer_inputs(wl)
    M, K = li.x.shape
    El, N2, _ = li.w13.shape
    need = moe.moe_workspace_size(min(chunk or M, M), K, N2 // 2, wl.topk, El)
    ws_full = torch.full((need + 4096,), SENT, dtype=torch.uint8, device="cuda")
    o_full, o = guarded(M, K, torch.bfloat16)
    moe.moe_forward_chunked(dev(li.x), dev(li.topk_ids), dev(li.topk_weights), dev(li.w13), dev(li.w13_scale),
                            dev(li.w2), dev(li.w2_scale), wl.E, chunk_size=chunk, out=o, workspace=ws_full[:need])
    torch.cuda.synchronize()
    assert untouched(o_full, M)
    assert bool((ws_full[need:] == SENT).all())
    ref = oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2, li.w2_scale,
                                 wl.E, chunk_size=chunk)
    from helpers import host_bits, layer_tolerance
    layer_tolerance(host_bits(o), ref)
