"""int64 top-k ids (the dtype torch.topk returns): every entry point that reads ids has an
_i64 twin. Results must equal the oracle's (which reads ids at 64 bits) and the int32
path's bit for bit; an id past the int32 range is a bad id, never a truncated alias."""
import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
import oracle
from helpers import dev, host, host_bits, layer_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def plant_wide_ids(ids, seed, every=97):
    """int64 copy of ids with some entries moved past the int32 range: 2**32 + id (which
    a 32-bit cut would read as id), 2**40 and -(2**32) + 1. Returns (ids64, n_planted)."""
    out = ids.astype(np.int64).reshape(-1).copy()
    rng = np.random.default_rng(seed)
    pos = np.arange(out.size)[::every]
    pos = pos[rng.permutation(len(pos))]
    kinds = np.array([2**32, 2**40, -(2**32) + 1], np.int64)
    for j, p in enumerate(pos):
        out[p] = out[p] + kinds[0] if j % 3 == 0 else kinds[j % 3]
    return out.reshape(ids.shape), len(pos)


def misaligned(t):
    """The same values at an address 8 bytes past a 16-byte boundary (the count kernel's
    scalar path)."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    flat[1:] = t.reshape(-1)
    return flat[1:].view(t.shape)


@pytest.mark.parametrize("M,topk,E,El,aligned", [(1, 1, 1, 1, True), (129, 2, 8, 8, True), (1000, 8, 128, 64, True),
                                                 (2049, 8, 128, 128, True), (5001, 8, 128, 128, False),
                                                 (70000, 8, 128, 64, True), (3, 3, 16, 16, False)])
def test_count_i64(M, topk, E, El, aligned):
    ids, _ = mi.route(M, E, topk, seed=M)
    m = None if El == E else mi.expert_map(E, El)
    ids64, planted = plant_wide_ids(ids, seed=M)
    ref, bad = oracle.count(ids64, E, El, m)
    assert bad == planted
    d = dev(ids64)
    if not aligned:
        d = misaligned(d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = moe.moe_count_expert_tokens(d, E, El, None if m is None else dev(m), err_count=err)
    assert (host(got) == ref).all()
    assert int(err.item()) == bad


@pytest.mark.parametrize("M,topk,E,El,count_here", [(1, 8, 128, 128, False), (300, 8, 128, 64, True),
                                                    (5000, 8, 128, 128, False), (5000, 8, 128, 37, True)])
def test_scatter_i64(M, topk, E, El, count_here):
    K = 256
    ids, w = mi.route(M, E, topk, seed=M + 1, zipf_s=1.2)
    m = None if El == E else (mi.expert_map(E, El) if El == E // 2 else mi.random_expert_map(E, El, seed=2))
    ids64, _ = plant_wide_ids(ids, seed=M + 1, every=53)
    x = mi.hidden_states(M, K, seed=M)
    r = oracle.scatter(x, ids64, w, E, El, m)
    md = None if m is None else dev(m)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if count_here:
        cnt = torch.full((El,), -3, dtype=torch.int32, device="cuda")
    else:
        cnt = moe.moe_count_expert_tokens(dev(ids64), E, El, md)
    a, sa, offs, s2d = moe.moe_scatter(dev(x), dev(ids64), dev(w), E, El, cnt, md, count_here=count_here,
                                       err_count=err)
    torch.cuda.synchronize()
    assert (host(cnt) == r["counts"]).all()
    if count_here:
        assert int(err.item()) == r["bad"] > 0
    assert (host(offs) == r["offsets"]).all()
    assert (host(s2d) == r["src2dst"]).all()
    rows = r["src2dst"].reshape(-1)
    rows = rows[rows >= 0]
    assert (host(a)[rows] == r["a"][rows]).all()
    assert (host(sa)[rows].view(np.uint32) == r["a_scale"][rows].view(np.uint32)).all()


def test_scatter_noalloc_i64():
    M, topk, E, El, K = 2000, 8, 128, 128, 256
    ids, w = mi.route(M, E, topk, seed=4)
    ids64, _ = plant_wide_ids(ids, seed=4)
    x = mi.hidden_states(M, K, seed=4)
    r = oracle.scatter(x, ids64, w, E, El)
    cnt = moe.moe_count_expert_tokens(dev(ids64), E, El)
    cap = moe.moe_rp_cap(M, topk, El)
    a = torch.empty(cap, K, dtype=torch.uint8, device="cuda")
    sa = torch.empty(cap, K // 128, dtype=torch.float32, device="cuda")
    offs = torch.empty(El + 1, dtype=torch.int32, device="cuda")
    s2d = torch.empty(M, topk, dtype=torch.int32, device="cuda")
    moe.moe_scatter_noalloc(dev(x), dev(ids64), dev(w), E, El, cnt, a, sa, offs, s2d)
    torch.cuda.synchronize()
    assert (host(offs) == r["offsets"]).all()
    assert (host(s2d) == r["src2dst"]).all()
    rows = r["src2dst"].reshape(-1)
    rows = rows[rows >= 0]
    assert (host(a)[rows] == r["a"][rows]).all()
    assert (host(sa)[rows].view(np.uint32) == r["a_scale"][rows].view(np.uint32)).all()


@pytest.mark.parametrize("wl_name,chunk", [("tiny", None), ("tiny", 16), ("decode", None)])
def test_layer_i64_equals_i32(wl_name, chunk):
    """The layer with int64 ids: bit-identical to the int32 call on ids that fit, and,
    with wide ids planted, bit-identical to the int32 call where those slots carry another
    bad id (both drop them), with the same bad-id count; within tolerance of the oracle."""
    wl = {"tiny": mi.TINY, "decode": mi.QWEN3_DECODE}[wl_name]
    li = mi.make_layer_inputs(wl)
    wts = (dev(li.w13), dev(li.w13_scale), dev(li.w2), dev(li.w2_scale))
    m = None if li.expert_map is None else dev(li.expert_map)
    x, tw = dev(li.x), dev(li.topk_weights)
    run = lambda ids, err=None: moe.moe_forward_chunked(x, ids, tw, *wts, wl.E, expert_map=m, chunk_size=chunk,
                                                        err_count=err)
    ref32 = host_bits(run(dev(li.topk_ids)))
    got = host_bits(run(dev(li.topk_ids.astype(np.int64))))
    assert (got == ref32).all()

    ids64, planted = plant_wide_ids(li.topk_ids, seed=11, every=7)
    ids32 = np.where((ids64 >= 0) & (ids64 < wl.E), ids64, wl.E + 3).astype(np.int32)
    ids32[ids64 == -1] = -1
    e64 = torch.zeros(1, dtype=torch.int32, device="cuda")
    e32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = host_bits(run(dev(ids64), e64))
    want = host_bits(run(dev(ids32), e32))
    torch.cuda.synchronize()
    assert (got == want).all()
    assert int(e64.item()) == int(e32.item()) == planted
    if wl_name == "tiny":
        ref = oracle.forward_chunked(li.x, ids64, li.topk_weights, li.w13, li.w13_scale, li.w2, li.w2_scale, wl.E,
                                     expert_map=li.expert_map, chunk_size=chunk)
        layer_tolerance(got, ref)


def test_forward_host_i64():
    wl = mi.TINY
    li = mi.make_layer_inputs(wl)
    wts = (dev(li.w13), dev(li.w13_scale), dev(li.w2), dev(li.w2_scale))
    ids64, _ = plant_wide_ids(li.topk_ids, seed=5, every=11)
    want = host_bits(moe.moe_forward_chunked(dev(li.x), dev(ids64), dev(li.topk_weights), *wts, wl.E))
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    xh = torch.from_numpy(li.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ev = torch.cuda.Event()
    out = moe.moe_forward_host(xh, pin(ids64), pin(li.topk_weights), *wts, wl.E, done=ev)
    ev.synchronize()
    assert (out.view(torch.int16).numpy().view(np.uint16) == want).all()
