"""The allocation-free scatter entry point (moe_scatter_noalloc).

It exists for callers that cannot allocate device memory -- engines that plan every
buffer at start-up and forbid allocation while serving, or runtimes that only pass
inputs and outputs -- and keeps its scratch in a fixed array inside the library. These
tests call it through the C ABI and require its outputs to equal moe_scatter's (the
scatter outputs are integers and FP8 codes, compared bit for bit) on two calls in a
row with different inputs, so that the shared scratch left by the first call cannot
leak into the second. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _case(M, K, E, topk, seed, local=None):
    x = mi.hidden_states(M, K, seed)
    ids, w = mi.route(M, E, topk, seed=seed, zipf_s=1.2)
    m = mi.expert_map(E, local)
    El = E if local is None else local
    return _dev(x), _dev(ids), _dev(w), (None if m is None else _dev(m)), El


def _run_both(x, ids, w, m, E, El):
    M, K = x.shape
    topk = ids.shape[1]
    counts = moe.moe_count_expert_tokens(ids, E, El, m)
    ref = moe.moe_scatter(x, ids, w, E, El, counts, m)
    cap = moe.moe_rp_cap(M, topk, El)
    # output buffers pre-filled with junk: the entry point must write every kept row
    a = torch.full((cap, K), 0x55, dtype=torch.uint8, device="cuda")
    sa = torch.full((cap, K // 128), 7.0, dtype=torch.float32, device="cuda")
    offs = torch.full((El + 1,), -9, dtype=torch.int32, device="cuda")
    s2d = torch.full((M, topk), -9, dtype=torch.int32, device="cuda")
    st = moe.lib().moe_scatter_noalloc(
        ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
        topk, None if m is None else ctypes.c_void_p(m.data_ptr()), E, El, ctypes.c_void_p(counts.data_ptr()),
        0, moe.MOE_QUANT_FP8_1X128, ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(sa.data_ptr()),
        ctypes.c_void_p(offs.data_ptr()), ctypes.c_void_p(s2d.data_ptr()), cap,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, moe.status_string(st)
    torch.cuda.synchronize()
    ra, rsa, roffs, rs2d = (t.cpu().numpy() for t in ref)
    got_s2d = s2d.cpu().numpy()
    assert (got_s2d == rs2d).all()
    assert (offs.cpu().numpy() == roffs).all()
    rows = rs2d.reshape(-1)
    rows = rows[rows >= 0]
    assert (a.cpu().numpy()[rows] == ra[rows]).all()
    assert (sa.cpu().numpy()[rows].view(np.uint32) == rsa[rows].view(np.uint32)).all()


def test_noalloc_scatter_matches_scatter_on_two_calls():
    # several scatter blocks, so the fixed scratch is really used; the second call has
    # fewer experts and another routing, over the first call's leftover scratch
    x, ids, w, m, El = _case(4096, 2048, 128, 8, seed=31)
    _run_both(x, ids, w, m, 128, El)
    x, ids, w, m, El = _case(3001, 384, 128, 8, seed=32, local=64)
    _run_both(x, ids, w, m, 128, El)


def test_noalloc_scatter_refuses_problems_beyond_its_scratch():
    # 1024 local experts x 157 scatter blocks (160000 slots) > 65536 entries: refused on
    # the host with MOE_ERR_SCRATCH_LIMIT, nothing enqueued
    p = ctypes.c_void_p(256)
    st = moe.lib().moe_scatter_noalloc(p, 20000, 128, p, p, 8, None, 1024, 1024, p, 0, 1, p, p, p, p,
                                       moe.moe_rp_cap(20000, 8, 1024), None)
    assert st == 5
    assert "fixed scratch" in moe.status_string(st)
