"""moe_forward_host: the layer with the batch in pinned host memory, its copies on the
library's own streams. Its output must equal moe_forward_chunked's bit for bit, for
several calls in flight at once (they alternate the workspace's two staging slots), with
completion signalled by events or by moe_host_wait."""
import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
from helpers import dev, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def batches(li, n):
    """n different batches of the workload's shape: token order rotated and activations
    rescaled per batch (routing rows move with their tokens)."""
    out = []
    for v in range(n):
        x = mi.bf16_bits(np.roll(mi.bf16_to_f32(li.x), 5 * v, axis=0) * np.float32(1 + 0.25 * v))
        out.append((x, np.roll(li.topk_ids, 5 * v, axis=0), np.roll(li.topk_weights, 5 * v, axis=0)))
    return out


def pinned(a):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.pin_memory()


@pytest.mark.parametrize("name,chunk", [("tiny", None), ("tiny", 16), ("decode", None)])
def test_forward_host_equals_device(name, chunk):
    wl = {"tiny": mi.TINY, "decode": mi.QWEN3_DECODE}[name]
    li = mi.make_layer_inputs(wl)
    w = dict(w13=dev(li.w13), s13=dev(li.w13_scale), w2=dev(li.w2), s2=dev(li.w2_scale),
             m=None if li.expert_map is None else dev(li.expert_map))
    bs = batches(li, 3)
    refs = []
    for x, ids, tw in bs:
        out = moe.moe_forward_chunked(dev(x), dev(ids), dev(tw), w["w13"], w["s13"], w["w2"], w["s2"], wl.E,
                                      expert_map=w["m"], chunk_size=chunk)
        torch.cuda.synchronize()
        refs.append(host_bits(out))
    assert not all((refs[0] == r).all() for r in refs[1:])  # the batches differ

    M, K = li.x.shape
    El, N2, _ = li.w13.shape
    ws = torch.empty(moe.moe_host_workspace_size(M, K, N2 // 2, wl.topk, El, chunk or M), dtype=torch.uint8,
                     device="cuda")
    hin = [tuple(pinned(a) for a in b) for b in bs]
    for completion in ("events", "host_wait"):
        outs, evs = [], []
        for x, ids, tw in hin:  # three calls in flight; the slots alternate 0, 1, 0
            ev = torch.cuda.Event() if completion == "events" else None
            outs.append(moe.moe_forward_host(x, ids, tw, w["w13"], w["s13"], w["w2"], w["s2"], wl.E,
                                             expert_map=w["m"], chunk_size=chunk, workspace=ws, done=ev))
            evs.append(ev)
        if completion == "events":
            for ev in evs:
                ev.synchronize()
        else:
            moe.moe_host_wait()
            torch.cuda.current_stream().synchronize()
        for got, ref in zip(outs, refs):
            assert (got.view(torch.int16).numpy().view(np.uint16) == ref).all()


def test_forward_host_needs_pinned_host_tensors():
    li = mi.make_layer_inputs(mi.TINY)
    args = (torch.from_numpy(li.x.view(np.int16)).view(torch.bfloat16), pinned(li.topk_ids),
            pinned(li.topk_weights), dev(li.w13), dev(li.w13_scale), dev(li.w2), dev(li.w2_scale), mi.TINY.E)
    with pytest.raises(ValueError):
        moe.moe_forward_host(*args)  # hidden_states is pageable


def test_forward_host_interleaved_sizes_share_one_workspace():
    """Large and small batches alternate on one workspace sized for the largest, several
    calls in flight: a call whose size differs from the previous one places its staging
    slots elsewhere, and must not overwrite bytes an earlier call is still using."""
    wl = mi.QWEN3_DECODE
    li = mi.make_layer_inputs(wl)
    K, E, topk = wl.K, wl.E, wl.topk
    El, N2, _ = li.w13.shape
    w = dict(w13=dev(li.w13), s13=dev(li.w13_scale), w2=dev(li.w2), s2=dev(li.w2_scale))
    sizes = [2048, 64, 2048, 7, 1500, 2048, 1, 2048, 640]
    chunk = 512
    bs = []
    for i, M in enumerate(sizes):
        ids, tw = mi.route(M, E, topk, 100 + i, 1.2)
        bs.append((mi.hidden_states(M, K, 100 + i), ids, tw))
    refs = []
    for x, ids, tw in bs:
        out = moe.moe_forward_chunked(dev(x), dev(ids), dev(tw), w["w13"], w["s13"], w["w2"], w["s2"], E,
                                      chunk_size=chunk)
        torch.cuda.synchronize()
        refs.append(host_bits(out))
    ws = torch.empty(moe.moe_host_workspace_size(max(sizes), K, N2 // 2, topk, El, chunk), dtype=torch.uint8,
                     device="cuda")
    hin = [tuple(pinned(a) for a in b) for b in bs]
    outs, evs = [], []
    for x, ids, tw in hin:  # all calls in flight before any wait
        ev = torch.cuda.Event()
        outs.append(moe.moe_forward_host(x, ids, tw, w["w13"], w["s13"], w["w2"], w["s2"], E, chunk_size=chunk,
                                         workspace=ws, done=ev))
        evs.append(ev)
    for ev in evs:
        ev.synchronize()
    for i, (got, ref) in enumerate(zip(outs, refs)):
        assert (got.view(torch.int16).numpy().view(np.uint16) == ref).all(), f"batch {i} (M={sizes[i]})"
