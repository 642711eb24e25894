"""CUDA-graph capture: the entry points enqueue only kernels (and a memset) on the
caller's stream, with no allocation or synchronisation, so a serving loop can capture
the layer once and replay it. Replays on new batch contents must equal eager calls bit
for bit."""
import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
from helpers import dev, host, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def batches(li, n):
    """n batches of the workload's shape: tokens rolled and rescaled, routing rolled."""
    out = []
    for v in range(n):
        x = mi.bf16_bits(np.roll(mi.bf16_to_f32(li.x), 3 * v + 1, axis=0) * np.float32(1 + 0.5 * v))
        out.append((x, np.roll(li.topk_ids, 7 * v + 1, axis=0), np.roll(li.topk_weights, 7 * v + 1, axis=0)))
    return out


def capture(fn):
    """Warm fn up on a side stream, then capture one call of it into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("name,chunk", [("tiny", None), ("tiny", 16), ("decode", None), ("chunked", 128)])
def test_layer_graph_replay_equals_eager(name, chunk):
    wl = {"tiny": mi.TINY, "decode": mi.QWEN3_DECODE, "chunked": mi.QWEN3_CHUNKED}[name]
    li = mi.make_layer_inputs(wl)
    if name == "chunked":  # 40 chunks of 128 tokens (the last one ragged) keep the test short
        M = 40 * 128 - 77
        li.x, li.topk_ids, li.topk_weights = li.x[:M], li.topk_ids[:M], li.topk_weights[:M]
    wts = (dev(li.w13), dev(li.w13_scale), dev(li.w2), dev(li.w2_scale))
    m = None if li.expert_map is None else dev(li.expert_map)
    M, K = li.x.shape
    El, N2, _ = li.w13.shape
    topk = li.topk_ids.shape[1]
    # static buffers the graph is captured on
    x, ids, tw = dev(li.x), dev(li.topk_ids), dev(li.topk_weights)
    out = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(moe.moe_workspace_size(min(chunk or M, M), K, N2 // 2, topk, El), dtype=torch.uint8,
                     device="cuda")
    call = lambda: moe.moe_forward_chunked(x, ids, tw, *wts, wl.E, expert_map=m, chunk_size=chunk, out=out,
                                           workspace=ws)
    g = capture(call)
    for bx, bids, btw in batches(li, 3):
        want = host_bits(moe.moe_forward_chunked(dev(bx), dev(bids), dev(btw), *wts, wl.E, expert_map=m,
                                                 chunk_size=chunk))
        x.copy_(dev(bx))
        ids.copy_(dev(bids))
        tw.copy_(dev(btw))
        g.replay()
        torch.cuda.synchronize()
        assert (host_bits(out) == want).all()
    assert moe.moe_device_error() == 0


@pytest.mark.parametrize("M", [100, 20000])  # one CTA / memset + many CTAs
def test_count_and_scatter_graph_replay(M):
    E, El, topk, K = 128, 128, 8, 256
    ids0, w0 = mi.route(M, E, topk, seed=1)
    x0 = mi.hidden_states(M, K, seed=1)
    ids, tw, x = dev(ids0), dev(w0), dev(x0)
    cnt = torch.empty(El, dtype=torch.int32, device="cuda")
    cap = moe.moe_rp_cap(M, topk, El)
    a = torch.empty(cap, K, dtype=torch.uint8, device="cuda")
    sa = torch.empty(cap, K // 128, dtype=torch.float32, device="cuda")
    offs = torch.empty(El + 1, dtype=torch.int32, device="cuda")
    s2d = torch.empty(M, topk, dtype=torch.int32, device="cuda")
    sws = torch.empty(moe.moe_scatter_workspace_size(M, topk, El), dtype=torch.uint8, device="cuda")

    def call():
        moe.moe_count_expert_tokens(ids, E, El, expert_num_tokens=cnt)
        moe.moe_scatter(x, ids, tw, E, El, cnt, rp_cap=cap, a_out=a, a_scale=sa, expert_offsets=offs,
                        src2dst=s2d, workspace=sws)

    g = capture(call)
    for seed in (2, 3):
        ids1, w1 = mi.route(M, E, topk, seed=seed, zipf_s=1.2)
        x1 = mi.hidden_states(M, K, seed=seed)
        c_ref = moe.moe_count_expert_tokens(dev(ids1), E, El)
        a_ref, sa_ref, off_ref, s2d_ref = moe.moe_scatter(dev(x1), dev(ids1), dev(w1), E, El, c_ref)
        ids.copy_(dev(ids1))
        tw.copy_(dev(w1))
        x.copy_(dev(x1))
        g.replay()
        torch.cuda.synchronize()
        assert (host(cnt) == host(c_ref)).all()
        assert (host(offs) == host(off_ref)).all()
        assert (host(s2d) == host(s2d_ref)).all()
        rows = host(s2d_ref).reshape(-1)
        rows = rows[rows >= 0]
        assert (host(a)[rows] == host(a_ref)[rows]).all()
        assert (host(sa)[rows] == host(sa_ref)[rows]).all()
