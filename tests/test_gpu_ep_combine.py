"""moe_ep_combine (the sum of the expert-parallel ranks' shares) against the oracle: bit
for bit on synthetic shares, and, fed with the shares of the layer run under several
expert_maps, equal to the oracle's single-GPU layer within the layer tolerance."""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_count_gb300 as moe
import moe_inputs as mi
import oracle
from helpers import dev, host_bits, layer_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("R,M,K", [(1, 1, 8), (2, 37, 128), (3, 1000, 2048), (8, 129, 384), (64, 5, 16)])
def test_combine_bit_exact(R, M, K):
    rng = np.random.default_rng(R * 1000 + M)
    parts = [mi.bf16_bits((rng.standard_normal((M, K)) * rng.uniform(0.01, 100, (M, 1))).astype(np.float32))
             for _ in range(R)]
    full = torch.full((M + 16, K), 0x5A5A, dtype=torch.int16, device="cuda")
    out = full[:M].view(torch.bfloat16)
    moe.moe_ep_combine([dev(p) for p in parts], out=out)
    torch.cuda.synchronize()
    assert (host_bits(out) == oracle.ep_combine(parts)).all()
    assert bool((full[M:] == 0x5A5A).all())  # nothing written past M rows


def test_combine_refuses_bad_arguments():
    L = moe.lib()
    p = torch.zeros(4, 8, dtype=torch.bfloat16, device="cuda")
    arr = (ctypes.c_void_p * 2)(p.data_ptr(), p.data_ptr())
    assert L.moe_ep_combine(arr, 0, 4, 8, ctypes.c_void_p(p.data_ptr()), None) == 1      # no parts
    assert L.moe_ep_combine(arr, 2, 4, 12, ctypes.c_void_p(p.data_ptr()), None) == 1     # K % 8
    assert L.moe_ep_combine(arr, 2, 4, 8, ctypes.c_void_p(p.data_ptr()), None) == 1      # out overlaps a part


@pytest.mark.parametrize("wl,ranks", [(mi.TINY, 2), (mi.TINY, 4), (mi.QWEN3_DECODE, 2)])
def test_expert_parallel_layer(wl, ranks):
    """Each simulated rank holds E / ranks consecutive experts (expert_map and its slice
    of the weights) and runs the layer; the combined shares are the layer."""
    li = mi.make_layer_inputs(wl)
    E, per = wl.E, wl.E // ranks
    x, ids, tw = dev(li.x), dev(li.topk_ids), dev(li.topk_weights)
    parts = []
    for r in range(ranks):
        m = np.full(E, -1, np.int32)
        m[r * per:(r + 1) * per] = np.arange(per)
        sl = slice(r * per, (r + 1) * per)
        parts.append(moe.moe_forward_chunked(x, ids, tw, dev(li.w13[sl]), dev(li.w13_scale[sl]), dev(li.w2[sl]),
                                             dev(li.w2_scale[sl]), E, expert_map=dev(m)))
    out = moe.moe_ep_combine(parts)
    torch.cuda.synchronize()
    ref = oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2, li.w2_scale, E)
    layer_tolerance(host_bits(out), ref)
