"""The C-ABI library builds, loads and exports every symbol of include/*.h, and its
host-side queries and argument checks behave as documented. No kernel is launched."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_count_gb300 as moe
    return moe.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert {"moe_count_expert_tokens", "moe_scatter", "moe_grouped_gemm_fp8", "moe_silu_mul_quant",
            "moe_gather_weight_reduce", "moe_forward_chunked"} <= names
    for n in names:
        assert hasattr(L, n), n


def test_binding_declares_every_symbol(L):
    import moe_expert_layer_count_gb300 as moe
    assert declared_symbols() <= set(moe.SIGNATURES)


def test_size_queries(L):
    import moe_expert_layer_count_gb300 as moe
    import oracle
    for Mc, topk, El in ((1, 8, 64), (128, 8, 64), (64, 8, 128), (8192, 8, 128), (3, 2, 1), (0, 8, 4)):
        assert moe.moe_rp_cap(Mc, topk, El) == oracle.rp_cap(Mc, topk, El)
    assert moe.moe_rp_cap(1, 0, 4) == -1
    assert moe.moe_workspace_size(128, 2048, 768, 8, 64) > 0
    assert moe.moe_workspace_size(128, 2000, 768, 8, 64) == 0          # K not a multiple of 128
    # per-chunk sizing: a smaller chunk never needs more
    assert moe.moe_workspace_size(1, 2048, 768, 8, 64) < moe.moe_workspace_size(128, 2048, 768, 8, 64)
    assert moe.status_string(0) == "ok"


def test_argument_checks_return_before_any_launch(L):
    # invalid arguments are refused on the host: nothing touches a device
    p = ctypes.c_void_p(16)
    assert L.moe_count_expert_tokens(p, 4, 0, None, 8, 8, p, None, None) == 1          # topk 0
    assert L.moe_count_expert_tokens(p, 4, 2, None, 8, 0, p, None, None) == 1          # El 0
    assert L.moe_count_expert_tokens(p, 4, 2, None, 8, 2000, p, None, None) == 1       # El > 1024
    assert L.moe_gather_weight_reduce(p, p, p, 4, 2, 100, 0, p, None) == 1             # K % 128
    assert L.moe_grouped_gemm_fp8(p, p, p, p, p, None, 4, 128, 384, 256, 2, p, p, None) == 1  # silu: n_out%256
    assert L.moe_silu_mul_quant(None, p, 4, 128, 128, p, p, None) == 1
    ws = ctypes.c_void_p(4096)
    # out overlapping the workspace is refused
    assert L.moe_forward_chunked(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 4, 0, ws,
                                 ws, 1 << 30, None, None) == 1
    # workspace too small
    assert L.moe_forward_chunked(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 4, 0, p,
                                 ws, 16, None, None) == 2
    # out overlapping hidden_states other than exactly, or the top-k ids / weights
    x, ids, tw = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    big = ctypes.c_void_p(1 << 40)
    for out in (ctypes.c_void_p((1 << 20) + 256), ids, ctypes.c_void_p((3 << 20) - 16)):
        assert L.moe_forward_chunked(x, ids, tw, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 4, 0, out,
                                     big, 1 << 30, None, None) == 1
    # the int64-id twins run the same checks
    assert L.moe_count_expert_tokens_i64(p, 4, 0, None, 8, 8, p, None, None) == 1      # topk 0
    assert L.moe_scatter_i64(p, 4, 100, p, p, 2, None, 8, 8, p, 0, None, 0, 1, p, p, p, p, 1 << 20, p,
                             1 << 20, None) == 1                                           # K % 128
    assert L.moe_scatter_noalloc_i64(p, 4, 128, p, p, 33, None, 8, 8, p, 0, 1, p, p, p, p, 1 << 20,
                                     None) == 1                                            # topk > 32
    assert L.moe_forward_chunked_i64(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 4, 0, ws,
                                     ws, 1 << 30, None, None) == 1
    assert L.moe_forward_host_i64(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 4, 0, p, p, 16,
                                  None, None, None) == 2


def test_binding_picks_the_entry_point_by_id_dtype():
    import torch
    import moe_expert_layer_count_gb300 as moe
    assert moe._ids_entry("moe_scatter", torch.zeros(1, dtype=torch.int32)) == "moe_scatter"
    assert moe._ids_entry("moe_scatter", torch.zeros(1, dtype=torch.int64)) == "moe_scatter_i64"
    with pytest.raises(TypeError):
        moe.moe_count_expert_tokens(torch.zeros(4, 2, dtype=torch.int16), 8, 8)


def test_host_entry_point_checks(L):
    import moe_expert_layer_count_gb300 as moe
    # two staging slots (x, ids with room for int64, weights, out) after the layer's own workspace
    lay = moe.moe_workspace_size(128, 2048, 768, 8, 64)
    slot = 128 * 2048 * 2 + 128 * 8 * 8 + 128 * 8 * 4 + 128 * 2048 * 2
    assert moe.moe_host_workspace_size(128, 2048, 768, 8, 64, 128) >= lay + 2 * slot
    assert moe.moe_host_workspace_size(128, 2000, 768, 8, 64, 128) == 0   # K not a multiple of 128
    assert moe.moe_host_workspace_size(0, 2048, 768, 8, 64, 128) == 0
    p = ctypes.c_void_p(16)
    # refused on the host before any copy or launch
    assert L.moe_forward_host(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 0, 4, 0, p, p, 1 << 30,
                              None, None, None) == 1                                   # topk 0
    assert L.moe_forward_host(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 4, 0, p, p, 16,
                              None, None, None) == 2                                   # workspace too small
    assert L.moe_forward_host(p, p, p, p, p, p, p, None, 8, 8, 0, 128, 128, 2, 4, 0, p, p, 16,
                              None, None, None) == 0                                   # M = 0: no-op


def test_every_entry_point_refuses_bad_arguments_on_the_host(L):
    """Each documented argument error returns its status before anything is enqueued
    (no device is touched: these calls run on a machine without a GPU)."""
    p, odd = ctypes.c_void_p(16), ctypes.c_void_p(8)  # 16-byte aligned / misaligned
    INVALID, SMALL, SCRATCH = 1, 2, 5
    # count: E < 1, top-k > 32, ids missing for M > 0
    assert L.moe_count_expert_tokens(p, 4, 2, None, 0, 1, p, None, None) == INVALID
    assert L.moe_count_expert_tokens(p, 4, 33, None, 64, 64, p, None, None) == INVALID
    assert L.moe_count_expert_tokens(None, 4, 2, None, 8, 8, p, None, None) == INVALID

    def scatter(M=4, K=128, topk=2, El=8, quant=1, x=p, rp_cap=1 << 20, ws_bytes=1 << 20, fn=L.moe_scatter):
        return fn(x, M, K, p, p, topk, None, 8, El, p, 0, None, 0, quant, p, p, p, p, rp_cap, p, ws_bytes, None)
    assert scatter(K=100) == INVALID                                 # K not a multiple of 128
    assert scatter(quant=7) == INVALID                               # unknown quantisation
    assert scatter(x=odd) == INVALID                                 # rows not 16-byte aligned
    assert scatter(rp_cap=L.moe_rp_cap(4, 2, 8) - 128) == INVALID    # row bound below moe_rp_cap
    assert scatter(M=1000, topk=8, ws_bytes=16) == SMALL             # many blocks, scratch too small
    assert scatter(K=100, fn=L.moe_scatter_i64) == INVALID
    # allocation-free scatter: more block histograms than its fixed scratch holds
    M, topk, El = 100000, 8, 1024
    assert L.moe_scatter_noalloc(p, M, 128, p, p, topk, None, El, El, p, 0, 1, p, p, p, p,
                                 L.moe_rp_cap(M, topk, El), None) == SCRATCH

    def gemm(El=4, rp_cap=256, n_out=256, k_in=256, epi=0, out=p):
        return L.moe_grouped_gemm_fp8(p, p, p, p, p, None, El, rp_cap, n_out, k_in, epi, out, p, None)
    assert gemm(epi=9) == INVALID                                    # unknown epilogue
    assert gemm(n_out=200) == INVALID                                # n_out not a multiple of 128
    assert gemm(rp_cap=200) == INVALID                               # row bound not a multiple of 128
    assert gemm(El=2000) == INVALID                                  # more than 1024 local experts
    assert gemm(out=odd) == INVALID                                  # output not 16-byte aligned
    # standalone SiLU-and-mul: N not a multiple of 128, misaligned input
    assert L.moe_silu_mul_quant(p, p, 4, 128, 100, p, p, None) == INVALID
    assert L.moe_silu_mul_quant(odd, p, 4, 128, 128, p, p, None) == INVALID
    # gather: top-k > 32, negative M, weights missing when they are applied here
    assert L.moe_gather_weight_reduce(p, p, p, 4, 33, 128, 0, p, None) == INVALID
    assert L.moe_gather_weight_reduce(p, p, p, -1, 2, 128, 0, p, None) == INVALID
    assert L.moe_gather_weight_reduce(p, p, None, 4, 2, 128, 0, p, None) == INVALID
    # whole layer: chunk size < 1, N not a multiple of 128; M = 0 is a no-op
    ws = ctypes.c_void_p(1 << 20)
    assert L.moe_forward_chunked(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 128, 2, 0, 0, p, ws, 1 << 30,
                                 None, None) == INVALID
    assert L.moe_forward_chunked(p, p, p, p, p, p, p, None, 8, 8, 4, 128, 100, 2, 4, 0, p, ws, 1 << 30,
                                 None, None) == INVALID
    assert L.moe_forward_chunked(p, p, p, p, p, p, p, None, 8, 8, 0, 128, 128, 2, 4, 0, p, ws, 1 << 30,
                                 None, None) == 0


def test_int32_row_indices_bound_the_sizes(L):
    """Slots and permuted rows are indexed with int32: sizes that would overflow them are
    refused on the host, by every entry point that builds such indices."""
    p = ctypes.c_void_p(16)
    INVALID = 1
    big_M = (1 << 31) // 8 + 1                      # M * top-8 > 2^31 - 1
    assert L.moe_count_expert_tokens(p, big_M, 8, None, 128, 128, p, None, None) == INVALID
    assert L.moe_count_expert_tokens_i64(p, big_M, 8, None, 128, 128, p, None, None) == INVALID
    assert L.moe_scatter(p, big_M, 128, p, p, 8, None, 128, 128, p, 0, None, 0, 1, p, p, p, p, 1 << 40, p,
                         1 << 40, None) == INVALID
    assert L.moe_scatter_noalloc(p, big_M, 128, p, p, 8, None, 128, 128, p, 0, 1, p, p, p, p, 1 << 40,
                                 None) == INVALID
    assert L.moe_gather_weight_reduce(p, p, p, big_M, 8, 128, 0, p, None) == INVALID
    assert L.moe_workspace_size(big_M, 128, 128, 8, 128) == 0
    # M * topk fits, but the padded row bound does not
    M = (1 << 31) // 8 - 1000
    assert L.moe_rp_cap(M, 8, 1024) > (1 << 31) - 1
    assert L.moe_count_expert_tokens(p, M, 8, None, 1024, 1024, p, None, None) == INVALID
    # a row bound past int32 on the GEMM and the standalone SiLU
    assert L.moe_grouped_gemm_fp8(p, p, p, p, p, None, 4, 1 << 31, 256, 256, 0, p, p, None) == INVALID
    assert L.moe_silu_mul_quant(p, p, 4, 1 << 31, 128, p, p, None) == INVALID
    # the scatter's own row bound must stay in int32 too
    assert L.moe_scatter(p, 4, 128, p, p, 2, None, 8, 8, p, 0, None, 0, 1, p, p, p, p, 1 << 31, p, 1 << 20,
                         None) == INVALID
