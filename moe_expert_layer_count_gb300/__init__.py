"""Fused Mixture-of-Experts layer hot path for GB300 (sm_103a).

A thin Python binding over the C ABI of ``include/moe_gb300.h`` (``libmoe_gb300.so``):
the functions below carry the C entry points' names and only marshal arguments
(torch tensors -> device pointers, sizes, the current CUDA stream). Every step of the
layer runs in the library's CUDA kernels; there is no fallback of any kind. If the
library is missing or was not built, importing the binding's functions raises.

The layer (vLLM PRs #20903, #20725, #20392): count_expert_num_tokens ->
ep_scatter with 1x128 FP8 quantisation -> block-scaled FP8 grouped GEMM (w13) ->
SiLU-and-mul requantisation -> grouped GEMM (w2) -> ep_gather with the top-k
weight-and-reduce, under a chunking loop that sizes the workspace per chunk.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_QUANT_NONE, MOE_QUANT_FP8_1X128 = 0, 1
MOE_EPI_BF16, MOE_EPI_F32, MOE_EPI_SILU_MUL_QUANT = 0, 1, 2

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib


_p, _i64, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

SIGNATURES = {
    "moe_status_string": ([_int], ctypes.c_char_p),
    "moe_kernel_launch_count": ([], ctypes.c_uint64),
    "moe_device_error": ([_int], _int),
    "moe_rp_cap": ([_i64, _int, _int], _i64),
    "moe_scatter_workspace_size": ([_i64, _int, _int], _sz),
    "moe_workspace_size": ([_i64, _int, _int, _int, _int], _sz),
    "moe_count_expert_tokens": ([_p, _i64, _int, _p, _int, _int, _p, _p, _p], _int),
    "moe_count_expert_tokens_i64": ([_p, _i64, _int, _p, _int, _int, _p, _p, _p], _int),
    "moe_scatter": ([_p, _i64, _int, _p, _p, _int, _p, _int, _int, _p, _int, _p, _int, _int, _p, _p, _p, _p,
                     _i64, _p, _sz, _p], _int),
    "moe_scatter_i64": ([_p, _i64, _int, _p, _p, _int, _p, _int, _int, _p, _int, _p, _int, _int, _p, _p, _p, _p,
                         _i64, _p, _sz, _p], _int),
    "moe_scatter_noalloc": ([_p, _i64, _int, _p, _p, _int, _p, _int, _int, _p, _int, _int, _p, _p, _p, _p, _i64,
                             _p], _int),
    "moe_scatter_noalloc_i64": ([_p, _i64, _int, _p, _p, _int, _p, _int, _int, _p, _int, _int, _p, _p, _p, _p,
                                 _i64, _p], _int),
    "moe_grouped_gemm_fp8": ([_p, _p, _p, _p, _p, _p, _int, _i64, _int, _int, _int, _p, _p, _p], _int),
    "moe_silu_mul_quant": ([_p, _p, _int, _i64, _int, _p, _p, _p], _int),
    "moe_gather_weight_reduce": ([_p, _p, _p, _i64, _int, _int, _int, _p, _p], _int),
    "moe_forward_chunked": ([_p, _p, _p, _p, _p, _p, _p, _p, _int, _int, _i64, _int, _int, _int, _i64, _int,
                             _p, _p, _sz, _p, _p], _int),
    "moe_forward_chunked_i64": ([_p, _p, _p, _p, _p, _p, _p, _p, _int, _int, _i64, _int, _int, _int, _i64, _int,
                                 _p, _p, _sz, _p, _p], _int),
    "moe_host_workspace_size": ([_i64, _int, _int, _int, _int, _i64], _sz),
    "moe_ep_combine": ([_p, _int, _i64, _int, _p, _p], _int),
    "moe_forward_host": ([_p, _p, _p, _p, _p, _p, _p, _p, _int, _int, _i64, _int, _int, _int, _i64, _int,
                          _p, _p, _sz, _p, _p, _p], _int),
    "moe_forward_host_i64": ([_p, _p, _p, _p, _p, _p, _p, _p, _int, _int, _i64, _int, _int, _int, _i64, _int,
                              _p, _p, _sz, _p, _p, _p], _int),
    "moe_host_wait": ([_p], _int),
}


def _declare(L):
    for name, (args, res) in SIGNATURES.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def _dt(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")


def _ids_entry(name: str, topk_ids) -> str:
    """The C entry point for the ids' dtype: `name` for int32, `name`_i64 for int64."""
    if topk_ids.dtype == torch.int32:
        return name
    if topk_ids.dtype == torch.int64:
        return name + "_i64"
    raise TypeError(f"topk_ids: expected torch.int32 or torch.int64, got {topk_ids.dtype}")


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_kernel_launch_count() -> int:
    return int(lib().moe_kernel_launch_count())


def moe_device_error(clear: bool = False) -> int:
    """The library's device error word (0 = fine); synchronises the device."""
    return int(lib().moe_device_error(int(bool(clear))))


def moe_rp_cap(chunk_M: int, topk: int, local_num_experts: int) -> int:
    return int(lib().moe_rp_cap(chunk_M, topk, local_num_experts))


def moe_scatter_workspace_size(M: int, topk: int, local_num_experts: int) -> int:
    return int(lib().moe_scatter_workspace_size(M, topk, local_num_experts))


def moe_workspace_size(chunk_M: int, K: int, N: int, topk: int, local_num_experts: int) -> int:
    return int(lib().moe_workspace_size(chunk_M, K, N, topk, local_num_experts))


# ------------------------------------------------------------------- entry points
def moe_count_expert_tokens(topk_ids, E, local_num_experts, expert_map=None, expert_num_tokens=None,
                            err_count=None, stream=None):
    """Tokens per local expert: int32 [local_num_experts]. topk_ids is int32 or int64."""
    fn = _ids_entry("moe_count_expert_tokens", topk_ids)
    _dt(expert_map, torch.int32, "expert_map")
    M, topk = topk_ids.shape
    if expert_num_tokens is None:
        expert_num_tokens = torch.empty(local_num_experts, dtype=torch.int32, device=topk_ids.device)
    _check(fn, getattr(lib(), fn)(
        _ptr(topk_ids), M, topk, _ptr(expert_map), E, local_num_experts, _ptr(expert_num_tokens),
        _ptr(err_count), _stream(stream)))
    return expert_num_tokens


def moe_scatter(hidden_states, topk_ids, topk_weights, E, local_num_experts, expert_num_tokens,
                expert_map=None, apply_router_weight_on_input=False, quant=MOE_QUANT_FP8_1X128,
                rp_cap=None, a_out=None, a_scale=None, expert_offsets=None, src2dst=None,
                workspace=None, count_here=False, err_count=None, stream=None):
    """Permute rows into expert-contiguous, 128-aligned blocks (+ FP8 1x128 quant).
    With count_here, expert_num_tokens is an output (the count step fused into the
    scatter). topk_ids is int32 or int64. Returns (a_out, a_scale, expert_offsets, src2dst)."""
    _dt(hidden_states, torch.bfloat16, "hidden_states")
    fn = _ids_entry("moe_scatter", topk_ids)
    _dt(topk_weights, torch.float32, "topk_weights")
    M, K = hidden_states.shape
    topk = topk_ids.shape[1]
    El = local_num_experts
    dev = hidden_states.device
    cap = moe_rp_cap(M, topk, El) if rp_cap is None else rp_cap
    if a_out is None:
        a_out = torch.empty(cap, K, dtype=torch.uint8 if quant else torch.bfloat16, device=dev)
    if a_scale is None and quant:
        a_scale = torch.empty(cap, K // 128, dtype=torch.float32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(El + 1, dtype=torch.int32, device=dev)
    if src2dst is None:
        src2dst = torch.empty(M, topk, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(moe_scatter_workspace_size(M, topk, El), dtype=torch.uint8, device=dev)
    _check(fn, getattr(lib(), fn)(
        _ptr(hidden_states), M, K, _ptr(topk_ids), _ptr(topk_weights), topk, _ptr(expert_map), E, El,
        _ptr(expert_num_tokens), int(bool(count_here)), _ptr(err_count), int(bool(apply_router_weight_on_input)),
        quant, _ptr(a_out), _ptr(a_scale), _ptr(expert_offsets), _ptr(src2dst), cap, _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return a_out, a_scale, expert_offsets, src2dst


def moe_scatter_noalloc(hidden_states, topk_ids, topk_weights, E, local_num_experts, expert_num_tokens,
                        a_out, a_scale, expert_offsets, src2dst, expert_map=None,
                        apply_router_weight_on_input=False, quant=MOE_QUANT_FP8_1X128, rp_cap=None, stream=None):
    """moe_scatter for callers that cannot allocate: every output buffer is the caller's,
    and the scratch is a fixed array inside the library (see the C header for its limit
    and for the rule that calls must not overlap on the GPU). topk_ids is int32 or int64.
    Returns the outputs."""
    _dt(hidden_states, torch.bfloat16, "hidden_states")
    fn = _ids_entry("moe_scatter_noalloc", topk_ids)
    M, K = hidden_states.shape
    topk = topk_ids.shape[1]
    cap = a_out.shape[0] if rp_cap is None else rp_cap
    _check(fn, getattr(lib(), fn)(
        _ptr(hidden_states), M, K, _ptr(topk_ids), _ptr(topk_weights), topk, _ptr(expert_map), E,
        local_num_experts, _ptr(expert_num_tokens), int(bool(apply_router_weight_on_input)), quant,
        _ptr(a_out), _ptr(a_scale), _ptr(expert_offsets), _ptr(src2dst), cap, _stream(stream)))
    return a_out, a_scale, expert_offsets, src2dst


def moe_grouped_gemm_fp8(a, a_scale, w, w_scale, expert_offsets, epilogue=MOE_EPI_BF16, out=None,
                         out_scale=None, stream=None, expert_num_tokens=None):
    """Block-scaled FP8 grouped GEMM over the permuted rows (see the C header). With
    expert_num_tokens, 32-row groups of padding rows are neither computed nor written."""
    _dt(a, torch.uint8, "a")
    _dt(w, torch.uint8, "w")
    rp_cap, k_in = a.shape
    El, n_out, _ = w.shape
    dev = a.device
    if out is None:
        if epilogue == MOE_EPI_SILU_MUL_QUANT:
            out = torch.empty(rp_cap, n_out // 2, dtype=torch.uint8, device=dev)
        else:
            out = torch.empty(rp_cap, n_out, device=dev,
                              dtype=torch.float32 if epilogue == MOE_EPI_F32 else torch.bfloat16)
    if out_scale is None and epilogue == MOE_EPI_SILU_MUL_QUANT:
        out_scale = torch.empty(rp_cap, n_out // 256, dtype=torch.float32, device=dev)
    _check("moe_grouped_gemm_fp8", lib().moe_grouped_gemm_fp8(
        _ptr(a), _ptr(a_scale), _ptr(w), _ptr(w_scale), _ptr(expert_offsets), _ptr(expert_num_tokens), El, rp_cap,
        n_out, k_in,
        epilogue, _ptr(out), _ptr(out_scale), _stream(stream)))
    return (out, out_scale) if epilogue == MOE_EPI_SILU_MUL_QUANT else out


def moe_silu_mul_quant(c1, expert_offsets, h=None, h_scale=None, stream=None):
    """h = silu(gate) * up, requantised 1x128 to FP8. Returns (h, h_scale)."""
    _dt(c1, torch.float32, "c1")
    rp_cap, N2 = c1.shape
    N = N2 // 2
    El = expert_offsets.numel() - 1
    if h is None:
        h = torch.empty(rp_cap, N, dtype=torch.uint8, device=c1.device)
    if h_scale is None:
        h_scale = torch.empty(rp_cap, N // 128, dtype=torch.float32, device=c1.device)
    _check("moe_silu_mul_quant", lib().moe_silu_mul_quant(
        _ptr(c1), _ptr(expert_offsets), El, rp_cap, N, _ptr(h), _ptr(h_scale), _stream(stream)))
    return h, h_scale


def moe_gather_weight_reduce(y, src2dst, topk_weights, apply_router_weight_on_input=False, out=None,
                             stream=None):
    """Unpermute + top-k weight-and-reduce: bf16 [M, K]."""
    _dt(y, torch.bfloat16, "y")
    M, topk = src2dst.shape
    K = y.shape[1]
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16, device=y.device)
    _check("moe_gather_weight_reduce", lib().moe_gather_weight_reduce(
        _ptr(y), _ptr(src2dst), _ptr(topk_weights), M, topk, K, int(bool(apply_router_weight_on_input)),
        _ptr(out), _stream(stream)))
    return out


def moe_forward_chunked(hidden_states, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, E,
                        expert_map=None, chunk_size=None, apply_router_weight_on_input=False, out=None,
                        workspace=None, err_count=None, stream=None):
    """The whole MoE layer under the chunking loop: bf16 [M, K]. topk_ids is int32 or int64."""
    _dt(hidden_states, torch.bfloat16, "hidden_states")
    fn = _ids_entry("moe_forward_chunked", topk_ids)
    _dt(topk_weights, torch.float32, "topk_weights")
    M, K = hidden_states.shape
    El, N2, _ = w13.shape
    topk = topk_ids.shape[1]
    chunk = M if chunk_size is None else int(chunk_size)
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16, device=hidden_states.device)
    if workspace is None:
        workspace = torch.empty(max(1, moe_workspace_size(max(1, min(chunk, M)), K, N2 // 2, topk, El)),
                                dtype=torch.uint8, device=hidden_states.device)
    _check(fn, getattr(lib(), fn)(
        _ptr(hidden_states), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13), _ptr(w13_scale), _ptr(w2),
        _ptr(w2_scale), _ptr(expert_map), E, El, M, K, N2 // 2, topk, max(1, chunk),
        int(bool(apply_router_weight_on_input)), _ptr(out), _ptr(workspace), workspace.numel(),
        _ptr(err_count), _stream(stream)))
    return out


def _hptr(t: torch.Tensor):
    """Address of a page-locked, contiguous host tensor."""
    if t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if not t.is_pinned():
        raise ValueError("expected a pinned (page-locked) host tensor")
    return ctypes.c_void_p(t.data_ptr())


def _event(done):
    if done is None:
        return None
    if done.cuda_event == 0:  # torch creates the CUDA event lazily, on its first record
        done.record()
    return ctypes.c_void_p(done.cuda_event)


def moe_host_workspace_size(M: int, K: int, N: int, topk: int, local_num_experts: int, chunk_size: int) -> int:
    return int(lib().moe_host_workspace_size(M, K, N, topk, local_num_experts, chunk_size))


def moe_forward_host(hidden_states, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, E, expert_map=None,
                     chunk_size=None, apply_router_weight_on_input=False, out=None, workspace=None, err_count=None,
                     stream=None, done=None):
    """The layer with the batch in pinned HOST memory (hidden_states, topk_ids,
    topk_weights and out are pinned CPU tensors); asynchronous: `out` holds the result
    once the torch.cuda.Event `done` has completed, or once the stream has passed a later
    moe_host_wait(). topk_ids is int32 or int64."""
    _dt(hidden_states, torch.bfloat16, "hidden_states")
    fn = _ids_entry("moe_forward_host", topk_ids)
    _dt(topk_weights, torch.float32, "topk_weights")
    M, K = hidden_states.shape
    El, N2, _ = w13.shape
    topk = topk_ids.shape[1]
    chunk = M if chunk_size is None else int(chunk_size)
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16).pin_memory()
    if workspace is None:
        workspace = torch.empty(max(1, moe_host_workspace_size(max(1, M), K, N2 // 2, topk, El, max(1, chunk))),
                                dtype=torch.uint8, device=w13.device)
    _check(fn, getattr(lib(), fn)(
        _hptr(hidden_states), _hptr(topk_ids), _hptr(topk_weights), _ptr(w13), _ptr(w13_scale), _ptr(w2),
        _ptr(w2_scale), _ptr(expert_map), E, El, M, K, N2 // 2, topk, max(1, chunk),
        int(bool(apply_router_weight_on_input)), _hptr(out), _ptr(workspace), workspace.numel(),
        _ptr(err_count), _stream(stream), _event(done)))
    return out


def moe_host_wait(stream=None):
    """Orders `stream` after every output copy moe_forward_host has enqueued so far."""
    _check("moe_host_wait", lib().moe_host_wait(_stream(stream)))


def moe_ep_combine(partials, out=None, stream=None):
    """Sum of the ranks' partial layer outputs (bf16 [M, K] CUDA tensors, in rank order):
    fp32 accumulation in ascending rank order, one rounding to bf16."""
    if not partials:
        raise ValueError("moe_ep_combine: no partial outputs")
    for p in partials:
        _dt(p, torch.bfloat16, "partials")
    M, K = partials[0].shape
    if any(tuple(p.shape) != (M, K) for p in partials):
        raise ValueError("moe_ep_combine: partial outputs of different shapes")
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16, device=partials[0].device)
    arr = (ctypes.c_void_p * len(partials))(*[_ptr(p).value for p in partials])
    _check("moe_ep_combine", lib().moe_ep_combine(arr, len(partials), M, K, _ptr(out), _stream(stream)))
    return out
