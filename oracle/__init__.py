"""CPU oracle of the fused-MoE layer hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg and
reference arm may import this package. The CUDA path never imports it, and it imports nothing from the
CUDA path: the two share only the seeded input generators of ``moe_inputs``.

The arithmetic lives in ``moe_oracle.c`` (plain C, built with gcc by ``build.py``);
this module only marshals numpy arrays into it. Each function's docstring names the
step of the vLLM pull-request pages it follows (see the header of ``moe_oracle.c``).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` against
hand-worked examples (``tests/golden/``), closed forms, invariants and independent
library routines.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
GROUP = 128

_libs = {}


def lib(parallel: bool = False) -> ctypes.CDLL:
    """The single-threaded oracle (the checker), or with parallel=True its OpenMP build
    (the timed CPU baseline; identical results)."""
    if parallel not in _libs:
        L = ctypes.CDLL(_build.build(parallel=parallel))
        _declare(L)
        _libs[parallel] = L
    return _libs[parallel]


def num_threads(parallel: bool = True) -> int:
    """Host threads the oracle's row loop runs on."""
    return int(lib(parallel).oracle_num_threads())


_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def _declare(L):
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.restype = ctypes.c_float
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_quant_row.argtypes = [_p, _int, _p, _p]
    L.oracle_quant_row.restype = None
    L.oracle_count.argtypes = [_p, _i64, _int, _p, _int, _int, _p]
    L.oracle_count.restype = _i64
    L.oracle_offsets.argtypes = [_p, _int, _p]
    L.oracle_offsets.restype = None
    L.oracle_rp_cap.argtypes = [_i64, _int, _int]
    L.oracle_rp_cap.restype = _i64
    L.oracle_scatter.argtypes = [_p, _i64, _int, _p, _p, _int, _p, _int, _int, _int, _int,
                                 _p, _p, _p, _p]
    L.oracle_scatter.restype = _i64
    L.oracle_grouped_gemm.argtypes = [_p, _p, _p, _p, _p, _p, _int, _int, _int, _p]
    L.oracle_grouped_gemm.restype = None
    L.oracle_silu_mul_quant.argtypes = [_p, _p, _p, _int, _int, _p, _p]
    L.oracle_silu_mul_quant.restype = None
    L.oracle_gather.argtypes = [_p, _p, _p, _i64, _int, _int, _int, _p]
    L.oracle_gather.restype = None
    L.oracle_forward_chunked.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _int, _int, _i64,
                                         _int, _int, _int, _i64, _int, _p]
    L.oracle_forward_chunked.restype = _i64
    L.oracle_forward_token.argtypes = [_i64, _p, _p, _p, _p, _p, _p, _p, _p, _int, _int,
                                       _int, _int, _int, _int, _p]
    L.oracle_forward_token.restype = None
    L.oracle_ep_combine.argtypes = [_p, _int, _i64, _int, _p]
    L.oracle_ep_combine.restype = None
    L.oracle_num_threads.argtypes = []
    L.oracle_num_threads.restype = _int


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ids(topk_ids) -> np.ndarray:
    """Top-k ids as int64 (the C side takes 64-bit ids; int32 ids widen exactly)."""
    a = np.asarray(topk_ids)
    if a.dtype.kind not in "iu":
        raise TypeError(f"topk_ids: expected an integer array, got {a.dtype}")
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------- formats
def e4m3_decode(code: int) -> float:
    """FP8 E4M3 value of one code, from the format definition."""
    return float(lib().oracle_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    """FP8 E4M3 code of an fp32 value: nearest, ties to even, saturating at +-448."""
    return int(lib().oracle_e4m3_encode(float(v)))


def quant_rows(x: np.ndarray):
    """1x128 quantisation of fp32 rows [R, K] -> (codes uint8 [R, K], scales fp32 [R, K/128])."""
    x = _c(x, np.float32)
    R, K = x.shape
    q = np.zeros((R, K), np.uint8)
    s = np.zeros((R, K // GROUP), np.float32)
    for r in range(R):
        lib().oracle_quant_row(_ptr(x[r]), K, _ptr(q[r]), _ptr(s[r]))
    return q, s


# ----------------------------------------------------------------------- the steps
def count(topk_ids, E, El, expert_map=None):
    """Step a1: tokens per local expert. Returns (counts int32 [El], n_bad_ids)."""
    ids = _ids(topk_ids)
    M, topk = ids.shape
    m = None if expert_map is None else _c(expert_map, np.int32)
    counts = np.zeros(El, np.int32)
    bad = lib().oracle_count(_ptr(ids), M, topk, _ptr(m), E, El, _ptr(counts))
    return counts, int(bad)


def offsets(counts):
    """Expert block starts, each a multiple of 128: int32 [El + 1]."""
    c = _c(counts, np.int32)
    off = np.zeros(len(c) + 1, np.int32)
    lib().oracle_offsets(_ptr(c), len(c), _ptr(off))
    return off


def rp_cap(Mc, topk, El) -> int:
    """Row bound of the permuted workspace for a chunk of Mc tokens."""
    return int(lib().oracle_rp_cap(Mc, topk, El))


def scatter(x_bits, topk_ids, topk_weights, E, El, expert_map=None,
            apply_router_weight_on_input=False, quant=True):
    """Step a2. Returns dict(a, a_scale, offsets, src2dst, bad); a is uint8 [Rp, K]
    (FP8 codes) when quant else uint16 bf16 bits [Rp, K]; padding rows are zero."""
    x = _c(x_bits, np.uint16)
    ids = _ids(topk_ids)
    w = _c(topk_weights, np.float32)
    M, K = x.shape
    topk = ids.shape[1]
    m = None if expert_map is None else _c(expert_map, np.int32)
    counts, _ = count(ids, E, El, m)
    Rp = int(offsets(counts)[-1])
    a = np.zeros((Rp, K), np.uint8 if quant else np.uint16)
    s = np.zeros((Rp, K // GROUP), np.float32)
    off = np.zeros(El + 1, np.int32)
    s2d = np.zeros((M, topk), np.int32)
    bad = lib().oracle_scatter(_ptr(x), M, K, _ptr(ids), _ptr(w), topk, _ptr(m), E, El,
                               int(bool(apply_router_weight_on_input)), int(bool(quant)),
                               _ptr(a), _ptr(s), _ptr(off), _ptr(s2d))
    return dict(a=a, a_scale=s, offsets=off, src2dst=s2d, counts=counts, bad=int(bad))


def grouped_gemm(a, a_scale, W, w_scale, offs, counts):
    """Steps a3/a5: block-scaled FP8 grouped GEMM over the kept rows, fp64 [Rp, Nout]."""
    a = _c(a, np.uint8)
    sa = _c(a_scale, np.float32)
    W = _c(W, np.uint8)
    sw = _c(w_scale, np.float32)
    offs = _c(offs, np.int32)
    counts = _c(counts, np.int32)
    El, Nout, Kin = W.shape
    C = np.zeros((a.shape[0], Nout), np.float64)
    lib().oracle_grouped_gemm(_ptr(a), _ptr(sa), _ptr(W), _ptr(sw), _ptr(offs), _ptr(counts),
                              El, Nout, Kin, _ptr(C))
    return C


def silu_mul_quant(c1_f32, offs, counts):
    """Step a4: h = silu(gate) * up, then 1x128 FP8 requantisation (kept rows only)."""
    c1 = _c(c1_f32, np.float32)
    R, N2 = c1.shape
    N = N2 // 2
    offs = _c(offs, np.int32)
    counts = _c(counts, np.int32)
    H = np.zeros((R, N), np.uint8)
    hs = np.zeros((R, N // GROUP), np.float32)
    lib().oracle_silu_mul_quant(_ptr(c1), _ptr(offs), _ptr(counts), len(counts), N, _ptr(H),
                                _ptr(hs))
    return H, hs


def gather(Y_bits, src2dst, topk_weights, apply_router_weight_on_input=False):
    """Step a6: unpermute + top-k weight-and-reduce, bf16 bits [M, K]."""
    Y = _c(Y_bits, np.uint16)
    s2d = _c(src2dst, np.int32)
    w = _c(topk_weights, np.float32)
    M, topk = s2d.shape
    K = Y.shape[1]
    out = np.zeros((M, K), np.uint16)
    lib().oracle_gather(_ptr(Y), _ptr(s2d), _ptr(w), M, topk, K,
                        int(bool(apply_router_weight_on_input)), _ptr(out))
    return out


def forward_chunked(x_bits, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, E,
                    expert_map=None, chunk_size=None, apply_router_weight_on_input=False, parallel=False):
    """Step a7: the whole layer under the chunking loop, bf16 bits [M, K] (parallel=True:
    the OpenMP build, same result)."""
    x = _c(x_bits, np.uint16)
    ids = _ids(topk_ids)
    w = _c(topk_weights, np.float32)
    w13 = _c(w13, np.uint8)
    s13 = _c(w13_scale, np.float32)
    w2 = _c(w2, np.uint8)
    s2 = _c(w2_scale, np.float32)
    m = None if expert_map is None else _c(expert_map, np.int32)
    M, K = x.shape
    El, N2, _ = w13.shape
    topk = ids.shape[1]
    chunk = M if chunk_size is None else int(chunk_size)
    out = np.zeros((M, K), np.uint16)
    bad = lib(parallel).oracle_forward_chunked(_ptr(x), _ptr(ids), _ptr(w), _ptr(w13), _ptr(s13),
                                       _ptr(w2), _ptr(s2), _ptr(m), E, El, M, K, N2 // 2, topk,
                                       max(chunk, 1), int(bool(apply_router_weight_on_input)),
                                       _ptr(out))
    if bad < 0:
        raise ValueError("oracle_forward_chunked: bad arguments")
    return out


def forward_tokens(tokens, x_bits, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, E,
                   expert_map=None, apply_router_weight_on_input=False):
    """The layer output of selected tokens, evaluated per token with no permutation.
    Returns bf16 bits [len(tokens), K]."""
    x = _c(x_bits, np.uint16)
    ids = _ids(topk_ids)
    w = _c(topk_weights, np.float32)
    w13 = _c(w13, np.uint8)
    s13 = _c(w13_scale, np.float32)
    w2 = _c(w2, np.uint8)
    s2 = _c(w2_scale, np.float32)
    m = None if expert_map is None else _c(expert_map, np.int32)
    K = x.shape[1]
    El, N2, _ = w13.shape
    topk = ids.shape[1]
    out = np.zeros((len(tokens), K), np.uint16)
    for i, t in enumerate(tokens):
        lib().oracle_forward_token(int(t), _ptr(x), _ptr(ids), _ptr(w), _ptr(w13), _ptr(s13),
                                   _ptr(w2), _ptr(s2), _ptr(m), E, El, K, N2 // 2, topk,
                                   int(bool(apply_router_weight_on_input)), _ptr(out[i]))
    return out


def ep_combine(parts):
    """Expert-parallel combine: the sum of the ranks' partial outputs (bf16 bits [M, K]
    each, in rank order), fp32 in ascending rank order, one rounding to bf16."""
    ps = [_c(p, np.uint16) for p in parts]
    M, K = ps[0].shape
    arr = (ctypes.c_void_p * len(ps))(*[p.ctypes.data for p in ps])
    out = np.zeros((M, K), np.uint16)
    lib().oracle_ep_combine(arr, len(ps), M, K, _ptr(out))
    return out
