"""Seeded synthetic inputs for the fused-MoE layer (hidden states, routing, FP8 weights).

This module is shared by the CUDA path's tests/bench and by the CPU oracle. It holds
none of the layer's own arithmetic (counting, permutation, activation quantisation,
GEMMs, activation, reduction): it only draws the layer's *inputs*, the way a model
checkpoint and a router would hand them over.

* Hidden states: N(0, 1), rounded to bf16 (returned as uint16 bit patterns).
* Router: logits N(0, 1) [+ a Zipf popularity bias], softmax in fp32, top-k with ties
  going to the lower expert id, the k weights renormalised to sum to 1 in fp32.
  The router itself is upstream of the fused-MoE kernels on the vLLM pages (the experts
  receive ``topk_ids``/``topk_weights``), so it is input generation here.
* Weights: N(0, 0.02) fp32, quantised per 128x128 block to FP8 e4m3 with an fp32 scale
  amax/448 -- the "-FP8" checkpoint format with ``--block-shape 128 128`` named in vLLM
  PR #20903 "[Kernel] DeepGemm MoE : Integrate triton permute / unpermute kernels",
  section "Optimizations". The cast uses torch's own float8_e4m3fn conversion (a library
  routine), so neither the oracle's nor the kernels' encoder is involved.

Everything is CPU-side numpy/torch; nothing here touches a GPU.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

BLOCK = 128  # the 128x128 weight block and the 1x128 activation group


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic MoE-layer problem, named by what it is."""
    name: str
    M: int                 # tokens
    K: int                 # hidden size
    N: int                 # moe intermediate size (0: permute/unpermute only)
    E: int                 # global experts
    topk: int
    seed: int
    zipf_s: float = 0.0    # 0: unbiased N(0,1) logits
    local_experts: Optional[int] = None  # experts [0, local_experts) are local, the rest -1
    chunk_size: Optional[int] = None     # None: one chunk
    apply_router_weight_on_input: bool = False

    @property
    def El(self) -> int:
        return self.E if self.local_experts is None else self.local_experts

    @property
    def chunk(self) -> int:
        return self.M if self.chunk_size is None else self.chunk_size


# The workloads: a tiny layer, a permute/unpermute-only pass, a
# Qwen3-30B-A3B-shaped layer (hidden 2048, moe intermediate 768, 128 experts, top-8)
# at decode size, at prefill size with skewed routing, and chunked with half the
# experts local, and a count-only pass over 2^20 tokens (33.5 MB of top-8 ids, large
# enough for the count kernel's bandwidth to mean something).
TINY = Workload("tiny_m64_k256_n256_e8_top2", M=64, K=256, N=256, E=8, topk=2, seed=0)
PERMUTE_ONLY = Workload("permute_only_m4096_k2048_e128_top8", M=4096, K=2048, N=0,
                        E=128, topk=8, seed=2)
QWEN3_DECODE = Workload("qwen3_30b_a3b_decode_m64", M=64, K=2048, N=768, E=128,
                        topk=8, seed=3)
QWEN3_PREFILL = Workload("qwen3_30b_a3b_prefill_m8192_zipf1.2", M=8192, K=2048, N=768,
                         E=128, topk=8, seed=4, zipf_s=1.2)
QWEN3_CHUNKED = Workload("qwen3_30b_a3b_chunked_m16385_c128_local64_zipf1.2", M=16385,
                         K=2048, N=768, E=128, topk=8, seed=5, zipf_s=1.2,
                         local_experts=64, chunk_size=128)
COUNT_ONLY = Workload("count_only_m1048576_e128_top8", M=1 << 20, K=128, N=0, E=128, topk=8,
                      seed=6)
# The same count pass over 2^23 tokens (268 MB of ids, twice the L2): its ids are the 2^20
# routing repeated eight times, so every step streams them from DRAM without an L2 flush.
COUNT_ONLY_LARGE = Workload("count_only_m8388608_e128_top8", M=1 << 23, K=128, N=0, E=128,
                            topk=8, seed=6)
WORKLOADS = {w.name: w for w in (TINY, PERMUTE_ONLY, QWEN3_DECODE, QWEN3_PREFILL,
                                 QWEN3_CHUNKED, COUNT_ONLY, COUNT_ONLY_LARGE)}


def is_count_only(wl: Workload) -> bool:
    return wl.name in (COUNT_ONLY.name, COUNT_ONLY_LARGE.name)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round-to-nearest-even, via torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def hidden_states(M: int, K: int, seed: int) -> np.ndarray:
    """bf16 [M, K] as uint16 bits, values ~ N(0, 1)."""
    return bf16_bits(_rng(seed, 1).standard_normal((M, K), dtype=np.float32))


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """log-popularity bias: expert popularity ~ rank^-s over a seeded permutation."""
    if s == 0.0:
        return np.zeros(E, np.float32)
    perm = _rng(seed, 2).permutation(E)          # perm[e] = rank-1 of expert e
    p = (perm + 1.0) ** (-s)
    p = p / p.sum()
    return np.log(p).astype(np.float32)


def route(M: int, E: int, topk: int, seed: int, zipf_s: float = 0.0):
    """Router outputs: topk_ids int32 [M, topk], topk_weights fp32 [M, topk]."""
    logits = _rng(seed, 3).standard_normal((M, E), dtype=np.float32)
    logits = logits + zipf_bias(E, zipf_s, seed)[None, :]
    probs = torch.softmax(torch.from_numpy(logits), dim=-1).numpy()
    # stable sort of -p: equal probabilities keep ascending expert id
    ids = np.argsort(-probs, axis=1, kind="stable")[:, :topk].astype(np.int32)
    w = np.take_along_axis(probs, ids, axis=1).astype(np.float32)
    w = (w / w.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(w)


def count_only_routing(wl: Workload):
    """The count-only workloads' top-k ids and weights: the 2^20-token routing of the
    workload's seed, repeated to the workload's M (a multiple of 2^20)."""
    ids, w = route(COUNT_ONLY.M, wl.E, wl.topk, wl.seed, wl.zipf_s)
    reps = wl.M // COUNT_ONLY.M
    if reps <= 1:
        return ids, w
    return np.ascontiguousarray(np.tile(ids, (reps, 1))), np.ascontiguousarray(np.tile(w, (reps, 1)))


def expert_map(E: int, local: Optional[int]) -> Optional[np.ndarray]:
    """Global id -> local id; experts [0, local) are this GPU's, the rest -1."""
    if local is None:
        return None
    m = np.full(E, -1, np.int32)
    m[:local] = np.arange(local, dtype=np.int32)
    return m


def random_expert_map(E: int, local: int, seed: int) -> np.ndarray:
    """A seeded random subset of `local` experts, numbered in ascending global id."""
    m = np.full(E, -1, np.int32)
    chosen = np.sort(_rng(seed, 4).choice(E, size=local, replace=False))
    m[chosen] = np.arange(local, dtype=np.int32)
    return m


def block_quant_weights(w: torch.Tensor):
    """fp32 [..., R, C] (R, C multiples of 128) -> (e4m3 codes uint8, fp32 scales
    [..., R/128, C/128]) with scale = amax/448 per 128x128 block."""
    *lead, R, C = w.shape
    b = w.reshape(*lead, R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    amax = b.abs().amax(dim=(-3, -1))                       # [..., R/128, C/128]
    scale = amax / 448.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    q = (b / safe[..., :, None, :, None]).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(*lead, R, C)
    return codes.numpy(), scale.to(torch.float32).numpy()


def expert_weights(E: int, rows: int, cols: int, seed: int, stream: int, std=0.02):
    """FP8 e4m3 weights [E, rows, cols] + fp32 block scales [E, rows/128, cols/128].
    Drawn expert by expert from one seeded torch generator."""
    g = torch.Generator().manual_seed(seed * 1000 + stream)
    codes = np.empty((E, rows, cols), np.uint8)
    scales = np.empty((E, rows // BLOCK, cols // BLOCK), np.float32)
    for e in range(E):
        w = torch.randn(rows, cols, generator=g, dtype=torch.float32) * std
        codes[e], scales[e] = block_quant_weights(w)
    return codes, scales


@dataclasses.dataclass
class LayerInputs:
    wl: Workload
    x: np.ndarray                  # bf16 bits [M, K]
    topk_ids: np.ndarray           # int32 [M, topk]
    topk_weights: np.ndarray       # fp32 [M, topk]
    expert_map: Optional[np.ndarray]  # int32 [E] or None
    w13: Optional[np.ndarray] = None  # e4m3 [El, 2N, K]
    w13_scale: Optional[np.ndarray] = None  # fp32 [El, 2N/128, K/128]
    w2: Optional[np.ndarray] = None   # e4m3 [El, K, N]
    w2_scale: Optional[np.ndarray] = None   # fp32 [El, K/128, N/128]


def make_layer_inputs(wl: Workload, with_weights: bool = True) -> LayerInputs:
    x = hidden_states(wl.M, wl.K, wl.seed)
    ids, w = route(wl.M, wl.E, wl.topk, wl.seed, wl.zipf_s)
    li = LayerInputs(wl, x, ids, w, expert_map(wl.E, wl.local_experts))
    if with_weights and wl.N > 0:
        li.w13, li.w13_scale = expert_weights(wl.El, 2 * wl.N, wl.K, wl.seed, 13)
        li.w2, li.w2_scale = expert_weights(wl.El, wl.K, wl.N, wl.seed, 2)
    return li
