"""Pins of the CPU oracle to things other than itself.

Hand-worked fixtures (tests/golden/), closed forms, invariants, the special cases that
reduce to a library routine (torch's float8_e4m3fn cast, numpy's stable sort / bincount
/ fp64 matmul, scipy's logistic function), and brute force on tiny inputs. Each test is
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, swapped gate/up halves, an unstable order) fails at least one.
No GPU is used.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import moe_inputs as mi
from conftest import read_golden

G = 128


def torch_e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def torch_f32_to_e4m3(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def bf16_round(v: np.ndarray) -> np.ndarray:
    """fp32 values rounded to bf16 (returned as fp32), via torch's cast."""
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16).float().numpy()


# ------------------------------------------------------------------------ E4M3 format
def test_e4m3_golden_codes():
    for code_hex, val in read_golden("e4m3_codes.txt"):
        got = oracle.e4m3_decode(int(code_hex, 16))
        if val == "nan":
            assert math.isnan(got), code_hex
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code_hex


def test_e4m3_golden_rounding():
    for v, code_hex in read_golden("e4m3_rounding.txt"):
        assert oracle.e4m3_encode(float(v)) == int(code_hex, 16), v


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_e4m3_to_f32(codes)
    got = np.array([oracle.e4m3_decode(c) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan].view(np.uint32) == ref[~nan].view(np.uint32)).all()


def test_e4m3_roundtrip_all_codes():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(7)
    # log-uniform magnitudes across the whole range incl. subnormals, both signs,
    # below the 464 midpoint where torch's (non-saturating) cast and ours agree
    mag = np.exp(rng.uniform(np.log(1e-4), np.log(463.0), 20000)).astype(np.float32)
    v = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    # exact midpoints between neighbouring codes exercise ties-to-even
    vals = np.sort(torch_e4m3_to_f32(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((vals[1:].astype(np.float64) + vals[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ref = torch_f32_to_e4m3(v)
    got = np.array([oracle.e4m3_encode(x) for x in v], np.uint8)
    assert (got == ref).all()


def test_e4m3_encode_is_nearest_by_brute_force():
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    fv = np.array([oracle.e4m3_decode(c) for c in finite], np.float64)
    rng = np.random.default_rng(8)
    for x in rng.uniform(-460, 460, 500).astype(np.float32):
        d = np.abs(fv - float(x))
        best = finite[d == d.min()]
        got = oracle.e4m3_encode(float(x))
        if len(best) == 1:
            assert got == best[0]
        else:  # a tie (or +-0): the even mantissa wins
            assert got in best and (got & 1) == 0


# ------------------------------------------------------------------ 1x128 quantisation
def test_quant_constant_rows():
    for v in (1.0, -3.25, 1e-3, 300.0):
        q, s = oracle.quant_rows(np.full((1, 256), v, np.float32))
        assert (q == (0x7E if v > 0 else 0xFE)).all()
        assert (s == np.float32(abs(v)) / np.float32(448)).all()


def test_quant_zero_row_and_exact_powers():
    q, s = oracle.quant_rows(np.zeros((1, 128), np.float32))
    assert (q == 0).all() and (s == 0).all()
    # amax 448 -> scale exactly 1: codes are the plain e4m3 encodings
    x = np.zeros((1, 128), np.float32)
    x[0, :6] = [448.0, 224.0, 1.0, -1.0, 0.5, 16.0]
    q, s = oracle.quant_rows(x)
    assert s[0, 0] == 1.0
    assert list(q[0, :6]) == [0x7E, 0x76, 0x38, 0xB8, 0x30, 0x58]
    assert (q[0, 6:] == 0).all()


def test_quant_groups_are_independent_and_match_torch():
    rng = np.random.default_rng(9)
    x = bf16_round(rng.standard_normal((16, 512)).astype(np.float32) * rng.uniform(0.01, 10, (16, 1)))
    x[3, 128:256] = 0.0
    q, s = oracle.quant_rows(x)
    xg = x.reshape(16, 4, 128)
    amax = np.abs(xg).max(axis=2)
    s_ref = (amax / np.float32(448.0)).astype(np.float32)
    assert (s.view(np.uint32) == s_ref.view(np.uint32)).all()
    safe = np.where(s_ref > 0, s_ref, np.float32(1))
    q_ref = torch_f32_to_e4m3((xg / safe[:, :, None]).astype(np.float32)).reshape(16, 512)
    assert (q == q_ref).all()


# ------------------------------------------------------------------- count / offsets
def _golden_route():
    d = {r[0]: [int(v) for v in r[1:]] for r in read_golden("route_small.txt")}
    return d


def test_count_offsets_scatter_golden():
    d = _golden_route()
    ids = np.array(d["topk_ids"], np.int32).reshape(3, 2)
    x = mi.bf16_bits(np.arange(3 * 128, dtype=np.float32).reshape(3, 128) / 64.0)
    w = np.full((3, 2), 0.5, np.float32)
    for case, E, El, m in (("A", 4, 4, None), ("B", 4, 2, np.array(d["B.expert_map"], np.int32))):
        counts, bad = oracle.count(ids, E, El, m)
        assert bad == 0
        assert list(counts) == d[f"{case}.counts"]
        assert list(oracle.offsets(counts)) == d[f"{case}.offsets"]
        r = oracle.scatter(x, ids, w, E, El, m, quant=False)
        assert list(r["src2dst"].reshape(-1)) == d[f"{case}.src2dst"]
        assert list(r["offsets"]) == d[f"{case}.offsets"]


@pytest.mark.parametrize("M,topk,E,local", [(1, 1, 1, None), (127, 2, 8, None), (129, 8, 128, None),
                                            (1000, 8, 128, 64), (300, 4, 16, "random")])
def test_count_matches_bincount_and_sums(M, topk, E, local):
    ids, _ = mi.route(M, E, topk, seed=M)
    if local == "random":
        m = mi.random_expert_map(E, 5, seed=3)
        El = 5
    else:
        m = mi.expert_map(E, local)
        El = E if local is None else local
    counts, bad = oracle.count(ids, E, El, m)
    assert bad == 0
    loc = ids.reshape(-1) if m is None else m[ids.reshape(-1)]
    loc = loc[loc >= 0]
    assert (counts == np.bincount(loc, minlength=El)).all()
    if m is None:
        assert counts.sum() == M * topk
    else:
        assert counts.sum() == int((m[ids] >= 0).sum())


def test_count_bad_ids_are_dropped_and_counted():
    ids = np.array([[0, -1], [5, 1], [-7, 1]], np.int32)
    counts, bad = oracle.count(ids, 4, 4)
    assert list(counts) == [1, 2, 0, 0] and bad == 2


def test_int64_ids_are_not_truncated():
    """64-bit top-k ids follow the same rule: kept when in [0, E), -1 silent, anything
    else dropped and counted. An id that would alias a small expert if cut to 32 bits
    (2**32 + 1 -> 1) must be dropped, not counted for that expert."""
    ids = np.array([[2**32 + 1, 1], [-1, 2**33], [-(2**32) + 2, 3], [2**62, 0]], np.int64)
    counts, bad = oracle.count(ids, 4, 4)
    assert list(counts) == [1, 1, 0, 1] and bad == 4
    x = mi.bf16_bits(np.ones((4, 128), np.float32))
    r = oracle.scatter(x, ids, np.full((4, 2), 0.5, np.float32), 4, 4, quant=False)
    # kept slots (flat 1, 5, 7) in stable order within their experts; the rest dropped
    assert list(r["src2dst"].reshape(-1)) == [-1, 128, -1, -1, -1, 256, -1, 0]
    assert r["bad"] == 4
    # ids that fit in 32 bits give the same answer from int32 and int64 arrays
    small = np.array([[0, 3], [2, -1], [9, 1]], np.int64)
    for got, want in zip(oracle.count(small, 4, 4), oracle.count(small.astype(np.int32), 4, 4)):
        assert np.array_equal(got, want)


def test_offsets_closed_form_and_rp_cap_bound():
    rng = np.random.default_rng(1)
    for _ in range(50):
        El = int(rng.integers(1, 200))
        counts = rng.integers(0, 400, El).astype(np.int32)
        counts[rng.random(El) < 0.3] = 0
        off = oracle.offsets(counts)
        assert off[0] == 0 and (off % 128 == 0).all()
        assert (np.diff(off) >= counts).all() and (np.diff(off) - counts < 128).all()
        assert off[-1] == sum(-(-int(c) // 128) * 128 for c in counts)
    # rp_cap: hand-evaluated roundup128(Mc*topk + min(El, Mc*topk) * 127)
    for (Mc, topk, El), cap in {(1, 8, 64): 1024, (128, 8, 64): 9216, (64, 8, 128): 16768,
                                (8192, 8, 128): 81792, (3, 2, 1): 256}.items():
        assert oracle.rp_cap(Mc, topk, El) == cap
        # the widest spread (every expert one slot more than a multiple of 128) fits
        n = Mc * topk
        spread = np.zeros(El, np.int32)
        for i in range(n):
            spread[i % El] += 1
        assert oracle.offsets(spread)[-1] <= cap


# ------------------------------------------------------------------------- scatter
@pytest.mark.parametrize("local", [None, 64, "random"])
def test_scatter_is_the_stable_order(local):
    M, topk, E, K = 300, 8, 128, 128
    ids, w = mi.route(M, E, topk, seed=11, zipf_s=1.2)
    if local == "random":
        m, El = mi.random_expert_map(E, 40, seed=2), 40
    else:
        m, El = mi.expert_map(E, local), (E if local is None else local)
    x = mi.hidden_states(M, K, seed=5)
    r = oracle.scatter(x, ids, w, E, El, m, quant=False)
    s2d = r["src2dst"].reshape(-1)
    loc = ids.reshape(-1) if m is None else m[ids.reshape(-1)]
    keep = loc >= 0
    assert (s2d[~keep] == -1).all()
    # unique stable order: numpy's stable argsort on the local expert id
    flat = np.nonzero(keep)[0]
    order = flat[np.argsort(loc[flat], kind="stable")]
    counts = np.bincount(loc[flat], minlength=El)
    off = oracle.offsets(counts)
    expect = np.empty(len(order), np.int64)
    pos = 0
    for l in range(El):
        expect[pos:pos + counts[l]] = off[l] + np.arange(counts[l])
        pos += counts[l]
    got = np.full(M * topk, -1, np.int64)
    got[order] = expect
    assert (s2d == got).all()
    # copied rows: row dst of the bf16 buffer is x[t]
    a = r["a"]
    for i in flat[:200]:
        assert (a[s2d[i]] == x[i // topk]).all()


def test_scatter_gather_identity_bf16():
    """quant off, identity experts (Y = A), weights summing to 1: gather(scatter(x)) == x."""
    M, topk, E, K = 257, 8, 16, 256
    ids, w = mi.route(M, E, topk, seed=4)
    x = mi.hidden_states(M, K, seed=6)
    r = oracle.scatter(x, ids, w, E, E, quant=False)
    out = oracle.gather(r["a"], r["src2dst"], w)
    assert (out == x).all()


def test_scatter_gather_identity_fp8():
    """With FP8 1x128 quant and experts Y = bf16(dequant(A)), the layer gives
    bf16(dequant(quant(x))), quant done here with torch's e4m3 cast."""
    M, topk, E, K = 200, 4, 8, 384
    ids, w = mi.route(M, E, topk, seed=12)
    x = mi.hidden_states(M, K, seed=13)
    r = oracle.scatter(x, ids, w, E, E, quant=True)
    a, sa = r["a"], r["a_scale"]
    Y = mi.bf16_bits(torch_e4m3_to_f32(a) * np.repeat(sa, 128, axis=1))
    out = oracle.gather(Y, r["src2dst"], w)
    xf = mi.bf16_to_f32(x).reshape(M, K // 128, 128)
    s = (np.abs(xf).max(axis=2) / np.float32(448)).astype(np.float32)
    q = torch_e4m3_to_f32(torch_f32_to_e4m3((xf / s[:, :, None]).astype(np.float32)))
    ref = mi.bf16_bits((q * s[:, :, None]).reshape(M, K))
    # values, not bits: the fp32 accumulator starts at +0, so a -0 input comes back as +0
    assert (mi.bf16_to_f32(out) == mi.bf16_to_f32(ref)).all()


def test_apply_router_weight_on_input_topk1():
    M, K, E = 64, 128, 4
    ids, _ = mi.route(M, E, 1, seed=3)
    w = np.full((M, 1), 1.0, np.float32)
    x = mi.hidden_states(M, K, seed=3)
    r = oracle.scatter(x, ids, w, E, E, apply_router_weight_on_input=True, quant=False)
    assert (oracle.gather(r["a"], r["src2dst"], w * 7, apply_router_weight_on_input=True) == x).all()
    w2 = np.full((M, 1), 0.5, np.float32)
    r2 = oracle.scatter(x, ids, w2, E, E, apply_router_weight_on_input=True, quant=False)
    half = mi.bf16_bits(mi.bf16_to_f32(x) * 0.5)
    assert (oracle.gather(r2["a"], r2["src2dst"], w2, apply_router_weight_on_input=True) == half).all()


def test_gather_weights_and_dropped_slots():
    # two rows of Y, token 0 takes 0.25*Y0 + 0.75*Y1, token 1 has no kept slot
    Y = mi.bf16_bits(np.array([[4.0, -8.0], [2.0, 1.0]], np.float32))
    s2d = np.array([[0, 1], [-1, -1]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]], np.float32)
    out = mi.bf16_to_f32(oracle.gather(Y, s2d, w))
    assert list(out[0]) == [2.5, -1.25] and list(out[1]) == [0.0, 0.0]


def test_gather_sums_in_fp32_in_ascending_k():
    """Reading C8: the weighted rows are added in fp32 in ascending k. Rows 1, 2^-24, -1
    with weights 1: in ascending fp32 order 1 + 2^-24 rounds to 1 (a tie, to even) and
    the sum is 0; any other order (or an fp64 or pairwise sum) gives 2^-24."""
    Y = mi.bf16_bits(np.array([[1.0, 0.0], [2.0 ** -24, 0.0], [-1.0, 0.0]], np.float32))
    w = np.ones((1, 3), np.float32)
    assert mi.bf16_to_f32(oracle.gather(Y, np.array([[0, 1, 2]], np.int32), w))[0, 0] == 0.0
    # the same rows in descending order: -1 + 2^-24 is exact in fp32, + 1 leaves 2^-24
    assert mi.bf16_to_f32(oracle.gather(Y, np.array([[2, 1, 0]], np.int32), w))[0, 0] == np.float32(2.0 ** -24)


def test_gather_rounds_product_and_sum_separately():
    """Reading C8: each weighted row is rounded to fp32 before it is added (no fused
    multiply-add). The second product p = w1 * y1 lies just above 2^-24 (half an ulp of
    1.0) and rounds to exactly 2^-24, so 1 + fl(p) is a tie that rounds to 1 and the
    third row (-1) leaves 0; a fused 1 + p would round up to 1 + 2^-23 and leave 2^-23."""
    from fractions import Fraction
    y1 = np.float32(2.0 ** -24 * (1 + 2.0 ** -7))   # a bf16 value
    w1 = np.float32(0.9922481179237366)             # one fp32 step above 1/(1 + 2^-7)
    p = Fraction(float(w1)) * Fraction(float(y1))
    half_ulp = Fraction(2) ** -24
    assert half_ulp < p < half_ulp * (1 + Fraction(2) ** -24)   # exact product just above the tie
    assert np.float32(w1) * np.float32(y1) == np.float32(2.0 ** -24)
    Y = mi.bf16_bits(np.array([[1.0, 0.0], [float(y1), 0.0], [-1.0, 0.0]], np.float32))
    assert mi.bf16_to_f32(Y)[1, 0] == y1
    w = np.array([[1.0, w1, 1.0]], np.float32)
    assert mi.bf16_to_f32(oracle.gather(Y, np.array([[0, 1, 2]], np.int32), w))[0, 0] == 0.0


# --------------------------------------------------------------------------- GEMMs
def _dequant_weights(W, S):
    El, R, C = W.shape
    return torch_e4m3_to_f32(W).astype(np.float64) * np.repeat(np.repeat(S, 128, 1), 128, 2)


def test_grouped_gemm_single_expert_is_dense_matmul():
    """E=1, topk=1: the grouped GEMM reduces to one dense block-scaled GEMM; checked
    against numpy's fp64 matmul of the dequantised operands (Nout != Kin so that a
    transposed operand or a swapped scale index fails)."""
    rng = np.random.default_rng(3)
    R, Kin, Nout = 200, 384, 256
    x = rng.standard_normal((R, Kin)).astype(np.float32) * rng.uniform(0.1, 5, (R, 1)).astype(np.float32)
    a, sa = oracle.quant_rows(x)
    W, S = mi.block_quant_weights(torch.randn(1, Nout, Kin, generator=torch.Generator().manual_seed(1)))
    S = S * np.array([1.0, 3.0, 0.5], np.float32)[None, None, :]   # distinct per-block scales
    S = (S * np.array([1.0, 2.0], np.float32)[None, :, None]).astype(np.float32)
    offs = np.array([0, 256], np.int32)
    counts = np.array([R], np.int32)
    A = np.zeros((256, Kin), np.uint8)
    A[:R] = a
    SA = np.zeros((256, Kin // 128), np.float32)
    SA[:R] = sa
    C = oracle.grouped_gemm(A, SA, W, S, offs, counts)
    a_deq = torch_e4m3_to_f32(a).astype(np.float64) * np.repeat(sa, 128, axis=1)
    ref = a_deq @ _dequant_weights(W, S)[0].T
    np.testing.assert_allclose(C[:R], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert (C[R:] == 0).all()


def test_grouped_gemm_identity_weights_is_exact():
    """W = block-diagonal 1.0 codes with scale 1: C[r, j] = a_scale[r, j/128] * A[r, j]."""
    rng = np.random.default_rng(4)
    El, K = 3, 256
    counts = np.array([5, 0, 130], np.int32)
    offs = oracle.offsets(counts)
    R = int(offs[-1])
    x = rng.standard_normal((R, K)).astype(np.float32)
    A, SA = oracle.quant_rows(x)
    W = np.zeros((El, K, K), np.uint8)
    for l in range(El):
        np.fill_diagonal(W[l], 0x38)
    S = np.ones((El, 2, 2), np.float32)
    C = oracle.grouped_gemm(A, SA, W, S, offs, counts)
    exact = torch_e4m3_to_f32(A).astype(np.float64) * np.repeat(SA, 128, axis=1)
    for l in range(El):
        rows = slice(offs[l], offs[l] + counts[l])
        assert (C[rows] == exact[rows]).all()


def test_grouped_gemm_uses_each_experts_weights():
    """Two experts with weights scaled differently: rows of expert l see expert l only."""
    rng = np.random.default_rng(5)
    K, Nout = 128, 128
    counts = np.array([3, 4], np.int32)
    offs = oracle.offsets(counts)
    x = rng.standard_normal((256, K)).astype(np.float32)
    A, SA = oracle.quant_rows(x)
    W1, S1 = mi.block_quant_weights(torch.randn(1, Nout, K, generator=torch.Generator().manual_seed(2)))
    W = np.concatenate([W1, W1])
    S = np.concatenate([S1, S1 * 4]).astype(np.float32)
    C = oracle.grouped_gemm(A, SA, W, S, offs, counts)
    np.testing.assert_allclose(C[128:132], 4 * oracle.grouped_gemm(A, SA, W1.repeat(2, 0), S1.repeat(2, 0),
                                                                   offs, counts)[128:132], rtol=1e-12)


# --------------------------------------------------------------------------- SiLU
def test_silu_mul_quant_closed_forms():
    N = 128
    counts = np.array([4], np.int32)
    offs = oracle.offsets(counts)
    c1 = np.zeros((128, 2 * N), np.float32)
    c1[0, :N] = 0.0; c1[0, N:] = 5.0            # gate 0 -> h = 0
    c1[1, :N] = 1.0; c1[1, N:] = 2.0            # silu(1)*2, constant row
    c1[2, :N] = 2.0; c1[2, N:] = 1.0            # silu(2)*1 (catches swapped halves)
    rng = np.random.default_rng(6)
    c1[3] = rng.standard_normal(2 * N).astype(np.float32) * 3
    H, hs = oracle.silu_mul_quant(c1, offs, counts)
    assert (H[0] == 0).all() and hs[0, 0] == 0
    for r, (g, u) in ((1, (1.0, 2.0)), (2, (2.0, 1.0))):
        h = np.float32(g * expit(g) * u)
        assert (H[r] == 0x7E).all()
        assert hs[r, 0] == np.float32(h) / np.float32(448)
    g, u = c1[3, :N].astype(np.float64), c1[3, N:].astype(np.float64)
    h = (g * expit(g) * u).astype(np.float32)
    s = np.float32(np.abs(h).max()) / np.float32(448)
    assert hs[3, 0] == s
    assert (H[3] == torch_f32_to_e4m3(h / s)).all()


# ------------------------------------------------------------------------ the layer
@pytest.fixture(scope="module")
def tiny():
    return mi.make_layer_inputs(mi.TINY)


def test_layer_chunked_equals_per_token_brute_force(tiny):
    li = tiny
    E = li.wl.E
    args = (li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2, li.w2_scale, E)
    full = oracle.forward_chunked(*args)
    per_tok = oracle.forward_tokens(range(li.wl.M), *args)
    assert (full == per_tok).all()
    for chunk in (1, 7, 64, 100):
        assert (oracle.forward_chunked(*args, chunk_size=chunk) == full).all()
    assert np.abs(mi.bf16_to_f32(full)).max() > 0


def test_layer_local_experts_is_partial_sum(tiny):
    """Expert-parallel split: the outputs of two complementary expert_maps sum to the
    single-GPU output (up to bf16 rounding of each partial)."""
    li = tiny
    E = li.wl.E
    x, ids, w = li.x, li.topk_ids, li.topk_weights
    full = mi.bf16_to_f32(oracle.forward_chunked(x, ids, w, li.w13, li.w13_scale, li.w2, li.w2_scale, E))
    parts = []
    for lo in (0, 4):
        m = np.full(E, -1, np.int32)
        m[lo:lo + 4] = np.arange(4)
        sl = slice(lo, lo + 4)
        parts.append(mi.bf16_to_f32(oracle.forward_chunked(
            x, ids, w, li.w13[sl], li.w13_scale[sl], li.w2[sl], li.w2_scale[sl], E, expert_map=m)))
    np.testing.assert_allclose(parts[0] + parts[1], full, atol=2e-2 * np.abs(full).max())


def test_layer_single_expert_matches_numpy_pipeline():
    """E=1, topk=1, weight 1: the layer is quant -> dense GEMM -> SiLU-and-mul -> quant ->
    dense GEMM, written here with numpy matmuls, scipy's logistic and torch's e4m3 cast."""
    M, K, N = 40, 256, 256
    x = mi.hidden_states(M, K, seed=21)
    ids = np.zeros((M, 1), np.int32)
    w = np.ones((M, 1), np.float32)
    W13, S13 = mi.expert_weights(1, 2 * N, K, seed=21, stream=1)
    W2, S2 = mi.expert_weights(1, K, N, seed=21, stream=2)
    got = mi.bf16_to_f32(oracle.forward_chunked(x, ids, w, W13, S13, W2, S2, 1))

    def q(v):
        v = v.reshape(v.shape[0], -1, 128)
        s = (np.abs(v).max(axis=2) / np.float32(448)).astype(np.float32)
        c = torch_e4m3_to_f32(torch_f32_to_e4m3((v / s[:, :, None]).astype(np.float32)))
        return (c.astype(np.float64) * s[:, :, None]).reshape(v.shape[0], -1)

    a = q(mi.bf16_to_f32(x))
    c1 = (a @ _dequant_weights(W13, S13)[0].T).astype(np.float32).astype(np.float64)
    h = (c1[:, :N] * expit(c1[:, :N]) * c1[:, N:]).astype(np.float32)
    y = bf16_round((q(h) @ _dequant_weights(W2, S2)[0].T).astype(np.float32))
    ref = y
    err = np.abs(got - ref)
    assert err.max() <= 2e-2 * np.abs(ref).max()
    assert err.sum() / np.abs(ref).sum() <= 5e-3


def test_openmp_build_equals_single_threaded():
    """The OpenMP build (the timed CPU baseline) only spreads independent rows over
    threads: its layer output is bit-identical to the single-threaded checker's."""
    li = mi.make_layer_inputs(mi.TINY)
    wl = li.wl
    args = (li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2, li.w2_scale, wl.E)
    for chunk in (None, 7):
        single = oracle.forward_chunked(*args, chunk_size=chunk)
        par = oracle.forward_chunked(*args, chunk_size=chunk, parallel=True)
        assert (single == par).all()
    assert oracle.num_threads(parallel=False) == 1
    assert oracle.num_threads(parallel=True) >= 1


def test_ep_combine_pins():
    """Expert-parallel combine: one share is returned unchanged; shares of exactly
    representable values add exactly; and the fp32 sum runs in ascending rank order:
    2^24 + 1 + 1 - 2^24 is 0 that way (2^24 + 1 rounds to 2^24 in fp32, twice), while a
    pairwise sum would give 2."""
    rng = np.random.default_rng(0)
    x = mi.bf16_bits(rng.standard_normal((5, 16)).astype(np.float32))
    assert (oracle.ep_combine([x]) == x).all()
    a = mi.bf16_bits(np.full((2, 8), 1.5, np.float32))
    b = mi.bf16_bits(np.full((2, 8), -0.25, np.float32))
    c = mi.bf16_bits(np.full((2, 8), 4.0, np.float32))
    assert (mi.bf16_to_f32(oracle.ep_combine([a, b, c])) == 5.25).all()
    big = mi.bf16_bits(np.full((1, 8), 2.0 ** 24, np.float32))
    one = mi.bf16_bits(np.full((1, 8), 1.0, np.float32))
    neg = mi.bf16_bits(np.full((1, 8), -(2.0 ** 24), np.float32))
    assert (mi.bf16_to_f32(oracle.ep_combine([big, one, one, neg])) == 0.0).all()
    assert (mi.bf16_to_f32(oracle.ep_combine([one, one, big, neg])) == 2.0).all()
    # one rounding at the end: 1 + 2^-8 (not a bf16) arises only inside the sum
    s = oracle.ep_combine([one, mi.bf16_bits(np.full((1, 8), 2.0 ** -8, np.float32))])
    assert (mi.bf16_to_f32(s) == 1.0).all()  # 1 + 2^-8 is a tie in bf16: rounds to even (1.0)


def test_ep_combine_of_expert_shares_is_the_layer(tiny):
    """Shares from four expert subsets (2 experts each) sum to the single-GPU layer
    output up to the bf16 rounding of each share."""
    li = tiny
    E = li.wl.E
    full = mi.bf16_to_f32(oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale,
                                                 li.w2, li.w2_scale, E))
    parts = []
    for lo in range(0, E, 2):
        m = np.full(E, -1, np.int32)
        m[lo:lo + 2] = np.arange(2)
        sl = slice(lo, lo + 2)
        parts.append(oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13[sl], li.w13_scale[sl],
                                            li.w2[sl], li.w2_scale[sl], E, expert_map=m))
    got = mi.bf16_to_f32(oracle.ep_combine(parts))
    err = np.abs(got - full)
    assert err.max() <= 2e-2 * np.abs(full).max() and err.sum() <= 5e-3 * np.abs(full).sum()
