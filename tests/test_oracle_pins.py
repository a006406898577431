"""Pins of the CPU oracle against things other than itself.

Each pin is chosen so that a plausible mistake in the oracle (a swapped
nibble, a wrong group index, a transposed operand, a dropped top-k weight, a
wrong zero point, an unstable routing order, a wrong rounding mode) fails at
least one test here. The references are: hand-derived fixtures under
tests/golden/, closed forms, invariants, special cases that reduce to a
library dense GEMM, and brute-force per-token loops written independently in
plain Python.
"""

import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as mo
from w4a16_int4_moe_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- BF16 ----

def test_bf16_rounding_golden():
    g = _load("bf16_rounding.json")
    for c in g["cases"]:
        assert int(oracle.f64_to_bf16_bits(np.array([c["x"]]))[0]) == c["bits"], c


def test_bf16_rounding_matches_torch_on_float32_inputs():
    # Library reference: torch's float32 -> bfloat16 conversion is RNE. Inputs
    # are float32 values so no double rounding is involved.
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        # exact ties: a BF16 value plus half its spacing
        (np.float32(1.0) + np.float32(2.0 ** -8) * (2 * rng.integers(0, 64, 500) + 1)).astype(np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_decode_closed_form():
    bits = np.array([0x3F80, 0xC000, 0x4300, 0x0000, 0x8000, 0x3F00, 0x7F80], dtype=np.uint16)
    v = oracle.bf16_bits_to_f64(bits)
    assert list(v[:6]) == [1.0, -2.0, 128.0, 0.0, -0.0, 0.5]
    assert math.isinf(v[6]) and v[6] > 0


# ------------------------------------------------------------ weights -----

def test_nibble_order_and_zero_point_golden():
    g = _load("nibble_order.json")
    k = g["k"]
    q = np.frombuffer(bytes.fromhex(g["q_row_hex"]), dtype=np.uint8).reshape(1, 1, k // 2)
    s = np.array(g["scale_bits"], dtype=np.uint16).reshape(1, 1, k // 32)
    for c in g["cases"]:
        x = np.zeros(k, dtype=np.float32)
        if c.get("x_all_ones"):
            x[:] = 1.0
        else:
            x[c["x_onehot_k"]] = 1.0
        xb = wl.to_bf16_bits(x.reshape(1, k))
        out = oracle.indexed_gate_up(xb, np.array([[0]], np.int32), q, s)
        assert out[0, 0] == c["expected"], c


def test_dequant_closed_form_each_code_and_group():
    # Every code 0..15 in every position of two groups with distinct scales:
    # W = (q - 8) * s[group].
    k = 64
    codes = np.tile(np.arange(16, dtype=np.uint8), 4)            # k -> k % 16
    q = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8).reshape(1, 1, k // 2)
    scales = np.array([0.25, 3.0], dtype=np.float32)               # exact in BF16
    s = wl.to_bf16_bits(scales).reshape(1, 1, 2)
    w = oracle.dequant_weights(q, s)[0, 0]
    want = (codes.astype(np.float64) - 8.0) * np.repeat(scales.astype(np.float64), 32)
    np.testing.assert_array_equal(w, want)


def test_all_zero_point_codes_give_exact_zero():
    p = wl.uniform_problem(16, 64, 32, 4, 2, seed=3)
    q_gu = np.full_like(p.q_gu, 0x88)
    q_dn = np.full_like(p.q_dn, 0x88)
    g, g_bits, a_bits, y = oracle.moe_layer(p.x, p.topk_ids, p.topk_weights, q_gu, p.s_gu, q_dn, p.s_dn)
    routed = ~np.isnan(g[:, 0])
    assert np.all(g[routed] == 0.0)
    assert np.all(y == 0.0)


def _torch_dequant(q, s):
    """Independent decode for the dense special case: torch bit operations."""
    qt = torch.from_numpy(q.astype(np.int64))
    lo, hi = qt & 15, qt >> 4
    codes = torch.stack([lo, hi], dim=-1).reshape(*q.shape[:-1], q.shape[-1] * 2).double()
    st = torch.from_numpy(s.astype(np.int32)).bitwise_left_shift(16).view(torch.float32).double()
    return (codes - 8.0) * st.repeat_interleave(32, dim=-1)


def test_single_expert_top1_is_a_dense_gemm():
    # E = 1, top-1, weight 1: gate_up is X @ W^T and down is A @ Wd^T.
    rng = np.random.default_rng(7)
    t, h, inter = 24, 96, 64
    q_gu, s_gu = wl.random_weights(rng, 1, 2 * inter, h)
    q_dn, s_dn = wl.random_weights(rng, 1, h, inter)
    x = wl.random_activations(rng, t, h)
    ids = np.zeros((t, 1), np.int32)
    w = np.ones((t, 1), np.float32)
    g, g_bits, a_bits, y = oracle.moe_layer(x, ids, w, q_gu, s_gu, q_dn, s_dn)
    xt = torch.from_numpy(x.astype(np.int32)).bitwise_left_shift(16).view(torch.float32).double()
    dense_g = torch.matmul(xt, _torch_dequant(q_gu, s_gu)[0].T).numpy()
    np.testing.assert_allclose(g, dense_g, rtol=1e-12, atol=1e-12)
    at = torch.from_numpy(a_bits.astype(np.int32)).bitwise_left_shift(16).view(torch.float32).double()
    dense_y = torch.matmul(at, _torch_dequant(q_dn, s_dn)[0].T).numpy()
    np.testing.assert_allclose(y, dense_y, rtol=1e-12, atol=1e-12)


# ------------------------------------------------- brute force, per token --

def _py_bf16(bits):
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _py_round_bf16(v):
    """Round a Python float to BF16 with Python's own round-half-even."""
    if v == 0.0 or math.isnan(v) or math.isinf(v):
        return v
    m, e = math.frexp(v)
    e = max(e, -125)
    return round(v * 2.0 ** (8 - e)) * 2.0 ** (e - 8)


def _py_code(qrow, k):
    byte = int(qrow[k // 2])
    return (byte & 15) if k % 2 == 0 else (byte >> 4)


def _py_weight(q, s, e, n, k):
    return (_py_code(q[e][n], k) - 8) * _py_bf16(s[e][n][k // 32])


def _brute_layer(p):
    """Per-token dense evaluation in pure Python, independent of the oracle."""
    t_n, topk, h, inter = p.tokens, p.topk, p.hidden, p.inter
    g_all = {}
    y = [[0.0] * h for _ in range(t_n)]
    for t in range(t_n):
        for k in range(topk):
            e = int(p.topk_ids[t][k])
            if not (0 <= e < p.num_experts):
                continue
            xs = [_py_bf16(p.x[t][j]) for j in range(h)]
            g = [sum(xs[j] * _py_weight(p.q_gu, p.s_gu, e, n, j) for j in range(h))
                 for n in range(2 * inter)]
            g_all[t * topk + k] = g
            gb = [_py_round_bf16(v) for v in g]
            a = [_py_round_bf16(gb[j] / (1.0 + math.exp(-gb[j])) * gb[inter + j]) for j in range(inter)]
            wt = float(np.float32(p.topk_weights[t][k]))
            for n in range(h):
                y[t][n] += wt * sum(a[j] * _py_weight(p.q_dn, p.s_dn, e, n, j) for j in range(inter))
    return g_all, np.array(y)


@pytest.mark.parametrize("seed,topk,experts", [(0, 2, 4), (1, 3, 5)])
def test_brute_force_per_token_layer(seed, topk, experts):
    p = wl.uniform_problem(6, 64, 32, experts, topk, seed=seed)
    # one non-local slot, to check skipping
    p.topk_ids[2, 0] = -1
    g, g_bits, a_bits, y = oracle.moe_layer(p.x, p.topk_ids, p.topk_weights,
                                            p.q_gu, p.s_gu, p.q_dn, p.s_dn)
    g_ref, y_ref = _brute_layer(p)
    for i, row in g_ref.items():
        np.testing.assert_allclose(g[i], row, rtol=1e-12, atol=1e-12)
    assert np.all(np.isnan(g[2 * topk + 0]))
    np.testing.assert_allclose(y, y_ref, rtol=1e-10, atol=1e-10)


def test_down_is_linear_in_topk_weights():
    p = wl.uniform_problem(12, 64, 32, 4, 2, seed=5)
    _, _, a_bits, y1 = oracle.moe_layer(p.x, p.topk_ids, p.topk_weights, p.q_gu, p.s_gu, p.q_dn, p.s_dn)
    y2 = oracle.indexed_down(a_bits, p.topk_ids, 2.0 * p.topk_weights, p.q_dn, p.s_dn)
    np.testing.assert_array_equal(y2, 2.0 * y1)
    # zeroing the second slot's weight equals dropping that slot
    w = p.topk_weights.copy()
    w[:, 1] = 0.0
    ids = p.topk_ids.copy()
    ids[:, 1] = -1
    np.testing.assert_allclose(oracle.indexed_down(a_bits, p.topk_ids, w, p.q_dn, p.s_dn),
                               oracle.indexed_down(a_bits, ids, p.topk_weights, p.q_dn, p.s_dn),
                               rtol=0, atol=0)


def test_column_subset_equals_full_evaluation():
    p = wl.uniform_problem(20, 128, 64, 4, 2, seed=9)
    cols = np.array([0, 5, 77, 127])
    full = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu)
    sub = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu, cols=cols)
    np.testing.assert_array_equal(sub, full[:, cols])


# -------------------------------------------------------------- silu ------

def test_silu_golden_and_gate_up_order():
    g = _load("silu.json")
    for c in g["cases"]:
        gu = wl.to_bf16_bits(np.array([[c["gate"], c["up"]]], np.float32))
        a = oracle.silu_and_mul(gu)
        if "bits" in c:
            assert int(a[0, 0]) == c["bits"], c
        else:
            assert oracle.bf16_bits_to_f64(a)[0, 0] == c["value"]


def test_silu_odd_identity():
    # silu(x) - silu(-x) = x exactly in real arithmetic; with BF16 rounding of
    # both outputs the difference stays within one BF16 spacing of x.
    x = np.linspace(-6, 6, 97).astype(np.float32)
    xb = wl.to_bf16_bits(x)
    xv = oracle.bf16_bits_to_f64(xb)
    ones = wl.to_bf16_bits(np.ones_like(x))
    pos = oracle.bf16_bits_to_f64(oracle.silu_and_mul(np.stack([xb, ones], 1)))[:, 0]
    neg = oracle.bf16_bits_to_f64(oracle.silu_and_mul(
        np.stack([wl.to_bf16_bits(-x), ones], 1)))[:, 0]
    assert np.all(np.abs((pos - neg) - xv) <= 2.0 ** -7 * np.maximum(np.abs(xv), 1.0))


# -------------------------------------------------------------- align -----

def test_align_golden():
    g = _load("align_small.json")
    for case in (g, g["cases_with_nonlocal"]):
        s, e, n = oracle.moe_align_block_size(np.array(case["topk_ids"]), case["num_experts"],
                                              case["block_m"], case["capacity"])
        assert s.tolist() == case["sorted_ids"]
        assert e.tolist() == case["expert_ids"]
        assert int(n[0]) == case["num_tokens_padded"]


@pytest.mark.parametrize("seed,tokens,topk,experts,bm", [(0, 100, 4, 16, 16), (1, 257, 8, 48, 32),
                                                         (2, 64, 2, 8, 64), (3, 31, 8, 384, 16)])
def test_align_properties(seed, tokens, topk, experts, bm):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, experts + 3, size=(tokens, topk)).astype(np.int32)
    numel = ids.size
    cap = -(-(numel + experts * (bm - 1)) // bm) * bm
    s, e, n = oracle.moe_align_block_size(ids, experts, bm, cap)
    flat = ids.reshape(-1)
    counts = np.array([(flat == x).sum() for x in range(experts)])
    # closed form of the padded total
    assert int(n[0]) == int(sum(-(-c // bm) * bm for c in counts))
    total = int(n[0])
    body = s[:total]
    valid = body[body < numel]
    local = np.nonzero((flat >= 0) & (flat < experts))[0]
    # permutation: every local row exactly once
    np.testing.assert_array_equal(np.sort(valid), local)
    assert np.all(s[total:] == numel)
    # per block: one expert, rows of that expert, ascending, sentinel only at the tail
    blocks = body.reshape(-1, bm)
    assert e.size == cap // bm and np.all(e[blocks.shape[0]:] == -1)
    prev_e = -1
    for b, row in enumerate(blocks):
        ex = e[b]
        assert ex >= prev_e
        prev_e = ex
        real = row[row < numel]
        assert np.all(flat[real] == ex)
        assert np.all(np.diff(real) > 0)
        k = real.size
        assert np.all(row[k:] == numel)
    # within an expert, rows are ascending across its blocks too
    for x in range(experts):
        rows = body[(np.repeat(e[:blocks.shape[0]], bm) == x) & (body < numel)]
        assert np.all(np.diff(rows) > 0)


# ------------------------------------------------------------ grouped -----

def test_grouped_contiguous_matches_row_by_row():
    rng = np.random.default_rng(11)
    q, s = wl.random_weights(rng, 3, 40, 64)
    m_expert = np.array([0, 0, 0, -1, 2, 2, -1, -1, 1], np.int32)
    a = wl.random_activations(rng, m_expert.size, 64)
    c = oracle.grouped_contiguous(a, m_expert, q, s)
    for r, e in enumerate(m_expert):
        if e < 0:
            assert np.all(np.isnan(c[r]))
            continue
        xs = [_py_bf16(v) for v in a[r]]
        want = [sum(xs[j] * _py_weight(q, s, e, n, j) for j in range(64)) for n in range(40)]
        np.testing.assert_allclose(c[r], want, rtol=1e-12, atol=1e-12)


def test_grouped_masked_matches_row_by_row():
    rng = np.random.default_rng(12)
    q, s = wl.random_weights(rng, 3, 24, 32)
    masked_m = np.array([2, 0, 4], np.int32)
    a = wl.random_activations(rng, 3, 4, 32)
    c = oracle.grouped_masked(a, masked_m, q, s)
    for e in range(3):
        for r in range(4):
            if r >= masked_m[e]:
                assert np.all(np.isnan(c[e, r]))
                continue
            xs = [_py_bf16(v) for v in a[e, r]]
            want = [sum(xs[j] * _py_weight(q, s, e, n, j) for j in range(32)) for n in range(24)]
            np.testing.assert_allclose(c[e, r], want, rtol=1e-12, atol=1e-12)


def test_indexed_equals_grouped_on_the_same_rows():
    # The same expert rows evaluated through the indexed and the contiguous
    # definitions agree exactly (both are the plain per-row GEMM).
    p = wl.uniform_problem(10, 64, 32, 3, 2, seed=13)
    g = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu)
    flat = p.topk_ids.reshape(-1)
    rows = np.argsort(flat, kind="stable")
    a = p.x[rows // p.topk]
    c = oracle.grouped_contiguous(a, flat[rows], p.q_gu, p.s_gu)
    np.testing.assert_array_equal(c, g[rows])


# ------------------------------------------- planted mistakes are caught --

def test_planted_nibble_swap_is_caught(monkeypatch):
    def swapped(q_packed):
        q = np.asarray(q_packed, dtype=np.uint8)
        codes = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
        codes[..., 0::2] = q >> 4
        codes[..., 1::2] = q & 15
        return codes
    monkeypatch.setattr(mo, "unpack_codes", swapped)
    with pytest.raises(AssertionError):
        test_nibble_order_and_zero_point_golden()


def test_planted_group_index_mistake_is_caught(monkeypatch):
    real = mo.dequant_weights

    def wrong(q_packed, scales_bits):
        codes = mo.unpack_codes(q_packed).astype(np.float64)
        s = mo.bf16_bits_to_f64(scales_bits)
        return (codes - 8) * np.tile(s, (1,) * (s.ndim - 1) + (32,))   # k % G instead of k // G
    monkeypatch.setattr(mo, "dequant_weights", wrong)
    monkeypatch.setattr(oracle, "dequant_weights", wrong)
    with pytest.raises(AssertionError):
        test_dequant_closed_form_each_code_and_group()
    with pytest.raises(AssertionError):
        test_brute_force_per_token_layer(0, 2, 4)
    monkeypatch.setattr(mo, "dequant_weights", real)


def test_planted_dropped_topk_weight_is_caught(monkeypatch):
    real = mo.indexed_down

    def unweighted(a_bits, topk_ids, topk_weights, q, s, cols=None):
        return real(a_bits, topk_ids, np.ones_like(topk_weights), q, s, cols)
    monkeypatch.setattr(mo, "indexed_down", unweighted)
    with pytest.raises(AssertionError):
        test_brute_force_per_token_layer(0, 2, 4)


# ------------------------------------------------------------ top-k routing --

def test_topk_softmax_golden_tie_and_local_ids():
    # hand-derived: logits 1, 3, 3, 0.5; the two 3s tie -> lower id first;
    # renormalised over the pair their softmax weights are 1/2 each
    lg = np.array([[1.0, 3.0, 3.0, 0.5]])
    ids, w = oracle.topk_softmax(lg, 2)
    assert ids.tolist() == [[1, 2]]
    np.testing.assert_allclose(w, [[0.5, 0.5]], rtol=0, atol=1e-15)
    # this GPU holds global experts 2..3: expert 1 is another GPU's
    ids, _ = oracle.topk_softmax(lg, 2, expert_offset=2, num_local_experts=2)
    assert ids.tolist() == [[-1, 0]]
    # without renormalisation the weights are the plain softmax values
    _, w = oracle.topk_softmax(lg, 2, renormalize=False)
    e = np.exp([1.0, 3.0, 3.0, 0.5])
    np.testing.assert_allclose(w, [[e[1] / e.sum(), e[2] / e.sum()]], rtol=1e-15)


def test_topk_softmax_all_experts_is_the_library_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((5, 9))
    ids, w = oracle.topk_softmax(lg, 9, renormalize=False)
    for t in range(5):
        np.testing.assert_allclose(w[t], softmax(lg[t])[ids[t]], rtol=1e-12)
        assert sorted(ids[t].tolist()) == list(range(9))
        assert np.all(np.diff(lg[t][ids[t]]) <= 0)


def test_topk_softmax_brute_force_over_subsets():
    import itertools
    rng = np.random.default_rng(8)
    for t in range(20):
        lg = rng.standard_normal((1, 7))
        k = int(rng.integers(1, 5))
        ids, w = oracle.topk_softmax(lg, k)
        best = max(itertools.combinations(range(7), k), key=lambda c: lg[0, list(c)].sum())
        assert set(ids[0].tolist()) == set(best)
        assert abs(w.sum() - 1.0) < 1e-12 and np.all(w > 0)
        assert np.all(np.diff(w[0]) <= 1e-15)            # larger logit, larger weight first


def test_topk_softmax_masked_experts_golden():
    # hand-derived: logits 0, -inf, 1, -inf with k = 3: only experts 2 and 0
    # can be chosen (larger logit first); their softmax weights are e/(1+e)
    # and 1/(1+e) (the masked experts have probability 0), already summing to
    # 1; the third slot finds no expert: id -1, weight 0
    lg = np.array([[0.0, -np.inf, 1.0, -np.inf]])
    ids, w = oracle.topk_softmax(lg, 3)
    assert ids.tolist() == [[2, 0, -1]]
    e = np.e
    np.testing.assert_allclose(w, [[e / (1 + e), 1 / (1 + e), 0.0]], rtol=1e-15, atol=0)
    # every expert masked: no slot is routed
    ids, w = oracle.topk_softmax(np.full((1, 4), -np.inf), 2)
    assert ids.tolist() == [[-1, -1]] and w.tolist() == [[0.0, 0.0]]


def test_planted_ascending_topk_is_caught(monkeypatch):
    import oracle.moe_oracle as om
    real = om.np.lexsort
    monkeypatch.setattr(om.np, "lexsort", lambda keys: real((keys[0], -keys[1])))
    lg = np.array([[1.0, 3.0, 3.0, 0.5]])
    ids, _ = om.topk_softmax(lg, 2)
    assert ids.tolist() != [[1, 2]]
