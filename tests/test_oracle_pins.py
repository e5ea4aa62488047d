"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each pin compares the oracle with something fixed independently of it:
hand-derived values (tests/golden), closed forms, brute force from the
definition of an exact top-k, a different library routine, and the formats'
definitions.  ``test_planted_mistakes_are_caught`` plants plausible bugs in the
oracle (on the CPU) and checks that every one of them fails at least one pin.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle.indexer_topk as orc
from indexer_topk_long_gb300 import datagen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


class _Bundle:
    """Minimal fp64-exact input bundle (values representable in bf16)."""

    def __init__(self, q, w, keys, positions):
        self.dtype = "bf16"
        self.q = datagen.bf16_bits(np.asarray(q, np.float32))
        self.k = datagen.bf16_bits(np.asarray(keys, np.float32))
        self.w = np.asarray(w, np.float32)
        self.positions = np.asarray(positions, np.int32)


class _Fp8Bundle:
    """Input bundle of e4m3 codes with fp32 per-token scales."""

    def __init__(self, q_codes, q_scale, w, k_codes, k_scale, positions):
        self.dtype = "fp8"
        self.q = np.asarray(q_codes, np.uint8)
        self.k = np.asarray(k_codes, np.uint8)
        self.q_scale = np.asarray(q_scale, np.float32)
        self.k_scale = np.asarray(k_scale, np.float32)
        self.w = np.asarray(w, np.float32)
        self.positions = np.asarray(positions, np.int32)


def _hex(a):
    return np.vectorize(lambda c: int(c, 16))(np.asarray(a, dtype=object)).astype(np.uint8)


def _f(x):
    return -math.inf if x == "-inf" else float(x)


# ---------------------------------------------------------------------------
# Pins (each returns None on success, raises AssertionError on failure)
# ---------------------------------------------------------------------------

def pin_hand_examples():
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        for run in case["runs"]:
            b = _Bundle(case["q"], case["w"], case["keys"], run["positions"])
            idx, val = orc.indexer_topk(b, case["k"])
            np.testing.assert_array_equal(idx, np.array(run["idx"], np.int32), err_msg=case["name"])
            exp = np.array([[_f(x) for x in row] for row in run["score"]], np.float32)
            np.testing.assert_array_equal(val, exp, err_msg=case["name"])
        # every score of the fully visible case
        b = _Bundle(case["q"], case["w"], case["keys"], [len(case["keys"]) - 1] * len(case["q"]))
        for t, row in enumerate(case["all_scores"]):
            np.testing.assert_allclose(orc.full_scores(b, t), row, rtol=0, atol=0)


def pin_basis_keys():
    """Keys = unit basis vectors e_i: I[t, i] = sum_h w[t,h] * max(0, q[t,h,i])."""
    rng = np.random.default_rng(5)
    H, d, T = 4, 6, 3
    q = rng.integers(-4, 5, size=(T, H, d)).astype(np.float32)
    w = rng.integers(1, 8, size=(T, H)).astype(np.float32) / 4
    keys = np.eye(d, dtype=np.float32)
    b = _Bundle(q, w, keys, [d - 1] * T)
    for t in range(T):
        expect = [sum(w[t, h] * max(0.0, q[t, h, i]) for h in range(H)) for i in range(d)]
        np.testing.assert_array_equal(orc.full_scores(b, t), np.array(expect))


def pin_identical_heads_closed_form():
    """All heads equal to a: I[t, s] = (sum_h w[t,h]) * max(0, a . k[s])."""
    rng = np.random.default_rng(6)
    H, d, S = 5, 8, 40
    a = rng.integers(-3, 4, size=d).astype(np.float32)
    q = np.broadcast_to(a, (1, H, d)).copy()
    w = (rng.integers(1, 9, size=(1, H)) / 8).astype(np.float32)
    keys = rng.integers(-3, 4, size=(S, d)).astype(np.float32)
    b = _Bundle(q, w, keys, [S - 1])
    expect = float(w.sum()) * np.maximum(keys.astype(np.float64) @ a.astype(np.float64), 0)
    np.testing.assert_array_equal(orc.full_scores(b, 0), expect)


def _dominates(Ia, a, Ib, b):
    """a precedes b in the exact top-k order: higher score, then lower index."""
    return Ia > Ib or (Ia == Ib and a < b)


def pin_bruteforce_subsets():
    """Enumerate every k-subset; the answer is the unique subset A such that each
    member of A precedes each non-member.  Output order = number of visible keys
    that precede each member (no sort routine involved)."""
    rng = np.random.default_rng(7)
    for trial in range(40):
        S = int(rng.integers(1, 10))
        H, d = 2, 3
        q = rng.integers(-2, 3, size=(1, H, d)).astype(np.float32)
        w = (rng.integers(1, 4, size=(1, H)) / 2).astype(np.float32)
        keys = rng.integers(-2, 3, size=(S, d)).astype(np.float32)
        pos = int(rng.integers(0, S + 2))
        k = int(rng.integers(1, 6))
        b = _Bundle(q, w, keys, [pos])
        V = min(pos + 1, S)
        I = [sum(float(w[0, h]) * max(0.0, float(np.dot(q[0, h].astype(np.float64), keys[s].astype(np.float64))))
                 for h in range(H)) for s in range(V)]
        n = min(k, V)
        winners = [A for A in itertools.combinations(range(V), n)
                   if all(_dominates(I[a], a, I[c], c) for a in A for c in range(V) if c not in A)]
        assert len(winners) == 1
        A = winners[0]
        rank = {a: sum(_dominates(I[c], c, I[a], a) for c in range(V)) for a in A}
        expect_idx = [None] * n
        for a, r in rank.items():
            expect_idx[r] = a
        idx, val = orc.indexer_topk(b, k)
        assert list(idx[0, :n]) == expect_idx, (trial, I, idx)
        assert all(x == -1 for x in idx[0, n:])
        np.testing.assert_array_equal(val[0, :n], np.array([I[a] for a in expect_idx], np.float32))
        assert np.all(np.isneginf(val[0, n:]))


def pin_retrieval_vs_torch_topk():
    """H=1, w=1, no ReLU, no mask is a plain inner product: compare with
    torch.matmul + torch.topk (a different library) on tie-free data."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    n, d, N, k = 5, 24, 300, 17
    qf = rng.standard_normal((n, d)).astype(np.float32)
    cf = rng.standard_normal((N, d)).astype(np.float32)
    qb, cb = datagen.bf16_bits(qf), datagen.bf16_bits(cf)
    idx, val = orc.retrieval_topk(qb, cb, k, block=64)
    qt = torch.from_numpy(qb.view(np.int16).copy()).view(torch.bfloat16).double()
    ct = torch.from_numpy(cb.view(np.int16).copy()).view(torch.bfloat16).double()
    tv, ti = torch.topk(qt @ ct.T, k, dim=1)
    np.testing.assert_array_equal(idx, ti.numpy().astype(np.int32))
    np.testing.assert_array_equal(val, tv.numpy().astype(np.float32))


def pin_fp_formats():
    with open(os.path.join(GOLDEN, "fp_formats.json")) as f:
        g = json.load(f)
    for code, v in g["bf16"]:
        got = orc.bf16_to_f64(np.array([int(code, 16)], np.uint16))[0]
        assert got == float(v), (code, got, v)
    for code, v in g["e4m3"]:
        got = orc.e4m3_to_f64(np.array([int(code, 16)], np.uint8))[0]
        if v == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(v), (code, got, v)


def pin_fp8_bundle_is_scaled_product():
    """fp8 bundle: the widened value is code value times its own token's scale."""
    codes = np.array([[0x38, 0x40, 0xB8, 0x01], [0x38, 0x40, 0xB8, 0x01]], np.uint8)   # 1, 2, -1, 2^-9
    b = _Fp8Bundle(codes.reshape(2, 1, 4), [0.25, 8.0], np.ones((2, 1)), codes, [4.0, 0.5], [1, 1])
    q, w = orc.widen_queries(b)
    k = orc.widen_keys(b)
    np.testing.assert_array_equal(q[0, 0], [0.25, 0.5, -0.25, 0.25 * 2 ** -9])
    np.testing.assert_array_equal(q[1, 0], [8.0, 16.0, -8.0, 8 * 2 ** -9])
    np.testing.assert_array_equal(k[0], [4.0, 8.0, -4.0, 4 * 2 ** -9])
    np.testing.assert_array_equal(k[1], [0.5, 1.0, -0.5, 0.5 * 2 ** -9])
    np.testing.assert_array_equal(w, np.ones((2, 1)))


def pin_fp8_hand_examples():
    """Hand-derived e4m3 indexer case with per-token scales (tests/golden)."""
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["fp8_cases"]
    for case in cases:
        qc, kc = _hex(case["q_codes"]), _hex(case["k_codes"])
        for run in case["runs"]:
            b = _Fp8Bundle(qc, case["q_scale"], case["w"], kc, case["k_scale"], run["positions"])
            idx, val = orc.indexer_topk(b, case["k"])
            np.testing.assert_array_equal(idx, np.array(run["idx"], np.int32), err_msg=case["name"])
            np.testing.assert_array_equal(val, np.array(run["score"], np.float32), err_msg=case["name"])
        b = _Fp8Bundle(qc, case["q_scale"], case["w"], kc, case["k_scale"], [len(kc) - 1] * len(qc))
        for t, row in enumerate(case["all_scores"]):
            np.testing.assert_array_equal(orc.full_scores(b, t), row)


def _fp8_random_bundle(rng, T, H, d, S, pow2_scales=True):
    qv = rng.standard_normal((T, H, d)) * 4
    kv = rng.standard_normal((S, d)) * 4
    qc, kc = datagen.e4m3_codes(qv), datagen.e4m3_codes(kv)
    if pow2_scales:
        qs = np.exp2(rng.integers(-3, 4, size=T)).astype(np.float32)
        ks = np.exp2(rng.integers(-3, 4, size=S)).astype(np.float32)
    else:
        qs = np.ones(T, np.float32)
        ks = np.ones(S, np.float32)
    w = (rng.standard_normal((T, H)) / 4).astype(np.float32)   # either sign
    return _Fp8Bundle(qc, qs, w, kc, ks, np.full(T, S - 1))


def pin_fp8_scale_homogeneity():
    """ReLU(a x) = a ReLU(x) for a > 0, so the score with per-token scales is
    q_scale[t] * k_scale[s] times the score of the bare codes.  Power-of-two
    scales keep both sides exact."""
    rng = np.random.default_rng(10)
    T, H, d, S = 3, 4, 8, 20
    b = _fp8_random_bundle(rng, T, H, d, S)
    bare = _Fp8Bundle(b.q, np.ones(T), b.w, b.k, np.ones(S), b.positions)
    for t in range(T):
        expect = orc.full_scores(bare, t) * float(b.q_scale[t]) * b.k_scale.astype(np.float64)
        np.testing.assert_array_equal(orc.full_scores(b, t), expect)


def pin_fp8_matches_bf16_of_same_values():
    """An e4m3 code times a power-of-two scale is exactly a bf16 value (3 vs 7
    mantissa bits): the fp8 bundle and the bf16 bundle of the same real
    numbers (codes decoded by torch's float8_e4m3fn, not by the oracle) must
    give identical top-k results."""
    rng = np.random.default_rng(11)
    T, H, d, S, k = 4, 3, 8, 40, 7
    b = _fp8_random_bundle(rng, T, H, d, S)
    b.positions = np.array([5, 17, 30, 39], np.int32)
    qv = _e4m3_by_torch(b.q) * b.q_scale[:, None, None].astype(np.float64)
    kv = _e4m3_by_torch(b.k) * b.k_scale[:, None].astype(np.float64)
    bf = _Bundle(qv.astype(np.float32), b.w, kv.astype(np.float32), b.positions)
    assert np.array_equal(orc.bf16_to_f64(bf.q), qv) and np.array_equal(orc.bf16_to_f64(bf.k), kv)
    i8, v8 = orc.indexer_topk(b, k)
    i16, v16 = orc.indexer_topk(bf, k)
    np.testing.assert_array_equal(i8, i16)
    np.testing.assert_array_equal(v8, v16)


def _e4m3_by_torch(codes):
    """e4m3 values decoded by a different library (torch.float8_e4m3fn)."""
    torch = pytest.importorskip("torch")
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).double().numpy()


def pin_invariants_gaussian():
    """On a generated tiny chunk: the returned set dominates the rest, no index
    beyond the query's position, min(k, V) valid distinct entries."""
    inp = datagen.make_indexer_inputs(T=6, first_pos=90, S=100, H=4, d=16, seed=3)
    idx, val = orc.indexer_topk(inp, 16)
    for t in range(6):
        I = orc.full_scores(inp, t)
        V = I.shape[0]
        n = min(16, V)
        got = idx[t, :n]
        assert len(set(got.tolist())) == n and got.max() <= inp.positions[t]
        rest = np.setdiff1d(np.arange(V), got)
        if rest.size:
            assert I[got].min() >= I[rest].max()


PINS = [pin_hand_examples, pin_basis_keys, pin_identical_heads_closed_form, pin_bruteforce_subsets,
        pin_retrieval_vs_torch_topk, pin_fp_formats, pin_fp8_bundle_is_scaled_product,
        pin_fp8_hand_examples, pin_fp8_scale_homogeneity, pin_fp8_matches_bf16_of_same_values,
        pin_invariants_gaussian]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin
# ---------------------------------------------------------------------------

def _mut_no_relu(q_t, w_t, keys, relu=True):
    return (keys @ q_t.T) @ w_t


def _mut_relu_after_sum(q_t, w_t, keys, relu=True):
    return np.maximum((keys @ q_t.T) @ w_t, 0.0)


def _mut_heads_reversed(q_t, w_t, keys, relu=True):
    return np.maximum(keys @ q_t[::-1].T, 0.0) @ w_t


def _mut_unweighted(q_t, w_t, keys, relu=True):
    return np.maximum(keys @ q_t.T, 0.0).sum(axis=1)


def _mut_causal_strict(pos, S, causal):
    return min(int(pos), S) if causal else S


def _mut_drop_last_key(pos, S, causal):
    return max(0, min(int(pos) + 1, S) - 1) if causal else S - 1


def _mut_ties_high_index(scores, k):
    V = scores.shape[0]
    order = np.lexsort((-np.arange(V), -scores))
    n = min(k, V)
    idx = np.full(k, -1, np.int32)
    val = np.full(k, -np.inf, np.float32)
    idx[:n] = order[:n]
    val[:n] = scores[order[:n]]
    return idx, val


def _mut_ascending(scores, k):
    V = scores.shape[0]
    order = np.lexsort((np.arange(V), scores))
    n = min(k, V)
    idx = np.full(k, -1, np.int32)
    val = np.full(k, -np.inf, np.float32)
    idx[:n] = order[:n]
    val[:n] = scores[order[:n]]
    return idx, val


def _mut_w_transposed(inputs):
    q, w = ORIG["widen_queries"](inputs)
    return q, (w.T if w.shape[0] == w.shape[1] else w[::-1])


def _q_codes(inputs):
    return ORIG["e4m3_to_f64"](inputs.q)


def _mut_q_scale_dropped(inputs):
    if inputs.dtype != "fp8":
        return ORIG["widen_queries"](inputs)
    return _q_codes(inputs), np.asarray(inputs.w, np.float64)


def _mut_k_scale_dropped(inputs):
    if inputs.dtype != "fp8":
        return ORIG["widen_keys"](inputs)
    return ORIG["e4m3_to_f64"](inputs.k)


def _mut_q_scale_on_head_axis(inputs):
    if inputs.dtype != "fp8":
        return ORIG["widen_queries"](inputs)
    qs = np.asarray(inputs.q_scale, np.float64)
    return _q_codes(inputs) * qs[None, :, None], np.asarray(inputs.w, np.float64)


def _mut_q_scale_of_wrong_query(inputs):
    if inputs.dtype != "fp8":
        return ORIG["widen_queries"](inputs)
    qs = np.asarray(inputs.q_scale, np.float64)[::-1]
    return _q_codes(inputs) * qs[:, None, None], np.asarray(inputs.w, np.float64)


def _mut_k_scale_of_wrong_key(inputs):
    if inputs.dtype != "fp8":
        return ORIG["widen_keys"](inputs)
    ks = np.asarray(inputs.k_scale, np.float64)[::-1]
    return ORIG["e4m3_to_f64"](inputs.k) * ks[:, None]


def _mut_w_scaled_twice(inputs):
    q, w = ORIG["widen_queries"](inputs)
    if inputs.dtype != "fp8":
        return q, w
    return q, w * np.asarray(inputs.q_scale, np.float64)[:, None]


def _mut_e4m3_bias8(codes):
    return ORIG["e4m3_to_f64"](codes) / 2.0


def _mut_bf16_shift(bits):
    b32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
    return b32.view(np.float32).astype(np.float64)


ORIG = {name: getattr(orc, name) for name in
        ["scores_one_query", "visible_count", "exact_topk_row", "widen_queries", "widen_keys",
         "e4m3_to_f64", "bf16_to_f64"]}

MUTANTS = [
    ("scores_one_query", _mut_no_relu),
    ("scores_one_query", _mut_relu_after_sum),
    ("scores_one_query", _mut_heads_reversed),
    ("scores_one_query", _mut_unweighted),
    ("visible_count", _mut_causal_strict),
    ("visible_count", _mut_drop_last_key),
    ("exact_topk_row", _mut_ties_high_index),
    ("exact_topk_row", _mut_ascending),
    ("widen_queries", _mut_w_transposed),
    ("widen_queries", _mut_q_scale_dropped),
    ("widen_keys", _mut_k_scale_dropped),
    ("widen_queries", _mut_q_scale_on_head_axis),
    ("widen_queries", _mut_q_scale_of_wrong_query),
    ("widen_keys", _mut_k_scale_of_wrong_key),
    ("widen_queries", _mut_w_scaled_twice),
    ("e4m3_to_f64", _mut_e4m3_bias8),
    ("bf16_to_f64", _mut_bf16_shift),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_planted_mistakes_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(orc, name, mutant)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures >= 1, f"mutant {mutant.__name__} of {name} passed every pin"
