"""e4m3 chunks in the scorer's general form (more than 4 queries).

Against the oracle's fp64 scores with the floating-point tolerance rule, on
ragged chunks (partial query groups and partial CTAs), chunks whose blocks are
split along the keys, both signs of w, and an overflowing candidate list; the
dense scorer of the decoupled path must return the fused path's scores bit for
bit.
"""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_tolerant, to_device

pytestmark = pytest.mark.gpu


def _fused_and_decoupled(inp, k, **cfg):
    import torch
    op = IndexerTopK(max_T=inp.T, max_S=inp.S, k=k, dtype="fp8", enable_decoupled=1, **cfg)
    d = to_device(inp)
    idx, sc = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, q_scale=d["q_scale"],
                 k_scale=d["k_scale"])
    torch.cuda.synchronize()
    st = op.stats()
    di, ds = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=k,
                          q_scale=d["q_scale"], k_scale=d["k_scale"])
    torch.cuda.synchronize()
    st_dec = op.stats()
    op.close()
    assert st["device_status"] == 0 and st_dec["device_status"] == 0
    return (idx.cpu().numpy(), sc.cpu().numpy(), di.cpu().numpy(), ds.cpu().numpy(), st)


@pytest.mark.parametrize("T,S,k", [(5, 9000, 1024), (6, 20000, 2048), (7, 12345, 700),
                                   (8, 30000, 2048), (13, 40000, 2048), (100, 60000, 2048)])
def test_fp8_ragged_chunks(T, S, k):
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, dtype="fp8", seed=700 + T)
    idx, sc, di, ds, st = _fused_and_decoupled(inp, k)
    assert st["n_overflow"] == 0
    check_tolerant(inp, idx, sc, k)
    np.testing.assert_array_equal(di, idx)
    np.testing.assert_array_equal(ds, sc)


def test_fp8_signed_weights_and_spread_positions():
    """w of either sign, queries spread over the
    cache so their key ranges differ within a CTA."""
    T, S, k = 27, 50000, 1500
    rng = np.random.default_rng(71)
    pos = np.sort(rng.integers(2000, S, size=T)).astype(np.int32)
    inp = datagen.make_indexer_inputs(T=T, first_pos=0, S=S, dtype="fp8", seed=71, positions=pos)
    inp.w[::3] = -inp.w[::3]
    inp.w[1::5, ::2] = -inp.w[1::5, ::2]
    idx, sc, di, ds, _ = _fused_and_decoupled(inp, k)
    check_tolerant(inp, idx, sc, k)
    np.testing.assert_array_equal(di, idx)
    np.testing.assert_array_equal(ds, sc)


def test_fp8_waves_and_split_tail():
    """More query blocks than SMs with a partial last wave: the tail blocks are
    split along the keys (global histograms, shared counts)."""
    T, S, k = 1000, 24576, 2048
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, dtype="fp8", seed=72)
    idx, sc, di, ds, st = _fused_and_decoupled(inp, k)
    assert st["n_overflow"] == 0
    rows = sorted({0, 1, 5, 6, 7, 499, 500, 995, 996, 997, 998, 999})
    check_tolerant(inp, idx, sc, k, queries=rows)
    np.testing.assert_array_equal(di, idx)
    np.testing.assert_array_equal(ds, sc)


def test_fp8_overflow_rescue():
    """A tiny candidate list overflows; the rescued queries are exact."""
    T, S, k = 11, 30000, 600
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, dtype="fp8", seed=73)
    idx, sc, _, _, st = _fused_and_decoupled(inp, k, cand_cap=1024, refresh_interval=0, n_bins=32)
    assert st["n_overflow"] > 0
    check_tolerant(inp, idx, sc, k)


def _fp8_integer_inputs(T, S, seed):
    """e4m3 codes of small integers (-3..3 are exact in e4m3) with per-token
    power-of-two scales and power-of-two weights: every product and partial
    sum is exact in fp32, so the kernel must return the oracle's result bit
    for bit."""
    import oracle.indexer_topk as orc
    base = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=True, seed=seed)
    q8 = datagen.e4m3_codes(orc.bf16_to_f64(base.q)).reshape(base.q.shape)
    k8 = datagen.e4m3_codes(orc.bf16_to_f64(base.k)).reshape(base.k.shape)
    qs = np.ldexp(np.ones(T, np.float32), -(np.arange(T) % 3)).astype(np.float32)
    ks = np.ldexp(np.ones(S, np.float32), (np.arange(S) % 5) - 2).astype(np.float32)
    return datagen.IndexerInputs("fp8", q8, k8, base.w, base.positions, qs, ks)


@pytest.mark.parametrize("T,S,k", [(1, 300000, 2048), (3, 9001, 256), (4, 20000, 300),
                                   (37, 30001, 1000), (1300, 20000, 512)])
def test_fp8_integer_codes_exact(T, S, k):
    from parity import check_exact
    inp = _fp8_integer_inputs(T, S, seed=800 + T)
    idx, sc, di, ds, st = _fused_and_decoupled(inp, k)
    assert st["n_overflow"] == 0
    rows = None if T < 100 else sorted({0, 1, 7, 8, 640, 647, T - 2, T - 1})
    check_exact(inp, idx, sc, k, queries=rows)
    np.testing.assert_array_equal(di, idx)
    np.testing.assert_array_equal(ds, sc)
