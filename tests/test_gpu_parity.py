"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small cases are compared element by element for every query; they span
several 128-key tiles, partial query blocks (T not a multiple of 8) and ragged
key tails (S not a multiple of 128).  Integer-valued inputs must match
bit-exactly; Gaussian inputs within the stated tolerances (tests/parity.py).
"""
import numpy as np
import pytest

import oracle.indexer_topk as orc
from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, check_tolerant, to_device

pytestmark = pytest.mark.gpu


def _run(inp, k, op=None, prev=None, **cfg):
    import torch
    own = op is None
    if own:
        op = IndexerTopK(max_T=max(inp.T, 1), max_S=inp.S, k=k, dtype=inp.dtype, **cfg)
    d = to_device(inp)
    idx, sc = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, prev_topk=prev,
                 q_scale=d["q_scale"], k_scale=d["k_scale"])
    torch.cuda.synchronize()
    st = op.stats()
    if own:
        op.close()
    assert st["device_status"] == 0, st
    return idx.cpu().numpy(), sc.cpu().numpy(), st


def test_tiny_integer_exact():
    inp = datagen.workload_inputs("tiny", integer=True)
    idx, sc, st = _run(inp, 2048)
    check_exact(inp, idx, sc, 2048)
    assert st["n_overflow"] == 0


def test_tiny_gaussian_bf16():
    inp = datagen.workload_inputs("tiny")
    idx, sc, _ = _run(inp, 2048)
    check_tolerant(inp, idx, sc, 2048)


@pytest.mark.parametrize("T,S,k,seed", [(20, 5000, 256, 1), (9, 777, 64, 2), (33, 3001, 1000, 3)])
def test_ragged_integer_exact(T, S, k, seed):
    # positions spread over the whole cache: some queries see fewer than k keys
    rng = np.random.default_rng(seed)
    pos = np.sort(rng.integers(0, S, size=T)).astype(np.int32)
    pos[-1] = S - 1
    inp = datagen.make_indexer_inputs(T=T, first_pos=0, S=S, integer=True, seed=seed, positions=pos)
    idx, sc, _ = _run(inp, k)
    check_exact(inp, idx, sc, k)


@pytest.mark.parametrize("T,S,k", [(20, 5000, 256), (64, 20000, 2048)])
def test_ragged_gaussian(T, S, k):
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, seed=T)
    idx, sc, _ = _run(inp, k)
    check_tolerant(inp, idx, sc, k)


def test_decoupled_matches_oracle_and_fused():
    import torch
    inp = datagen.make_indexer_inputs(T=24, first_pos=4000, S=4100, integer=True, seed=7)
    op = IndexerTopK(max_T=24, max_S=4100, k=512, enable_decoupled=1)
    d = to_device(inp)
    i1, s1 = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=512)
    i2, s2 = op(d["q"], d["w"], d["k_cache"], d["positions"], k=512)
    torch.cuda.synchronize()
    op.close()
    check_exact(inp, i1.cpu().numpy(), s1.cpu().numpy(), 512)
    assert torch.equal(i1, i2) and torch.equal(s1, s2)


def test_decoupled_gaussian():
    import torch
    inp = datagen.make_indexer_inputs(T=16, first_pos=9000, S=9016, seed=8)
    op = IndexerTopK(max_T=16, max_S=9016, k=2048, enable_decoupled=1)
    d = to_device(inp)
    i1, s1 = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=2048)
    i2, s2 = op(d["q"], d["w"], d["k_cache"], d["positions"], k=2048)
    torch.cuda.synchronize()
    op.close()
    check_tolerant(inp, i1.cpu().numpy(), s1.cpu().numpy(), 2048)
    # both paths select from the same fp32 scores: identical results
    assert torch.equal(i1, i2) and torch.equal(s1, s2)


def test_result_independent_of_sample_bins_and_refresh():
    """Sample, bin count and refresh cadence change the speed, never the result."""
    import torch
    inp = datagen.make_indexer_inputs(T=16, first_pos=12000, S=12016, seed=9)
    d = to_device(inp)
    outs = []
    variants = [dict(), dict(n_bins=64), dict(refresh_interval=0), dict(refresh_interval=7),
                dict(sample_size=300)]
    for cfg in variants:
        op = IndexerTopK(max_T=16, max_S=12016, k=1024, **cfg)
        outs.append(op(d["q"], d["w"], d["k_cache"], d["positions"], k=1024))
        op.close()
    # previous-chunk sample built from the first result, and an all-invisible sample
    op = IndexerTopK(max_T=16, max_S=12016, k=1024)
    smp = op.make_sample(outs[0][0], 12016, 3072)
    outs.append(op(d["q"], d["w"], d["k_cache"], d["positions"], k=1024, prev_topk=smp))
    late = torch.arange(12016 - 64, 12016, dtype=torch.int32, device="cuda")   # beyond most positions
    outs.append(op(d["q"], d["w"], d["k_cache"], d["positions"], k=1024, prev_topk=late))
    torch.cuda.synchronize()
    op.close()
    for i, (a, b) in enumerate(outs[1:]):
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1]), f"variant {i + 1}"
    check_tolerant(inp, outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy(), 1024)


def test_scan_order_does_not_change_results():
    """More query blocks than SMs, so CTAs of later waves start their key scan
    at the filter's sweep position and wrap around; with refresh_interval=0 the
    sweep counter never advances and every CTA scans from the first tile.  Both
    orders (and a sparser refresh) must give the same bits, and the oracle's."""
    import torch
    T, S = 2432, 40000          # 304 query blocks: two waves of 152
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=True, seed=21)
    d = to_device(inp)
    outs = []
    for cfg in (dict(refresh_interval=0), dict(), dict(refresh_interval=7)):
        op = IndexerTopK(max_T=T, max_S=S, k=512, **cfg)
        outs.append(op(d["q"], d["w"], d["k_cache"], d["positions"], k=512))
        torch.cuda.synchronize()
        assert op.stats()["device_status"] == 0
        op.close()
    for i, (a, b) in enumerate(outs[1:]):
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1]), f"variant {i + 1}"
    qs = [0, 1, 607, 1215, 1823, 2400, T - 2, T - 1]
    check_exact(inp, outs[1][0].cpu().numpy(), outs[1][1].cpu().numpy(), 512, queries=qs)


def test_overflow_is_rescued_exactly():
    inp = datagen.make_indexer_inputs(T=12, first_pos=3000, S=3100, integer=True, seed=10)
    idx, sc, st = _run(inp, 300, cand_cap=320, refresh_interval=0, n_bins=32)
    assert st["n_overflow"] > 0
    check_exact(inp, idx, sc, 300)


def test_degenerate_scores():
    """All-zero queries (every score 0: the lowest indices win), zero weight
    rows, and negative weights."""
    inp = datagen.make_indexer_inputs(T=10, first_pos=2000, S=2010, integer=True, seed=12)
    inp.q[0] = 0            # bf16 bit pattern 0 = +0.0
    inp.w[1] = 0
    inp.w[2] = -inp.w[2]
    idx, sc, _ = _run(inp, 128)
    check_exact(inp, idx, sc, 128)


def test_fp8_tiny():
    inp = datagen.workload_inputs("tiny", dtype="fp8")
    idx, sc, _ = _run(inp, 2048)
    check_tolerant(inp, idx, sc, 2048)


def test_make_sample_ranking():
    import torch
    S = 5000
    rng = np.random.default_rng(13)
    prev = rng.integers(-1, S, size=(40, 64)).astype(np.int32)
    op = IndexerTopK(max_T=8, max_S=S, k=64)
    got = op.make_sample(torch.from_numpy(prev).cuda(), S, 300).cpu().numpy()
    op.close()
    counts = np.bincount(prev[prev >= 0], minlength=S)
    chosen = np.flatnonzero(counts > 0)
    order = chosen[np.lexsort((-chosen, -counts[chosen]))]   # count desc, id desc
    assert len(np.unique(got)) == 300
    np.testing.assert_array_equal(np.sort(got[np.isin(got, order)]), np.sort(order[:300]))


def test_make_sample_pads_with_unselected_ids():
    """Fewer selected ids than asked for: all of them, then distinct unselected ones."""
    import torch
    S = 3000
    rng = np.random.default_rng(17)
    prev = rng.integers(0, S, size=(4, 16)).astype(np.int32)
    prev[0, :3] = -1
    op = IndexerTopK(max_T=8, max_S=S, k=64)
    got = op.make_sample(torch.from_numpy(prev).cuda(), S, 500).cpu().numpy()
    op.close()
    chosen = np.unique(prev[prev >= 0])
    assert len(np.unique(got)) == 500 and got.min() >= 0 and got.max() < S
    assert np.isin(chosen, got).all()


def test_empty_chunk_and_k_larger_than_visible():
    import torch
    inp = datagen.make_indexer_inputs(T=8, first_pos=0, S=700, integer=True, seed=14)
    idx, sc, _ = _run(inp, 1024)           # every query sees <= 8 keys
    check_exact(inp, idx, sc, 1024)
    op = IndexerTopK(max_T=8, max_S=700, k=16)
    d = to_device(inp)
    e_idx = torch.empty((0, 16), dtype=torch.int32, device="cuda")
    e_sc = torch.empty((0, 16), dtype=torch.float32, device="cuda")
    op(d["q"][:0], d["w"][:0], d["k_cache"], d["positions"][:0], k=16, out=(e_idx, e_sc))
    torch.cuda.synchronize()
    op.close()


@pytest.mark.parametrize("T,S,integer", [(1, 300000, True), (5, 300000, False), (16, 200003, True)])
def test_decode_small_chunks_split_over_keys(T, S, integer):
    """Few queries against a long cache (decode-like): the query block's keys are
    split over many CTAs that share the candidate count and histogram."""
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=integer, seed=40 + T)
    idx, sc, st = _run(inp, 2048)
    assert st["n_overflow"] == 0
    if integer:
        check_exact(inp, idx, sc, 2048)
    else:
        check_tolerant(inp, idx, sc, 2048)
