"""Parity helpers for GPU tests: inputs to device tensors, exact and tolerant
comparison of top-k results against the CPU oracle.

Tolerances (floating-point mode): a returned score s must be within
1e-4 * (1 + |s_oracle|) of the oracle's fp64 score of the same key, and the
returned key set must equal the oracle's except for swaps among keys whose
oracle score lies within 2e-4 * (1 + |s_k|) of the k-th largest score s_k.
Integer-valued inputs make every fp32 partial sum exact, so there the results
must be bit-identical.
"""
from __future__ import annotations

import numpy as np

import oracle.indexer_topk as orc

SCORE_RTOL = 1e-4
TIE_BAND = 2e-4


def to_device(inp, device="cuda"):
    import torch
    dev = torch.device(device)
    if inp.dtype == "bf16":
        q = torch.from_numpy(np.ascontiguousarray(inp.q).view(np.int16)).to(dev)
        k = torch.from_numpy(np.ascontiguousarray(inp.k).view(np.int16)).to(dev)
        qs = ks = None
    else:
        q = torch.from_numpy(np.ascontiguousarray(inp.q)).to(dev)
        k = torch.from_numpy(np.ascontiguousarray(inp.k)).to(dev)
        qs = torch.from_numpy(inp.q_scale).to(dev)
        ks = torch.from_numpy(inp.k_scale).to(dev)
    w = torch.from_numpy(np.ascontiguousarray(inp.w)).to(dev)
    pos = torch.from_numpy(np.ascontiguousarray(inp.positions)).to(dev)
    return dict(q=q, w=w, k_cache=k, positions=pos, q_scale=qs, k_scale=ks)


def check_row_tolerant(idx, score, I, k, where=""):
    """One query: GPU (idx, score) vs the oracle's fp64 visible scores I."""
    V = I.shape[0]
    n = min(k, V)
    assert np.all(idx[n:] == -1), f"{where}: padding indices"
    assert np.all(np.isneginf(score[n:])), f"{where}: padding scores"
    got = idx[:n].astype(np.int64)
    assert np.all(got >= 0) and np.all(got < V), f"{where}: index out of the visible range"
    assert len(np.unique(got)) == n, f"{where}: duplicate indices"
    s_or = I[got]
    err = np.abs(score[:n].astype(np.float64) - s_or)
    bad = err > SCORE_RTOL * (1 + np.abs(s_or))
    assert not bad.any(), f"{where}: {bad.sum()} scores off, max err {err.max():.3g}"
    # output order: by the kernel's own scores, descending, ties by index
    sc = score[:n]
    assert np.all((sc[:-1] > sc[1:]) | ((sc[:-1] == sc[1:]) & (got[:-1] < got[1:]))), \
        f"{where}: output not sorted"
    ref_idx, _ = orc.exact_topk_row(I, k)
    ref = ref_idx[:n].astype(np.int64)
    s_k = I[ref[-1]]
    band = TIE_BAND * (1 + abs(s_k))
    missing = np.setdiff1d(ref, got)
    extra = np.setdiff1d(got, ref)
    assert len(missing) == len(extra)
    assert np.all(np.abs(I[missing] - s_k) <= band), f"{where}: missing keys outside the tie band"
    assert np.all(np.abs(I[extra] - s_k) <= band), f"{where}: extra keys outside the tie band"
    return len(missing)


def check_tolerant(inp, idx, score, k, queries=None, keys64=None, causal=True, relu=True):
    """All (or the chosen) queries of a chunk; returns the number of tie swaps."""
    idx = np.asarray(idx)
    score = np.asarray(score)
    rows = range(inp.T) if queries is None else queries
    kk = orc.widen_keys(inp) if keys64 is None else keys64
    swaps = 0
    for t in rows:
        I = orc.full_scores(inp, t, causal=causal, relu=relu, keys64=kk)
        swaps += check_row_tolerant(idx[t], score[t], I, k, where=f"query {t}")
    return swaps


def check_exact(inp, idx, score, k, queries=None):
    """Bit-exact comparison (integer-valued inputs); GPU rows are [T, k]."""
    ref_idx, ref_score = orc.indexer_topk(inp, k, queries=queries)
    rows = slice(None) if queries is None else list(queries)
    np.testing.assert_array_equal(np.asarray(idx)[rows], ref_idx)
    np.testing.assert_array_equal(np.asarray(score)[rows], ref_score)
