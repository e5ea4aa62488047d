"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Each chunk runs with the previous chunk's top-3k as the sample (the previous
chunk is run first, as the prefill would).  The CPU oracle checks a seeded
subset of queries element by element (always the first and last query of the
chunk, 64 queries per chunk); every query is checked for the invariants that
hold at any size (sorted output, distinct indices, no index beyond the query's
position, exactly min(k, V) valid entries), and the same-GPU decoupled
baseline -- a second, independent selection path over the same fp32 scores --
must return identical results for all queries.  An integer-valued 128K chunk
pair (heavy score ties) must match the oracle bit for bit: it drives the
Select stage's crowded boundary bins at prefill scale.  The vector-retrieval workload
runs at its full size too (sampled queries against the oracle's fp64 scores
over the whole corpus, every query against the decoupled path).
"""
import numpy as np
import pytest

import oracle.indexer_topk as orc
from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, check_row_tolerant, check_tolerant, to_device

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _invariants(idx, sc, positions, S, k):
    V = np.minimum(positions.astype(np.int64) + 1, S)
    n = np.minimum(V, k)
    T = idx.shape[0]
    cols = np.arange(k)[None, :]
    valid = cols < n[:, None]
    assert np.all((idx >= 0) == valid), "valid-entry count"
    assert np.all(np.isneginf(sc[~valid])), "padding scores"
    assert np.all(idx[valid] <= np.repeat(positions, n)), "index beyond the query's position"
    s_sorted = np.sort(idx, axis=1)
    dup = (s_sorted[:, 1:] == s_sorted[:, :-1]) & (s_sorted[:, 1:] >= 0)
    assert not dup.any(), "duplicate index"
    a, b = sc[:, :-1], sc[:, 1:]
    ia, ib = idx[:, :-1], idx[:, 1:]
    both = valid[:, 1:]
    ok = (a > b) | ((a == b) & (ia < ib))
    assert np.all(ok[both]), "output order"
    del T


def _sample_queries(T, n, seed):
    rng = np.random.default_rng(seed)
    q = set(rng.choice(T, size=n - 2, replace=False).tolist()) | {0, T - 1}
    return sorted(q)


def _chunk_pair(prev_name, cur_name, dtype, n_check, decoupled, integer=False):
    import torch
    wl = datagen.WORKLOADS[cur_name]
    keys = datagen.keys_fp32(wl.S, wl.d)
    prev = datagen.workload_inputs(prev_name, dtype=dtype, keys=keys, integer=integer)
    cur = datagen.workload_inputs(cur_name, dtype=dtype, keys=keys, integer=integer)
    op = IndexerTopK(max_T=wl.T, max_S=wl.S, k=wl.k, dtype=dtype,
                     enable_decoupled=1 if decoupled else 0)
    dp, dc = to_device(prev), to_device(cur)
    S_prev = prev.S
    ks = None if dc["k_scale"] is None else dc["k_scale"][:S_prev]
    p_idx, p_sc = op(dp["q"], dp["w"], dc["k_cache"][:S_prev], dp["positions"], k=wl.k,
                     q_scale=dp["q_scale"], k_scale=ks)
    sample = op.make_sample(p_idx, wl.S, 3 * wl.k)
    idx, sc = op(dc["q"], dc["w"], dc["k_cache"], dc["positions"], k=wl.k, prev_topk=sample,
                 q_scale=dc["q_scale"], k_scale=dc["k_scale"])
    torch.cuda.synchronize()
    st = op.stats()
    assert st["device_status"] == 0 and st["visible_pairs"] == wl.visible_pairs
    out = {"idx": idx.cpu().numpy(), "sc": sc.cpu().numpy(), "stats": st,
           "prev_idx": p_idx.cpu().numpy(), "prev_sc": p_sc.cpu().numpy()}
    if decoupled:
        d_idx, d_sc = op.decoupled(dc["q"], dc["w"], dc["k_cache"], dc["positions"], k=wl.k,
                                   q_scale=dc["q_scale"], k_scale=dc["k_scale"])
        torch.cuda.synchronize()
        out["dec_identical"] = bool(torch.equal(d_idx, idx) and torch.equal(d_sc, sc))
    op.close()
    del dp, dc
    torch.cuda.empty_cache()
    keys64 = orc.widen_keys(cur)
    q = _sample_queries(wl.T, n_check, 7)
    qp = _sample_queries(prev.T, 4, 8)
    if integer:
        # exact fp32 sums: indices and scores bit for bit, ties to the lower index
        check_exact(cur, out["idx"], out["sc"], wl.k, queries=q)
        check_exact(prev, out["prev_idx"], out["prev_sc"], wl.k, queries=qp)
    else:
        check_tolerant(cur, out["idx"], out["sc"], wl.k, queries=q, keys64=keys64)
        # the previous chunk, too (its sample was random)
        check_tolerant(prev, out["prev_idx"], out["prev_sc"], wl.k, queries=qp,
                       keys64=keys64[:prev.S])
    _invariants(out["idx"], out["sc"], cur.positions, wl.S, wl.k)
    _invariants(out["prev_idx"], out["prev_sc"], prev.positions, prev.S, wl.k)
    return out


def test_128k_two_consecutive_chunks():
    out = _chunk_pair("128k_chunk1", "128k_chunk2", "bf16", 64, decoupled=True)
    assert out["dec_identical"]
    assert out["stats"]["n_overflow"] == 0


def test_128k_two_consecutive_chunks_integer():
    """Integer-valued q, k and power-of-two w: every score is exact, and the
    k-th score is shared by many keys, so Select's boundary bin is crowded.
    Bit-exact against the oracle on 64 sampled queries, identical to the
    decoupled path on all 8192."""
    out = _chunk_pair("128k_chunk1", "128k_chunk2", "bf16", 64, decoupled=True, integer=True)
    assert out["dec_identical"]


def test_256k_chunk():
    out = _chunk_pair("256k_prev", "256k", "bf16", 64, decoupled=True)
    assert out["dec_identical"]
    assert out["stats"]["n_overflow"] == 0


def test_1m_chunk_bf16():
    out = _chunk_pair("1m_prev", "1m", "bf16", 64, decoupled=True)
    assert out["dec_identical"]
    assert out["stats"]["n_overflow"] == 0


def test_1m_chunk_fp8():
    out = _chunk_pair("1m_prev", "1m", "fp8", 64, decoupled=True)
    assert out["dec_identical"]
    assert out["stats"]["n_overflow"] == 0


def test_retrieval_full_size():
    """Vector retrieval at the full workload size: 1024 queries x 8,388,608
    corpus rows, d = 768, k = 1000, sample 3000 -- the configuration bench.py
    times.  Sampled queries against the oracle's fp64 scores over the whole
    corpus; every query against the same-GPU decoupled path (same fp32 scores,
    independent selection) and the invariants."""
    import torch
    T, N, d, k = 1024, 8388608, 768, 1000
    q, c = datagen.retrieval_inputs_torch(N, T, d, seed=20260715, device="cuda")
    op = IndexerTopK(max_T=T, max_S=N, k=k, heads=1, dim=d, sample_size=3000, enable_decoupled=1)
    qi, ci = q.view(torch.int16), c.view(torch.int16)
    w = torch.ones((T, 1), dtype=torch.float32, device="cuda")
    idx, sc = op(qi, w, ci, None, k=k)
    torch.cuda.synchronize()
    st = op.stats()
    assert st["device_status"] == 0 and st["visible_pairs"] == T * N
    d_idx, d_sc = op.decoupled(qi, w, ci, None, k=k)
    torch.cuda.synchronize()
    if st["n_overflow"] == 0:
        assert torch.equal(d_idx, idx) and torch.equal(d_sc, sc)
    op.close()
    del d_idx, d_sc
    idx_h, sc_h = idx.cpu().numpy(), sc.cpu().numpy()
    _invariants(idx_h, sc_h, np.full(T, N - 1, np.int32), N, k)
    qb = qi.cpu().numpy().view(np.uint16)
    cb = ci.cpu().numpy().view(np.uint16)
    del q, c, qi, ci, idx, sc
    torch.cuda.empty_cache()
    rows = _sample_queries(T, 4, 9)
    I = orc.retrieval_scores(qb, cb, rows=rows)
    for r, t in enumerate(rows):
        check_row_tolerant(idx_h[t], sc_h[t], I[r], k, where=f"query {t}")
