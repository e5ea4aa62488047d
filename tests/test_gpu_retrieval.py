"""Vector-retrieval variant (one head, plain inner product, no causal mask):
the CUDA path against the oracle's retrieval_topk.

Sizes span several corpus tiles and query blocks with ragged tails
(corpus not a multiple of 128, queries not a multiple of 256).  Integer-valued
inputs make the fp32 dot products exact, so those cases must match bit for bit
(including the lower-index rule on the many exact ties).
"""
import numpy as np
import pytest

import oracle.indexer_topk as orc
from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_row_tolerant

pytestmark = pytest.mark.gpu


def _inputs(T, N, d, seed, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        q = rng.integers(-3, 4, size=(T, d)).astype(np.float32)
        c = rng.integers(-3, 4, size=(N, d)).astype(np.float32)
    else:
        c = datagen.retrieval_corpus_block(0, N, d=d, n_centroids=64, seed=seed, block=4096)
        q = datagen.retrieval_queries(T, d=d, n_centroids=64, seed=seed)
    return datagen.bf16_bits(q), datagen.bf16_bits(c)


def _run(qb, cb, k, **cfg):
    import torch
    T, d = qb.shape
    N = cb.shape[0]
    op = IndexerTopK(max_T=T, max_S=N, k=k, heads=1, dim=d, **cfg)
    q = torch.from_numpy(qb.view(np.int16)).cuda()
    c = torch.from_numpy(cb.view(np.int16)).cuda()
    w = torch.ones((T, 1), dtype=torch.float32, device="cuda")
    idx, sc = op(q, w, c, None, k=k)
    torch.cuda.synchronize()
    out = {"idx": idx.cpu().numpy(), "sc": sc.cpu().numpy(), "stats": op.stats()}
    if cfg.get("enable_decoupled"):
        di, ds = op.decoupled(q, w, c, None, k=k)
        out["dec_equal"] = bool(torch.equal(di, idx) and torch.equal(ds, sc))
    torch.cuda.synchronize()
    op.close()
    assert out["stats"]["device_status"] == 0
    return out


@pytest.mark.parametrize("T,N,k", [(40, 30001, 1000), (300, 20000, 100)])
def test_retrieval_gaussian(T, N, k):
    qb, cb = _inputs(T, N, 768, seed=T)
    out = _run(qb, cb, k, enable_decoupled=1)
    # same fp32 scores, same selection (a rescued query would be recomputed on
    # CUDA cores, so equality is only required without overflow)
    assert out["stats"]["n_overflow"] == 0 and out["dec_equal"]
    S = orc.bf16_to_f64(qb) @ orc.bf16_to_f64(cb).T
    for t in range(T):
        check_row_tolerant(out["idx"][t], out["sc"][t], S[t], k, where=f"query {t}")


def test_retrieval_integer_exact():
    qb, cb = _inputs(20, 9000, 256, seed=5, integer=True)
    out = _run(qb, cb, 500)
    ref_idx, ref_sc = orc.retrieval_topk(qb, cb, 500)
    np.testing.assert_array_equal(out["idx"], ref_idx)
    np.testing.assert_array_equal(out["sc"], ref_sc)


def test_retrieval_overflow_rescued():
    qb, cb = _inputs(10, 5000, 768, seed=6, integer=True)
    out = _run(qb, cb, 300, cand_cap=320, refresh_interval=0, n_bins=32)
    assert out["stats"]["n_overflow"] > 0
    ref_idx, ref_sc = orc.retrieval_topk(qb, cb, 300)
    np.testing.assert_array_equal(out["idx"], ref_idx)
    np.testing.assert_array_equal(out["sc"], ref_sc)


@pytest.mark.parametrize("k", [2048, 4096, 8192])
def test_retrieval_large_k(k):
    """k from 1024 to 8192, the range of the pages' retrieval comparison."""
    qb, cb = _inputs(48, 100003, 768, seed=k)
    out = _run(qb, cb, k, enable_decoupled=1)
    assert out["stats"]["n_overflow"] == 0 and out["dec_equal"]
    S = orc.bf16_to_f64(qb) @ orc.bf16_to_f64(cb).T
    for t in range(0, 48, 5):
        check_row_tolerant(out["idx"][t], out["sc"][t], S[t], k, where=f"query {t}")


def test_retrieval_segments_overflow_rescued():
    """Several corpus ranges per query (one list segment each) with segments far
    too small: the overflowed queries are recomputed exactly."""
    qb, cb = _inputs(12, 100003, 256, seed=8, integer=True)
    out = _run(qb, cb, 300, cand_cap=600)
    assert out["stats"]["n_overflow"] > 0
    ref_idx, ref_sc = orc.retrieval_topk(qb, cb, 300)
    np.testing.assert_array_equal(out["idx"], ref_idx)
    np.testing.assert_array_equal(out["sc"], ref_sc)


def test_retrieval_relu_scores():
    """One head with ReLU (the retrieval kernel's ReLU form) against the
    oracle's plain definition with H = 1, w = 1, no mask."""
    qb, cb = _inputs(33, 20011, 256, seed=9, integer=True)
    T, d = qb.shape
    out = _run(qb, cb, 400, relu=1)
    inp = datagen.IndexerInputs(dtype="bf16", q=qb.reshape(T, 1, d), k=cb,
                                w=np.ones((T, 1), np.float32), positions=np.zeros(T, np.int32))
    ref_idx, ref_sc = orc.indexer_topk(inp, 400, causal=False, relu=True)
    np.testing.assert_array_equal(out["idx"], ref_idx)
    np.testing.assert_array_equal(out["sc"], ref_sc)
