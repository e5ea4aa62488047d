"""Small chunks (T <= 8) and the sample-id preparation, on the GPU against the
oracle.

T <= 4 runs the scorer's alternating form (one query group, narrower MMA,
two accumulators alternating between tiles, deeper key ring); T = 5..7 the
general form with a partial second group.  The sample ids go through a bitmap
of the key range, so duplicates, out-of-range ids and calls with different
cache lengths on one handle must not change any result.
"""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, check_tolerant, to_device

pytestmark = pytest.mark.gpu


def _call(op, inp, k, prev=None):
    import torch
    d = to_device(inp)
    idx, sc = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, prev_topk=prev,
                 q_scale=d["q_scale"], k_scale=d["k_scale"])
    torch.cuda.synchronize()
    assert op.stats()["device_status"] == 0
    return idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("T,S,integer", [(2, 90001, True), (3, 100000, True), (4, 70000, False),
                                         (6, 50000, True), (7, 65536, False)])
def test_small_chunks_fused(T, S, integer):
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=integer, seed=300 + T)
    op = IndexerTopK(max_T=T, max_S=S, k=2048)
    idx, sc = _call(op, inp, 2048)
    # and again with the previous call's selection as the sample
    import torch
    prev = op.make_sample(torch.from_numpy(idx).cuda(), S, 6144)
    idx2, sc2 = _call(op, inp, 2048, prev)
    op.close()
    np.testing.assert_array_equal(idx, idx2)
    np.testing.assert_array_equal(sc, sc2)
    if integer:
        check_exact(inp, idx, sc, 2048)
    else:
        check_tolerant(inp, idx, sc, 2048)


@pytest.mark.parametrize("T", [1, 3, 6])
def test_small_chunks_decoupled(T):
    """The dense scorer in the same forms (decoupled baseline) against the oracle."""
    import torch
    S = 40000
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=True, seed=320 + T)
    d = to_device(inp)
    op = IndexerTopK(max_T=T, max_S=S, k=512, enable_decoupled=1)
    idx, sc = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=512)
    torch.cuda.synchronize()
    op.close()
    check_exact(inp, idx.cpu().numpy(), sc.cpu().numpy(), 512)


def test_messy_sample_ids_do_not_change_results():
    """Duplicates, -1, ids past the cache and a full-size list as the sample."""
    import torch
    T, S, k = 5, 30000, 700
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=True, seed=333)
    op = IndexerTopK(max_T=T, max_S=S, k=k)
    ref = _call(op, inp, k)
    rng = np.random.default_rng(5)
    ids = rng.integers(-5, S + 5000, size=16384).astype(np.int32)
    ids[:4000] = ids[4000:8000]            # many duplicates
    ids[100:200] = -1
    out = _call(op, inp, k, torch.from_numpy(ids).cuda())
    np.testing.assert_array_equal(out[0], ref[0])
    np.testing.assert_array_equal(out[1], ref[1])
    same = np.full(3000, 17, dtype=np.int32)   # one key, 3000 times
    out = _call(op, inp, k, torch.from_numpy(same).cuda())
    np.testing.assert_array_equal(out[0], ref[0])
    op.close()
    check_exact(inp, ref[0], ref[1], k)


def test_one_handle_different_cache_lengths():
    """Calls with a long, a short and again a long cache on one handle."""
    k = 300
    op = IndexerTopK(max_T=8, max_S=60000, k=k)
    for S, seed in [(60000, 341), (9000, 342), (60000, 343), (1500, 344)]:
        inp = datagen.make_indexer_inputs(T=8, first_pos=S - 8, S=S, integer=True, seed=seed)
        idx, sc = _call(op, inp, k)
        check_exact(inp, idx, sc, k)
    op.close()


@pytest.mark.parametrize("T,S", [(1, 70000), (3, 40001)])
def test_small_chunks_fp8(T, S):
    """e4m3 q/k in the alternating form (its deeper key ring sits in the unused
    query rows of the e4m3 layout)."""
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, dtype="fp8", seed=360 + T)
    op = IndexerTopK(max_T=T, max_S=S, k=1024, dtype="fp8", enable_decoupled=1)
    idx, sc = _call(op, inp, 1024)
    import torch
    d = to_device(inp)
    di, ds = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=1024,
                          q_scale=d["q_scale"], k_scale=d["k_scale"])
    torch.cuda.synchronize()
    op.close()
    np.testing.assert_array_equal(di.cpu().numpy(), idx)
    np.testing.assert_array_equal(ds.cpu().numpy(), sc)
    check_tolerant(inp, idx, sc, 1024)
