"""The decoupled baseline's row select (and the overflow rescue, which uses the
same select on a recomputed row) on rows that take each of its paths: spread
scores (equal-width bins over the row's range, boundary bin in shared memory),
rows with no spread (every score equal: the crowded-bin radix fallback), rows
with one huge tie group, and rows with fewer visible keys than k.  Integer
inputs: bit-exact against the oracle, and identical to the fused path."""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, to_device

pytestmark = pytest.mark.gpu


def _both(inp, k):
    import torch
    op = IndexerTopK(max_T=inp.T, max_S=inp.S, k=k, enable_decoupled=1)
    d = to_device(inp)
    i1, s1 = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=k)
    i2, s2 = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k)
    torch.cuda.synchronize()
    op.close()
    return i1.cpu().numpy(), s1.cpu().numpy(), i2.cpu().numpy(), s2.cpu().numpy()


def test_row_select_paths():
    T, S, k = 12, 20000, 1500
    pos = np.array([19999, 19998, 19990, 15000, 9000, 4097, 4096, 1499, 700, 20, 0, 19999], np.int32)
    inp = datagen.make_indexer_inputs(T=T, first_pos=0, S=S, integer=True, seed=91, positions=pos)
    inp.q[1] = 0                       # no spread: every visible score is 0 (radix fallback)
    inp.w[2] = 0                       # the same through zero weights
    inp.q[3] = inp.q[3] * 0            # likewise, 15001 equal scores
    # one huge tie group: keys copied so that thousands share the top scores
    inp.k[5000:14000] = inp.k[5000]
    i1, s1, i2, s2 = _both(inp, k)
    check_exact(inp, i1, s1, k)
    np.testing.assert_array_equal(i1, i2)
    np.testing.assert_array_equal(s1, s2)


def test_row_select_gaussian_many_rows():
    """Gaussian rows over a few k, the bucket path's usual case."""
    import torch
    from parity import check_tolerant
    T, S = 40, 30000
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, seed=92)
    for k in (1, 37, 2048, 8192):
        op = IndexerTopK(max_T=T, max_S=S, k=k, enable_decoupled=1)
        d = to_device(inp)
        i1, s1 = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=k)
        i2, s2 = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k)
        torch.cuda.synchronize()
        op.close()
        assert torch.equal(i1, i2) and torch.equal(s1, s2), k
        check_tolerant(inp, i1.cpu().numpy(), s1.cpu().numpy(), k, queries=[0, 17, 39])
