"""The allocation-free decoupled entry point against the handle-based one.

ltk_decoupled_topk_noalloc exists for callers that cannot call cudaMalloc
(an engine that owns all device memory through its own pool, or a path that
cannot take cudaMalloc's implicit device synchronisation): it keeps its score
matrix in a static device array instead of a handle's workspace.  This file is
collected last so that a failure here does not hide any other test.
"""
import ctypes

import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen, ltk
from parity import check_row_tolerant, to_device
import oracle.indexer_topk as orc

pytestmark = pytest.mark.gpu


def _noalloc(lib, d, T, S, k, dtype=0, causal=1):
    import torch
    oi = torch.empty((T, k), dtype=torch.int32, device="cuda")
    os_ = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ptr = lambda t: None if t is None else t.data_ptr()
    st = lib.ltk_decoupled_topk_noalloc(dtype, causal, ptr(d["q"]), ptr(d["q_scale"]), ptr(d["w"]),
                                        ptr(d["k_cache"]), ptr(d["k_scale"]), ptr(d["positions"]),
                                        T, S, k, ptr(oi), ptr(os_),
                                        torch.cuda.current_stream().cuda_stream)
    return st, oi, os_


@pytest.mark.parametrize("calls", [[(12, 5000, 512, 21), (40, 20000, 2048, 22)]])
def test_noalloc_matches_handle_entry_point(calls):
    import torch
    lib = ltk.load_library()
    for T, S, k, seed in calls:            # two calls in a row share the static array
        inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, seed=seed)
        d = to_device(inp)
        st, i1, s1 = _noalloc(lib, d, T, S, k)
        assert st == 0
        op = IndexerTopK(max_T=T, max_S=S, k=k, enable_decoupled=1)
        i2, s2 = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=k)
        torch.cuda.synchronize()
        op.close()
        a_idx, a_sc = i1.cpu().numpy(), s1.cpu().numpy()
        b_idx, b_sc = i2.cpu().numpy(), s2.cpu().numpy()
        keys64 = orc.widen_keys(inp)
        for t in range(T):
            I = orc.full_scores(inp, t, keys64=keys64)
            check_row_tolerant(a_idx[t], a_sc[t], I, k, where=f"noalloc query {t}")
            check_row_tolerant(b_idx[t], b_sc[t], I, k, where=f"handle query {t}")
            # against the handle-based entry point, with the tests' tolerance:
            # same keys except near-tie swaps (both checked above), and equal
            # scores within 1e-4 * (1 + |s|) wherever the keys agree
            agree = a_idx[t] == b_idx[t]
            valid = agree & (b_idx[t] >= 0)
            assert agree[b_idx[t] < 0].all()
            assert np.all(np.abs(a_sc[t][valid] - b_sc[t][valid]) <= 1e-4 * (1 + np.abs(b_sc[t][valid])))


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = ltk.load_library()
    assert lib.ltk_decoupled_topk_noalloc(0, 1, None, None, None, None, None, None,
                                          8192, 1 << 20, 16, None, None, None) == 1
