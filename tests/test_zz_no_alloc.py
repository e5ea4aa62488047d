"""The allocation-free decoupled entry point against the handle-based one.

ltk_decoupled_topk_noalloc exists for callers that cannot call cudaMalloc
(an engine that owns all device memory through its own pool, or a path that
cannot take cudaMalloc's implicit device synchronisation): it keeps its score
matrix in a static device array instead of a handle's workspace.  This file is
collected last so that a failure here does not hide any other test.
"""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen, ltk
from parity import check_row_tolerant, to_device
import oracle.indexer_topk as orc

pytestmark = pytest.mark.gpu


def _compare(inp, k, a_idx, a_sc, b_idx, b_sc, causal):
    keys64 = orc.widen_keys(inp)
    for t in range(inp.T):
        I = orc.full_scores(inp, t, causal=causal, keys64=keys64)
        check_row_tolerant(a_idx[t], a_sc[t], I, k, where=f"noalloc query {t}")
        check_row_tolerant(b_idx[t], b_sc[t], I, k, where=f"handle query {t}")
        # against the handle-based entry point, with the tests' tolerance:
        # same keys except near-tie swaps (both checked above), and equal
        # scores within 1e-4 * (1 + |s|) wherever the keys agree
        agree = a_idx[t] == b_idx[t]
        valid = agree & (b_idx[t] >= 0)
        assert agree[b_idx[t] < 0].all()
        assert np.all(np.abs(a_sc[t][valid] - b_sc[t][valid]) <= 1e-4 * (1 + np.abs(b_sc[t][valid])))


# Each case is two calls in a row: the second reuses the static array the
# first one filled (different sizes, so stale scores would show).
CASES = {
    "bf16_causal": [(12, 5000, 512, 21, "bf16", True), (40, 20000, 2048, 22, "bf16", True)],
    "fp8_causal": [(9, 7000, 700, 23, "fp8", True), (33, 30000, 2048, 24, "fp8", True)],
    "bf16_no_mask": [(5, 9000, 1000, 25, "bf16", False), (17, 3000, 300, 26, "bf16", False)],
}


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_noalloc_matches_handle_entry_point(case):
    import torch
    for T, S, k, seed, dtype, causal in CASES[case]:
        inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, seed=seed, dtype=dtype)
        d = to_device(inp)
        i1, s1, status = ltk.decoupled_noalloc(d["q"], d["w"], d["k_cache"], d["positions"], k=k,
                                               dtype=dtype, causal=causal, q_scale=d["q_scale"],
                                               k_scale=d["k_scale"])
        op = IndexerTopK(max_T=T, max_S=S, k=k, dtype=dtype, causal=1 if causal else 0,
                         enable_decoupled=1)
        i2, s2 = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"] if causal else None,
                              k=k, q_scale=d["q_scale"], k_scale=d["k_scale"])
        torch.cuda.synchronize()
        op.close()
        assert int(status.item()) == 0
        _compare(inp, k, i1.cpu().numpy(), s1.cpu().numpy(), i2.cpu().numpy(), s2.cpu().numpy(),
                 causal)


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = ltk.load_library()
    assert lib.ltk_decoupled_topk_noalloc(0, 1, None, None, None, None, None, None,
                                          8192, 1 << 20, 16, None, None, None, None) == 1
