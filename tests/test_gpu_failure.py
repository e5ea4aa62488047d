"""Failure handling without faulting the GPU.

With debug flag 1 the Filter kernel's producer issues no key-tile loads (a
barrier that nothing completes).  Every wait in the kernel is bounded: the
MMA warp's wait expires after about 2 s, it raises the CTA's abort flag and
the device status, the other roles leave their loops, TMEM is freed and the
kernel returns.  The host must read LTK_ERR_TIMEOUT, and the context must stay
usable: a normal call right after returns exact results.
"""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    inp = datagen.make_indexer_inputs(T=8, first_pos=2000, S=2008, integer=True, seed=31)
    d = to_device(inp)
    bad = IndexerTopK(max_T=8, max_S=2008, k=64, debug_flags=1)
    bad(d["q"], d["w"], d["k_cache"], d["positions"], k=64)
    torch.cuda.synchronize()
    assert bad.stats()["device_status"] == 5          # LTK_ERR_TIMEOUT
    bad.close()
    good = IndexerTopK(max_T=8, max_S=2008, k=64)
    idx, sc = good(d["q"], d["w"], d["k_cache"], d["positions"], k=64)
    torch.cuda.synchronize()
    assert good.stats()["device_status"] == 0
    good.close()
    check_exact(inp, idx.cpu().numpy(), sc.cpu().numpy(), 64)
