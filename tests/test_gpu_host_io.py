"""ltk_indexer_topk_host: the same call with every buffer in pinned host memory
(the library stages inputs to the device, runs the path, copies results
back).  Results must equal the device-buffer call's and match the oracle."""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, check_tolerant, to_device

pytestmark = pytest.mark.gpu


def _host(t):
    return None if t is None else t.cpu().pin_memory()


@pytest.mark.parametrize("dtype,integer", [("bf16", True), ("fp8", False)])
def test_host_buffers_match_device_call_and_oracle(dtype, integer):
    import torch
    T, S, k = 21, 7000, 700
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, dtype=dtype, integer=integer, seed=81)
    op = IndexerTopK(max_T=T, max_S=S, k=k, dtype=dtype, enable_host_io=1)
    d = to_device(inp)
    di, ds = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, q_scale=d["q_scale"],
                k_scale=d["k_scale"])
    h = {key: _host(v) for key, v in d.items()}
    hi, hs = op.topk_host(h["q"], h["w"], h["k_cache"], h["positions"], k=k, q_scale=h["q_scale"],
                          k_scale=h["k_scale"])
    # and with a previous-chunk sample given as host ids
    smp = _host(op.make_sample(di, S, 2100))
    hi2, hs2 = op.topk_host(h["q"], h["w"], h["k_cache"], h["positions"], k=k, prev_topk=smp,
                            q_scale=h["q_scale"], k_scale=h["k_scale"])
    torch.cuda.synchronize()
    assert op.stats()["device_status"] == 0
    op.close()
    assert hi.device.type == "cpu"
    np.testing.assert_array_equal(hi.numpy(), di.cpu().numpy())
    np.testing.assert_array_equal(hs.numpy(), ds.cpu().numpy())
    np.testing.assert_array_equal(hi2.numpy(), hi.numpy())
    np.testing.assert_array_equal(hs2.numpy(), hs.numpy())
    if integer:
        check_exact(inp, hi.numpy(), hs.numpy(), k)
    else:
        check_tolerant(inp, hi.numpy(), hs.numpy(), k)
