"""The fused call captured in a CUDA graph (stream capture) and replayed.

The call makes no host synchronisation and no allocation, so one decode-size
call can be captured once and replayed: the replay must give the eager
results, and it must read the input buffers at replay time (new contents,
same pointers, new results).
"""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, to_device

pytestmark = pytest.mark.gpu


def test_capture_and_replay_matches_eager():
    import torch
    T, S, k = 3, 40000, 512
    inp = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=True, seed=71)
    inp2 = datagen.make_indexer_inputs(T=T, first_pos=S - T, S=S, integer=True, seed=72)
    d = to_device(inp)
    op = IndexerTopK(max_T=T, max_S=S, k=k)
    first = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k)
    sample = op.make_sample(first[0], S, 3 * k)
    out = (torch.empty((T, k), dtype=torch.int32, device="cuda"),
           torch.empty((T, k), dtype=torch.float32, device="cuda"))
    call = lambda: op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, prev_topk=sample, out=out)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                      # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = (out[0].cpu().numpy().copy(), out[1].cpu().numpy().copy())
    check_exact(inp, eager[0], eager[1], k)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out[0].fill_(-7)
    out[1].fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out[0].cpu().numpy(), eager[0])
    np.testing.assert_array_equal(out[1].cpu().numpy(), eager[1])
    assert op.stats()["device_status"] == 0

    # same buffers, new contents: the replay scores the new inputs
    d2 = to_device(inp2)
    for name in ("q", "w", "k_cache"):
        d[name].copy_(d2[name])
    g.replay()
    torch.cuda.synchronize()
    check_exact(inp2, out[0].cpu().numpy(), out[1].cpu().numpy(), k)
    op.close()
