"""CUDA-core engine (bin map fused into the score, scores recovered through the
inverse affine map) against the oracle, for the standard shape and for shapes
the tensor-core kernels do not serve.

delta is a power of two on this engine, so w * delta and the inverse map are
exact: on integer-valued inputs the results must match the oracle bit for bit,
and the fused path must return exactly the decoupled (dense) path's scores.
Floating-point inputs use the tolerance rule.
"""
import numpy as np
import pytest

from indexer_topk_long_gb300 import IndexerTopK, datagen
from parity import check_exact, check_tolerant, to_device

pytestmark = pytest.mark.gpu


def _run(inp, k, **cfg):
    import torch
    op = IndexerTopK(max_T=inp.T, max_S=inp.S, k=k, heads=inp.q.shape[1], dim=inp.q.shape[2],
                     dtype=inp.dtype, **cfg)
    d = to_device(inp)
    idx, sc = op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, q_scale=d["q_scale"],
                 k_scale=d["k_scale"])
    torch.cuda.synchronize()
    st = op.stats()
    out = {"idx": idx.cpu().numpy(), "sc": sc.cpu().numpy(), "stats": st}
    if cfg.get("enable_decoupled"):
        di, ds = op.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=k,
                              q_scale=d["q_scale"], k_scale=d["k_scale"])
        torch.cuda.synchronize()
        out["dec_idx"], out["dec_sc"] = di.cpu().numpy(), ds.cpu().numpy()
    op.close()
    assert st["device_status"] == 0
    return out


def test_standard_shape_on_cuda_cores():
    inp = datagen.make_indexer_inputs(T=24, first_pos=6000, S=6024, seed=51)
    out = _run(inp, 1024, engine=2, enable_decoupled=1)
    check_tolerant(inp, out["idx"], out["sc"], 1024)
    check_tolerant(inp, out["dec_idx"], out["dec_sc"], 1024)


@pytest.mark.parametrize("H,d,dtype,integer", [(32, 64, "bf16", False), (16, 256, "fp8", False),
                                               (8, 128, "bf16", True), (3, 40, "bf16", False),
                                               (32, 64, "bf16", True), (64, 128, "bf16", True)])
def test_other_shapes(H, d, dtype, integer):
    inp = datagen.make_indexer_inputs(T=13, first_pos=3000, S=3013, H=H, d=d, dtype=dtype,
                                      integer=integer, seed=H * d)
    # (64, 128) is the tensor-core shape: force the CUDA-core engine there
    out = _run(inp, 512, enable_decoupled=1, **({"engine": 2} if (H, d) == (64, 128) else {}))
    assert out["stats"]["n_overflow"] == 0
    if integer:
        check_exact(inp, out["idx"], out["sc"], 512)
        check_exact(inp, out["dec_idx"], out["dec_sc"], 512)
    else:
        check_tolerant(inp, out["idx"], out["sc"], 512)
    # the inverse map returns the dense path's own fp32 scores
    np.testing.assert_array_equal(out["idx"], out["dec_idx"])
    np.testing.assert_array_equal(out["sc"], out["dec_sc"])


def test_decode_split_on_cuda_cores():
    inp = datagen.make_indexer_inputs(T=2, first_pos=199998, S=200000, H=32, d=64, seed=52)
    out = _run(inp, 2048)
    check_tolerant(inp, out["idx"], out["sc"], 2048)


def test_decode_split_on_cuda_cores_integer():
    """Key ranges split over many CTAs (global histogram), integer inputs: bit-exact."""
    inp = datagen.make_indexer_inputs(T=3, first_pos=131069, S=131072, H=16, d=64, integer=True,
                                      seed=54)
    out = _run(inp, 2048)
    check_exact(inp, out["idx"], out["sc"], 2048)


def test_overflow_rescue_generic_shape():
    inp = datagen.make_indexer_inputs(T=6, first_pos=2500, S=2506, H=24, d=48, seed=53)
    out = _run(inp, 200, cand_cap=256, refresh_interval=0, n_bins=32)
    assert out["stats"]["n_overflow"] > 0
    check_tolerant(inp, out["idx"], out["sc"], 200)
