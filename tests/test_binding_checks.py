"""The Python binding's argument checks (no GPU): every tensor's device,
layout, element type and element count is checked before a call reaches the
C library, whose plain pointers carry no size, so a short or mistyped tensor
cannot make a kernel read or write past its end."""
import pytest
import torch

from indexer_topk_long_gb300.ltk import check_inputs

H, D = 64, 128


def _args(T=5, S=300, dtype="bf16", k=16):
    code = torch.int16 if dtype == "bf16" else torch.uint8
    a = dict(q=torch.zeros((T, H, D), dtype=code), w=torch.zeros((T, H), dtype=torch.float32),
             k_cache=torch.zeros((S, D), dtype=code),
             positions=torch.arange(S - T, S, dtype=torch.int32),
             out=(torch.empty((T, k), dtype=torch.int32), torch.empty((T, k), dtype=torch.float32)))
    if dtype == "fp8":
        a["q_scale"] = torch.ones(T, dtype=torch.float32)
        a["k_scale"] = torch.ones(S, dtype=torch.float32)
    return a


def _check(dtype="bf16", causal=True, k=16, heads=H, dim=D, **a):
    return check_inputs(heads, dim, dtype, causal, k=k, device_type="cpu", **a)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_well_formed_calls_pass(dtype):
    assert _check(dtype, **_args(dtype=dtype)) == (5, 300)
    a = _args(dtype=dtype)
    a["prev_topk"] = torch.arange(40, dtype=torch.int32)
    assert _check(dtype, **a) == (5, 300)


def test_empty_chunk_needs_no_positions_or_scales():
    a = _args(T=0, dtype="fp8")
    a["positions"] = a["q_scale"] = a["k_scale"] = None
    assert _check("fp8", **a) == (0, 300)


def test_one_head_retrieval_shapes():
    T, N, d = 4, 1000, 768
    a = dict(q=torch.zeros((T, d), dtype=torch.bfloat16), w=torch.ones((T, 1)),
             k_cache=torch.zeros((N, d), dtype=torch.bfloat16))
    assert _check("bf16", causal=False, heads=1, dim=d, **a) == (T, N)


@pytest.mark.parametrize("field,bad,msg", [
    ("w", torch.zeros((5, H), dtype=torch.bfloat16), "float32"),
    ("w", torch.zeros((5, H - 1), dtype=torch.float32), "elements"),
    ("positions", torch.arange(5, dtype=torch.int64), "int32"),
    ("positions", torch.arange(4, dtype=torch.int32), "elements"),
    ("q", torch.zeros((5, H, D), dtype=torch.float32), "2-byte"),
    ("q", torch.zeros((5, D, H), dtype=torch.int16).transpose(1, 2), "contiguous"),
    ("k_cache", torch.zeros((300, D - 8), dtype=torch.int16), "elements"),
    ("prev_topk", torch.arange(10, dtype=torch.int64), "int32"),
    ("out", (torch.empty((5, 15), dtype=torch.int32), torch.empty((5, 16))), "elements"),
    ("out", (torch.empty((5, 16), dtype=torch.int32), torch.empty((5, 16), dtype=torch.float64)),
     "float32"),
])
def test_malformed_tensor_rejected(field, bad, msg):
    a = _args()
    a[field] = bad
    with pytest.raises(ValueError, match=msg):
        _check(**a)


def test_causal_handle_requires_positions():
    a = _args()
    a["positions"] = None
    with pytest.raises(ValueError, match="positions"):
        _check(**a)
    assert _check(causal=False, **a) == (5, 300)


@pytest.mark.parametrize("field", ["q_scale", "k_scale"])
def test_e4m3_requires_fp32_scales(field):
    a = _args(dtype="fp8")
    a[field] = None
    with pytest.raises(ValueError, match=field):
        _check("fp8", **a)
    a = _args(dtype="fp8")
    a[field] = a[field].double()
    with pytest.raises(ValueError, match="float32"):
        _check("fp8", **a)


def test_wrong_device_rejected():
    with pytest.raises(ValueError, match="expected a cuda tensor"):
        check_inputs(H, D, "bf16", True, k=16, device_type="cuda", **_args())
