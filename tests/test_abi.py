"""The C-ABI library: loads, exports every function include/ltk.h declares, and
validates arguments on the host before touching the GPU (no GPU needed)."""
import ctypes

import pytest

from indexer_topk_long_gb300 import ltk


def test_exports_every_declared_function(ltk_lib):
    names = ltk.header_functions()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(ltk_lib, n)]
    assert not missing, missing
    assert set(names) == set(ltk._SIGS), "binding signatures out of sync with the header"


def test_abi_version_and_status_strings(ltk_lib):
    assert ltk_lib.ltk_abi_version() == 2
    assert ltk_lib.ltk_status_string(0) == b"ok"
    assert ltk_lib.ltk_status_string(5) == b"device wait timed out"


def _cfg(**kw):
    cfg = ltk.config_defaults(64, 128, 2048, 8192, 1 << 20)
    for k, v in kw.items():
        setattr(cfg, k, v)
    return cfg


def test_config_defaults(ltk_lib):
    cfg = _cfg()
    assert (cfg.heads, cfg.dim, cfg.k, cfg.relu, cfg.causal, cfg.n_bins) == (64, 128, 2048, 1, 1, 512)
    assert cfg.refresh_interval == 1 and cfg.sample_size == 0 and cfg.dtype == ltk.LTK_BF16


def test_workspace_sizing(ltk_lib):
    base = ltk.workspace_bytes(_cfg())
    # candidate lists dominate: 8192 queries x derived cap x 8 bytes
    assert 1 << 30 < base < 4 << 30
    dec = ltk.workspace_bytes(_cfg(enable_decoupled=1))
    assert dec - base == 8192 * (1 << 20) * 4          # the full fp32 score matrix
    small = ltk.workspace_bytes(_cfg(max_T=32, max_S=8192))
    assert small < base


@pytest.mark.parametrize("field,value,status", [
    ("k", 0, 1), ("k", 8193, 1), ("max_S", 0, 1), ("max_S", 1 << 31, 1), ("n_bins", 100, 1),
    ("n_bins", 16, 1), ("dtype", 7, 1), ("sample_size", 20000, 1), ("heads", 256, 6),
    ("dim", 12, 6), ("dim", 8192, 6), ("n_bins", 8192, 6), ("debug_flags", 2, 1), ("engine", 3, 1),
])
def test_invalid_configs_rejected_on_host(ltk_lib, field, value, status):
    cfg = _cfg(**{field: value})
    out = ctypes.c_ulonglong(0)
    assert ltk_lib.ltk_workspace_bytes(ctypes.byref(cfg), ctypes.byref(out)) == status
    h = ctypes.c_void_p()
    assert ltk_lib.ltk_create(ctypes.byref(cfg), ctypes.byref(h)) == status
    assert not h.value


def test_fp8_allows_more_bins(ltk_lib):
    cfg = _cfg(dtype=ltk.LTK_FP8_E4M3, n_bins=2048)
    out = ctypes.c_ulonglong(0)
    assert ltk_lib.ltk_workspace_bytes(ctypes.byref(cfg), ctypes.byref(out)) == 0


def test_null_handle_calls_rejected(ltk_lib):
    assert ltk_lib.ltk_create(None, None) == 1
    assert ltk_lib.ltk_indexer_topk(None, None, None, None, None, None, None, 1, 10, None, 0, 1,
                                    None, None, None) == 1
    assert ltk_lib.ltk_decoupled_topk(None, None, None, None, None, None, None, 1, 10, 1,
                                      None, None, None) == 1
    assert ltk_lib.ltk_get_stats(None, None) == 1
    assert ltk_lib.ltk_set_timing(None, 1) == 1
    ltk_lib.ltk_destroy(None)


@pytest.mark.parametrize("heads,dim,engine,status", [
    (32, 64, 0, 0), (32, 64, 1, 6), (32, 64, 2, 0), (64, 128, 2, 0), (1, 768, 0, 0), (1, 768, 2, 0),
    (200, 64, 0, 6), (64, 4104, 0, 6)])
def test_engine_selection_on_host(ltk_lib, heads, dim, engine, status):
    cfg = _cfg(heads=heads, dim=dim, engine=engine)
    if heads == 1:
        cfg.relu, cfg.causal, cfg.n_bins = 0, 0, 64
    out = ctypes.c_ulonglong(0)
    assert ltk_lib.ltk_workspace_bytes(ctypes.byref(cfg), ctypes.byref(out)) == status
