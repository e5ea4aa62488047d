"""Thin ctypes binding over libltk.so (argument marshalling only).

Every step of the path runs in the library's CUDA kernels; this module only
checks tensor shapes/dtypes, passes device pointers and the current CUDA
stream, and raises on a non-zero status.  There is no fallback: if the library
is missing the calls fail.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "ltk.h")

LTK_BF16, LTK_FP8_E4M3 = 0, 1
STATUS = {0: "LTK_OK", 1: "LTK_ERR_ARG", 2: "LTK_ERR_CUDA", 3: "LTK_ERR_NOMEM",
          4: "LTK_ERR_OVERFLOW", 5: "LTK_ERR_TIMEOUT", 6: "LTK_ERR_UNSUPPORTED"}


class LtkError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class Config(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int), ("dim", ctypes.c_int), ("dtype", ctypes.c_int),
                ("relu", ctypes.c_int), ("causal", ctypes.c_int), ("max_T", ctypes.c_int),
                ("max_S", ctypes.c_longlong), ("k", ctypes.c_int), ("n_bins", ctypes.c_int),
                ("cand_cap", ctypes.c_int), ("sample_size", ctypes.c_int),
                ("seed", ctypes.c_ulonglong), ("refresh_interval", ctypes.c_int),
                ("enable_decoupled", ctypes.c_int), ("rescue_rows", ctypes.c_int),
                ("enable_host_io", ctypes.c_int), ("engine", ctypes.c_int),
                ("debug_flags", ctypes.c_int)]


class Stats(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("S", ctypes.c_longlong), ("k", ctypes.c_int),
                ("visible_pairs", ctypes.c_longlong), ("cand_written", ctypes.c_longlong),
                ("cand_max", ctypes.c_int), ("n_overflow", ctypes.c_int),
                ("device_status", ctypes.c_int), ("ms_sample", ctypes.c_float),
                ("ms_filter", ctypes.c_float), ("ms_select", ctypes.c_float),
                ("ms_rescue", ctypes.c_float), ("ms_total", ctypes.c_float),
                ("timed_calls", ctypes.c_int), ("launches", ctypes.c_longlong)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
_SIGS = {
    "ltk_abi_version": (_I, []),
    "ltk_status_string": (ctypes.c_char_p, [_I]),
    "ltk_config_init": (_I, [ctypes.POINTER(Config), _I, _I, _I, _I, _LL]),
    "ltk_workspace_bytes": (_I, [ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_ulonglong)]),
    "ltk_create": (_I, [ctypes.POINTER(Config), ctypes.POINTER(_P)]),
    "ltk_destroy": (None, [_P]),
    "ltk_set_timing": (_I, [_P, _I]),
    "ltk_random_sample": (_I, [_P, _LL, _I, _P, _P]),
    "ltk_make_sample": (_I, [_P, _P, _I, _I, _LL, _I, _P, _P]),
    "ltk_indexer_topk": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _LL, _P, _I, _I, _P, _P, _P]),
    "ltk_indexer_topk_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _LL, _P, _I, _I, _P, _P, _P]),
    "ltk_decoupled_topk": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _LL, _I, _P, _P, _P]),
    "ltk_get_stats": (_I, [_P, ctypes.POINTER(Stats)]),
    "ltk_decoupled_topk_noalloc": (_I, [_I, _I, _P, _P, _P, _P, _P, _P, _I, _LL, _I, _P, _P, _P, _P]),
    "ltk_litedsa_pack": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
}

_LIB = None


def library_path() -> str:
    return os.path.join(PKG, "libltk.so")


def load_library() -> ctypes.CDLL:
    """Load the in-tree libltk.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise LtkError(2, f"{path} is not built (python -m indexer_topk_long_gb300._build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/ltk.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ltk_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, what: str) -> None:
    if status != 0:
        raise LtkError(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream_handle(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _tensor_ok(t, name: str, numel: int, elem_size: int, device_type: str,
               dtype=None, device_index=None) -> None:
    """One tensor argument: device, contiguity, element size (and type) and
    element count, so that the kernels behind the plain pointers of the C ABI
    never read or write past the tensor's end."""
    if t.device.type != device_type:
        raise ValueError(f"{name}: expected a {device_type} tensor, got one on {t.device}")
    if device_index is not None and t.device.index != device_index:
        raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{device_index}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.element_size() != elem_size or (dtype is not None and t.dtype != dtype):
        want = str(dtype).replace("torch.", "") if dtype is not None else f"{elem_size}-byte"
        raise ValueError(f"{name}: expected {want} elements, got {t.dtype}")
    if t.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {t.numel()} (shape {tuple(t.shape)})")


def check_inputs(heads: int, dim: int, dtype: str, causal: bool, q, w, k_cache, positions=None,
                 q_scale=None, k_scale=None, prev_topk=None, out=None, k: int | None = None,
                 device_type: str = "cuda", device_index=None) -> tuple[int, int]:
    """Validates the tensors of one indexer call before anything is enqueued.

    T = q.shape[0] queries and S = k_cache.shape[0] keys; q holds T * heads *
    dim codes (2-byte bf16 or 1-byte e4m3), k_cache S * dim codes, w T * heads
    fp32 weights, positions T int32 (required by a causal handle), q_scale T
    and k_scale S fp32 (e4m3), prev_topk int32 key ids, out (int32, fp32) with
    T * k elements each.  Every tensor must be contiguous and on
    ``device_type``.  Raises ValueError; returns (T, S)."""
    import torch
    T, S = int(q.shape[0]), int(k_cache.shape[0])
    code = 2 if dtype == "bf16" else 1
    dev = dict(device_type=device_type, device_index=device_index)
    _tensor_ok(q, "q", T * heads * dim, code, **dev)
    _tensor_ok(k_cache, "k_cache", S * dim, code, **dev)
    _tensor_ok(w, "w", T * heads, 4, dtype=torch.float32, **dev)
    if positions is not None:
        _tensor_ok(positions, "positions", T, 4, dtype=torch.int32, **dev)
    elif causal and T > 0:
        raise ValueError("positions: required by a causal handle")
    if dtype == "fp8":
        for t, name, n in ((q_scale, "q_scale", T), (k_scale, "k_scale", S)):
            if t is not None:
                _tensor_ok(t, name, n, 4, dtype=torch.float32, **dev)
            elif T > 0:
                raise ValueError(f"{name}: required for e4m3 inputs")
    if prev_topk is not None:
        _tensor_ok(prev_topk, "prev_topk", prev_topk.numel(), 4, dtype=torch.int32, **dev)
    if out is not None:
        n = T * int(k)
        _tensor_ok(out[0], "out[0] (indices)", n, 4, dtype=torch.int32, **dev)
        _tensor_ok(out[1], "out[1] (scores)", n, 4, dtype=torch.float32, **dev)
    return T, S


def _index_matrix_ok(t, name: str) -> None:
    """A [rows, cols] int32 CUDA tensor of key indices on the current device."""
    import torch
    if t.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D [rows, k] tensor, got shape {tuple(t.shape)}")
    _tensor_ok(t, name, t.numel(), 4, "cuda", dtype=torch.int32,
               device_index=torch.cuda.current_device())


def config_defaults(heads=64, dim=128, k=2048, max_T=8192, max_S=1 << 20) -> Config:
    lib = load_library()
    cfg = Config()
    _check(lib.ltk_config_init(ctypes.byref(cfg), heads, dim, k, max_T, max_S), "ltk_config_init")
    return cfg


def workspace_bytes(cfg: Config) -> int:
    lib = load_library()
    out = ctypes.c_ulonglong(0)
    _check(lib.ltk_workspace_bytes(ctypes.byref(cfg), ctypes.byref(out)), "ltk_workspace_bytes")
    return out.value


def litedsa_pack(topk_idx, group: int, stream=None):
    """LiteDSA packing of a [T, k] int32 CUDA tensor of selected indices.

    Returns (union [ceil(T/group), group*k] int32, lengths [ceil(T/group)] int32,
    masks [T, ceil(group*k/32)] int32 holding the uint32 bit patterns)."""
    import torch
    lib = load_library()
    _index_matrix_ok(topk_idx, "topk_idx")
    T, k = int(topk_idx.shape[0]), int(topk_idx.shape[1])
    n_groups = (T + group - 1) // group
    words = (group * k + 31) // 32
    dev = topk_idx.device
    union = torch.empty((n_groups, group * k), dtype=torch.int32, device=dev)
    lens = torch.empty((n_groups,), dtype=torch.int32, device=dev)
    masks = torch.empty((T, words), dtype=torch.int32, device=dev)
    _check(lib.ltk_litedsa_pack(_ptr(topk_idx), T, k, group, _ptr(union), _ptr(lens), _ptr(masks),
                                _stream_handle(stream)), "ltk_litedsa_pack")
    return union, lens, masks


def decoupled_noalloc(q, w, k_cache, positions=None, k: int = 2048, dtype: str = "bf16",
                      causal: bool = True, q_scale=None, k_scale=None, out=None, status=None,
                      stream=None):
    """ltk_decoupled_topk_noalloc: the decoupled top-k (H = 64, d = 128) with its
    score matrix in the library's static device array -- for callers that must
    not allocate device memory (T * S <= 4,194,304).  Tensors are checked like
    every other entry point's before the call.  Returns (idx int32 [T, k],
    score fp32 [T, k], status int32 [1]); status holds LTK_ERR_TIMEOUT (5) once
    the stream has run the call if a bounded device wait expired, else 0."""
    import torch
    lib = load_library()
    k = int(k)
    T, S = check_inputs(64, 128, dtype, causal, q, w, k_cache, positions, q_scale, k_scale,
                        None, out, k, device_type="cuda", device_index=torch.cuda.current_device())
    if out is None:
        out = (torch.empty((T, k), dtype=torch.int32, device=q.device),
               torch.empty((T, k), dtype=torch.float32, device=q.device))
    if status is None:
        status = torch.empty((1,), dtype=torch.int32, device=q.device)
    _tensor_ok(status, "status", 1, 4, "cuda", dtype=torch.int32,
               device_index=torch.cuda.current_device())
    code = {"bf16": LTK_BF16, "fp8": LTK_FP8_E4M3}[dtype]
    _check(lib.ltk_decoupled_topk_noalloc(code, 1 if causal else 0, _ptr(q), _ptr(q_scale), _ptr(w),
                                          _ptr(k_cache), _ptr(k_scale),
                                          _ptr(positions) if causal else None, T, S, k,
                                          _ptr(out[0]), _ptr(out[1]), _ptr(status),
                                          _stream_handle(stream)),
           "ltk_decoupled_topk_noalloc")
    return out[0], out[1], status


class IndexerTopK:
    """Owns one ltk handle (and its device workspace) on the current device."""

    def __init__(self, max_T: int, max_S: int, k: int = 2048, heads: int = 64, dim: int = 128,
                 dtype: str = "bf16", **overrides):
        self.lib = load_library()
        cfg = config_defaults(heads, dim, k, max_T, max_S)
        cfg.dtype = {"bf16": LTK_BF16, "fp8": LTK_FP8_E4M3}[dtype]
        for key, val in overrides.items():
            if not hasattr(cfg, key):
                raise TypeError(f"unknown config field {key}")
            setattr(cfg, key, val)
        h = ctypes.c_void_p()
        _check(self.lib.ltk_create(ctypes.byref(cfg), ctypes.byref(h)), "ltk_create")
        self.cfg = cfg
        self.h = h
        self.dtype = dtype

    # -- helpers ---------------------------------------------------------
    def _check(self, device_type, q, w, k_cache, positions, q_scale, k_scale, prev_topk, out, k):
        import torch
        idx = torch.cuda.current_device() if device_type == "cuda" else None
        return check_inputs(self.cfg.heads, self.cfg.dim, self.dtype, bool(self.cfg.causal), q, w,
                            k_cache, positions, q_scale, k_scale, prev_topk, out, k,
                            device_type=device_type, device_index=idx)

    def _outputs(self, T, k, device, out):
        import torch
        if out is not None:
            return out
        return (torch.empty((T, k), dtype=torch.int32, device=device),
                torch.empty((T, k), dtype=torch.float32, device=device))

    # -- API -----------------------------------------------------------------
    def topk(self, q, w, k_cache, positions=None, k: int | None = None, prev_topk=None,
             q_scale=None, k_scale=None, out=None, stream=None):
        """Fused exact top-k; returns (idx int32 [T,k], score fp32 [T,k])."""
        k = int(k or self.cfg.k)
        T, S = self._check("cuda", q, w, k_cache, positions, q_scale, k_scale, prev_topk, out, k)
        oi, os_ = self._outputs(T, k, q.device, out)
        n_prev = 0 if prev_topk is None else int(prev_topk.numel())
        _check(self.lib.ltk_indexer_topk(self.h, _ptr(q), _ptr(q_scale), _ptr(w), _ptr(k_cache),
                                         _ptr(k_scale), _ptr(positions), T, S, _ptr(prev_topk),
                                         n_prev, k, _ptr(oi), _ptr(os_), _stream_handle(stream)),
               "ltk_indexer_topk")
        return oi, os_

    __call__ = topk

    def topk_host(self, q, w, k_cache, positions=None, k: int | None = None, prev_topk=None,
                  q_scale=None, k_scale=None, out=None, stream=None):
        """Same as topk, but all tensors live in (pinned) host memory."""
        import torch
        k = int(k or self.cfg.k)
        T, S = self._check("cpu", q, w, k_cache, positions, q_scale, k_scale, prev_topk, out, k)
        if out is None:
            out = (torch.empty((T, k), dtype=torch.int32, pin_memory=True),
                   torch.empty((T, k), dtype=torch.float32, pin_memory=True))
        n_prev = 0 if prev_topk is None else int(prev_topk.numel())
        _check(self.lib.ltk_indexer_topk_host(self.h, _ptr(q), _ptr(q_scale), _ptr(w),
                                              _ptr(k_cache), _ptr(k_scale), _ptr(positions), T, S,
                                              _ptr(prev_topk), n_prev, k, _ptr(out[0]),
                                              _ptr(out[1]), _stream_handle(stream)),
               "ltk_indexer_topk_host")
        return out

    def decoupled(self, q, w, k_cache, positions=None, k: int | None = None, q_scale=None,
                  k_scale=None, out=None, stream=None):
        """Decoupled baseline: materialised scores + row radix select."""
        k = int(k or self.cfg.k)
        T, S = self._check("cuda", q, w, k_cache, positions, q_scale, k_scale, None, out, k)
        oi, os_ = self._outputs(T, k, q.device, out)
        _check(self.lib.ltk_decoupled_topk(self.h, _ptr(q), _ptr(q_scale), _ptr(w), _ptr(k_cache),
                                           _ptr(k_scale), _ptr(positions), T, S, k, _ptr(oi),
                                           _ptr(os_), _stream_handle(stream)),
               "ltk_decoupled_topk")
        return oi, os_

    def random_sample(self, S: int, n: int, stream=None):
        import torch
        out = torch.empty(n, dtype=torch.int32, device="cuda")
        _check(self.lib.ltk_random_sample(self.h, S, n, _ptr(out), _stream_handle(stream)),
               "ltk_random_sample")
        return out

    def make_sample(self, prev_idx, S: int, n: int | None = None, stream=None):
        import torch
        n = int(n or min(3 * self.cfg.k, 16384))
        if prev_idx is not None:
            _index_matrix_ok(prev_idx, "prev_idx")
        out = torch.empty(n, dtype=torch.int32, device="cuda")
        T_prev, k_prev = (int(prev_idx.shape[0]), int(prev_idx.shape[1])) if prev_idx is not None else (0, 0)
        _check(self.lib.ltk_make_sample(self.h, _ptr(prev_idx), T_prev, k_prev, S, n, _ptr(out),
                                        _stream_handle(stream)), "ltk_make_sample")
        return out

    def set_timing(self, enable: bool = True) -> None:
        _check(self.lib.ltk_set_timing(self.h, 1 if enable else 0), "ltk_set_timing")

    def stats(self) -> dict:
        st = Stats()
        _check(self.lib.ltk_get_stats(self.h, ctypes.byref(st)), "ltk_get_stats")
        return st.as_dict()

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.ltk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
