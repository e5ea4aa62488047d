"""GB300-native fused Indexer-TopK (LiteTopK-style sample / filter / select).

The compute path lives in the CUDA library ``libltk.so`` (sources in ``csrc/``,
C ABI in ``include/ltk.h``); ``ltk`` is a thin ctypes binding over it.
"""
from .ltk import IndexerTopK, LtkError, litedsa_pack, load_library, library_path  # noqa: F401
