"""Kara decode-time KV-cache compression on GB300 (sm_103a).

The work runs in ``libkara.so`` (hand-written CUDA, C ABI in include/kara.h);
``decode_kv_cache_03_gb300.kara`` is its ctypes binding and raises on import if
the library is missing.  ``decode_kv_cache_03_gb300.build`` compiles it.
``Compressor`` wraps the workspace and error word for one cache.  Names are
resolved lazily so that the build module can be imported before the library
exists.
"""
from __future__ import annotations

import importlib

_LAZY = {
    "kara": ("kara", None),
    "Compressor": ("compressor", "Compressor"),
    "periodic": ("periodic", None),
    "BlockPool": ("periodic", "BlockPool"),
    "PeriodicSchedule": ("periodic", "PeriodicSchedule"),
    "KaraError": ("kara", "KaraError"),
    "kara_plan": ("kara", "kara_plan"),
    "kara_workspace_size": ("kara", "kara_workspace_size"),
    "kara_score": ("kara", "kara_score"),
    "kara_select": ("kara", "kara_select"),
    "kara_compact": ("kara", "kara_compact"),
    "kara_compress_batch": ("kara", "kara_compress_batch"),
    "kara_get_error": ("kara", "kara_get_error"),
    "kara_decode_attention": ("kara", "kara_decode_attention"),
    "kara_decode_workspace_size": ("kara", "kara_decode_workspace_size"),
}

__all__ = sorted(_LAZY)


def __getattr__(name):
    if name not in _LAZY:
        raise AttributeError(name)
    mod, attr = _LAZY[name]
    m = importlib.import_module(f".{mod}", __name__)
    return m if attr is None else getattr(m, attr)
