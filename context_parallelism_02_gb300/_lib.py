"""ctypes loader and raw signatures of libcp (include/cp.h).

The library must exist: there is no fallback path.  Build it with
``python -m context_parallelism_02_gb300.build`` (or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

from . import build as _build

CP_OK = 0
CP_EINVAL = -1
CP_EHEADS = -2
CP_EUNSUPPORTED = -3
CP_ECUDA = -4
CP_ETIMEOUT = -5
CP_ESMEM = -6
CP_EBOUNDS = -7

CP_LAYOUT_CONTIGUOUS = 0
CP_LAYOUT_ZIGZAG = 1
CP_LAYOUT_STRIPED = 2
CP_F32 = 0
CP_BF16 = 1
CP_BWD_NOALLOC_MAX_ROWS = 4 * 1024 * 1024

# name -> (restype, argtypes); mirrors include/cp.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_F = ctypes.c_float
SIGNATURES = {
    "cp_shard_map": (_I, [_L, _I, _I, _P]),
    "cp_schedule_pairs": (_I, [_L, _I, _I, _I, _P, _P]),
    "ring_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I, _I, _I, _I, _F, _P]),
    "ring_attn_fwd_rank": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I, _I, _I, _I, _F, _I,
                                _I, _P]),
    "flash_block_step": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I, _I, _I, _I, _I,
                              _I, _F, _I, _P]),
    "ring_attn_fwd_split": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I, _I, _I, _I, _F, _I,
                                 _I, _I, _P, ctypes.c_size_t, _P]),
    "ring_attn_fwd_split_workspace": (ctypes.c_size_t, [_I, _I, _L, _I, _I]),
    "cp_fwd_split_count": (_I, [_I, _I, _L, _I, _I, _I, _I, _I, _I, _I]),
    "ring_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I, _I, _I,
                           _I, _F, _P, ctypes.c_size_t, _P]),
    "ring_attn_bwd_workspace": (ctypes.c_size_t, [_I, _I, _L]),
    "usp_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I, _I, _I, _I, _I, _F, _P,
                          ctypes.c_size_t, _P]),
    "usp_attn_fwd_workspace": (ctypes.c_size_t, [_I, _I, _L, _I, _I]),
    "ring_attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _L, _I, _I,
                                   _I, _I, _I, _F, _P]),
    "lse_merge": (_I, [_P, _P, _P, _P, _P, _P, _L, _I, _P]),
    "lse_merge_n": (_I, [_P, _P, _I, _L, _I, _P, _P, _P]),
    "ulysses_seq_to_head": (_I, [_P, _P, _I, _L, _I, _I, _I, _I, _I, _P]),
    "ulysses_head_to_seq": (_I, [_P, _P, _I, _L, _I, _I, _I, _I, _I, _P]),
    "cp_get_error": (_I, [_P]),
    "cp_strerror": (ctypes.c_char_p, [_I]),
    "cp_debug_wait_timeout": (_I, [ctypes.c_uint64, _P]),
    "cp_debug_set_wait_limit": (_I, [ctypes.c_uint64]),
    "cp_debug_set_grid_limit": (_I, [_I]),
}

_lock = threading.RLock()
_libs = {}                 # variant -> loaded library
_active = "default"        # the variant load() returns (see variant())
_VARIANTS = {"default": (_build.LIB, {}), "debug_bounds": (_build.LIB_DEBUG_BOUNDS, {"debug_bounds": True})}


class CpError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (code {code})")


def lib_path(variant: str | None = None) -> str:
    return _VARIANTS[variant or _active][0]


def load(build_if_missing: bool = False, variant: str | None = None):
    """Load libcp.so (raises if it is missing: no fallback exists).  ``variant``
    "debug_bounds" loads the checking build (default: the active variant)."""
    v = variant or _active
    with _lock:
        if v not in _libs:
            path, opts = _VARIANTS[v]
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(
                        f"libcp.so not found at {path}; build it with "
                        "`python -m context_parallelism_02_gb300.build`")
                _build.build(**opts)
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _libs[v] = lib
    return _libs[v]


@contextlib.contextmanager
def variant(name: str):
    """Route every binding call inside the block to the ``name`` build of libcp
    (built if missing), e.g. ``with variant("debug_bounds"): ...``."""
    global _active
    with _lock:
        prev = _active
        load(build_if_missing=True, variant=name)
        _active = name
    try:
        yield _libs[name]
    finally:
        _active = prev


def strerror(code: int) -> str:
    try:
        return load().cp_strerror(code).decode()
    except Exception:  # noqa: BLE001 - message lookup must not mask the real error
        return f"status {code}"


def check(code: int, what: str):
    if code != CP_OK:
        raise CpError(code, what)
