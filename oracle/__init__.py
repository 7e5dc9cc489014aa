"""fp64 CPU oracle for ring / context-parallel attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never does: the CUDA library
has no fallback to it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent
rows); this module compiles it with gcc on first use and wraps it with
numpy.  Every function cites the passage it follows in ``oracle.c``.

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against values and properties the pages or the mathematics fix (library
attention in fp64, the exactness claim across N and layouts, row sums,
constant V, exact pair-count identities, the printed 4-GPU ring table,
finite differences, and the permutation's index formula).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CONTIGUOUS = 0
ZIGZAG = 1
STRIPED = 2


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            P = ctypes.c_void_p
            lib.or_shard_pos.argtypes = [i64, i32, i32, P]
            lib.or_ring_source_table.argtypes = [i32, P]
            lib.or_pair_counts.argtypes = [i64, i32, i32, i32, P]
            lib.or_attn_fwd.argtypes = [P, P, P, i32, i32, i32, i64, i32, i32, dbl,
                                        i64, P, i64, i64, P, P]
            lib.or_ring_fwd.argtypes = [P, P, P, i32, i32, i32, i64, i32, i32, i32, i32,
                                        dbl, P, P]
            lib.or_block_step.argtypes = [P, P, P, i32, i32, i32, i64, i32, i32, i32, i32,
                                          i32, i32, dbl, i32, P, P]
            lib.or_lse_merge.argtypes = [P, P, P, P, i64, i32, P, P]
            lib.or_lse_merge_n.argtypes = [P, P, i32, i64, i32, P, P]
            lib.or_ulysses_seq_to_head.argtypes = [P, P, i32, i64, i32, i32, i32, i32, i32]
            lib.or_ulysses_head_to_seq.argtypes = [P, P, i32, i64, i32, i32, i32, i32, i32]
            lib.or_attn_bwd.argtypes = [P, P, P, P, i32, i32, i32, i64, i32, i32, dbl,
                                        i64, P, i64, P, P, P, P]
            lib.or_num_threads.argtypes = []
            for f in ("or_shard_pos", "or_ring_source_table", "or_pair_counts", "or_attn_fwd",
                      "or_ring_fwd", "or_block_step", "or_lse_merge", "or_ulysses_seq_to_head",
                      "or_ulysses_head_to_seq", "or_attn_bwd", "or_num_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):          # torch tensor: exact up-conversion of its values
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def num_threads() -> int:
    return _load().or_num_threads()


def shard_pos(S: int, N: int, layout: int) -> np.ndarray:
    """Global position of each local row: ``pos[r, t]`` (int64, [N, S/N])."""
    out = np.zeros(S, dtype=np.int64)
    _check(_load().or_shard_pos(S, N, layout, _ptr(out)), "shard_pos")
    return out.reshape(N, S // N)


def ring_source_table(N: int) -> np.ndarray:
    """``src[k, r]``: the rank whose KV block rank r holds at ring step k."""
    out = np.zeros(N * N, dtype=np.int32)
    _check(_load().or_ring_source_table(N, _ptr(out)), "ring_source_table")
    return out.reshape(N, N)


def pair_counts(S: int, N: int, layout: int, causal: bool) -> np.ndarray:
    """Masked-in (query, key) pairs per (rank, step), int64 ``[N, N]``."""
    out = np.zeros(N * N, dtype=np.int64)
    _check(_load().or_pair_counts(S, N, layout, int(causal), _ptr(out)), "pair_counts")
    return out.reshape(N, N)


def attn_fwd(q, k, v, causal: bool, scale: float | None = None, rows=None,
             klo: int = 0, khi: int | None = None):
    """O1, definitional attention in fp64.

    q ``[B,S,Hq,D]``, k/v ``[B,S,Hkv,D]`` (any float dtype, up-converted).
    ``rows``: optional query positions (int64); keys restricted to [klo, khi).
    Returns out ``[B, nrows, Hq, D]`` and lse ``[B, Hq, nrows]`` (fp64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if rows is None:
        nrows, rp = S, None
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rp = rows_arr.size, _ptr(rows_arr)
    out = np.zeros((B, nrows, Hq, D))
    lse = np.zeros((B, Hq, nrows))
    rc = _load().or_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, int(causal),
                             float(scale), nrows, rp, klo, S if khi is None else khi,
                             _ptr(out), _ptr(lse))
    _check(rc, "attn_fwd")
    return out, lse


def ring_fwd(q, k, v, N: int, layout: int, causal: bool, scale: float | None = None):
    """O2, explicit ring emulation; returns (out [B,S,Hq,D], lse [B,Hq,S]) fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, S, Hq, D))
    lse = np.zeros((B, Hq, S))
    rc = _load().or_ring_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, N, int(causal),
                             layout, float(scale), _ptr(out), _ptr(lse))
    _check(rc, "ring_fwd")
    return out, lse


def block_step(q_shard, k_blk, v_blk, S: int, N: int, layout: int, causal: bool, rank: int,
               source: int, out=None, lse=None, scale: float | None = None):
    """One ring step of one device on shard-local buffers (fp64).

    q_shard ``[B, C, Hq, D]`` holds rank ``rank``'s queries, k_blk / v_blk
    ``[B, C, Hkv, D]`` rank ``source``'s keys and values, each in local order
    (C = S / N).  ``out`` ``[B, C, Hq, D]`` / ``lse`` ``[B, Hq, C]`` is the
    running state (None: start from the empty state).  Returns the new
    (out, lse); the arguments are not modified.
    """
    q, k, v = _f64(q_shard), _f64(k_blk), _f64(v_blk)
    B, C, Hq, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    acc = out is not None
    o = _f64(out).copy() if acc else np.zeros((B, C, Hq, D))
    l_ = _f64(lse).copy() if acc else np.zeros((B, Hq, C))
    rc = _load().or_block_step(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, N, layout,
                               int(causal), rank, source, float(scale), int(acc), _ptr(o), _ptr(l_))
    _check(rc, "block_step")
    return o, l_


def lse_merge(out_a, lse_a, out_b, lse_b):
    """Merge two normalised partials over disjoint key sets (fp64)."""
    out_a, lse_a, out_b, lse_b = _f64(out_a), _f64(lse_a), _f64(out_b), _f64(lse_b)
    rows = lse_a.size
    D = out_a.size // rows
    out = np.zeros_like(out_a)
    lse = np.zeros_like(lse_a)
    _check(_load().or_lse_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), rows, D,
                                _ptr(out), _ptr(lse)), "lse_merge")
    return out, lse


def lse_merge_n(out_parts, lse_parts):
    """Merge n normalised partials over disjoint key sets (fp64):
    out_parts [n, rows, D], lse_parts [n, rows] -> (out [rows, D], lse [rows])."""
    out_parts, lse_parts = _f64(out_parts), _f64(lse_parts)
    n, rows = lse_parts.shape
    D = out_parts.size // max(n * rows, 1)
    out = np.zeros((rows, D))
    lse = np.zeros(rows)
    _check(_load().or_lse_merge_n(_ptr(out_parts), _ptr(lse_parts), n, rows, D, _ptr(out),
                                  _ptr(lse)), "lse_merge_n")
    return out, lse


def _raw(x) -> np.ndarray:
    """Raw bytes of a tensor/array as a contiguous numpy array (dtype kept by size)."""
    if hasattr(x, "detach"):
        t = x.detach().to("cpu").contiguous()
        return t.view(_torch_int_view(t)).numpy()
    return np.ascontiguousarray(x)


def _torch_int_view(t):
    import torch
    return {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()]


def ulysses_seq_to_head(x, N: int, layout: int):
    """``[N, B, S/N, H, D]`` rank-major shards -> ``[N, B, S, H/N, D]`` head groups."""
    a = _raw(x)
    Nn, B, L, H, D = a.shape
    assert Nn == N
    S = N * L
    y = np.zeros((N, B, S, H // N, D), dtype=a.dtype)
    _check(_load().or_ulysses_seq_to_head(_ptr(a), _ptr(y), B, S, H, D, N, layout,
                                          a.dtype.itemsize), "ulysses_seq_to_head")
    return y


def ulysses_head_to_seq(y, N: int, layout: int):
    """Inverse of :func:`ulysses_seq_to_head`."""
    a = _raw(y)
    Nn, B, S, hg, D = a.shape
    assert Nn == N
    H = hg * N
    x = np.zeros((N, B, S // N, H, D), dtype=a.dtype)
    _check(_load().or_ulysses_head_to_seq(_ptr(a), _ptr(x), B, S, H, D, N, layout,
                                          a.dtype.itemsize), "ulysses_head_to_seq")
    return x


def attn_bwd(q, k, v, dout, causal: bool, qrows, krows, scale: float | None = None):
    """Closed-form gradient of sum(dO * out) in fp64 on row slices.

    Returns dq ``[B, nq, Hq, D]`` for query positions ``qrows`` and dk, dv
    ``[B, nk, Hkv, D]`` for key positions ``krows``.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qr = np.ascontiguousarray(qrows, dtype=np.int64)
    kr = np.ascontiguousarray(krows, dtype=np.int64)
    dq = np.zeros((B, qr.size, Hq, D))
    dk = np.zeros((B, kr.size, Hkv, D))
    dv = np.zeros((B, kr.size, Hkv, D))
    rc = _load().or_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, Hq, Hkv, S, D,
                             int(causal), float(scale), qr.size, _ptr(qr), kr.size, _ptr(kr),
                             _ptr(dq), _ptr(dk), _ptr(dv))
    _check(rc, "attn_bwd")
    return dq, dk, dv
