"""Python binding of libcp: same names as the C ABI, argument marshalling only.

Tensors are torch tensors on the current CUDA device (torch supplies device
memory and streams); every computation runs in libcp's CUDA kernels.  Outputs
are allocated with torch when not given.  Each call is asynchronous on the
current torch stream (or ``stream``), like the C call.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import CP_BF16, CP_F32, CpError, check  # noqa: F401

_DT = {torch.float32: CP_F32, torch.bfloat16: CP_BF16}


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda_contig(name, t):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_out_contig(name, t):
    # an output may also be pinned host memory, which the kernels address directly
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def cp_shard_map(S: int, N: int, layout: int) -> np.ndarray:
    """Global position of each local row, int32 ``[N, S/N]`` (host)."""
    out = np.zeros(S, dtype=np.int32)
    check(_lib.load().cp_shard_map(S, N, layout, out.ctypes.data_as(ctypes.c_void_p)),
          "cp_shard_map")
    return out.reshape(N, S // N)


def cp_schedule_pairs(S: int, N: int, layout: int, causal: bool):
    """(masked-in pairs, executed 128x128 tile pairs) per (rank, step), int64 ``[N, N]``."""
    pairs = np.zeros(N * N, dtype=np.int64)
    tiles = np.zeros(N * N, dtype=np.int64)
    check(_lib.load().cp_schedule_pairs(S, N, layout, int(causal),
                                        pairs.ctypes.data_as(ctypes.c_void_p),
                                        tiles.ctypes.data_as(ctypes.c_void_p)),
          "cp_schedule_pairs")
    return pairs.reshape(N, N), tiles.reshape(N, N)


def ring_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, N: int, layout: int,
                  causal: bool = True, scale: float | None = None, out=None, lse=None,
                  stream=None, rank_range: tuple[int, int] | None = None):
    """Ring / context-parallel attention forward; returns (out, lse).

    q ``[B,S,Hq,D]``, k/v ``[B,S,Hkv,D]`` (fp32 or bf16, global order);
    out like q, lse ``[B,Hq,S]`` fp32.  ``out`` and ``lse`` may be pinned host
    tensors: the kernels then write the result straight into host memory.
    ``rank_range=(lo, hi)`` restricts the computed queries to virtual ranks
    [lo, hi) (``ring_attn_fwd_rank``).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(name, t)
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype float32 or bfloat16")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _need_out_contig("out", out)
    _need_out_contig("lse", lse)
    sc = -1.0 if scale is None else float(scale)
    L = _lib.load()
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, N, int(causal),
            layout, _DT[q.dtype], sc)
    if rank_range is None:
        rc = L.ring_attn_fwd(*args, ctypes.c_void_p(_stream(stream)))
        check(rc, "ring_attn_fwd")
    else:
        rc = L.ring_attn_fwd_rank(*args, rank_range[0], rank_range[1],
                                  ctypes.c_void_p(_stream(stream)))
        check(rc, "ring_attn_fwd_rank")
    return out, lse


def flash_block_step(q, k, v, rank: int, source: int, N: int, S: int, layout: int,
                     causal: bool = True, scale: float | None = None, out_acc=None, lse_acc=None,
                     out_final=None, accumulate: bool = True, stream=None):
    """One ring step on shard-local buffers: rank ``rank``'s queries against the
    KV block of rank ``source``, merged into the running state; returns
    (out_acc, lse_acc).

    q ``[B, C, Hq, D]`` and k/v ``[B, C, Hkv, D]`` (C = S / N) are in the local
    row order of their ranks (``cp_shard_map``); out_acc ``[B, C, Hq, D]`` and
    lse_acc ``[B, Hq, C]`` are fp32 (allocated when None, which requires
    ``accumulate=False``).  ``out_final`` (optional, q's dtype) receives the
    merged output rounded to that dtype.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(name, t)
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype float32 or bfloat16")
    B, C, Hq, D = q.shape
    Hkv = k.shape[2]
    if (out_acc is None or lse_acc is None) and accumulate:
        raise ValueError("accumulate=True needs the running state out_acc and lse_acc")
    if out_acc is None:
        out_acc = torch.empty((B, C, Hq, D), dtype=torch.float32, device=q.device)
    if lse_acc is None:
        lse_acc = torch.empty((B, Hq, C), dtype=torch.float32, device=q.device)
    for name, t in (("out_acc", out_acc), ("lse_acc", lse_acc)):
        _need_cuda_contig(name, t)
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    if out_final is not None:
        _need_cuda_contig("out_final", out_final)
        if out_final.dtype != q.dtype:
            raise ValueError("out_final must have q's dtype")
    sc = -1.0 if scale is None else float(scale)
    rc = _lib.load().flash_block_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out_acc), _ptr(lse_acc),
                                      _ptr(out_final), B, Hq, Hkv, S, D, N, rank, source,
                                      int(causal), layout, _DT[q.dtype], sc, int(accumulate),
                                      ctypes.c_void_p(_stream(stream)))
    check(rc, "flash_block_step")
    return out_acc, lse_acc


def cp_fwd_split_count(B: int, Hq: int, S: int, D: int, N: int, layout: int, causal: bool = True,
                       rank_range: tuple[int, int] | None = None, num_sms: int | None = None) -> int:
    """Number of splits for :func:`ring_attn_fwd_split` (host-side dispatch
    simulation); ``num_sms`` defaults to the current CUDA device's SM count."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    lo, hi = (0, N) if rank_range is None else rank_range
    rc = _lib.load().cp_fwd_split_count(B, Hq, S, D, N, int(causal), layout, lo, hi, int(num_sms))
    if rc < 1:
        check(rc, "cp_fwd_split_count")
    return rc


def ring_attn_fwd_split_workspace(B: int, Hq: int, S: int, D: int, n_split: int) -> int:
    return int(_lib.load().ring_attn_fwd_split_workspace(B, Hq, S, D, n_split))


def ring_attn_fwd_split(q, k, v, N: int, layout: int, causal: bool = True, n_split: int | None = None,
                        scale: float | None = None, out=None, lse=None, workspace=None, stream=None,
                        rank_range: tuple[int, int] | None = None):
    """Split-KV ring forward (bf16): every query tile's key walk cut into
    ``n_split`` pieces on separate blocks, merged by log-sum-exp; returns
    (out, lse).  ``n_split=None`` takes :func:`cp_fwd_split_count`;
    ``workspace`` (at least ``ring_attn_fwd_split_workspace`` bytes) is
    allocated with torch if None."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(name, t)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    lo, hi = (0, N) if rank_range is None else rank_range
    if n_split is None:
        n_split = cp_fwd_split_count(B, Hq, S, D, N, layout, causal, (lo, hi))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _need_cuda_contig("out", out)
    _need_cuda_contig("lse", lse)
    ws_bytes = ring_attn_fwd_split_workspace(B, Hq, S, D, n_split) if n_split >= 1 else 0
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    sc = -1.0 if scale is None else float(scale)
    rc = _lib.load().ring_attn_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                         S, D, N, int(causal), layout, _DT.get(q.dtype, -1), sc, lo,
                                         hi, n_split, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         ctypes.c_void_p(_stream(stream)))
    check(rc, "ring_attn_fwd_split")
    return out, lse


def usp_attn_fwd(q, k, v, n_ulysses: int, n_ring: int, layout: int, causal: bool = True,
                 scale: float | None = None, out=None, lse=None, workspace=None, stream=None):
    """Attention on an n_ulysses x n_ring grid of virtual ranks (USP): heads split
    by the Ulysses relayout, ring attention over n_ring ranks in each head group."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(name, t)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    ws_bytes = int(_lib.load().usp_attn_fwd_workspace(Hq, Hkv, S, D, _DT[q.dtype]))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    sc = -1.0 if scale is None else float(scale)
    rc = _lib.load().usp_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S,
                                  D, n_ulysses, n_ring, int(causal), layout, _DT[q.dtype], sc,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  ctypes.c_void_p(_stream(stream)))
    check(rc, "usp_attn_fwd")
    return out, lse


def ring_attn_bwd_workspace(B: int, Hq: int, S: int) -> int:
    return int(_lib.load().ring_attn_bwd_workspace(B, Hq, S))


def ring_attn_bwd(q, k, v, out, lse, dout, N: int, layout: int, causal: bool = True,
                  scale: float | None = None, dq=None, dk=None, dv=None, workspace=None,
                  stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out) for :func:`ring_attn_fwd`
    (bf16 on the tensor cores, or fp32 with fp64 arithmetic).

    ``workspace``: optional caller-owned device buffer of at least
    ``ring_attn_bwd_workspace(B, Hq, S)`` bytes (allocated with torch if None).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse), ("dout", dout)):
        _need_cuda_contig(name, t)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = ring_attn_bwd_workspace(B, Hq, S)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    sc = -1.0 if scale is None else float(scale)
    rc = _lib.load().ring_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, S, D, N, int(causal),
                                   layout, _DT[q.dtype], sc, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   ctypes.c_void_p(_stream(stream)))
    check(rc, "ring_attn_bwd")
    return dq, dk, dv


def ring_attn_bwd_noalloc(q, k, v, out, lse, dout, N: int, layout: int, causal: bool = True,
                          scale: float | None = None, dq=None, dk=None, dv=None, stream=None):
    """:func:`ring_attn_bwd` without a workspace, for callers that cannot
    allocate device memory: the library keeps the scratch in a fixed 16 MiB
    device array (B * Hq * S <= CP_BWD_NOALLOC_MAX_ROWS).  Pass dq, dk, dv to
    keep this call free of allocations (torch allocates them here otherwise).
    Calls that overlap on the GPU share that array and race."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse), ("dout", dout)):
        _need_cuda_contig(name, t)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    sc = -1.0 if scale is None else float(scale)
    rc = _lib.load().ring_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                           _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv,
                                           S, D, N, int(causal), layout, _DT[q.dtype], sc,
                                           ctypes.c_void_p(_stream(stream)))
    check(rc, "ring_attn_bwd_noalloc")
    return dq, dk, dv


def lse_merge(out_a, lse_a, out_b, lse_b, out=None, lse=None, stream=None):
    """Merge two fp32 partials over disjoint key sets; returns (out, lse)."""
    for name, t in (("out_a", out_a), ("lse_a", lse_a), ("out_b", out_b), ("lse_b", lse_b)):
        _need_cuda_contig(name, t)
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    rows = lse_a.numel()
    D = out_a.numel() // max(rows, 1)
    if out is None:
        out = torch.empty_like(out_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    rc = _lib.load().lse_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out),
                               _ptr(lse), rows, D, ctypes.c_void_p(_stream(stream)))
    check(rc, "lse_merge")
    return out, lse


def lse_merge_n(out_parts, lse_parts, out=None, lse=None, stream=None):
    """Merge n fp32 partials over disjoint key sets in one pass:
    out_parts [n, rows, D], lse_parts [n, rows] -> (out [rows, D], lse [rows])."""
    for name, t in (("out_parts", out_parts), ("lse_parts", lse_parts)):
        _need_cuda_contig(name, t)
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    n, rows = lse_parts.shape[0], lse_parts[0].numel()
    D = out_parts.numel() // max(n * rows, 1)
    if out is None:
        out = torch.empty(rows, D, dtype=torch.float32, device=out_parts.device)
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=out_parts.device)
    rc = _lib.load().lse_merge_n(_ptr(out_parts), _ptr(lse_parts), n, rows, D, _ptr(out),
                                 _ptr(lse), ctypes.c_void_p(_stream(stream)))
    check(rc, "lse_merge_n")
    return out, lse


def ulysses_seq_to_head(x: torch.Tensor, N: int, layout: int, y=None, stream=None):
    """``[N, B, S/N, H, D]`` rank-major shards -> ``[N, B, S, H/N, D]`` head groups."""
    _need_cuda_contig("x", x)
    Nn, B, Lr, H, D = x.shape
    if Nn != N:
        raise ValueError("x.shape[0] must equal N")
    if y is None:
        y = torch.empty((N, B, N * Lr, H // N if H % N == 0 else 1, D), dtype=x.dtype,
                        device=x.device)
    rc = _lib.load().ulysses_seq_to_head(_ptr(x), _ptr(y), B, N * Lr, H, D, N, layout,
                                         x.element_size(), ctypes.c_void_p(_stream(stream)))
    check(rc, "ulysses_seq_to_head")
    return y


def ulysses_head_to_seq(y: torch.Tensor, N: int, layout: int, x=None, stream=None):
    """Inverse of :func:`ulysses_seq_to_head`."""
    _need_cuda_contig("y", y)
    Nn, B, S, hg, D = y.shape
    if Nn != N:
        raise ValueError("y.shape[0] must equal N")
    if x is None:
        x = torch.empty((N, B, S // N, hg * N, D), dtype=y.dtype, device=y.device)
    rc = _lib.load().ulysses_head_to_seq(_ptr(y), _ptr(x), B, S, hg * N, D, N, layout,
                                         y.element_size(), ctypes.c_void_p(_stream(stream)))
    check(rc, "ulysses_head_to_seq")
    return x


def cp_get_error(stream=None) -> int:
    """Synchronise the stream and read+clear the device error word (a status code)."""
    return _lib.load().cp_get_error(ctypes.c_void_p(_stream(stream)))


def cp_strerror(code: int) -> str:
    return _lib.strerror(code)


def cp_debug_set_wait_limit(limit_ns: int):
    """Test hook: bound (ns) of the pipeline waits of later tensor-core launches
    in this process; 0 restores the 2 s default (drains always keep 2 s)."""
    check(_lib.load().cp_debug_set_wait_limit(int(limit_ns)), "cp_debug_set_wait_limit")


def cp_debug_set_grid_limit(max_blocks: int):
    """Test hook: the tensor-core forward launches at most ``max_blocks`` blocks
    (each running several work items); 0 restores the default grid."""
    check(_lib.load().cp_debug_set_grid_limit(int(max_blocks)), "cp_debug_set_grid_limit")


def cp_debug_wait_timeout(limit_ns: int, stream=None):
    check(_lib.load().cp_debug_wait_timeout(limit_ns, ctypes.c_void_p(_stream(stream))),
          "cp_debug_wait_timeout")
