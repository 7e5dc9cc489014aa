"""ring_attn_bwd_noalloc: the backward for callers that cannot allocate.

Some callers (plugins that may only touch buffers their host hands them,
code bound to a foreign memory pool or a fixed budget) cannot provide
ring_attn_bwd's workspace.  ring_attn_bwd_noalloc keeps that scratch in a
fixed device array inside the library.  These tests call it through the C
ABI and check it against ring_attn_bwd on two calls in a row (the second
call finds the first call's leftovers in the shared array).  Both calls run
the same deterministic kernels on the same Delta, so the gradients must be
equal bit for bit.

This file is collected last on purpose, so that a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from context_parallelism_02_gb300 import _lib, api, inputs
from context_parallelism_02_gb300.inputs import STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", [ZIG, STR])
def test_noalloc_matches_workspace_backward_twice(cuda_dev, layout):
    w = Workload("noalloc", 2, 4, 2, 1600, 128, 4, layout, True, torch.bfloat16, seed=61,
                 with_grad=True)
    q, k, v, do = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    out, lse = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    ref = api.ring_attn_bwd(q, k, v, out, lse, do, w.N, w.layout, True)
    for _ in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in ref)
        api.ring_attn_bwd_noalloc(q, k, v, out, lse, do, w.N, w.layout, True, dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
        assert api.cp_get_error() == 0
        for got, exp in zip((dq, dk, dv), ref):
            assert torch.isfinite(got.float()).all()
            assert torch.equal(got, exp)


def test_noalloc_second_shape_after_larger_call(cuda_dev):
    """A smaller problem after a larger one: stale scratch does not leak in."""
    for S, Hq in ((4096, 8), (1024, 2)):
        w = Workload("noalloc2", 1, Hq, Hq, S, 64, 2, ZIG, True, torch.bfloat16, seed=62,
                     with_grad=True)
        q, k, v, do = (t.to(cuda_dev) for t in inputs.make_qkv(w))
        out, lse = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
        ref = api.ring_attn_bwd(q, k, v, out, lse, do, w.N, w.layout, True)
        got = api.ring_attn_bwd_noalloc(q, k, v, out, lse, do, w.N, w.layout, True)
        torch.cuda.synchronize()
        for g_, e in zip(got, ref):
            assert torch.equal(g_, e)


def test_noalloc_rejects_oversize(cuda_dev):
    """B * Hq * S above the fixed scratch is refused before anything runs."""
    L = _lib.load()
    S = 2 * _lib.CP_BWD_NOALLOC_MAX_ROWS          # one head, B=1: twice the limit
    p = ctypes.c_void_p(16)
    rc = L.ring_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, 1, S, 128, 1, 1, 0, 1, -1.0,
                                 None)
    assert rc == _lib.CP_EINVAL
