"""The failure path of the pipelined tensor-core kernels, run for real without
a GPU fault.

cp_debug_set_wait_limit shortens the bound of every pipeline wait of the
kernels launched afterwards to a few nanoseconds, while the waits that drain
a block's copies and MMAs before it exits keep their 2 s bound.  The first
wait that is not already satisfied then runs out: the block records
CP_ETIMEOUT, drains, frees its tensor memory and returns.  Each test checks
that status, restores the default bound, and checks that the next ordinary
call on the same context still matches the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from conftest import check_bf16
from context_parallelism_02_gb300 import CP_ETIMEOUT, api, inputs, ring
from context_parallelism_02_gb300.inputs import STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu

SHORT_NS = 1


def _times_out(fn):
    """Run fn with the pipeline waits bounded by SHORT_NS; return the status."""
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    api.cp_debug_set_wait_limit(SHORT_NS)
    try:
        fn()
        rc = api.cp_get_error()
    finally:
        api.cp_debug_set_wait_limit(0)
    return rc


@pytest.mark.parametrize("layout", [ZIG, STR])
def test_forward_aborts_and_context_survives(cuda_dev, oracle, layout):
    w = Workload("abort_fwd", 1, 2, 2, 2048, 128, 4, layout, True, torch.bfloat16, seed=111)
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))
    assert _times_out(lambda: api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, True)) == CP_ETIMEOUT
    out, lse = api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    ref, lref = oracle.attn_fwd(q, k, v, True)
    check_bf16(out.float().cpu().numpy(), lse.cpu().numpy(), ref, lref, f"after abort, layout {layout}")


def test_split_and_step_forward_abort(cuda_dev, oracle):
    w = Workload("abort_split", 1, 2, 2, 2048, 128, 4, ZIG, True, torch.bfloat16, seed=112)
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))
    assert _times_out(lambda: api.ring_attn_fwd_split(gq, gk, gv, w.N, w.layout, True,
                                                      n_split=3)) == CP_ETIMEOUT
    qs, ks, vs = (ring.shard(t, 1, w.N, w.layout) for t in (gq, gk, gv))
    assert _times_out(lambda: api.flash_block_step(qs, ks, vs, 1, 1, w.N, w.S, w.layout, True,
                                                   accumulate=False)) == CP_ETIMEOUT
    out, lse = ring.ring_attention_emulated(gq, gk, gv, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    ref, lref = oracle.attn_fwd(q, k, v, True)
    check_bf16(out.float().cpu().numpy(), lse.cpu().numpy(), ref, lref, "per-step ring after abort")


def test_backward_aborts_and_context_survives(cuda_dev, oracle):
    w = Workload("abort_bwd", 1, 2, 2, 1024, 128, 4, ZIG, True, torch.bfloat16, seed=113,
                 with_grad=True)
    q, k, v, do = inputs.make_qkv(w)
    gq, gk, gv, gdo = (t.to(cuda_dev) for t in (q, k, v, do))
    out, lse = api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, True)
    assert _times_out(lambda: api.ring_attn_bwd(gq, gk, gv, out, lse, gdo, w.N, w.layout,
                                                True)) == CP_ETIMEOUT
    dq, dk, dv = api.ring_attn_bwd(gq, gk, gv, out, lse, gdo, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    rows = np.arange(w.S)
    for got, ref in zip((dq, dk, dv), oracle.attn_bwd(q, k, v, do, True, rows, rows)):
        e = np.abs(got.float().cpu().numpy() - ref)
        assert e.max() <= 1e-2 * np.abs(ref).max() and e.mean() <= 1e-3 * np.abs(ref).max()


def test_wait_limit_hook_validation(cuda_dev):
    with pytest.raises(api.CpError):
        api.cp_debug_set_wait_limit(3_000_000_000)
    api.cp_debug_set_wait_limit(0)
