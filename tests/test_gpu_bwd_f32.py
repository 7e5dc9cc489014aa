"""GPU parity of the fp32 ring_attn_bwd (precision path, fp64 arithmetic)
against the fp64 oracle gradient, through the C ABI.

Bound: 1e-4 per element, taken relative to max(1, |ref|).  The kernel works
in fp64 from fp32 inputs, so what remains is the fp32 rounding of its inputs
and outputs: of dq/dk/dv themselves (2^-24 relative) and of the forward's lse
and out that it reads.  An lse near 40 (the q x 8 variant) carries an fp32
rounding of ~2.4e-6 that enters exp(s - lse) as a relative error, so for
gradients of size tens the bound has to be relative, as for the bf16
large-logit forward check.
"""
import numpy as np
import pytest
import torch

from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu

F32_GRAD_TOL = 1e-4


def _grads(w, dev):
    q, k, v, do = inputs.make_qkv(w)
    gq, gk, gv, gdo = (t.to(dev) for t in (q, k, v, do))
    out, lse = api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, w.causal)
    dq, dk, dv = api.ring_attn_bwd(gq, gk, gv, out, lse, gdo, w.N, w.layout, w.causal)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    assert dq.dtype == torch.float32
    return (q, k, v, do), (dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy())


def _check(name, got, ref):
    assert np.isfinite(got).all(), name
    rel = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert rel.max() <= F32_GRAD_TOL, (name, rel.max())


@pytest.mark.parametrize("qscale", [1.0, 8.0])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
def test_tiny_fp32_bwd(cuda_dev, oracle, layout, causal, qscale):
    """The tiny workload (B=1, H=2, S=512, D=64, N=4) in fp32, every row."""
    w = inputs.TINY.with_(layout=layout, causal=causal, q_scale=qscale, with_grad=True)
    (q, k, v, do), (dq, dk, dv) = _grads(w, cuda_dev)
    rows = np.arange(w.S)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, causal, rows, rows)
    _check("dq", dq, rq)
    _check("dk", dk, rk)
    _check("dv", dv, rv)


F32_CASES = [
    # name, B, Hq, Hkv, S, D, N, layout, causal
    ("gqa_ragged_d128", 2, 4, 2, 200, 128, 4, ZIG, True),     # chunks of 25: ragged tiles
    ("d64_cont_noncausal", 1, 3, 1, 96, 64, 3, CONT, False),
    ("n1_plain", 1, 1, 1, 70, 128, 1, CONT, True),
    ("n8_zig_tiny_chunks", 1, 2, 2, 64, 64, 8, ZIG, True),   # chunks of 4 rows
    ("str_gqa_ragged", 2, 4, 2, 200, 128, 4, STR, True),
    ("str_n3_c23", 1, 2, 1, 69, 64, 3, STR, True),
]


@pytest.mark.parametrize("case", F32_CASES, ids=[c[0] for c in F32_CASES])
def test_fp32_bwd_shapes(cuda_dev, oracle, case):
    name, B, Hq, Hkv, S, D, N, layout, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, torch.float32, seed=61, with_grad=True)
    (q, k, v, do), (dq, dk, dv) = _grads(w, cuda_dev)
    rows = np.arange(S)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, causal, rows, rows)
    _check(name + " dq", dq, rq)
    _check(name + " dk", dk, rk)
    _check(name + " dv", dv, rv)


def test_fp32_bwd_independent_of_n_and_layout(cuda_dev):
    """The gradient does not depend on the sharding ("What it does not change"):
    fp32 results for N in {1, 2, 4, 8} and every layout agree to 1e-5."""
    base = Workload("f32inv", 1, 2, 2, 256, 64, 1, CONT, True, torch.float32, seed=62, with_grad=True)
    q, k, v, do = (t.to(cuda_dev) for t in inputs.make_qkv(base))
    res = []
    for N in (1, 2, 4, 8):
        for layout in (CONT, ZIG, STR):
            out, lse = api.ring_attn_fwd(q, k, v, N, layout, True)
            res.append(api.ring_attn_bwd(q, k, v, out, lse, do, N, layout, True))
    torch.cuda.synchronize()
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert (a - b).abs().max().item() <= 1e-5
