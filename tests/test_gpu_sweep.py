"""Seeded random sweep of shapes through the C ABI, against the fp64 oracle:
forward and backward, bf16 and fp32, every layout, causal or not, GQA groups,
D = 64 and 128, ragged chunks.  Each case is drawn from a fixed seed, so the
sweep is the same on every run.

Bounds: forward as in test_gpu_fwd.py (bf16: |err| <= 1e-2 plus the half-ulp
of the bf16 output per element, mean <= 1e-3, |lse err| <= 1e-3; fp32: 1e-5); backward as in
test_gpu_bwd.py (bf16: 1e-2 / 1e-3 of max |ref|) and test_gpu_bwd_f32.py
(fp32: 1e-4 relative to max(1, |ref|)).
"""
import numpy as np
import pytest
import torch

from conftest import F32_TOL, check_bf16
from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import Workload

pytestmark = pytest.mark.gpu


def _draw_case(i):
    rng = np.random.default_rng(1000 + i)
    layout = int(rng.integers(0, 3))
    N = int(rng.choice([1, 2, 3, 4, 5, 8]))
    per = 2 * N if layout == 1 else N
    chunk = int(rng.choice([8, 37, 64, 100, 128, 129, 200, 256]))
    S = per * chunk
    grp = int(rng.choice([1, 2, 4]))
    Hkv = int(rng.choice([1, 2]))
    Hq = grp * Hkv
    B = int(rng.choice([1, 2]))
    D = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 4) > 0)
    dtype = torch.float32 if rng.integers(0, 4) == 0 else torch.bfloat16
    if dtype == torch.float32:     # the precision path: keep the fp64-arithmetic kernels quick
        S = per * min(chunk, 64)
    return Workload(f"sweep{i}", B, Hq, Hkv, S, D, N, layout, causal, dtype, seed=2000 + i,
                    with_grad=True)


CASES = [_draw_case(i) for i in range(48)]


def _ids(w):
    return (f"{w.name}-L{w.layout}-N{w.N}-S{w.S}-B{w.B}-H{w.Hq}/{w.Hkv}-D{w.D}-"
            f"{'c' if w.causal else 'nc'}-{'f32' if w.dtype == torch.float32 else 'bf16'}")


@pytest.mark.parametrize("w", CASES, ids=[_ids(w) for w in CASES])
def test_sweep_fwd_bwd(cuda_dev, oracle, w):
    q, k, v, do = inputs.make_qkv(w)
    gq, gk, gv, gdo = (t.to(cuda_dev) for t in (q, k, v, do))
    out, lse = api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, w.causal)
    dq, dk, dv = api.ring_attn_bwd(gq, gk, gv, out, lse, gdo, w.N, w.layout, w.causal)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    ref, lref = oracle.attn_fwd(q, k, v, w.causal)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rows = np.arange(w.S)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, w.causal, rows, rows)
    grads = [g.float().cpu().numpy() for g in (dq, dk, dv)]
    if w.dtype == torch.float32:
        assert np.abs(o - ref).max() <= F32_TOL and np.abs(l - lref).max() <= F32_TOL
        for g, r in zip(grads, (rq, rk, rv)):
            assert (np.abs(g - r) / np.maximum(1.0, np.abs(r))).max() <= 1e-4
    else:
        check_bf16(o, l, ref, lref, _ids(w))
        for g, r in zip(grads, (rq, rk, rv)):
            scale = np.abs(r).max()
            e = np.abs(g - r)
            assert e.max() <= 1e-2 * scale and e.mean() <= 1e-3 * scale, (e.max(), scale)
