"""GPU parity of usp_attn_fwd (Unified Sequence Parallelism: n_ulysses x
n_ring virtual ranks, "Sequence Parallelism in LLMs", "Unified Sequence
Parallelism (USP / 2D SP)") through the C ABI.

USP computes attention over all keys, so the fp64 oracle's definitional
attention is the reference (bf16: |err| <= 1e-2 plus the half-ulp of the
bf16 output per element, mean <= 1e-3, |lse err| <= 1e-3; fp32: 1e-5).  Each head group runs the same ring
kernel as ring_attn_fwd with N = n_ring, so the two are also compared bit
for bit.
"""
import numpy as np
import pytest
import torch

from conftest import F32_TOL, check_bf16
from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu

CASES = [
    # name, n_ulysses, n_ring, layout, B, Hq, Hkv, S, D, dtype, causal
    ("u2_r4_zig_gqa", 2, 4, ZIG, 1, 4, 2, 1024, 128, torch.bfloat16, True),
    ("u4_r2_cont_b2", 4, 2, CONT, 2, 8, 4, 512, 64, torch.bfloat16, True),
    ("u2_r2_striped", 2, 2, STR, 1, 4, 4, 768, 128, torch.bfloat16, True),
    ("u1_r4_ring_only", 1, 4, ZIG, 1, 2, 2, 512, 64, torch.bfloat16, True),
    ("u4_r1_ulysses_only", 4, 1, CONT, 1, 4, 4, 256, 64, torch.bfloat16, False),
    ("u2_r3_ragged", 2, 3, ZIG, 1, 2, 2, 600, 128, torch.bfloat16, True),    # chunks of 100 rows
    ("u2_r2_fp32", 2, 2, ZIG, 1, 2, 2, 512, 64, torch.float32, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_usp_matches_oracle_and_ring(cuda_dev, oracle, case):
    name, nu, nr, layout, B, Hq, Hkv, S, D, dt, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, nr, layout, causal, dt, seed=71)
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))
    out, lse = api.usp_attn_fwd(gq, gk, gv, nu, nr, layout, causal)
    ring_out, ring_lse = api.ring_attn_fwd(gq, gk, gv, nr, layout, causal)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    assert torch.equal(out, ring_out) and torch.equal(lse, ring_lse), name
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    if dt == torch.float32:
        assert np.abs(o - ref).max() <= F32_TOL and np.abs(l - lref).max() <= F32_TOL
    else:
        check_bf16(o, l, ref, lref, f"usp {name}")


def test_usp_gqa_workload_sampled(cuda_dev, oracle):
    """The GQA workload's shapes (Hq=32, Hkv=8, S=32768, D=128, zigzag) on a
    4 x 2 grid (4 Ulysses head groups of 8 query / 2 kv heads, ring of 2):
    bitwise equal to the ring over 2 ranks; sampled rows against the oracle."""
    w = inputs.GQA32K.with_(N=2)
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))
    out, lse = api.usp_attn_fwd(gq, gk, gv, 4, 2, w.layout, True)
    ring_out, ring_lse = api.ring_attn_fwd(gq, gk, gv, 2, w.layout, True)
    torch.cuda.synchronize()
    assert torch.equal(out, ring_out) and torch.equal(lse, ring_lse)
    rows = np.sort(np.random.default_rng(9).choice(w.S, 24, replace=False))
    ref, lref = oracle.attn_fwd(q, k, v, True, rows=rows)
    o = out.float().cpu().numpy()[:, rows]
    check_bf16(o, lse.cpu().numpy()[:, :, rows], ref, lref, "usp 4x2 GQA S=32768 sampled rows")
