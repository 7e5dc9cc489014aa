"""Small parity cases under the debug-bounds build of libcp.

That build (-DCP_DEBUG_BOUNDS) checks, in the tensor-core kernels, every TMA
tile coordinate and every output row index against the tensor's extents; a
value out of range would be recorded as CP_EBOUNDS in the error word and
replaced by an in-range one (no trap).  It stands in for a memory checker:
these runs must end with no such record, and with results that still match
the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from conftest import check_bf16
from context_parallelism_02_gb300 import _lib, api, build, inputs, ring
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_bounds(cuda_dev):
    build.build(debug_bounds=True)
    with _lib.variant("debug_bounds") as lib:
        assert api.cp_get_error() == 0
        yield lib


CASES = [
    # name, B, Hq, Hkv, S, D, N, layout, causal
    ("zig_gqa_ragged_c200", 2, 4, 2, 1600, 128, 4, ZIG, True),
    ("cont_d64_ragged", 1, 2, 1, 1000, 64, 4, CONT, True),
    ("str_n3_c97_d64", 1, 2, 2, 291, 64, 3, STR, True),
    ("str_gqa_ragged_c400", 2, 4, 2, 1600, 128, 4, STR, True),
    ("zig_noncausal_n2", 1, 2, 2, 1536, 128, 2, ZIG, False),
    ("zig_n16_c65", 1, 1, 1, 2080, 128, 16, ZIG, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forward_backward_in_bounds(debug_bounds, oracle, cuda_dev, case):
    name, B, Hq, Hkv, S, D, N, layout, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, torch.bfloat16, seed=121,
                 with_grad=True)
    q, k, v, do = inputs.make_qkv(w)
    gq, gk, gv, gdo = (t.to(cuda_dev) for t in (q, k, v, do))
    out, lse = api.ring_attn_fwd(gq, gk, gv, N, layout, causal)
    osp, lsp = api.ring_attn_fwd_split(gq, gk, gv, N, layout, causal, n_split=3)
    ost, lst = ring.ring_attention_emulated(gq, gk, gv, N, layout, causal)
    dq, dk, dv = api.ring_attn_bwd(gq, gk, gv, out, lse, gdo, N, layout, causal)
    # the persistent instantiations too: 3 blocks take every item in turn
    api.cp_debug_set_grid_limit(3)
    try:
        outp, lsep = api.ring_attn_fwd(gq, gk, gv, N, layout, causal)
        ospp, _ = api.ring_attn_fwd_split(gq, gk, gv, N, layout, causal, n_split=3)
        ostp, _ = ring.ring_attention_emulated(gq, gk, gv, N, layout, causal)
        torch.cuda.synchronize()
    finally:
        api.cp_debug_set_grid_limit(0)
    assert api.cp_get_error() == 0          # in particular no CP_EBOUNDS
    assert torch.equal(outp, out) and torch.equal(lsep, lse)
    assert torch.equal(ospp, osp) and torch.equal(ostp, ost)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    for tag, o, l_ in (("ring", out, lse), ("split", osp, lsp), ("step", ost, lst)):
        check_bf16(o.float().cpu().numpy(), l_.cpu().numpy(), ref, lref, f"debug-bounds {name} {tag}")
    rows = np.arange(S)
    for got, r in zip((dq, dk, dv), oracle.attn_bwd(q, k, v, do, causal, rows, rows)):
        e = np.abs(got.float().cpu().numpy() - r)
        assert e.max() <= 1e-2 * np.abs(r).max() and e.mean() <= 1e-3 * np.abs(r).max()
