"""The forward kernel's work distribution does not change its results.

A launch of the tensor-core forward (ring, split-KV and per-step modes) runs
its work items -- query tiles, times the splits -- either one per thread
block or several per block, in alternating rounds over the longest-first
order (the default when there are at most 16 items per SM).  Each item is
computed the same way whichever block runs it, so the outputs must be equal
bit for bit for every grid; cp_debug_set_grid_limit picks the grid.  With a
few blocks every block runs many items in a row, including the empty ones of
split and step launches, which exercises the phase bookkeeping that carries
across items.
"""
import numpy as np
import pytest
import torch

from conftest import check_bf16
from context_parallelism_02_gb300 import api, inputs, ring
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu

ONE_PER_ITEM = 1 << 30
GRIDS = [ONE_PER_ITEM, 1, 3, 7]

CASES = [
    # name, B, Hq, Hkv, S, D, N, layout, causal
    ("zig_gqa_ragged_c200", 2, 4, 2, 1600, 128, 4, ZIG, True),
    ("cont_d64_ragged", 1, 2, 1, 1000, 64, 4, CONT, True),
    ("str_n3_c97_d64", 1, 2, 2, 291, 64, 3, STR, True),
    ("zig_noncausal_n2", 1, 2, 2, 1536, 128, 2, ZIG, False),
    ("str_n16_c130", 1, 1, 1, 2080, 128, 16, STR, True),
]


def _with_grid(grid, fn):
    api.cp_debug_set_grid_limit(grid)
    try:
        res = fn()
        torch.cuda.synchronize()
    finally:
        api.cp_debug_set_grid_limit(0)
    assert api.cp_get_error() == 0
    return res


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_grid_does_not_change_results(cuda_dev, oracle, case):
    name, B, Hq, Hkv, S, D, N, layout, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, torch.bfloat16, seed=131)
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))

    def run():
        fwd = api.ring_attn_fwd(gq, gk, gv, N, layout, causal)
        spl = api.ring_attn_fwd_split(gq, gk, gv, N, layout, causal, n_split=5)
        stp = ring.ring_attention_emulated(gq, gk, gv, N, layout, causal)
        return [t.clone() for pair in (fwd, spl, stp) for t in pair]

    ref_run = _with_grid(ONE_PER_ITEM, run)
    for grid in GRIDS[1:]:
        got = _with_grid(grid, run)
        for a, b in zip(got, ref_run):
            assert torch.equal(a, b), (name, grid)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    check_bf16(ref_run[0].float().cpu().numpy(), ref_run[1].cpu().numpy(), ref, lref, f"grid test {name}")


def test_s8192_persistent_default_matches_one_block_per_item(cuda_dev):
    """S=8192 (512 items for 152 SMs): the default persistent grid against one
    block per item, bit for bit."""
    w = inputs.S8K
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    run = lambda: [t.clone() for t in api.ring_attn_fwd(q, k, v, w.N, w.layout, True)]
    a = _with_grid(0, run)
    b = _with_grid(ONE_PER_ITEM, run)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
