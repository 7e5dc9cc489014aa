"""GPU parity of the split-KV forward (ring_attn_fwd_split, through the C ABI)
against the fp64 oracle.

Each query tile's key walk is cut into n_split pieces whose normalised partials
are merged by log-sum-exp, so the result is the attention of the unsplit
forward up to rounding: the same bf16 bounds apply (|err| <= 1e-2 plus the
half-ulp of the bf16 output per element, mean <= 1e-3, |lse err| <= 1e-3).
"""
import numpy as np
import pytest
import torch

from conftest import BF16_LSE, check_bf16, check_bf16_pair
from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu


def _check_bf16(out, lse, ref, lref, what=""):
    check_bf16(out, lse, ref, lref, what)


def _split(w, dev, n_split, rank_range=None, out=None, lse=None):
    q, k, v = inputs.make_qkv(w)
    o, l = api.ring_attn_fwd_split(q.to(dev), k.to(dev), v.to(dev), w.N, w.layout, w.causal,
                                   n_split=n_split, rank_range=rank_range, out=out, lse=lse)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    return (q, k, v), o, l


CASES = [
    # name, B, Hq, Hkv, S, D, N, layout, causal
    ("zig_s2048_n4", 1, 2, 2, 2048, 128, 4, ZIG, True),
    ("gqa_ragged_c200", 2, 4, 2, 1600, 128, 4, ZIG, True),
    ("d64_ragged_cont", 1, 2, 1, 1000, 64, 4, CONT, True),
    ("cont_noncausal_n3", 1, 3, 3, 1200, 128, 3, CONT, False),
    ("str_gqa_ragged", 2, 4, 2, 1600, 128, 4, STR, True),
    ("str_d64_n8", 1, 2, 1, 2048, 64, 8, STR, True),
    ("n1_plain", 1, 2, 2, 4096, 128, 1, CONT, True),
]


@pytest.mark.parametrize("n_split", [2, 3, 7])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_split_matches_oracle(cuda_dev, oracle, case, n_split):
    name, B, Hq, Hkv, S, D, N, layout, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, torch.bfloat16, seed=71)
    (q, k, v), o, l = _split(w, cuda_dev, n_split)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    _check_bf16(o.float().cpu().numpy(), l.cpu().numpy(), ref, lref, f"{name} n_split={n_split}")


@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
def test_more_splits_than_tiles(cuda_dev, oracle, layout):
    """n_split = 64 on walks of 1 to 8 tiles: most splits are empty and carry
    (0, -inf), which the merge drops."""
    w = Workload("many", 1, 2, 2, 1024, 128, 4, layout, True, torch.bfloat16, seed=72)
    (q, k, v), o, l = _split(w, cuda_dev, 64)
    ref, lref = oracle.attn_fwd(q, k, v, True)
    _check_bf16(o.float().cpu().numpy(), l.cpu().numpy(), ref, lref, f"layout={layout}")


@pytest.mark.parametrize("layout", [ZIG, STR, CONT])
def test_rank_ranges(cuda_dev, oracle, layout):
    """One launch per virtual rank fills every row; rows of other ranks are not
    touched by a rank's launch."""
    w = Workload("ranks", 1, 2, 2, 4096, 128, 4, layout, True, torch.bfloat16, seed=73)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    out = torch.full_like(q, 7.0)
    lse = torch.full((1, 2, w.S), 7.0, dtype=torch.float32, device=cuda_dev)
    pos = api.cp_shard_map(w.S, w.N, layout)
    for r in range(w.N):
        api.ring_attn_fwd_split(q, k, v, w.N, layout, True, n_split=3, out=out, lse=lse,
                                rank_range=(r, r + 1))
        torch.cuda.synchronize()
        done = np.sort(pos[: r + 1].reshape(-1))
        todo = np.setdiff1d(np.arange(w.S), done)
        assert (out[0, todo].float() == 7.0).all() and (lse[0][:, todo] == 7.0).all()
    assert api.cp_get_error() == 0
    ref, lref = oracle.attn_fwd(q.cpu(), k.cpu(), v.cpu(), True)
    _check_bf16(out.float().cpu().numpy(), lse.cpu().numpy(), ref, lref, f"layout={layout}")


def test_one_split_is_the_unsplit_forward(cuda_dev):
    w = Workload("one", 2, 4, 2, 2048, 128, 4, ZIG, True, torch.bfloat16, seed=74)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    o1 = torch.zeros_like(q)
    l1 = torch.zeros((w.B, w.Hq, w.S), dtype=torch.float32, device=cuda_dev)
    o2 = torch.zeros_like(o1)
    l2 = torch.zeros_like(l1)
    api.ring_attn_fwd(q, k, v, w.N, w.layout, True, out=o1, lse=l1, rank_range=(1, 3))
    api.ring_attn_fwd_split(q, k, v, w.N, w.layout, True, n_split=1, out=o2, lse=l2,
                            rank_range=(1, 3))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_deterministic_and_close_to_unsplit(cuda_dev):
    """Two split runs agree bit for bit; the split and unsplit results agree to
    bf16 rounding."""
    w = Workload("det", 1, 4, 4, 8192, 128, 8, ZIG, True, torch.bfloat16, seed=75)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    a = api.ring_attn_fwd_split(q, k, v, w.N, w.layout, True, n_split=5)
    b = api.ring_attn_fwd_split(q, k, v, w.N, w.layout, True, n_split=5)
    u = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    check_bf16_pair(a[0].float().cpu().numpy(), u[0].float().cpu().numpy(), "split vs unsplit")
    assert (a[1] - u[1]).abs().max().item() <= BF16_LSE


def test_large_logit_split(cuda_dev, oracle):
    """q x 8: the partials' lse differ by tens, the merge weights span e^-40."""
    w = Workload("qx8", 1, 2, 2, 2048, 128, 4, ZIG, True, torch.bfloat16, seed=76, q_scale=8.0)
    (q, k, v), o, l = _split(w, cuda_dev, 4)
    ref, lref = oracle.attn_fwd(q, k, v, True)
    _check_bf16(o.float().cpu().numpy(), l.cpu().numpy(), ref, lref, "qx8")


@pytest.mark.parametrize("rank,n_split", [(0, 4), (15, None)])
def test_long_one_rank(cuda_dev, oracle, rank, n_split):
    """One rank of the S=131072, H=8, D=128, N=16 zigzag ring (the per-rank
    launch a device of a real ring would run), at 4 splits and at the chosen
    count: sampled rows of that rank against the oracle."""
    w = inputs.LONG128K
    if n_split is None:
        n_split = api.cp_fwd_split_count(w.B, w.Hq, w.S, w.D, w.N, w.layout, True, (rank, rank + 1))
        assert n_split == 2
    (q, k, v), o, l = _split(w, cuda_dev, n_split, rank_range=(rank, rank + 1))
    pos = np.sort(api.cp_shard_map(w.S, w.N, w.layout)[rank])
    rng = np.random.default_rng(rank)
    rows = np.unique(np.concatenate([pos[:2], pos[-2:], pos[len(pos) // 2 - 1: len(pos) // 2 + 1],
                                     rng.choice(pos, 8, replace=False)]))
    ref, lref = oracle.attn_fwd(q, k, v, True, rows=rows)
    _check_bf16(o.float().cpu().numpy()[:, rows], l.cpu().numpy()[:, :, rows], ref, lref,
                f"rank {rank} n_split={n_split}")
