"""GPU parity at tensor sizes whose element indices pass 2^31 and 2^32 (the
maximum-size edge case): every kernel must form its offsets in 64 bits.

Inputs are drawn on the device from a seeded generator (a host draw of 5.4
billion values would take minutes); the oracle sees the same values, copied
back for the sampled batch and heads only.  Attention is independent per
(batch, head), and the gradient of a kv head depends only on the query heads
of its group, so slicing the inputs that way leaves the oracle's result for
the sampled rows unchanged.
"""
import numpy as np
import pytest
import torch

from conftest import check_bf16
from context_parallelism_02_gb300 import api
from context_parallelism_02_gb300.inputs import ZIGZAG as ZIG

pytestmark = pytest.mark.gpu

# q, out, dO, dq: 5 x 65536 x 128 x 128 = 5.37e9 elements (> 2^32)
B, S, HQ, HKV, D, N = 5, 65536, 128, 8, 128, 8
GRP = HQ // HKV


def _draw(shape, gen, dev):
    x = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    for b in range(shape[0]):   # per batch: an fp32 temporary of one batch only
        x[b] = torch.randn(shape[1:], generator=gen, device=dev).to(torch.bfloat16)
    return x


def test_fwd_bwd_beyond_2_32_elements(cuda_dev, oracle):
    gen = torch.Generator(device=cuda_dev).manual_seed(81)
    q = _draw((B, S, HQ, D), gen, cuda_dev)
    k = _draw((B, S, HKV, D), gen, cuda_dev)
    v = _draw((B, S, HKV, D), gen, cuda_dev)
    do = _draw((B, S, HQ, D), gen, cuda_dev)
    assert q.numel() > 2 ** 32
    out, lse = api.ring_attn_fwd(q, k, v, N, ZIG, True)
    dq, dk, dv = api.ring_attn_bwd(q, k, v, out, lse, do, N, ZIG, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    b = B - 1                                   # the last batch: offsets past 2^32
    g = HKV - 1                                 # the last kv head and its query heads
    heads = list(range(g * GRP, (g + 1) * GRP))
    rng = np.random.default_rng(81)
    rows = np.unique(np.concatenate([[0, S // 2 - 1, S // 2, S - 1], rng.integers(0, S, 6)]))
    qs = q[b:b + 1, :, heads].cpu()
    ks, vs = k[b:b + 1, :, g:g + 1].cpu(), v[b:b + 1, :, g:g + 1].cpu()
    dos = do[b:b + 1, :, heads].cpu()
    ref, lref = oracle.attn_fwd(qs, ks, vs, True, rows=rows)
    got = out[b:b + 1][:, rows][:, :, heads].float().cpu().numpy()
    lgot = lse[b:b + 1][:, heads][:, :, rows].cpu().numpy()
    check_bf16(got, lgot, ref, lref, "out beyond 2^32 elements (last batch, last kv group)")
    # dq on the sampled query rows; dk, dv on late keys (few queries see them)
    krows = np.array([S - 300, S - 129, S - 2, S - 1])
    rq, rk, rv = oracle.attn_bwd(qs, ks, vs, dos, True, rows, krows)
    for name, t, r, sel, idx in (("dq", dq, rq, heads, rows), ("dk", dk, rk, [g], krows),
                                 ("dv", dv, rv, [g], krows)):
        got = t[b:b + 1][:, idx][:, :, sel].float().cpu().numpy()
        err = np.abs(got - r)
        assert np.isfinite(got).all(), name
        assert err.max() <= 1e-2 * max(1.0, np.abs(r).max()), (name, err.max(), np.abs(r).max())


def test_lse_merge_n_beyond_2_31_elements(cuda_dev, oracle):
    """n = 2 partials of 17.8M rows x D = 128 (2.3e9 floats each)."""
    rows, n = 17_825_792, 2
    gen = torch.Generator(device=cuda_dev).manual_seed(82)
    xs = torch.randn((n, rows, D), generator=gen, device=cuda_dev)
    ls = torch.randn((n, rows), generator=gen, device=cuda_dev) * 2.0
    assert xs[0].numel() > 2 ** 31
    o, lo = api.lse_merge_n(xs, ls)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    rng = np.random.default_rng(82)
    sel = np.unique(np.concatenate([[0, rows - 1, rows // 2], rng.integers(0, rows, 64)]))
    rx, rl = oracle.lse_merge_n(xs[:, sel].cpu().numpy(), ls[:, sel].cpu().numpy())
    got, lgot = o[sel].cpu().numpy(), lo[sel].cpu().numpy()
    tol = (n + 2) * 2.0 ** -23 * max(1.0, float(np.abs(rx).max()))
    assert np.abs(got - rx).max() <= tol
    assert np.abs(lgot - rl).max() <= 1e-5


@pytest.mark.parametrize("layout", [0, 1])
def test_ulysses_beyond_2_31_elements(cuda_dev, oracle, layout):
    """seq->head of a [8][1][65536][72][128] bf16 tensor (4.8e9 elements):
    sampled rows against the layout's shard map, and the round trip bitwise."""
    n, b, s, h, d = 8, 1, 524288, 72, 128
    gen = torch.Generator(device=cuda_dev).manual_seed(83)
    x = torch.randint(-1000, 1000, (n, b, s // n, h, d), generator=gen, device=cuda_dev,
                      dtype=torch.int16).to(torch.bfloat16)
    assert x.numel() > 2 ** 32
    y = api.ulysses_seq_to_head(x, n, layout)
    torch.cuda.synchronize()
    pos = oracle.shard_pos(s, n, layout)          # pos[r][t]: global position of local row t
    rng = np.random.default_rng(83)
    for r, t in zip(rng.integers(0, n, 24), rng.integers(0, s // n, 24)):
        p = int(pos[r][t])
        for grp in (0, n - 1):
            want = x[r, 0, t, grp * (h // n):(grp + 1) * (h // n)]
            assert torch.equal(y[grp, 0, p], want), (r, t, grp)
    x2 = api.ulysses_head_to_seq(y, n, layout)
    torch.cuda.synchronize()
    assert torch.equal(x, x2)
    assert api.cp_get_error() == 0
