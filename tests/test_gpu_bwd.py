"""GPU parity of ring_attn_bwd (through the C ABI) against the fp64 oracle
gradient.

The pages give no gradient tolerance.  The bound used here follows from the
arithmetic: P and dS are rounded to bf16 before the tensor-core products
(relative half-ulp 2^-9) and dq/dk/dv are rounded to bf16 at the end, so the
error of an output element is a small multiple of 2^-9 times the size of the
gradient; with max|ref| the largest reference entry of the checked slice,
max|err| <= 1e-2 * max|ref| and mean|err| <= 1e-3 * max|ref|.
"""
import numpy as np
import pytest
import torch

from conftest import record_grad
from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu

GRAD_MAX = 1e-2
GRAD_MEAN = 1e-3


def _grads(w, dev):
    q, k, v, do = inputs.make_qkv(w)
    gq, gk, gv, gdo = (t.to(dev) for t in (q, k, v, do))
    out, lse = api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, w.causal)
    dq, dk, dv = api.ring_attn_bwd(gq, gk, gv, out, lse, gdo, w.N, w.layout, w.causal)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    return (q, k, v, do), (dq.float().cpu().numpy(), dk.float().cpu().numpy(),
                           dv.float().cpu().numpy())


def _check(name, got, ref):
    record_grad(name, got, ref)
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert np.isfinite(got).all(), name
    assert err.max() <= GRAD_MAX * scale, (name, err.max(), scale)
    assert err.mean() <= GRAD_MEAN * scale, (name, err.mean(), scale)


SMALL = [
    # name, B, Hq, Hkv, S, D, N, layout, causal
    ("s1024_n4_zig", 1, 2, 2, 1024, 128, 4, ZIG, True),
    ("gqa_ragged_c200", 2, 4, 2, 1600, 128, 4, ZIG, True),
    ("d64_ragged_cont", 1, 2, 1, 1000, 64, 4, CONT, True),
    ("noncausal_n2", 1, 2, 2, 1536, 128, 2, ZIG, False),
    ("n1_plain", 1, 2, 2, 640, 128, 1, CONT, True),
    ("chunk_below_tile", 1, 2, 2, 512, 64, 4, ZIG, True),
    ("n8_zig", 1, 2, 2, 4096, 128, 8, ZIG, True),
    ("str_s1024_n4", 1, 2, 2, 1024, 128, 4, STR, True),
    ("str_gqa_ragged_c400", 2, 4, 2, 1600, 128, 4, STR, True),
    ("str_d64_n8", 1, 2, 1, 2048, 64, 8, STR, True),
    ("str_noncausal", 1, 2, 2, 1536, 128, 2, STR, False),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_bwd(cuda_dev, oracle, case):
    name, B, Hq, Hkv, S, D, N, layout, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, torch.bfloat16, seed=51,
                 with_grad=True)
    (q, k, v, do), (dq, dk, dv) = _grads(w, cuda_dev)
    rows = np.arange(S)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, causal, rows, rows)
    _check(name + " dq", dq, rq)
    _check(name + " dk", dk, rk)
    _check(name + " dv", dv, rv)


def test_bwd_deterministic_and_layout_free(cuda_dev):
    """No atomics: two runs are bitwise equal; N and layout change only rounding."""
    base = Workload("bdet", 1, 2, 2, 2048, 128, 4, ZIG, True, torch.bfloat16, seed=52,
                    with_grad=True)
    q, k, v, do = (t.to(cuda_dev) for t in inputs.make_qkv(base))
    res = []
    for N, layout in ((4, ZIG), (4, ZIG), (1, CONT), (8, CONT)):
        out, lse = api.ring_attn_fwd(q, k, v, N, layout, True)
        res.append(api.ring_attn_bwd(q, k, v, out, lse, do, N, layout, True))
    torch.cuda.synchronize()
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
    for other in res[2:]:
        for a, b in zip(res[0], other):
            scale = a.float().abs().max()
            assert (a.float() - b.float()).abs().max() <= 2 * GRAD_MAX * scale


def test_bwd_full_size_slices_and_invariants(cuda_dev, oracle):
    """B=2, H=16, S=32768, D=128, N=8, zigzag, causal.

    Oracle gradient on slices, for two heads of both batches: dq on 1024
    random query rows; dk/dv on three key slices -- the first 1024 keys (seen
    by every query, folded over all 8 ranks and all their ring steps), 512
    keys from the middle of a middle chunk, and the last 512 keys (seen by the
    fewest queries).

    At full size, two identities of the exact gradient (fp64 sums of the bf16
    results): every row of P sums to 1, so sum_j dV_j = sum_i dO_i; and
    sum_j dS_ij = 0 for every i, so sum_j dK_j = 0 (per batch, head, column).
    The residual of each comes from rounding only: dK and dV are rounded to
    bf16 (half-ulp 2^-9 relative) and so are the P and dS entering them, with
    errors of either sign, so the residual grows like the root sum of squares
    (rss) of the summed terms times ~2^-9.  The bound allows 2^-4 of the rss,
    far below what a dropped or duplicated tile would leave (a whole term)."""
    w = inputs.BWD32K
    (q, k, v, do), (dq, dk, dv) = _grads(w, cuda_dev)
    heads = [0, 5]
    sq, sk, sv, sdo = (t[:, :, heads] for t in (q, k, v, do))
    rng = np.random.default_rng(7)
    qrows = np.sort(rng.choice(w.S, 1024, replace=False))
    c = w.S // (2 * w.N)                       # zigzag chunk: 2048 keys
    mid = 7 * c + c // 2                       # chunk 7 (rank 7's first chunk)
    krows = np.concatenate([np.arange(0, 1024), np.arange(mid - 256, mid + 256),
                            np.arange(w.S - 512, w.S)])
    rq, rk, rv = oracle.attn_bwd(sq, sk, sv, sdo, True, qrows, krows)
    _check("dq slice", dq[:, qrows][:, :, heads], rq)
    for name, sel in (("first 1024 keys", slice(0, 1024)), ("middle chunk keys", slice(1024, 1536)),
                      ("last 512 keys", slice(1536, 2048))):
        _check(f"dk {name}", dk[:, krows[sel]][:, :, heads], rk[:, sel])
        _check(f"dv {name}", dv[:, krows[sel]][:, :, heads], rv[:, sel])
    # identities at full size
    dv64, dk64 = dv.astype(np.float64), dk.astype(np.float64)
    do64 = do.double().numpy()
    res_v = np.abs(dv64.sum(axis=1) - do64.sum(axis=1))
    rss_v = np.sqrt((dv64 ** 2).sum(axis=1) + (do64 ** 2).sum(axis=1))
    res_k = np.abs(dk64.sum(axis=1))
    rss_k = np.sqrt((dk64 ** 2).sum(axis=1))
    print(f"dV identity residual / rss: max {(res_v / rss_v).max():.3e}; "
          f"dK identity residual / rss: max {(res_k / rss_k).max():.3e}")
    assert (res_v <= 2.0 ** -4 * rss_v).all(), (res_v / rss_v).max()
    assert (res_k <= 2.0 ** -4 * rss_k).all(), (res_k / rss_k).max()


def test_bwd_medium_deterministic_and_identities(cuda_dev):
    """B=1, H=8, S=16384, D=128, N=8, zigzag, causal: a backward of 1024
    dK/dV blocks (several per SM) run twice.  The two calls are bitwise equal
    (no atomics, a fixed order of every sum), and the gradients satisfy the
    two exact identities of the full-size test (sum_j dV_j = sum_i dO_i,
    sum_j dK_j = 0 per head and column) within the same rounding bound."""
    w = Workload("bmed", 1, 8, 8, 16384, 128, 8, ZIG, True, torch.bfloat16, seed=57, with_grad=True)
    q, k, v, do = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    out, lse = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    first = api.ring_attn_bwd(q, k, v, out, lse, do, w.N, w.layout, True)
    second = api.ring_attn_bwd(q, k, v, out, lse, do, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    for a, b in zip(first, second):
        assert torch.equal(a, b)
    _, dk, dv = (t.double().cpu().numpy() for t in first)
    do64 = do.double().cpu().numpy()
    res_v = np.abs(dv.sum(axis=1) - do64.sum(axis=1))
    rss_v = np.sqrt((dv ** 2).sum(axis=1) + (do64 ** 2).sum(axis=1))
    res_k = np.abs(dk.sum(axis=1))
    rss_k = np.sqrt((dk ** 2).sum(axis=1))
    assert (res_v <= 2.0 ** -4 * rss_v).all(), (res_v / rss_v).max()
    assert (res_k <= 2.0 ** -4 * rss_k).all(), (res_k / rss_k).max()
