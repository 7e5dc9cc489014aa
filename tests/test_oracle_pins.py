"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a library routine, a value printed on the pages, a closed form, an
invariant the pages state, or brute force on tiny inputs.

Sources are cited by page title and section.
"""
import math
import os

import numpy as np
import pytest
import torch

from context_parallelism_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CONT, ZIG, STR = 0, 1, 2


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.empty(shape, dtype=torch.float64).normal_(generator=g) * scale)


def _sdpa(q, k, v, causal, scale=None):
    """Library attention (torch, fp64, CPU) in BSHD with contiguous GQA groups."""
    Hq, Hkv = q.shape[2], k.shape[2]
    qt, kt, vt = (x.permute(0, 2, 1, 3) for x in (q, k, v))
    if Hq != Hkv:
        kt = kt.repeat_interleave(Hq // Hkv, dim=1)
        vt = vt.repeat_interleave(Hq // Hkv, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o.permute(0, 2, 1, 3)


def _shards(x, S, N, layout, pos_fn):
    """Rank-local shards of a global-order [B, S, H, D] array (numpy), with the
    local row order given by pos_fn(r) (global positions of rank r's rows)."""
    return [np.ascontiguousarray(x[:, pos_fn(r)]) for r in range(N)]


def _positions(S, N, layout):
    """An independent restatement of the page's sharding (not the oracle's
    mapper): contiguous blocks of S/N; zigzag chunks r and 2N-1-r of S/(2N);
    striped positions r, r+N, r+2N, ..."""
    def pos(r):
        if layout == CONT:
            return np.arange(r * (S // N), (r + 1) * (S // N))
        if layout == STR:
            return np.arange(r, S, N)
        c = S // (2 * N)
        return np.concatenate([np.arange(r * c, (r + 1) * c),
                               np.arange((2 * N - 1 - r) * c, (2 * N - r) * c)])
    return pos


# ---------------------------------------------------------------- (a) brute force / library


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv,S,D", [(2, 2, 96, 16), (4, 2, 64, 8), (2, 2, 130, 64)])
@pytest.mark.parametrize("qscale", [1.0, 8.0])
def test_attn_fwd_matches_library(oracle, causal, Hq, Hkv, S, D, qscale):
    q = _rand((2, S, Hq, D), 1, qscale)
    k = _rand((2, S, Hkv, D), 2)
    v = _rand((2, S, Hkv, D), 3)
    out, lse = oracle.attn_fwd(q, k, v, causal)
    ref = _sdpa(q, k, v, causal).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse against scipy's logsumexp of scores built with einsum
    from scipy.special import logsumexp
    kk = np.repeat(k.numpy(), Hq // Hkv, axis=2)
    s = np.einsum("bihd,bjhd->bhij", q.numpy(), kk) / math.sqrt(D)
    if causal:
        s = np.where(np.tril(np.ones((S, S), bool))[None, None], s, -np.inf)
    np.testing.assert_allclose(lse, logsumexp(s, axis=-1), rtol=0, atol=1e-11)


def test_attn_fwd_rows_and_key_range(oracle):
    """Row subsets and key ranges agree with the full computation."""
    q, k, v = _rand((1, 80, 2, 8), 4), _rand((1, 80, 2, 8), 5), _rand((1, 80, 2, 8), 6)
    out, lse = oracle.attn_fwd(q, k, v, True)
    rows = np.array([0, 7, 40, 79])
    o2, l2 = oracle.attn_fwd(q, k, v, True, rows=rows)
    np.testing.assert_array_equal(o2, out[:, rows])
    np.testing.assert_array_equal(l2, lse[:, :, rows])
    # key range [0, 80) is the whole row; an empty range gives (0, -inf)
    o3, l3 = oracle.attn_fwd(q, k, v, True, rows=np.array([5]), klo=10, khi=80)
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))


# ---------------------------------------------------------------- (b) exactness across N, layout


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_ring_equals_definition(oracle, N, layout, causal):
    """"Sequence and Context Parallelism", "What it does not change": the
    distributed result equals single-device attention (nothing approximated)."""
    S = 128
    q, k, v = _rand((1, S, 4, 16), 7), _rand((1, S, 2, 16), 8), _rand((1, S, 2, 16), 9)
    out1, lse1 = oracle.attn_fwd(q, k, v, causal)
    out2, lse2 = oracle.ring_fwd(q, k, v, N, layout, causal)
    np.testing.assert_allclose(out2, out1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse1, rtol=0, atol=1e-12)


def test_ring_tiny_workload_all_variants(oracle):
    """The tiny workload (S=512, D=64, N=4): ring == definition for both
    layouts, causal and not, and for the q x 8 large-logit variant."""
    w = inputs.TINY
    for qscale in (1.0, 8.0):
        q, k, v = inputs.make_qkv(w.with_(q_scale=qscale))
        for causal in (True, False):
            ref, lref = oracle.attn_fwd(q, k, v, causal)
            for layout in (CONT, ZIG, STR):
                o, l = oracle.ring_fwd(q, k, v, w.N, layout, causal)
                assert np.max(np.abs(o - ref)) < 1e-12
                assert np.max(np.abs(l - lref)) < 1e-11


# ---------------------------------------------------------------- (c) rows of P sum to 1


@pytest.mark.parametrize("causal", [True, False])
def test_row_sums(oracle, causal):
    S, D = 200, 32
    q, k, v = _rand((1, S, 2, D), 10, 3.0), _rand((1, S, 2, D), 11), _rand((1, S, 2, D), 12)
    _, lse = oracle.ring_fwd(q, k, v, 4, ZIG, causal)
    s = np.einsum("bihd,bjhd->bhij", q.numpy(), k.numpy()) / math.sqrt(D)
    p = np.exp(s - lse[..., None])
    if causal:
        p = np.where(np.tril(np.ones((S, S), bool))[None, None], p, 0.0)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- (d) constant V


@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
def test_constant_v(oracle, layout):
    S, D = 64, 16
    q, k = _rand((1, S, 2, D), 13), _rand((1, S, 2, D), 14)
    c = np.linspace(-1, 1, D)
    v = np.broadcast_to(c, (1, S, 2, D)).copy()
    for N in (1, 2, 4):
        out, _ = oracle.ring_fwd(q, k, v, N, layout, True)
        np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- (e) work identities


def _brute_counts(pos, causal):
    """Brute force: full mask matrix over positions, summed per (rank, source)."""
    N, L = pos.shape
    flat = pos.reshape(-1)
    mask = (flat[None, :] <= flat[:, None]) if causal else np.ones((flat.size, flat.size), bool)
    per = mask.reshape(N, L, N, L).sum(axis=(1, 3))        # [rank, source rank]
    out = np.zeros((N, N), np.int64)
    for r in range(N):
        for kk in range(N):
            out[r, kk] = per[r, (r - kk) % N]
    return out


@pytest.mark.parametrize("S,N", [(32, 4), (48, 2), (64, 8), (40, 1)])
@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
@pytest.mark.parametrize("causal", [True, False])
def test_pair_counts_brute_force(oracle, S, N, layout, causal):
    np.testing.assert_array_equal(oracle.pair_counts(S, N, layout, causal),
                                  _brute_counts(_page_pos(S, N, layout), causal))


def _striped_pos(S, N):
    """"Causal Masking and Load Balancing": token t goes to rank t mod P; a
    rank keeps its tokens in sequence order."""
    return np.array([[p for p in range(S) if p % N == r] for r in range(N)])


def _page_pos(S, N, layout):
    if layout == CONT:
        return np.arange(S).reshape(N, S // N)
    return _zigzag_pos(S, N) if layout == ZIG else _striped_pos(S, N)


def _zigzag_pos(S, N):
    c = S // (2 * N)
    chunks = np.arange(S).reshape(2 * N, c)
    return np.stack([np.concatenate([chunks[r], chunks[2 * N - 1 - r]]) for r in range(N)])


@pytest.mark.parametrize("S,N", [(512, 4), (8192, 8), (1024, 16)])
def test_pair_count_closed_forms(oracle, S, N):
    """Causal work per rank ("Context Parallelism", "The causal imbalance";
    "Sequence Parallelism in LLMs", "Causal Masking and Load Balancing").

    contiguous rank r: r*C^2 + C(C+1)/2 (imbalanced 1..N); zigzag: 2N c^2 + c
    for every rank; both sum to S(S+1)/2.  Per step, zigzag gives 2c^2 for
    k != 0 and 2c^2 + c at k = 0; contiguous gives C^2 if src < r,
    C(C+1)/2 if src == r, else 0."""
    C, c = S // N, S // (2 * N)
    cont = oracle.pair_counts(S, N, CONT, True)
    zig = oracle.pair_counts(S, N, ZIG, True)
    for r in range(N):
        assert cont[r].sum() == r * C * C + C * (C + 1) // 2
        assert zig[r].sum() == 2 * N * c * c + c
        for kk in range(N):
            src = (r - kk) % N
            exp_c = C * C if src < r else (C * (C + 1) // 2 if src == r else 0)
            assert cont[r, kk] == exp_c
            assert zig[r, kk] == (2 * c * c + c if kk == 0 else 2 * c * c)
    assert cont.sum() == zig.sum() == S * (S + 1) // 2
    # G15 reading: contiguous rank r has non-empty work on exactly r+1 steps
    for r in range(N):
        assert np.count_nonzero(cont[r]) == r + 1
    nc = oracle.pair_counts(S, N, ZIG, False)
    assert np.all(nc == C * C)


@pytest.mark.parametrize("S,N", [(512, 4), (8192, 8), (1024, 16), (96, 3)])
def test_striped_pair_count_closed_forms(oracle, S, N):
    """Striped partitioning ("Causal Masking and Load Balancing"): with C = S/N
    rows per rank, query r + N t sees the keys src + N u with u <= t - [src > r],
    so step k (src = (r - k) mod N) has C(C+1)/2 - C [src > r] pairs, rank r
    in total N C(C+1)/2 - C (N - 1 - r): every rank within C(N-1) pairs of
    every other ("equal causal density"), summing to S(S+1)/2."""
    C = S // N
    st = oracle.pair_counts(S, N, STR, True)
    for r in range(N):
        for kk in range(N):
            src = (r - kk) % N
            assert st[r, kk] == C * (C + 1) // 2 - (C if src > r else 0)
        assert st[r].sum() == N * C * (C + 1) // 2 - C * (N - 1 - r)
    assert st.sum() == S * (S + 1) // 2
    tot = st.sum(1)
    assert tot.max() - tot.min() == C * (N - 1)
    assert np.all(oracle.pair_counts(S, N, STR, False) == C * C)


def test_pair_counts_imbalance_example(oracle):
    """The worked example (S=8192, N=8): rank 0 attends to almost nothing,
    rank 7 to everything; zigzag makes every rank equal."""
    cont = oracle.pair_counts(8192, 8, CONT, True).sum(1)
    zig = oracle.pair_counts(8192, 8, ZIG, True).sum(1)
    assert cont[0] == 524_800 and cont[7] == 7_864_832
    assert np.all(zig == 4_194_816)


# ---------------------------------------------------------------- shard map and schedule (golden)


def test_shard_map_golden(oracle):
    pos = oracle.shard_pos(8192, 8, CONT)
    for r, first, last in _read_table("contiguous_imbalance_example.txt"):
        assert pos[r, 0] == first and pos[r, -1] == last
        np.testing.assert_array_equal(pos[r], np.arange(first, last + 1))
    S, N = 64, 4
    c = S // (2 * N)
    pz = oracle.shard_pos(S, N, ZIG)
    for r, a, b in _read_table("zigzag_chunks_n4.txt"):
        np.testing.assert_array_equal(pz[r], np.concatenate([np.arange(a * c, a * c + c),
                                                             np.arange(b * c, b * c + c)]))
    # every position appears exactly once
    assert sorted(pz.reshape(-1).tolist()) == list(range(S))
    # striped: rank p mod N holds position p
    for S, N in ((64, 4), (96, 3), (40, 8), (7, 1)):
        ps = oracle.shard_pos(S, N, STR)
        np.testing.assert_array_equal(ps, _striped_pos(S, N))
        assert sorted(ps.reshape(-1).tolist()) == list(range(S))


def test_ring_schedule_golden(oracle):
    src = oracle.ring_source_table(4)
    for step, gpu, blk in _read_table("ring_schedule_p4.txt"):
        assert src[step, gpu] == blk
    # every rank sees every block exactly once over N steps
    for N in (1, 3, 8, 16):
        t = oracle.ring_source_table(N)
        for r in range(N):
            assert sorted(t[:, r].tolist()) == list(range(N))


# ---------------------------------------------------------------- (g) merge


def test_merge_split_keys(oracle):
    """Two disjoint key halves computed separately and merged equal the whole
    ("Algorithmic Mechanics", online softmax rescaling)."""
    S = 96
    q, k, v = _rand((1, S, 2, 16), 15, 2.0), _rand((1, S, 2, 16), 16), _rand((1, S, 2, 16), 17)
    full, lfull = oracle.attn_fwd(q, k, v, False)
    oa, la = oracle.attn_fwd(q, k, v, False, klo=0, khi=40)
    ob, lb = oracle.attn_fwd(q, k, v, False, klo=40, khi=S)
    # lse layout [B,H,S] vs out [B,S,H,D]: merge row-wise in [B,H,S,D]
    def rows(o):
        return o.transpose(0, 2, 1, 3).reshape(-1, 16)
    om, lm = oracle.lse_merge(rows(oa), la.reshape(-1), rows(ob), lb.reshape(-1))
    np.testing.assert_allclose(om, rows(full), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lfull.reshape(-1), rtol=0, atol=1e-13)
    # commutative
    om2, lm2 = oracle.lse_merge(rows(ob), lb.reshape(-1), rows(oa), la.reshape(-1))
    np.testing.assert_allclose(om2, om, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(lm2, lm)
    # associative over a 3-way split
    o1, l1 = oracle.attn_fwd(q, k, v, False, klo=0, khi=30)
    o2, l2 = oracle.attn_fwd(q, k, v, False, klo=30, khi=70)
    o3, l3 = oracle.attn_fwd(q, k, v, False, klo=70, khi=S)
    x12, y12 = oracle.lse_merge(rows(o1), l1.reshape(-1), rows(o2), l2.reshape(-1))
    xa, ya = oracle.lse_merge(x12, y12, rows(o3), l3.reshape(-1))
    x23, y23 = oracle.lse_merge(rows(o2), l2.reshape(-1), rows(o3), l3.reshape(-1))
    xb, yb = oracle.lse_merge(rows(o1), l1.reshape(-1), x23, y23)
    np.testing.assert_allclose(xa, rows(full), rtol=0, atol=1e-13)
    np.testing.assert_allclose(xb, xa, rtol=0, atol=1e-13)
    np.testing.assert_allclose(ya, yb, rtol=0, atol=1e-13)


@pytest.mark.parametrize("cuts", [[0, 96], [0, 10, 96], [0, 5, 40, 41, 90, 96], [0, 1, 2, 3, 96]])
def test_merge_n_split_keys(oracle, cuts):
    """n disjoint key ranges computed separately and merged in one n-way step
    equal attention over all keys ("Algorithmic Mechanics": the log-sum-exp
    combination of partial results)."""
    S, D = 96, 16
    q, k, v = _rand((1, S, 2, D), 18, 2.0), _rand((1, S, 2, D), 19), _rand((1, S, 2, D), 20)
    full, lfull = oracle.attn_fwd(q, k, v, False)
    parts = [oracle.attn_fwd(q, k, v, False, klo=a, khi=b) for a, b in zip(cuts[:-1], cuts[1:])]
    outs = np.stack([o.transpose(0, 2, 1, 3).reshape(-1, D) for o, _ in parts])
    lses = np.stack([l.reshape(-1) for _, l in parts])
    om, lm = oracle.lse_merge_n(outs, lses)
    np.testing.assert_allclose(om, full.transpose(0, 2, 1, 3).reshape(-1, D), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lfull.reshape(-1), rtol=0, atol=1e-13)
    # independent of the order of the partials
    perm = np.arange(len(parts))[::-1]
    om2, lm2 = oracle.lse_merge_n(outs[perm], lses[perm])
    np.testing.assert_allclose(om2, om, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lm2, lm, rtol=0, atol=1e-14)


def test_merge_n_empty_partials(oracle):
    """Partials with lse = -inf carry no weight; all empty gives (0, -inf);
    n = 1 returns its input."""
    rng = np.random.default_rng(1)
    rows, D, n = 7, 4, 3
    outs = rng.standard_normal((n, rows, D))
    lses = rng.standard_normal((n, rows))
    lses[1, :] = -np.inf
    lses[:, 3] = -np.inf
    om, lm = oracle.lse_merge_n(outs, lses)
    keep = [0, 2]
    o2, l2 = oracle.lse_merge_n(outs[keep], lses[keep])
    np.testing.assert_array_equal(np.isneginf(lm), np.isneginf(l2))
    np.testing.assert_allclose(om, o2, rtol=0, atol=1e-15)
    assert np.all(om[3] == 0) and np.isneginf(lm[3])
    o1, l1 = oracle.lse_merge_n(outs[:1], lses[:1])
    fin = np.isfinite(lses[0])
    np.testing.assert_allclose(o1[fin], outs[0][fin], rtol=0, atol=1e-15)
    np.testing.assert_allclose(l1[fin], lses[0][fin], rtol=0, atol=1e-15)


def test_merge_neg_inf_identity(oracle):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 8))
    lx = rng.standard_normal(5)
    empty = np.zeros((5, 8))
    ninf = np.full(5, -np.inf)
    o, l = oracle.lse_merge(x, lx, empty + 7.0, ninf)
    np.testing.assert_array_equal(o, x)
    np.testing.assert_array_equal(l, lx)
    o, l = oracle.lse_merge(empty + 3.0, ninf, empty - 2.0, ninf)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_merge_closed_form_equal_lse(oracle):
    """Equal lse: the merge is the average and lse grows by ln 2."""
    a, b = np.ones((3, 4)), 3 * np.ones((3, 4))
    la = np.array([0.5, -2.0, 10.0])
    o, l = oracle.lse_merge(a, la, b, la)
    np.testing.assert_allclose(o, 2.0, atol=1e-15)
    np.testing.assert_allclose(l, la + math.log(2.0), atol=1e-15)


# ---------------------------------------------------------------- (h) Ulysses relayout


@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
@pytest.mark.parametrize("N,H", [(2, 4), (4, 8), (8, 8), (1, 3)])
def test_ulysses_against_slicing(oracle, N, H, layout):
    """"DeepSpeed Ulysses": rank g ends with the full sequence for heads
    [g*H/N, (g+1)*H/N), in global order; the second all-to-all inverts it."""
    B, S, D = 2, 16 * N, 4
    x = inputs.make_layout_tensor(N, B, S, H, D, torch.bfloat16, seed=3)
    y = oracle.ulysses_seq_to_head(x, N, layout)
    # global tensor assembled with numpy from the page's chunk definition
    xs = x.view(torch.int16).numpy()
    pos = _page_pos(S, N, layout)
    glob = np.zeros((B, S, H, D), np.int16)
    for r in range(N):
        glob[:, pos[r]] = xs[r]
    hg = H // N
    for g in range(N):
        np.testing.assert_array_equal(y[g], glob[:, :, g * hg:(g + 1) * hg])
    back = oracle.ulysses_head_to_seq(y, N, layout)
    np.testing.assert_array_equal(back, xs)


# ---------------------------------------------------------------- (i) backward


def _loss_grads_torch(q, k, v, do, causal):
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = _sdpa(q, k, v, causal)
    (out * do).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_bwd_matches_autograd(oracle, causal, Hq, Hkv):
    S, D = 48, 8
    q, k, v = _rand((2, S, Hq, D), 20), _rand((2, S, Hkv, D), 21), _rand((2, S, Hkv, D), 22)
    do = _rand((2, S, Hq, D), 23)
    gq, gk, gv = _loss_grads_torch(q, k, v, do, causal)
    rows = np.arange(S)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, rows, rows)
    np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, gk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, gv, rtol=0, atol=1e-12)
    # row slices agree with the full computation
    sl = np.array([3, 17, 40])
    dq2, dk2, dv2 = oracle.attn_bwd(q, k, v, do, causal, sl, sl)
    np.testing.assert_allclose(dq2, dq[:, sl], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk2, dk[:, sl], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv2, dv[:, sl], rtol=0, atol=1e-13)


def test_bwd_finite_difference(oracle):
    """Central differences of L = sum(dO * out) with h = 1e-6."""
    S, D, h = 12, 4, 1e-6
    q, k, v = _rand((1, S, 2, D), 30), _rand((1, S, 1, D), 31), _rand((1, S, 1, D), 32)
    do = _rand((1, S, 2, D), 33).numpy()
    rows = np.arange(S)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True, rows, rows)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, True)
        return float((o * do).sum())

    rng = np.random.default_rng(1)
    for name, base, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        arr = base.numpy()
        for _ in range(6):
            idx = tuple(rng.integers(0, n) for n in arr.shape)
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args = {"q": q.numpy(), "k": k.numpy(), "v": v.numpy()}
            args[name] = plus
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = minus
            lm = loss(args["q"], args["k"], args["v"])
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])


# ---------------------------------------------------------------- (j) special cases


def test_n1_is_plain_attention_and_noncausal_layout_free(oracle):
    S = 64
    q, k, v = _rand((1, S, 2, 8), 40), _rand((1, S, 2, 8), 41), _rand((1, S, 2, 8), 42)
    o1, _ = oracle.ring_fwd(q, k, v, 1, CONT, True)
    np.testing.assert_allclose(o1, _sdpa(q, k, v, True).numpy(), rtol=0, atol=1e-12)
    oc, lc = oracle.ring_fwd(q, k, v, 4, CONT, False)
    oz, lz = oracle.ring_fwd(q, k, v, 4, ZIG, False)
    np.testing.assert_allclose(oc, oz, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lc, lz, rtol=0, atol=1e-13)


def test_oracle_rejects_bad_shapes(oracle):
    with pytest.raises(ValueError):
        oracle.shard_pos(100, 3, CONT)
    with pytest.raises(ValueError):
        oracle.shard_pos(12, 4, ZIG)
    with pytest.raises(ValueError):
        oracle.pair_counts(12, 4, ZIG, True)
    with pytest.raises(ValueError):
        oracle.shard_pos(12, 5, STR)
    with pytest.raises(ValueError):
        oracle.shard_pos(12, 4, 3)


# ---------------------------------------------------------------- one ring step on local shards


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
@pytest.mark.parametrize("N", [1, 2, 3, 4])
def test_block_steps_compose_to_attention(oracle, N, layout, causal):
    """"What it does not change" / "Algorithmic Mechanics": the N ring steps of
    one device, block of rank (r - k) mod N at step k, from the empty state,
    give that device's rows of single-device attention (library SDPA)."""
    S = 48 * N if layout != ZIG else 24 * 2 * N
    q, k, v = _rand((2, S, 4, 8), 11), _rand((2, S, 2, 8), 12), _rand((2, S, 2, 8), 13)
    ref = _sdpa(q, k, v, causal).numpy()
    pos = _positions(S, N, layout)
    qs, ks, vs = (_shards(x.numpy(), S, N, layout, pos) for x in (q, k, v))
    for r in range(N):
        out = lse = None
        for step in range(N):
            src = (r - step) % N
            out, lse = oracle.block_step(qs[r], ks[src], vs[src], S, N, layout, causal, r, src,
                                         out, lse)
        np.testing.assert_allclose(out, ref[:, pos(r)], rtol=0, atol=1e-12)
        assert np.isfinite(lse).all()


def test_block_step_single_block_is_attention_over_its_keys(oracle):
    """Contiguous shards: one step against source src equals definitional
    attention restricted to src's key range (the oracle's O1 with a key range,
    itself pinned to library attention); rows that see no key of the block
    get the empty state (0, -inf)."""
    S, N = 96, 4
    C = S // N
    q, k, v = _rand((1, S, 2, 8), 21), _rand((1, S, 2, 8), 22), _rand((1, S, 2, 8), 23)
    for r in range(N):
        for src in range(N):
            out, lse = oracle.block_step(q[:, r * C:(r + 1) * C], k[:, src * C:(src + 1) * C],
                                         v[:, src * C:(src + 1) * C], S, N, CONT, True, r, src)
            rows = np.arange(r * C, (r + 1) * C)
            ref, lref = oracle.attn_fwd(q, k, v, True, rows=rows, klo=src * C, khi=(src + 1) * C)
            if src > r:   # every key of the block lies after every query
                assert np.all(out == 0) and np.all(np.isneginf(lse))
            else:
                np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse, lref, rtol=0, atol=1e-12)


def test_block_step_order_free_and_empty_block_identity(oracle):
    """The fold is the log-sum-exp merge, so the blocks can arrive in any order
    (results equal to rounding); a block no query sees leaves the state
    unchanged bit for bit."""
    S, N, layout = 128, 4, ZIG
    q, k, v = _rand((1, S, 2, 8), 31, 3.0), _rand((1, S, 2, 8), 32), _rand((1, S, 2, 8), 33)
    pos = _positions(S, N, layout)
    qs, ks, vs = (_shards(x.numpy(), S, N, layout, pos) for x in (q, k, v))
    r = 2
    res = []
    for order in ([0, 1, 2, 3], [3, 1, 0, 2]):
        out = lse = None
        for src in order:
            out, lse = oracle.block_step(qs[r], ks[src], vs[src], S, N, layout, True, r, src, out, lse)
        res.append((out, lse))
    np.testing.assert_allclose(res[0][0], res[1][0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(res[0][1], res[1][1], rtol=0, atol=1e-12)
    # contiguous, causal: rank 0 sees nothing of rank 3's block
    posc = _positions(S, N, CONT)
    qc, kc, vc = (_shards(x.numpy(), S, N, CONT, posc) for x in (q, k, v))
    out, lse = oracle.block_step(qc[0], kc[0], vc[0], S, N, CONT, True, 0, 0)
    out2, lse2 = oracle.block_step(qc[0], kc[3], vc[3], S, N, CONT, True, 0, 3, out, lse)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
