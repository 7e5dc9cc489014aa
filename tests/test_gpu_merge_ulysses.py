"""GPU parity of lse_merge, the Ulysses relayouts and the bounded-wait failure
path, through the C ABI."""
import numpy as np
import pytest
import torch

from context_parallelism_02_gb300 import CP_ETIMEOUT, api, inputs
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,D,ninf", [(1, 128, 0), (1000, 128, 0), (4097, 64, 7), (65536, 128, 5),
                                         (3, 4, 2)])
def test_lse_merge_matches_oracle(cuda_dev, oracle, rows, D, ninf):
    a, la, b, lb = inputs.make_merge_inputs(rows, D, seed=31, neg_inf_every=ninf)
    if ninf:   # also a row where both partials are empty
        la[0] = lb[0] = float("-inf")
    out, lse = api.lse_merge(*(t.to(cuda_dev) for t in (a, la, b, lb)))
    torch.cuda.synchronize()
    ref, lref = oracle.lse_merge(a, la, b, lb)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    assert np.abs(out - ref).max() <= 1e-6
    fin = np.isfinite(lref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - lref[fin]).max(initial=0) <= 1e-6
    if ninf:
        assert np.all(out[0] == 0) and np.isneginf(lse[0])


def test_lse_merge_in_place_and_full_size(cuda_dev, oracle):
    """The benchmark workload (rows = 1x8x131072, D = 128), out aliasing out_a;
    sampled rows checked against the oracle."""
    a, la, b, lb = inputs.make_merge_inputs()
    ga, gla, gb, glb = (t.to(cuda_dev) for t in (a, la, b, lb))
    out, lse = api.lse_merge(ga, gla, gb, glb, out=ga, lse=gla)
    torch.cuda.synchronize()
    rows = np.random.default_rng(3).integers(0, la.numel(), 4096)
    ref, lref = oracle.lse_merge(a[rows], la[rows], b[rows], lb[rows])
    assert np.abs(out[rows].cpu().numpy() - ref).max() <= 1e-6
    assert np.abs(lse[rows].cpu().numpy() - lref).max() <= 1e-6


def test_lse_merge_equals_attention_over_split_keys(cuda_dev, oracle):
    """Attention over keys [0, 40) and [40, S) merged equals attention over all."""
    S, D = 96, 64
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(1, S, 1, D, generator=g, dtype=torch.float64) for _ in range(3))
    oa, la = oracle.attn_fwd(q, k, v, False, klo=0, khi=40)
    ob, lb = oracle.attn_fwd(q, k, v, False, klo=40, khi=S)
    full, lfull = oracle.attn_fwd(q, k, v, False)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x.reshape(-1, D) if x.ndim == 4 else x.reshape(-1))).float().to(cuda_dev)
    out, lse = api.lse_merge(t(oa), t(la), t(ob), t(lb))
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy() - full.reshape(-1, D)).max() <= 1e-5
    assert np.abs(lse.cpu().numpy() - lfull.reshape(-1)).max() <= 1e-5


@pytest.mark.parametrize("n,rows,D,ninf", [(1, 1000, 128, 0), (2, 1000, 128, 3), (3, 4097, 64, 5),
                                           (4, 1, 4, 0), (16, 2049, 128, 7), (5, 333, 12, 2),
                                           (32, 64, 128, 9), (33, 257, 8, 4)])
def test_lse_merge_n_matches_oracle(cuda_dev, oracle, n, rows, D, ninf):
    outs, lses = inputs.make_merge_n_inputs(n, rows, D, seed=33, neg_inf_every=ninf)
    if ninf:
        lses[:, 1] = float("-inf")        # a row where every partial is empty
    out, lse = api.lse_merge_n(outs.to(cuda_dev), lses.to(cuda_dev))
    torch.cuda.synchronize()
    ref, lref = oracle.lse_merge_n(outs, lses)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    # fp32: n weighted terms and their sum, each rounded once (2^-24 relative),
    # plus the weights' own rounding: (n + 2) ulps of the largest input
    tol = (n + 2) * 2.0 ** -23 * max(1.0, float(outs.abs().max()))
    assert np.abs(out - ref).max() <= tol
    fin = np.isfinite(lref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - lref[fin]).max(initial=0) <= 1e-6
    if ninf:
        assert np.all(out[1] == 0) and np.isneginf(lse[1])


def test_lse_merge_n_equals_attention_and_in_place(cuda_dev, oracle):
    """Attention over 4 disjoint key ranges merged in one n-way pass equals
    attention over all keys; out and lse may alias the first partial."""
    S, D = 120, 64
    g = torch.Generator().manual_seed(6)
    q, k, v = (torch.randn(1, S, 2, D, generator=g, dtype=torch.float64) for _ in range(3))
    cuts = [0, 17, 60, 61, S]
    parts = [oracle.attn_fwd(q, k, v, False, klo=a, khi=b) for a, b in zip(cuts[:-1], cuts[1:])]
    outs = torch.from_numpy(np.stack([o.transpose(0, 2, 1, 3).reshape(-1, D) for o, _ in parts])).float()
    lses = torch.from_numpy(np.stack([l.reshape(-1) for _, l in parts])).float()
    go, gl = outs.to(cuda_dev), lses.to(cuda_dev)
    out, lse = api.lse_merge_n(go, gl, out=go[0], lse=gl[0])
    torch.cuda.synchronize()
    full, lfull = oracle.attn_fwd(q, k, v, False)
    assert np.abs(out.cpu().numpy() - full.transpose(0, 2, 1, 3).reshape(-1, D)).max() <= 1e-5
    assert np.abs(lse.cpu().numpy() - lfull.reshape(-1)).max() <= 1e-5


def test_lse_merge_n_full_size(cuda_dev, oracle):
    """rows = 1x8x131072, D = 128, n = 4 partials: sampled rows against the oracle."""
    outs, lses = inputs.make_merge_n_inputs(4)
    out, lse = api.lse_merge_n(outs.to(cuda_dev), lses.to(cuda_dev))
    torch.cuda.synchronize()
    rows = np.random.default_rng(4).integers(0, lses.shape[1], 4096)
    ref, lref = oracle.lse_merge_n(outs[:, rows], lses[:, rows])
    assert np.abs(out[rows].cpu().numpy() - ref).max() <= 6 * 2.0 ** -23 * float(outs.abs().max())
    assert np.abs(lse[rows].cpu().numpy() - lref).max() <= 1e-6


ULY = [
    # N, B, S, H, D, dtype, layout
    (2, 1, 64, 4, 8, torch.bfloat16, CONT),
    (4, 2, 128, 8, 16, torch.float32, ZIG),
    (8, 1, 256, 8, 128, torch.bfloat16, ZIG),
    (4, 1, 96, 4, 3, torch.bfloat16, CONT),      # 6-byte runs: narrow vectors
    (1, 1, 32, 3, 8, torch.float32, ZIG),
    (4, 2, 128, 8, 16, torch.bfloat16, STR),
    (8, 1, 256, 8, 128, torch.float32, STR),
    (3, 1, 96, 6, 5, torch.bfloat16, STR),
]


@pytest.mark.parametrize("case", ULY)
def test_ulysses_bit_exact(cuda_dev, oracle, case):
    N, B, S, H, D, dt, layout = case
    x = inputs.make_layout_tensor(N, B, S, H, D, dt, seed=41)
    y = api.ulysses_seq_to_head(x.to(cuda_dev), N, layout)
    torch.cuda.synchronize()
    ref = oracle.ulysses_seq_to_head(x, N, layout)
    assert np.array_equal(y.cpu().contiguous().view({2: torch.int16, 4: torch.int32}[x.element_size()]).numpy(), ref)
    back = api.ulysses_head_to_seq(y, N, layout)
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), x)


@pytest.mark.parametrize("name,H", [("q", 32), ("kv", 8)])
def test_ulysses_gqa_workload(cuda_dev, oracle, name, H):
    """The GQA workload's tensors (S=32768, N=8, zigzag): q [8][1][4096][32][128]
    and k/v [8][1][4096][8][128] bf16, both directions, bit-exact."""
    N, B, S, D = 8, 1, 32768, 128
    x = inputs.make_layout_tensor(N, B, S, H, D, torch.bfloat16, seed=42)
    gx = x.to(cuda_dev)
    y = api.ulysses_seq_to_head(gx, N, ZIG)
    back = api.ulysses_head_to_seq(y, N, ZIG)
    torch.cuda.synchronize()
    assert torch.equal(back, gx)
    ref = oracle.ulysses_seq_to_head(x, N, ZIG)
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), ref)


def test_bounded_wait_times_out_and_context_survives(cuda_dev):
    """A wait on a barrier nothing arrives at gives up after its limit; the
    error word reports CP_ETIMEOUT and the context keeps working."""
    assert api.cp_get_error() == 0
    api.cp_debug_wait_timeout(2_000_000)          # 2 ms
    assert api.cp_get_error() == CP_ETIMEOUT
    assert api.cp_get_error() == 0                # read clears it
    w = inputs.TINY.with_(dtype=torch.bfloat16)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    out, _ = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert api.cp_get_error() == 0
