"""GPU parity of ring_attn_fwd (through the C ABI) against the fp64 oracle.

Tolerances: bf16 inputs with fp32 accumulation -- |out err| <= 1e-2 plus the
half-ulp of the bf16 output rounding per element, mean |out err| <= 1e-3,
|lse err| <= 1e-3 (conftest.check_bf16); fp32 inputs -- 1e-5 on out and lse.
"""
import numpy as np
import pytest
import torch

from conftest import F32_TOL, check_bf16, check_bf16_pair, record_f32
from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu


def _run(w, dev, rank_range=None):
    q, k, v = inputs.make_qkv(w)
    out, lse = api.ring_attn_fwd(q.to(dev), k.to(dev), v.to(dev), w.N, w.layout, w.causal,
                                 rank_range=rank_range)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    return q, k, v, out.float().cpu().numpy(), lse.cpu().numpy()


def _check_bf16(out, lse, ref, lref, what=""):
    check_bf16(out, lse, ref, lref, what)


# ------------------------------------------------------------------ fp32 (tiny workload)


@pytest.mark.parametrize("qscale", [1.0, 8.0])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
def test_tiny_fp32(cuda_dev, oracle, layout, causal, qscale):
    w = inputs.TINY.with_(layout=layout, causal=causal, q_scale=qscale)
    q, k, v, out, lse = _run(w, cuda_dev)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    record_f32(f"tiny fp32 layout {layout} causal {causal} q x {qscale}", out, ref, lse, lref)
    assert np.abs(out - ref).max() <= F32_TOL
    assert np.abs(lse - lref).max() <= F32_TOL


def test_fp32_rows_sum_to_one(cuda_dev):
    """Rows of P recomputed from the GPU lse sum to 1 (to 1e-5)."""
    w = inputs.TINY
    q, k, v, out, lse = _run(w, cuda_dev)
    qd, kd = q.double().numpy(), k.double().numpy()
    s = np.einsum("bihd,bjhd->bhij", qd, kd) / np.sqrt(w.D)
    p = np.exp(s - lse[..., None].astype(np.float64))
    p = np.where(np.tril(np.ones((w.S, w.S), bool))[None, None], p, 0.0)
    assert np.abs(p.sum(-1) - 1.0).max() <= 1e-5


# ------------------------------------------------------------------ bf16, small shapes

SMALL = [
    # name, B, Hq, Hkv, S, D, N, layout, causal
    ("s1024_n4_zig", 1, 2, 2, 1024, 128, 4, ZIG, True),
    ("gqa_ragged_c200", 2, 4, 2, 1600, 128, 4, ZIG, True),
    ("d64_ragged_cont", 1, 2, 1, 1000, 64, 4, CONT, True),
    ("noncausal_n2", 1, 2, 2, 1536, 128, 2, ZIG, False),
    ("n1_plain", 1, 2, 2, 640, 128, 1, CONT, True),
    ("n8_exact_tiles", 1, 2, 2, 2048, 128, 8, ZIG, True),
    ("chunk_below_tile", 1, 2, 2, 512, 64, 4, ZIG, True),
    ("cont_noncausal_ragged", 1, 3, 3, 1200, 128, 3, CONT, False),
    ("n16_zig_small_chunks", 1, 1, 1, 2080, 128, 16, ZIG, True),
    # striped: every ring step crosses the causal diagonal
    ("str_s1024_n4", 1, 2, 2, 1024, 128, 4, STR, True),
    ("str_gqa_ragged_c400", 2, 4, 2, 1600, 128, 4, STR, True),
    ("str_d64_n8", 1, 2, 1, 2048, 64, 8, STR, True),
    ("str_noncausal_n2", 1, 2, 2, 1536, 128, 2, STR, False),
    ("str_n16_c130", 1, 1, 1, 2080, 128, 16, STR, True),
    ("str_n3_c97", 1, 2, 2, 291, 64, 3, STR, True),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_bf16(cuda_dev, oracle, case):
    name, B, Hq, Hkv, S, D, N, layout, causal = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, torch.bfloat16, seed=21)
    q, k, v, out, lse = _run(w, cuda_dev)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    _check_bf16(out, lse, ref, lref, name)


def test_large_logit_bf16(cuda_dev, oracle):
    """q scaled by 8: logits of tens, lse stays accurate (online rescaling).
    Rows become nearly one-hot, so |out| reaches the size of single v entries;
    the same bounds as every bf16 case (absolute max and mean)."""
    w = Workload("qx8", 1, 2, 2, 2048, 128, 4, ZIG, True, torch.bfloat16, seed=22, q_scale=8.0)
    q, k, v, out, lse = _run(w, cuda_dev)
    ref, lref = oracle.attn_fwd(q, k, v, True)
    _check_bf16(out, lse, ref, lref, "qx8 zigzag N=4")


def test_tiny_shape_bf16(cuda_dev, oracle):
    """The tiny workload's shapes in bf16 (chunks of 64 < one 128-row tile)."""
    for layout in (CONT, ZIG, STR):
        for causal in (True, False):
            w = inputs.TINY.with_(dtype=torch.bfloat16, layout=layout, causal=causal)
            q, k, v, out, lse = _run(w, cuda_dev)
            ref, lref = oracle.attn_fwd(q, k, v, causal)
            _check_bf16(out, lse, ref, lref, f"tiny bf16 {layout} {causal}")


def test_independent_of_n_and_layout(cuda_dev, oracle):
    """"What it does not change": the result is the same for every N and layout
    (up to rounding), and equals the oracle."""
    base = Workload("inv", 1, 2, 2, 4096, 128, 1, CONT, True, torch.bfloat16, seed=23)
    q, k, v = inputs.make_qkv(base)
    ref, lref = oracle.attn_fwd(q, k, v, True)
    outs = []
    for N in (1, 2, 4, 8):
        for layout in (CONT, ZIG, STR):
            o, l = api.ring_attn_fwd(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), N, layout, True)
            torch.cuda.synchronize()
            o = o.float().cpu().numpy()
            _check_bf16(o, l.cpu().numpy(), ref, lref, f"N={N} layout={layout}")
            outs.append(o)
    for o in outs[1:]:
        check_bf16_pair(o, outs[0], "N/layout independence")


@pytest.mark.parametrize("layout", [ZIG, STR])
def test_deterministic_and_rank_split(cuda_dev, layout):
    """Two runs are bitwise equal (no atomics), and running each virtual rank's
    queries separately reproduces the full launch bit for bit."""
    w = Workload("det", 1, 2, 2, 4096, 128, 4, layout, True, torch.bfloat16, seed=24)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    o1, l1 = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    o2, l2 = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    o3 = torch.zeros_like(o1)
    l3 = torch.zeros_like(l1)
    for r in range(w.N):
        api.ring_attn_fwd(q, k, v, w.N, w.layout, True, out=o3, lse=l3, rank_range=(r, r + 1))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_constant_v(cuda_dev):
    w = Workload("cv", 1, 2, 2, 2048, 128, 4, ZIG, True, torch.bfloat16, seed=25)
    q, k, _ = inputs.make_qkv(w)
    c = torch.linspace(-1, 1, w.D).to(torch.bfloat16)
    v = c.expand(1, w.S, 2, w.D).contiguous()
    out, _ = api.ring_attn_fwd(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), w.N, w.layout, True)
    torch.cuda.synchronize()
    assert (out.float().cpu() - c.float()).abs().max() <= 2 ** -7


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_outputs_in_pinned_host_memory(cuda_dev, dtype):
    """out and lse given as pinned host tensors: the kernels write the result
    straight into host memory, bitwise the same as into device buffers (bf16
    tensor-core path with a persistent and a one-block-per-item launch, and the
    fp32 path)."""
    for S, H in ((4096, 2), (8192, 8)) if dtype == torch.bfloat16 else ((512, 2),):
        w = Workload("host_out", 1, H, H, S, 128 if dtype == torch.bfloat16 else 64, 4, ZIG, True, dtype, seed=27 + S)
        q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
        ref_o, ref_l = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
        out_h = torch.full(q.shape, 7.0, dtype=dtype, pin_memory=True)
        lse_h = torch.full((w.B, w.Hq, w.S), 7.0, dtype=torch.float32, pin_memory=True)
        o, l = api.ring_attn_fwd(q, k, v, w.N, w.layout, True, out=out_h, lse=lse_h)
        torch.cuda.synchronize()
        assert api.cp_get_error() == 0
        assert o.data_ptr() == out_h.data_ptr() and not o.is_cuda
        assert torch.equal(out_h, ref_o.cpu()) and torch.equal(lse_h, ref_l.cpu())
    with pytest.raises(ValueError):
        api.ring_attn_fwd(q, k, v, w.N, w.layout, True, out=torch.empty(q.shape, dtype=dtype))   # not pinned


# ------------------------------------------------------------------ full-size workloads


def _sample_rows(S, N, layout, n_rand, seed):
    """Chunk boundaries (first/last rows of every chunk; for striped, the first
    and last rows of every rank and rows at tile edges) plus random rows."""
    rows = set()
    if layout == STR:
        for r in range(N):
            for t in (0, 127, 128, 255, 256, S // N - 1):
                if t < S // N:
                    rows.add(r + N * t)
    else:
        nch = N * (2 if layout == ZIG else 1)
        c = S // nch
        for ch in range(nch):
            rows.update({ch * c, ch * c + c - 1, ch * c + min(127, c - 1), ch * c + min(128, c - 1)})
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, S, n_rand).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def _check_sampled(w, dev, oracle, n_rand=16):
    q, k, v, out, lse = _run(w, dev)
    rows = _sample_rows(w.S, w.N, w.layout, n_rand, w.seed)
    ref, lref = oracle.attn_fwd(q, k, v, w.causal, rows=rows)
    _check_bf16(out[:, rows], lse[:, :, rows], ref, lref, f"{w.name} {len(rows)} sampled rows")
    return out, lse


def test_s8192_full(cuda_dev, oracle):
    """B=1, H=8, S=8192, D=128, N=8, zigzag, causal: every output row."""
    w = inputs.S8K
    q, k, v, out, lse = _run(w, cuda_dev)
    ref, lref = oracle.attn_fwd(q, k, v, True)
    _check_bf16(out, lse, ref, lref, w.name)


def test_gqa_s32768_sampled(cuda_dev, oracle):
    _check_sampled(inputs.GQA32K, cuda_dev, oracle)


@pytest.mark.parametrize("layout", [ZIG, CONT, STR])
def test_long_s131072_sampled(cuda_dev, oracle, layout):
    w = inputs.LONG128K.with_(layout=layout)
    _check_sampled(w, cuda_dev, oracle, n_rand=8)
