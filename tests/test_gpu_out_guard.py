"""The forward writes exactly its outputs: out and lse placed inside larger
buffers, between sentinel regions, come back bitwise equal to a plain
allocation and leave the sentinels untouched.  The output view is taken both
32-byte aligned (the kernel's 32-byte store path) and only 16-byte aligned
(its 16-byte fallback), for both head dimensions, in the one-block-per-unit
and the persistent launch; the same for the split forward's fp32 partials
(workspace) and the ring step's state (out_acc, lse_acc, out_final)."""
import pytest
import torch

from context_parallelism_02_gb300 import api, inputs
from context_parallelism_02_gb300.inputs import ZIGZAG as ZIG, STRIPED as STR, Workload

pytestmark = pytest.mark.gpu

PAD = 64   # sentinel elements before and after each view (plus the alignment shift)


def _guarded(shape, dtype, shift, device, fill):
    n = 1
    for s in shape:
        n *= s
    big = torch.full((PAD + shift + n + PAD,), fill, dtype=dtype, device=device)
    view = big[PAD + shift: PAD + shift + n].view(shape)
    return big, view


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shift", [0, 8])   # bf16 elements: 0 B (32-byte aligned) or 16 B
@pytest.mark.parametrize("S,layout", [(1024, ZIG), (8192, ZIG), (2048, STR)])
def test_forward_writes_only_its_outputs(cuda_dev, D, shift, S, layout):
    w = Workload("guard", 1, 4, 2, S, D, 4, layout, True, torch.bfloat16, seed=120 + D + shift)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    ref_out, ref_lse = api.ring_attn_fwd(q, k, v, w.N, w.layout, True)
    big_o, out = _guarded(q.shape, torch.bfloat16, shift, cuda_dev, 77.0)
    big_l, lse = _guarded((w.B, w.Hq, w.S), torch.float32, shift, cuda_dev, 77.0)
    assert out.data_ptr() % 16 == 0
    assert (out.data_ptr() % 32 == 0) == (shift == 0)
    api.ring_attn_fwd(q, k, v, w.N, w.layout, True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)
    for big, n in ((big_o, out.numel()), (big_l, lse.numel())):
        head = big[:PAD + shift]
        tail = big[PAD + shift + n:]
        assert bool((head == 77.0).all()) and bool((tail == 77.0).all())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shift_bytes", [0, 16])
def test_split_partials_stay_in_the_workspace(cuda_dev, shift_bytes, D):
    """The split forward's fp32 partials (32- or 16-byte aligned workspace)
    stay inside ring_attn_fwd_split_workspace bytes; the result is bitwise
    the same as with a plain workspace (32-byte aligned: the warp regroups its
    rows so that each store covers whole 128-byte pieces; 16-byte aligned:
    every lane writes its own row)."""
    w = Workload("guard_split", 1, 2, 2, 2048, D, 4, ZIG, True, torch.bfloat16, seed=131 + D)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    n_split = 3
    ref_out, ref_lse = api.ring_attn_fwd_split(q, k, v, w.N, w.layout, True, n_split=n_split)
    need = api.ring_attn_fwd_split_workspace(w.B, w.Hq, w.S, w.D, n_split)
    big = torch.full((256 + shift_bytes + need + 256,), 0xA5, dtype=torch.uint8, device=cuda_dev)
    ws = big[256 + shift_bytes: 256 + shift_bytes + need]
    assert ws.data_ptr() % 16 == 0 and (ws.data_ptr() % 32 == 0) == (shift_bytes == 0)
    out, lse = api.ring_attn_fwd_split(q, k, v, w.N, w.layout, True, n_split=n_split, workspace=ws)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    assert bool((big[:256 + shift_bytes] == 0xA5).all()) and bool((big[256 + shift_bytes + need:] == 0xA5).all())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shift", [0, 4])   # fp32 elements: 0 B or 16 B (bf16 out_final: twice as many)
def test_step_state_stays_in_its_buffers(cuda_dev, shift, D):
    """Two ring steps (flash_block_step) into out_acc / lse_acc / out_final views
    between sentinels, 32- or 16-byte aligned: bitwise the same as plain
    buffers, and the sentinels untouched.  The plain buffers take the regrouped
    loads and stores (32-byte aligned), so the 16-byte shift checks them
    against the per-lane path bit for bit."""
    from context_parallelism_02_gb300 import ring
    w = Workload("guard_step", 1, 4, 2, 4096, D, 4, ZIG, True, torch.bfloat16, seed=132 + D)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    r = 2
    qs = ring.shard(q, r, w.N, w.layout).contiguous()
    ks = [ring.shard(k, s, w.N, w.layout).contiguous() for s in range(w.N)]
    vs = [ring.shard(v, s, w.N, w.layout).contiguous() for s in range(w.N)]
    C = w.S // w.N

    def two_steps(oacc, lacc, ofin):
        for s in range(2):
            src = (r - s) % w.N
            api.flash_block_step(qs, ks[src], vs[src], r, src, w.N, w.S, w.layout, True, out_acc=oacc,
                                 lse_acc=lacc, out_final=ofin if s == 1 else None, accumulate=s > 0)

    ref = (torch.empty(w.B, C, w.Hq, w.D, device=cuda_dev), torch.empty(w.B, w.Hq, C, device=cuda_dev),
           torch.empty(w.B, C, w.Hq, w.D, device=cuda_dev, dtype=torch.bfloat16))
    two_steps(*ref)
    big_o, oacc = _guarded((w.B, C, w.Hq, w.D), torch.float32, shift, cuda_dev, 77.0)
    big_l, lacc = _guarded((w.B, w.Hq, C), torch.float32, shift, cuda_dev, 77.0)
    big_f, ofin = _guarded((w.B, C, w.Hq, w.D), torch.bfloat16, 2 * shift, cuda_dev, 77.0)
    two_steps(oacc, lacc, ofin)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    for got, want in zip((oacc, lacc, ofin), ref):
        assert torch.equal(got, want)
    for big, n, sh in ((big_o, oacc.numel(), shift), (big_l, lacc.numel(), shift), (big_f, ofin.numel(), 2 * shift)):
        assert bool((big[:PAD + sh] == 77.0).all()) and bool((big[PAD + sh + n:] == 77.0).all())
