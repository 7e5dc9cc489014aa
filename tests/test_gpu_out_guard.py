"""The forward writes exactly its outputs: out and lse placed inside larger
buffers, between sentinel regions, come back bitwise equal to a plain
allocation and leave the sentinels untouched.  The output view is taken both
32-byte aligned (the kernel's 32-byte store path) and only 16-byte aligned
(its 16-byte fallback), for both head dimensions, in the one-block-per-unit
and the persistent launch."""
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
