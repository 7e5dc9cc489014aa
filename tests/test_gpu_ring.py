"""GPU parity of flash_block_step (one ring step on shard-local buffers,
through the C ABI) and of the real-ring driver built on it.

  * Every (rank, step) of small rings against the fp64 oracle's one-step
    function: the running state after each step, and the final output against
    single-device attention.  bf16: conftest.check_bf16 bounds (the fp32
    state carries the same P rounding as the output); fp32: 1e-5.
  * The whole ring, all ranks emulated in one process, at the S=8192 and
    S=131072 workloads, against the oracle and against ring_attn_fwd.
  * Two processes on this GPU running the driver, blocks exchanged through
    pinned host memory over gloo (HostStagedTransport): each process's
    kernels run on their own, only the host exchange joins them.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from conftest import F32_TOL, check_bf16, check_bf16_pair
from context_parallelism_02_gb300 import api, inputs, ring
from context_parallelism_02_gb300.inputs import CONTIGUOUS as CONT, STRIPED as STR, ZIGZAG as ZIG, Workload

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BF, F32 = torch.bfloat16, torch.float32

CASES = [
    # name, B, Hq, Hkv, S, D, N, layout, causal, dtype, q_scale
    ("zig_n4_s1024", 1, 2, 2, 1024, 128, 4, ZIG, True, BF, 1.0),
    ("zig_gqa_ragged_c200", 2, 4, 2, 1600, 128, 4, ZIG, True, BF, 1.0),
    ("cont_d64_ragged_c250", 1, 2, 1, 1000, 64, 4, CONT, True, BF, 1.0),
    ("str_n4_c400", 1, 2, 2, 1600, 128, 4, STR, True, BF, 1.0),
    ("str_n3_c97_d64", 1, 2, 2, 291, 64, 3, STR, True, BF, 1.0),
    ("zig_noncausal_n2", 1, 2, 2, 1536, 128, 2, ZIG, False, BF, 1.0),
    ("n1_plain", 1, 2, 2, 640, 128, 1, CONT, True, BF, 1.0),
    ("zig_n8_c64_below_tile", 1, 2, 2, 1024, 128, 8, ZIG, True, BF, 1.0),
    ("zig_qx8", 1, 2, 2, 1024, 128, 4, ZIG, True, BF, 8.0),
    ("f32_tiny_zig", 1, 2, 2, 512, 64, 4, ZIG, True, F32, 1.0),
    ("f32_str_gqa", 1, 2, 1, 384, 64, 3, STR, True, F32, 1.0),
    ("f32_qx8_cont", 1, 2, 2, 512, 128, 4, CONT, True, F32, 8.0),
]


def _check_state(out, lse, ref, lref, dtype, what):
    if dtype == F32:
        fin = np.isfinite(lref)
        assert np.array_equal(np.isfinite(lse), fin), what
        assert np.abs(out - ref).max() <= F32_TOL, (what, np.abs(out - ref).max())
        assert np.abs(lse[fin] - lref[fin]).max(initial=0) <= F32_TOL, what
    else:
        check_bf16(out, lse, ref, lref, what)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_steps_match_oracle(cuda_dev, oracle, case):
    name, B, Hq, Hkv, S, D, N, layout, causal, dtype, qs = case
    w = Workload(name, B, Hq, Hkv, S, D, N, layout, causal, dtype, seed=101, q_scale=qs)
    q, k, v = inputs.make_qkv(w)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    shards = [[ring.shard(x, r, N, layout) for r in range(N)] for x in (q, k, v)]
    dq, dk, dv = ([t.to(cuda_dev) for t in xs] for xs in shards)
    for r in range(N):
        out_acc = torch.full((B, S // N, Hq, D), float("nan"), device=cuda_dev)
        lse_acc = torch.full((B, Hq, S // N), float("nan"), device=cuda_dev)
        final = torch.full_like(dq[r], float("nan"))
        o_ref = l_ref = None
        for step in range(N):
            src = (r - step) % N
            api.flash_block_step(dq[r], dk[src], dv[src], r, src, N, S, layout, causal,
                                 out_acc=out_acc, lse_acc=lse_acc,
                                 out_final=final if step == N - 1 else None, accumulate=step > 0)
            torch.cuda.synchronize()
            o_ref, l_ref = oracle.block_step(shards[0][r], shards[1][src], shards[2][src], S, N,
                                             layout, causal, r, src, o_ref, l_ref)
            _check_state(out_acc.cpu().numpy(), lse_acc.cpu().numpy(), o_ref, l_ref, dtype,
                         f"{name} rank {r} step {step} state")
        assert api.cp_get_error() == 0
        pos = ring.shard_positions(S, N, layout, r).numpy()
        f = final.float().cpu().numpy()
        if dtype == F32:
            assert np.abs(f - ref[:, pos]).max() <= F32_TOL
        else:
            check_bf16(f, lse_acc.cpu().numpy(), ref[:, pos], lref[:, :, pos],
                       f"{name} rank {r} final")


@pytest.mark.parametrize("layout", [CONT, ZIG, STR])
def test_first_step_without_visible_keys(cuda_dev, oracle, layout):
    """accumulate=0 on a block no query of the rank sees (contiguous: rank 0
    against rank 3's keys) writes the empty state; merging such a block into a
    state changes nothing, bit for bit."""
    S, N = 1024, 4
    w = Workload("empty", 1, 2, 2, S, 128, N, layout, True, BF, seed=102)
    q, k, v = (t.to(cuda_dev) for t in inputs.make_qkv(w))
    qs = [ring.shard(q, r, N, layout) for r in range(N)]
    ks = [ring.shard(k, r, N, layout) for r in range(N)]
    vs = [ring.shard(v, r, N, layout) for r in range(N)]
    out_acc, lse_acc = api.flash_block_step(qs[0], ks[0], vs[0], 0, 0, N, S, layout, True,
                                            accumulate=False)
    before = (out_acc.clone(), lse_acc.clone())
    api.flash_block_step(qs[0], ks[3], vs[3], 0, 3, N, S, layout, True, out_acc=out_acc,
                         lse_acc=lse_acc, accumulate=True)
    torch.cuda.synchronize()
    if layout == CONT:
        assert torch.equal(out_acc, before[0]) and torch.equal(lse_acc, before[1])
        o2, l2 = api.flash_block_step(qs[0], ks[3], vs[3], 0, 3, N, S, layout, True,
                                      accumulate=False)
        torch.cuda.synchronize()
        assert torch.all(o2 == 0) and torch.all(torch.isneginf(l2))
    assert api.cp_get_error() == 0


def test_emulated_ring_s8192_all_rows(cuda_dev, oracle):
    """B=1, H=8, S=8192, D=128, N=8, zigzag, causal: every output row of the
    per-step ring against the oracle and against the fused ring_attn_fwd."""
    w = inputs.S8K
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))
    out, lse = ring.ring_attention_emulated(gq, gk, gv, w.N, w.layout, True)
    fused, flse = api.ring_attn_fwd(gq, gk, gv, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    ref, lref = oracle.attn_fwd(q, k, v, True)
    o = out.float().cpu().numpy()
    check_bf16(o, lse.cpu().numpy(), ref, lref, "per-step ring S=8192 N=8 zigzag")
    check_bf16_pair(o, fused.float().cpu().numpy(), "per-step ring vs fused ring")


@pytest.mark.parametrize("layout", [ZIG, STR])
def test_emulated_ring_long_sampled(cuda_dev, oracle, layout):
    """S=131072, H=8, D=128, N=16 (256 step launches): sampled rows of every
    rank's first and last chunk rows against the oracle."""
    w = inputs.LONG128K.with_(layout=layout)
    q, k, v = inputs.make_qkv(w)
    gq, gk, gv = (t.to(cuda_dev) for t in (q, k, v))
    out, lse = ring.ring_attention_emulated(gq, gk, gv, w.N, w.layout, True)
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0
    pos = api.cp_shard_map(w.S, w.N, layout)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([pos[:, 0], pos[:, -1], rng.integers(0, w.S, 16)]))
    ref, lref = oracle.attn_fwd(q, k, v, True, rows=rows)
    check_bf16(out.float().cpu().numpy()[:, rows], lse.cpu().numpy()[:, :, rows], ref, lref,
               f"per-step ring S=131072 N=16 layout {layout} {len(rows)} sampled rows")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _host_staged_worker(rank, world, port, result, layout, dtype_name):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from context_parallelism_02_gb300 import api as api_, inputs as inputs_, ring as ring_
        dtype = getattr(torch, dtype_name)
        w = inputs_.Workload("host_staged", 1, 4, 2, 256 * world * 2, 128, world, layout, True,
                             dtype, seed=103)
        q, k, v = inputs_.make_qkv(w)
        dev = torch.device("cuda:0")
        qs, ks, vs = (ring_.shard(x, rank, world, layout).to(dev) for x in (q, k, v))
        times = ring_.StepTimes()
        out, lse = ring_.ring_attention(qs, ks, vs, rank=rank, N=world, S=w.S, layout=layout,
                                        causal=True, transport=ring_.HostStagedTransport(),
                                        times=times)
        torch.cuda.synchronize()
        result[rank] = (out.float().cpu().numpy(), lse.cpu().numpy(), api_.cp_get_error(),
                        len(times.compute_ms()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,layout,dtype_name", [(2, ZIG, "bfloat16"), (3, STR, "bfloat16"),
                                                     (2, CONT, "float32")])
def test_two_process_host_staged_ring(cuda_dev, oracle, world, layout, dtype_name):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    result = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_host_staged_worker, args=(r, world, port, result, layout, dtype_name))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    dtype = getattr(torch, dtype_name)
    w = Workload("host_staged", 1, 4, 2, 256 * world * 2, 128, world, layout, True, dtype, seed=103)
    q, k, v = inputs.make_qkv(w)
    ref, lref = oracle.attn_fwd(q, k, v, True)
    for r in range(world):
        o, l, err, nsteps = result[r]
        assert err == 0 and nsteps == world
        pos = ring.shard_positions(w.S, world, layout, r).numpy()
        if dtype == F32:
            assert np.abs(o - ref[:, pos]).max() <= F32_TOL
            assert np.abs(l - lref[:, :, pos]).max() <= F32_TOL
        else:
            check_bf16(o, l, ref[:, pos], lref[:, :, pos], f"host-staged ring of {world} rank {r}")
