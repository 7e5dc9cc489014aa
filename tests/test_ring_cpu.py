"""The real-ring driver (context_parallelism_02_gb300.ring) on CPU: N gloo
ranks on 127.0.0.1, CPU tensors, no GPU.

  * Exchange order: rank r must hold the block of rank (r - k) mod N at ring
    step k, as in the 4-GPU ring table of "Sequence Parallelism in LLMs"
    ("RingAttention and Blockwise Context Parallelism", tests/golden/
    ring_schedule_p4.txt), and the block it holds must be that rank's data.
  * Composition: the driver around the fp64 oracle's one-step function gives
    each rank its rows of single-device attention ("What it does not change").
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    return dist


def _record_worker(rank, world, port, result):
    dist = _init(rank, world, port)
    try:
        from context_parallelism_02_gb300 import ring
        B, C, H, D = 1, 6, 1, 4
        q = torch.zeros(B, C, H, D, dtype=torch.float64)
        # this rank's block carries its rank id (k) and 100 + rank id (v)
        k = torch.full((B, C, H, D), float(rank), dtype=torch.float64)
        v = torch.full((B, C, H, D), 100.0 + rank, dtype=torch.float64)
        seen = []

        def step(q_, k_, v_, out_acc, lse_acc, out_final, *, rank, source, N, S, layout, causal,
                 scale, accumulate):
            seen.append((source, float(k_[0, 0, 0, 0]), float(v_[0, -1, 0, -1]), accumulate,
                         out_final is not None))
            out_acc.zero_()
            lse_acc.zero_()

        ring.ring_attention(q, k, v, rank=rank, N=world, S=C * world, layout=0,
                            transport=ring.P2PTransport(), step=step,
                            state_dtype=torch.float64)
        result[rank] = seen
        # the caller's k, v are only read
        assert torch.all(k == rank) and torch.all(v == 100.0 + rank)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(worker, world, *args):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    result = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, result, *args)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    return dict(result)


def _golden_p4():
    table = {}
    with open(os.path.join(GOLDEN, "ring_schedule_p4.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                step, gpu, blk = (int(x) for x in line.split())
                table[(step, gpu)] = blk
    return table


@pytest.mark.parametrize("world", [2, 3, 4])
def test_exchange_order(world):
    res = _run(_record_worker, world)
    for r in range(world):
        seen = res[r]
        assert len(seen) == world
        for s, (src, kval, vval, acc, final) in enumerate(seen):
            assert src == (r - s) % world
            assert kval == src and vval == 100.0 + src      # the block held is src's data
            assert acc == (s > 0) and final == (s == world - 1)
    if world == 4:
        for (step, gpu), blk in _golden_p4().items():
            assert res[gpu][step][0] == blk


def _oracle_worker(rank, world, port, result, layout, causal, Hq, Hkv):
    dist = _init(rank, world, port)
    try:
        import oracle
        from context_parallelism_02_gb300 import inputs, ring
        S = 48 * world
        w = inputs.Workload("ring_cpu", 1, Hq, Hkv, S, 16, world, layout, causal, torch.float32,
                            seed=90 + world)
        q, k, v = (t.double() for t in inputs.make_qkv(w))

        def step(q_, k_, v_, out_acc, lse_acc, out_final, *, rank, source, N, S, layout, causal,
                 scale, accumulate):
            o, l_ = oracle.block_step(q_, k_, v_, S, N, layout, causal, rank, source,
                                      out_acc if accumulate else None,
                                      lse_acc if accumulate else None, scale)
            out_acc.copy_(torch.from_numpy(o))
            lse_acc.copy_(torch.from_numpy(l_))
            if out_final is not None:
                out_final.copy_(out_acc)

        out, lse = ring.ring_attention(ring.shard(q, rank, world, layout),
                                       ring.shard(k, rank, world, layout),
                                       ring.shard(v, rank, world, layout), rank=rank, N=world,
                                       S=S, layout=layout, causal=causal,
                                       transport=ring.P2PTransport(), step=step,
                                       state_dtype=torch.float64)
        result[rank] = (out.numpy(), lse.numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,layout,causal,Hq,Hkv", [(2, 1, True, 2, 2), (3, 2, True, 4, 2),
                                                        (4, 0, False, 2, 1), (4, 1, True, 2, 2)])
def test_ring_of_oracle_steps_is_attention(oracle, world, layout, causal, Hq, Hkv):
    from context_parallelism_02_gb300 import inputs, ring
    res = _run(_oracle_worker, world, layout, causal, Hq, Hkv)
    S = 48 * world
    w = inputs.Workload("ring_cpu", 1, Hq, Hkv, S, 16, world, layout, causal, torch.float32,
                        seed=90 + world)
    q, k, v = inputs.make_qkv(w)
    ref, lref = oracle.attn_fwd(q, k, v, causal)
    out = ring.unshard([torch.from_numpy(res[r][0]) for r in range(world)], world, layout)
    lse = ring.unshard([torch.from_numpy(res[r][1]) for r in range(world)], world, layout, dim=2)
    np.testing.assert_allclose(out.numpy(), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), lref, rtol=0, atol=1e-12)
