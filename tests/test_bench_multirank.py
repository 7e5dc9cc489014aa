"""The N>1 path of bench.py on CPU: two gloo ranks (no GPU).

bench.py runs one replica of the workload per GPU and reports the work of
all ranks over the slowest rank's time; these tests check that aggregation
with world_size 2 over gloo on 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, result):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(times[rank], world, "cpu")
        result[rank] = (ms_max, bench.job_value(1e12, world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(10.0, 12.5), (30.0, 3.0)])
def test_two_ranks_max_time_and_job_value(times):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    result = mgr.dict()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, result)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    slow = max(times)
    for r in range(world):
        ms_max, value = result[r]
        assert ms_max == slow
        assert abs(value - world * 1e12 / (slow * 1e-3) / 1e12) < 1e-9


def test_single_rank_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_value(2e12, 1, 1000.0) == 2.0


def _fake_extras():
    per = {"n_split_per_rank": [1] * 16, "ms_per_rank_split": [1.0] * 16,
           "split_max_rank_ms_vs_unsplit": [1.6, 1.7], "masked_in_pairs_per_rank": [4294508544] * 16,
           "work_max_over_mean": 1.0001144400448605, "ms_per_rank": [1.55] * 16,
           "time_max_over_mean": 1.0311458828609423, "ms_all_ranks": 23.352884928385418,
           "TFLOP/s_all_ranks": 1506.6507042785574, "executed_tiles_128x256": 2162688}
    return {
        "configs_fwd": {n: {"dtype": "bfloat16", "ms": 0.1331, "TFLOP/s": 1031.2, "masked_in_flops": 1}
                        for n in ("tiny_s512_d64_n4", "s8192_h8_d128_n8_zigzag_causal",
                                  "gqa_s32768_hq32_hkv8_d128_n8_zigzag_causal")},
        "lse_merge": {"rows": 1, "D": 128, "bytes": 1, "ms": 0.25, "GB/s": 6419.123, "frac_hbm": 0.9461},
        "lse_merge_n4": {"rows": 1, "D": 128, "n": 4, "bytes": 1, "ms": 0.43, "GB/s": 6233.1,
                         "frac_hbm": 0.92},
        "ulysses_q_gqa32k": {"seq_to_head": {"ms": 1.0, "GB/s": 6337.0, "frac_hbm": 0.934},
                             "head_to_seq": {"ms": 1.0, "GB/s": 6362.0, "frac_hbm": 0.94},
                             "bit_exact_roundtrip": True, "bytes": 1},
        "usp_gqa32k": {"grid": "n_ulysses x n_ring", **{k: {"ms": 5.8, "TFLOP/s": 1500.0}
                                                         for k in ("1x8", "2x4", "4x2", "8x1")}},
        "per_rank_long128k": {lay: dict(per) for lay in ("contiguous", "zigzag", "striped")},
        "split_kv_one_head_long128k": {"max_rank_ms_unsplit": 0.87, "max_rank_ms_split": 0.29},
        "ring_attn_bwd_bwd32k": {"ms": 24.29, "TFLOP/s": 905.13, "frac_bf16_burst": 0.4823,
                                 "executed_TFLOP/s": 1267.18},
    }


def test_compact_line_fits_the_kept_output():
    """The default bench line (extras as scalar summaries, HBM kernels last)
    stays well under the ~3 KB of stdout a caller's log tail keeps."""
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"hbm_gbs": 6785.2, "bf16_tflops": 1940.6, "bf16_tflops_sustained": 1736.5}
    full = _fake_extras()
    line = {"metric": bench.METRIC, "value": 1605.7175086641482, "unit": "TFLOP/s",
            "extras": bench.rounded(bench.compact_extras(full)),
            "hbm_kernels": bench.rounded(bench.hbm_summary(full, peaks))}
    text = json.dumps(line)
    assert len(text) < 2000, len(text)
    assert text.index('"hbm_kernels"') > text.index('"extras"')
    assert line["hbm_kernels"]["lse_merge"]["frac_hbm"] == 0.9461
    assert line["extras"]["long128k_zigzag_rank_time_max_over_mean"] == 1.031


def _ring_worker(rank, world, port, result):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from context_parallelism_02_gb300 import inputs, ring
        w = inputs.Workload("bench_ring_cpu", 1, 2, 2, 64 * world, 16, world, 1, True,
                            torch.float32, seed=7)
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

        sh = lambda x, r: ring.shard(x, r, world, w.layout)
        blocks = [(sh(k, r), sh(v, r)) for r in range(world)]
        m = bench.ring_measure(sh(q, rank), sh(k, rank), sh(v, rank), rank=rank, world=world,
                               S=w.S, layout=w.layout, causal=True, steps=2, warmup=1,
                               transport=ring.P2PTransport(), blocks=blocks, step=step,
                               state_dtype=torch.float64)
        result[rank] = m
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_real_ring_measurement_on_gloo():
    """bench.ring_measure's N > 1 logic (whole ring, compute alone, transfers
    alone, max over ranks) with gloo ranks on CPU and the oracle's step."""
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    result = mgr.dict()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_ring_worker, args=(r, world, port, result)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    for r in range(world):
        m = result[r]
        for key in ("ms_ring", "ms_compute", "ms_transfers"):
            assert m[key] > 0
        assert m["ms_ring"] == result[0]["ms_ring"]          # max over ranks
        assert m["hop_bytes"] == 2 * 1 * 64 * 2 * 16 * 8     # k and v shards (C = 64), fp64
