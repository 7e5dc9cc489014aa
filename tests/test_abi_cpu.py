"""CPU-side checks of the C ABI: the library loads, exports every entry point
that include/cp.h declares, and its host-only calls (shard map, schedule walk,
argument validation) behave as documented.  No compute call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

from context_parallelism_02_gb300 import _lib, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CONT, ZIG, STR = 0, 1, 2


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "cp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(cplib):
    names = _declared_symbols()
    assert {"ring_attn_fwd", "lse_merge", "ulysses_seq_to_head", "ulysses_head_to_seq",
            "cp_shard_map", "cp_get_error"} <= set(names)
    for n in names:
        assert hasattr(cplib, n), n
    # the Python binding knows the same set
    assert set(names) == set(_lib.SIGNATURES)


def test_debug_bounds_variant_builds_and_exports(cplib):
    """The -DCP_DEBUG_BOUNDS build compiles and exports the same entry points."""
    from context_parallelism_02_gb300 import build
    path = build.build(debug_bounds=True)
    assert path != _lib.lib_path("default")
    lib = _lib.load(variant="debug_bounds")
    for n in _declared_symbols():
        assert hasattr(lib, n), n
    assert lib.cp_strerror(-7) == _lib.load().cp_strerror(-7)


def test_library_is_in_tree(cplib):
    assert os.path.realpath(_lib.lib_path()).startswith(os.path.realpath(ROOT))


@pytest.mark.parametrize("S,N,layout", [(8192, 8, CONT), (64, 4, ZIG), (1600, 4, ZIG),
                                        (1000, 4, CONT), (48, 1, ZIG), (8192, 8, STR),
                                        (1000, 4, STR), (99, 3, STR)])
def test_shard_map_matches_oracle(cplib, oracle, S, N, layout):
    np.testing.assert_array_equal(api.cp_shard_map(S, N, layout), oracle.shard_pos(S, N, layout))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S,N,layout", [(512, 4, CONT), (512, 4, ZIG), (8192, 8, ZIG),
                                        (8192, 8, CONT), (1600, 4, ZIG), (1000, 4, CONT),
                                        (384, 1, ZIG), (96, 3, CONT), (512, 4, STR),
                                        (8192, 8, STR), (1000, 4, STR), (96, 3, STR),
                                        (4096, 16, STR)])
def test_schedule_pairs_match_oracle(cplib, oracle, S, N, layout, causal):
    """The kernel's tile schedule (tile skipping included) covers exactly the
    masked-in pairs of every (rank, step): bit-exact integer counts."""
    pairs, tiles = api.cp_schedule_pairs(S, N, layout, causal)
    np.testing.assert_array_equal(pairs, oracle.pair_counts(S, N, layout, causal))
    assert np.all(tiles >= 0)


def test_schedule_long_sequence_closed_forms(cplib):
    """S=131072, N=16: per-rank masked-in work, contiguous vs zigzag."""
    S, N = 131072, 16
    C, c = S // N, S // (2 * N)
    pc, tc = api.cp_schedule_pairs(S, N, CONT, True)
    pz, tz = api.cp_schedule_pairs(S, N, ZIG, True)
    for r in range(N):
        assert pc[r].sum() == r * C * C + C * (C + 1) // 2
        assert pz[r].sum() == 2 * N * c * c + c
    assert pc.sum() == pz.sum() == S * (S + 1) // 2
    assert pc.sum(1)[0] == 33_558_528 and pc.sum(1)[-1] == 1_040_191_488
    # executed (128-query x 256-key) tile pairs: equal per rank under zigzag; only
    # diagonal tiles are partial, so executed work is within 1 % of masked-in work
    per_rank = tz.sum(1)
    assert per_rank.max() - per_rank.min() <= 2
    full_pairs = S * (S + 1) // 2
    assert tz.sum() * 128 * 256 <= full_pairs * 1.01
    # striped: every step of every rank has C(C+1)/2 - C [src > r] pairs, so
    # every step (not only step 0) crosses the causal diagonal: each query row
    # of each step wastes fewer than 256 masked columns (3 % of the work here)
    ps, ts = api.cp_schedule_pairs(S, N, STR, True)
    for r in range(N):
        for k in range(N):
            src = (r - k) % N
            assert ps[r, k] == C * (C + 1) // 2 - (C if src > r else 0)
    assert ps.sum() == full_pairs
    assert np.all(ts == ts[0, 0])
    assert ts.sum() * 128 * 256 <= full_pairs + N * N * C * 256


def _call_fwd(**kw):
    a = dict(q=None, k=None, v=None, out=None, lse=None, B=1, Hq=2, Hkv=2, S=512, D=64, N=4,
             causal=1, layout=ZIG, dtype=1, scale=-1.0, stream=None)
    a.update(kw)
    return _lib.load().ring_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["Hq"],
                                     a["Hkv"], a["S"], a["D"], a["N"], a["causal"], a["layout"],
                                     a["dtype"], a["scale"], a["stream"])


def test_argument_validation_without_gpu(cplib):
    """Errors are returned before any CUDA call, so these run on a CPU-only box."""
    assert _call_fwd(Hq=3, Hkv=2) == _lib.CP_EINVAL           # Hq % Hkv
    assert _call_fwd(S=500, N=4) == _lib.CP_EINVAL            # zigzag needs S % 2N
    assert _call_fwd(S=510, N=4, layout=CONT) == _lib.CP_EINVAL
    assert _call_fwd(N=0) == _lib.CP_EINVAL
    assert _call_fwd(layout=3) == _lib.CP_EINVAL
    assert _call_fwd(layout=-1) == _lib.CP_EINVAL
    assert _call_fwd(S=510, N=4, layout=STR) == _lib.CP_EINVAL     # striped needs S % N
    assert _call_fwd(S=516, N=4, layout=STR) == _lib.CP_EINVAL     # null pointers (shape ok)
    assert _call_fwd(D=96) == _lib.CP_EUNSUPPORTED
    assert _call_fwd(dtype=7) == _lib.CP_EUNSUPPORTED
    assert _call_fwd() == _lib.CP_EINVAL                      # null pointers
    assert _call_fwd(B=0) == _lib.CP_OK                       # empty batch: no-op
    assert _call_fwd(S=0) == _lib.CP_OK                       # empty sequence: no-op
    L = _lib.load()
    # Ulysses head ceiling (P <= H): 6 heads cannot be split over 4 ranks
    assert L.ulysses_seq_to_head(None, None, 1, 64, 6, 8, 4, 0, 2, None) == _lib.CP_EHEADS
    assert L.ulysses_head_to_seq(None, None, 1, 64, 8, 8, 4, 1, 2, None) == _lib.CP_EINVAL
    assert L.ulysses_seq_to_head(None, None, 1, 64, 8, 8, 4, 0, 3, None) == _lib.CP_EINVAL
    assert L.lse_merge(None, None, None, None, None, None, 0, 128, None) == _lib.CP_OK
    assert L.lse_merge(None, None, None, None, None, None, 4, 6, None) == _lib.CP_EINVAL
    # USP: the Ulysses group size must divide the kv heads (P <= H_KV)
    assert L.usp_attn_fwd(None, None, None, None, None, 1, 8, 2, 512, 64, 4, 2, 1, 1, 1, -1.0,
                          None, 0, None) == _lib.CP_EHEADS
    assert L.usp_attn_fwd(None, None, None, None, None, 1, 8, 4, 512, 64, 4, 2, 1, 1, 1, -1.0,
                          None, 0, None) == _lib.CP_EINVAL          # null pointers / workspace
    assert L.usp_attn_fwd(None, None, None, None, None, 1, 8, 4, 500, 64, 4, 2, 1, 0, 1, -1.0,
                          None, 0, None) == _lib.CP_EINVAL          # S % n_ulysses
    assert L.usp_attn_fwd(None, None, None, None, None, 0, 8, 4, 512, 64, 4, 2, 1, 1, 1, -1.0,
                          None, 0, None) == _lib.CP_OK              # empty batch
    assert L.usp_attn_fwd_workspace(8, 4, 512, 64, 1) == (2 * 8 + 2 * 4) * 512 * 64 * 2
    assert L.lse_merge_n(None, None, 3, 0, 128, None, None, None) == _lib.CP_OK
    assert L.lse_merge_n(None, None, 0, 4, 128, None, None, None) == _lib.CP_EINVAL
    assert L.lse_merge_n(None, None, 3, 4, 6, None, None, None) == _lib.CP_EINVAL
    assert L.lse_merge_n(None, None, 3, 4, 128, None, None, None) == _lib.CP_EINVAL
    # split-KV forward (bf16 only); fake non-null addresses are never touched
    # because every check comes before the first CUDA call
    fake = 1 << 20
    split = lambda **kw: L.ring_attn_fwd_split(
        *(kw.get(n, fake) for n in ("q", "k", "v", "out", "lse")), kw.get("B", 1), 8, 8,
        kw.get("S", 8192), 128, kw.get("N", 8), 1, ZIG, kw.get("dtype", 1), -1.0, kw.get("lo", 0),
        kw.get("hi", 8), kw.get("n_split", 4), kw.get("ws", fake), kw.get("ws_bytes", 1 << 40), None)
    assert split(n_split=0) == _lib.CP_EINVAL
    assert split(n_split=65) == _lib.CP_EINVAL
    assert split(dtype=0) == _lib.CP_EUNSUPPORTED                     # CP_F32
    assert split(q=None) == _lib.CP_EINVAL
    assert split(ws=None) == _lib.CP_EINVAL
    assert split(ws=fake + 8) == _lib.CP_EINVAL                       # misaligned workspace
    need = L.ring_attn_fwd_split_workspace(1, 8, 8192, 128, 4)
    assert split(ws_bytes=need - 1) == _lib.CP_EINVAL
    assert split(lo=3, hi=3) == _lib.CP_EINVAL
    assert split(S=8200) == _lib.CP_EINVAL                            # zigzag: S % 2N
    assert split(B=0) == _lib.CP_OK                                   # empty batch
    # flash_block_step: rank, source and accumulate are checked first
    step = lambda **kw: L.flash_block_step(
        *(kw.get(n, fake) for n in ("q", "k", "v", "oacc", "lacc")), kw.get("final", None),
        kw.get("B", 1), 8, 8, kw.get("S", 8192), 128, kw.get("N", 8), kw.get("rank", 0),
        kw.get("src", 7), 1, kw.get("layout", ZIG), kw.get("dtype", 1), -1.0, kw.get("acc", 1), None)
    assert step(rank=8) == _lib.CP_EINVAL
    assert step(rank=-1) == _lib.CP_EINVAL
    assert step(src=8) == _lib.CP_EINVAL
    assert step(acc=2) == _lib.CP_EINVAL
    assert step(oacc=None) == _lib.CP_EINVAL
    assert step(lacc=None) == _lib.CP_EINVAL
    assert step(final=fake + 8) == _lib.CP_EINVAL                      # misaligned out_final
    assert step(S=8200) == _lib.CP_EINVAL                             # zigzag: S % 2N
    assert step(dtype=5) == _lib.CP_EUNSUPPORTED
    assert step(B=0) == _lib.CP_OK                                    # empty batch
    for code in (-6, -7):
        assert _lib.strerror(code) != _lib.strerror(-99)
    buf = np.zeros(8, np.int32)
    assert L.cp_shard_map(12, 4, ZIG, buf.ctypes.data_as(ctypes.c_void_p)) == _lib.CP_EINVAL
    assert L.cp_shard_map(1 << 40, 4, CONT, buf.ctypes.data_as(ctypes.c_void_p)) == _lib.CP_EINVAL
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(_lib.strerror(code), str) and _lib.strerror(code)


def test_split_workspace_size(cplib):
    L = _lib.load()
    for B, Hq, S, D, n in ((1, 8, 131072, 128, 4), (2, 3, 70, 64, 7), (1, 1, 1, 64, 1)):
        raw = n * B * S * Hq * (D + 1) * 4
        assert L.ring_attn_fwd_split_workspace(B, Hq, S, D, n) == (raw + 255) // 256 * 256
    assert L.ring_attn_fwd_split_workspace(1, 8, 4096, 96, 2) == 0
    assert L.ring_attn_fwd_split_workspace(1, 8, 4096, 128, 0) == 0
    assert L.ring_attn_fwd_split_workspace(1, 8, 4096, 128, 65) == 0
    assert L.ring_attn_fwd_split_workspace(1, 8, 1 << 31, 128, 4) == 0


def test_split_count_choice(cplib):
    """The split count from the dispatch simulation: 1 when the launch has many
    waves of units, more than 1 when a few long query tiles would hold the
    last wave, never above 32, and errors for what the split call rejects."""
    L = _lib.load()
    count = lambda B, Hq, S, N, layout, lo, hi, causal=1, D=128, sms=152: L.cp_fwd_split_count(
        B, Hq, S, D, N, causal, layout, lo, hi, sms)
    assert count(1, 8, 131072, 16, ZIG, 0, 16) == 1          # 8192 units: 54 waves
    assert count(2, 16, 32768, 8, ZIG, 0, 8) == 1
    assert count(1, 32, 32768, 8, ZIG, 0, 8) == 1
    # one rank of the 128k ring (512 units): the counts that timed fastest
    assert count(1, 8, 131072, 16, ZIG, 15, 16) == 2
    assert count(1, 8, 131072, 16, CONT, 15, 16) == 2
    assert count(1, 8, 131072, 16, CONT, 0, 1) == 1
    # one head of it: 64 units of up to 512 tiles for 152 SMs
    assert count(1, 1, 131072, 16, ZIG, 0, 1) >= 4
    # 128 equal units (non-causal, 256 tiles each) on 300 SMs: 2 splits fill
    # one wave exactly, 3 would need a second wave (the choice is not monotonic
    # in the SM count)
    assert count(1, 1, 65536, 4, ZIG, 0, 1, causal=0, sms=300) == 2
    assert count(1, 1, 65536, 4, ZIG, 0, 1, causal=0, sms=152) == 1
    for args in ((1, 1, 4096, 2, CONT, 0, 1), (3, 5, 1000, 4, STR, 1, 3), (1, 2, 640, 5, ZIG, 0, 5)):
        assert 1 <= count(*args) <= 32
    assert count(1, 8, 8192, 8, ZIG, 0, 8, sms=0) == _lib.CP_EINVAL
    assert count(1, 8, 8200, 8, ZIG, 0, 8) == _lib.CP_EINVAL
    assert count(1, 8, 8192, 8, ZIG, 4, 4) == _lib.CP_EINVAL
    assert count(1, 8, 8192, 8, ZIG, 0, 8, D=96) == _lib.CP_EUNSUPPORTED
