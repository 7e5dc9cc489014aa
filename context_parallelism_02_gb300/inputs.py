"""Seeded synthetic inputs for ring / context-parallel attention.

This module only draws numbers: it holds none of the attention arithmetic,
so that both the CUDA path and the fp64 oracle can take their inputs from it
without sharing any of the method.

Every tensor is drawn with ``torch.Generator(seed).normal_`` in fp32 on the
CPU, in the order q, k, v (then dO for the backward workload), and is then
cast to the workload's dtype.  The oracle up-converts the *cast* values to
fp64, so both sides see bit-identical inputs.

Layout is BSHD in global token order: q ``[B, S, Hq, D]``, k and v
``[B, S, Hkv, D]``.

The workloads follow the shapes the pages discuss: the worked imbalance
example of "Context Parallelism" (aiwiki, "The causal imbalance": rank 0
holds queries 0-1023 of an 8-rank split, i.e. S=8192, N=8), the GQA head
ceiling of "Sequence Parallelism in LLMs" (llms.blog, "Communication Cost and
Constraints": 8 KV heads), and the 128k-token context of the same page's
"Activation Memory Wall" section.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

CONTIGUOUS = 0
ZIGZAG = 1
STRIPED = 2
LAYOUT_NAMES = {CONTIGUOUS: "contiguous", ZIGZAG: "zigzag", STRIPED: "striped"}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    N: int
    layout: int
    causal: bool
    dtype: torch.dtype
    seed: int
    q_scale: float = 1.0          # multiplies q after the draw (large-logit variant)
    with_grad: bool = False       # also draw dO (backward workload)
    extra: dict = field(default_factory=dict, compare=False)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)


# The five workloads: tiny exact check, S=8k, GQA S=32k, long S=128k, fwd+bwd.
TINY = Workload("tiny_s512_d64_n4", B=1, Hq=2, Hkv=2, S=512, D=64, N=4,
                layout=ZIGZAG, causal=True, dtype=torch.float32, seed=0)
S8K = Workload("s8192_h8_d128_n8_zigzag_causal", B=1, Hq=8, Hkv=8, S=8192,
               D=128, N=8, layout=ZIGZAG, causal=True, dtype=torch.bfloat16, seed=1)
GQA32K = Workload("gqa_s32768_hq32_hkv8_d128_n8_zigzag_causal", B=1, Hq=32,
                  Hkv=8, S=32768, D=128, N=8, layout=ZIGZAG, causal=True,
                  dtype=torch.bfloat16, seed=2)
LONG128K = Workload("s131072_h8_d128_n16_zigzag_causal", B=1, Hq=8, Hkv=8,
                    S=131072, D=128, N=16, layout=ZIGZAG, causal=True,
                    dtype=torch.bfloat16, seed=3)
BWD32K = Workload("bwd_b2_s32768_h16_d128_n8_zigzag_causal", B=2, Hq=16,
                  Hkv=16, S=32768, D=128, N=8, layout=ZIGZAG, causal=True,
                  dtype=torch.bfloat16, seed=4, with_grad=True)

# lse_merge workload: rows = 1 x 8 x 131072, D = 128, fp32 partials, seed 5.
MERGE_ROWS = 1 * 8 * 131072
MERGE_D = 128
MERGE_SEED = 5


def draw(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.empty(shape, dtype=torch.float32).normal_(generator=gen)


def make_qkv(w: Workload):
    """Return (q, k, v[, dO]) on the CPU in ``w.dtype``, BSHD, global order."""
    g = torch.Generator().manual_seed(w.seed)
    q = draw((w.B, w.S, w.Hq, w.D), g)
    k = draw((w.B, w.S, w.Hkv, w.D), g)
    v = draw((w.B, w.S, w.Hkv, w.D), g)
    if w.q_scale != 1.0:
        q = q * w.q_scale
    out = [q.to(w.dtype), k.to(w.dtype), v.to(w.dtype)]
    if w.with_grad:
        out.append(draw((w.B, w.S, w.Hq, w.D), g).to(w.dtype))
    return tuple(out)


def make_merge_inputs(rows: int = MERGE_ROWS, D: int = MERGE_D, seed: int = MERGE_SEED,
                      neg_inf_every: int = 0):
    """Two fp32 partial results (out_a, lse_a, out_b, lse_b) for lse_merge.

    lse values are drawn N(0, 4) so that the two partials carry very
    different weights.  With ``neg_inf_every=k`` every k-th row of lse_a and
    every (k+1)-th row of lse_b is -inf (an empty partial).
    """
    g = torch.Generator().manual_seed(seed)
    out_a = draw((rows, D), g)
    lse_a = draw((rows,), g) * 2.0
    out_b = draw((rows, D), g)
    lse_b = draw((rows,), g) * 2.0
    if neg_inf_every:
        lse_a[::neg_inf_every] = float("-inf")
        lse_b[::neg_inf_every + 1] = float("-inf")
    return out_a, lse_a, out_b, lse_b


def make_merge_n_inputs(n: int, rows: int = MERGE_ROWS, D: int = MERGE_D, seed: int = MERGE_SEED,
                        neg_inf_every: int = 0):
    """n fp32 partial results (out_parts [n, rows, D], lse_parts [n, rows]) for
    lse_merge_n, drawn like make_merge_inputs (lse ~ N(0, 4)).  With
    ``neg_inf_every=k`` partial i has lse = -inf on every (k+i)-th row."""
    g = torch.Generator().manual_seed(seed)
    outs = draw((n, rows, D), g)
    lses = draw((n, rows), g) * 2.0
    if neg_inf_every:
        for i in range(n):
            lses[i, ::neg_inf_every + i] = float("-inf")
    return outs, lses


def make_layout_tensor(N: int, B: int, S: int, H: int, D: int, dtype: torch.dtype, seed: int):
    """A rank-major stack of N sequence shards, ``[N, B, S/N, H, D]``.

    Integer-valued draws (bit-exact in any dtype) so that a permutation can
    be compared byte for byte.
    """
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(-1000, 1000, (N, B, S // N, H, D), generator=g, dtype=torch.int32)
    return x.to(dtype)
