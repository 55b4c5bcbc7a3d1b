"""The comparison the GPU parity tests use (gpu_helpers.compare), checked on
the CPU with mistakes planted in the oracle's own results: a single wrong row
or element, which the whole-tensor relative error lets through, must fail
the per-row / per-element bound, while rounding-sized noise passes."""

import numpy as np

import oracle
import gpu_helpers
from gpu_helpers import TOL, compare, errors

import pytest


@pytest.fixture(autouse=True)
def _not_reported():
    """The planted comparisons stay out of the session's parity report."""
    n = len(gpu_helpers.REPORT)
    yield
    del gpu_helpers.REPORT[n:]


def _problem(seed=3, B=1, T=1024, Hq=4, Hkv=2, d=32, window=300):
    r = np.random.default_rng(seed)
    x = {"q": r.standard_normal((B, T, Hq, d)), "k": r.standard_normal((B, T, Hkv, d)),
         "v": r.standard_normal((B, T, Hkv, d)), "dO": r.standard_normal((B, T, Hq, d)),
         "gq": 1 + 0.1 * r.standard_normal(d), "gk": 1 + 0.1 * r.standard_normal(d)}
    kw = dict(window=window, causal=True, eps=1e-6)
    o, lse = oracle.attention_forward(x["q"], x["k"], x["v"], x["gq"], x["gk"], **kw)
    ref = oracle.attention_backward(x["q"], x["k"], x["v"], x["gq"], x["gk"], x["dO"], scales=True, **kw)
    ref["o"], ref["lse"] = o, lse
    return ref


@pytest.fixture(scope="module")
def ref():
    return _problem()


def _noisy(ref, rel=2e-3, seed=5):
    """The oracle's tensors with rounding-sized noise (rel times the typical
    element, a few times bf16's unit roundoff)."""
    r = np.random.default_rng(seed)
    out = {}
    for k in ("o", "lse", "dq", "dk", "dv", "dgq", "dgk"):
        t = np.asarray(ref[k])
        out[k] = t + rel * np.sqrt(np.mean(t * t)) * r.standard_normal(t.shape)
    return out


def test_rounding_sized_noise_passes(ref):
    compare(_noisy(ref), ref, TOL["bf16"])


def test_one_wrong_row_fails_the_row_bound_but_not_the_whole_tensor_bound(ref):
    got = _noisy(ref)
    # one (b, t, h) row of dq 50 % too large: 1 of 4096 rows
    got["dq"][0, 700, 2] *= 1.5
    frob, row, _ = errors(got["dq"], ref["dq"], row_scale=ref["dq_scale"])
    assert frob <= TOL["bf16"] < row
    with pytest.raises(AssertionError):
        compare(got, ref, TOL["bf16"])


def test_one_wrong_lse_element_fails_the_element_bound(ref):
    got = _noisy(ref)
    got["lse"][0, 1, 500] += np.log(2.0)   # half of a row's probability mass lost
    frob, row, _ = errors(got["lse"], ref["lse"], elementwise=True)
    assert frob <= TOL["bf16"] < row
    with pytest.raises(AssertionError):
        compare(got, ref, TOL["bf16"])


def test_one_wrong_key_row_of_dk_fails(ref):
    got = _noisy(ref)
    got["dk"][0, 129, 1] *= -1.0   # a sign error in one key row
    with pytest.raises(AssertionError):
        compare(got, ref, TOL["bf16"])
