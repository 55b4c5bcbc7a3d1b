"""The forward entry point that allocates nothing (swa_attn_fwd_noalloc).

Some callers cannot allocate device memory where they run the attention:
plug-ins whose host framework owns every allocation, services that must not
grow their memory after start-up, latency-critical paths that cannot afford
cudaMalloc's implicit device synchronisation. For them the library keeps the
forward's scratch in one fixed device array instead of a caller-provided
workspace. This test calls that entry point through the C ABI of both
libraries (bf16 tensor-core and fp32 debug build) and checks its outputs
against the float64 oracle and against the regular swa_attn_fwd (with a
workspace), within the parity tolerance of the other GPU tests, on two calls
in a row with different inputs (the array keeps the previous call's
contents, which must not leak into the next result).

The file is named so that pytest collects it last."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300 import build as swa_build
from sliding_window_gqa_qk_gb300.inputs import Problem, as_f64, make_inputs
from gpu_helpers import DTYPE, TOL, check

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024   # SWA_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def built():
    swa_build.build()


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_noalloc_forward_matches_oracle_and_workspace_forward_on_two_calls(kind):
    lib = swa.load(kind)
    dev = torch.device("cuda:0")
    p = Problem(B=1, T=300, Hq=4, Hkv=2, d=128, window=150, gain_std=0.1, ve=True, vocab=257)
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps,
                          p.ve_scale, p.vocab)
    assert 0 < swa.swa_attn_workspace_size(prm, 0, kind) <= SCRATCH_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    tol = TOL[kind]
    for layer in (1, 2):   # two calls in a row, different inputs
        x = make_inputs(p, layer=layer, dtype=DTYPE[kind])
        g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
        o_ws, lse_ws, _ = swa.attention_forward(
            g["q"], g["k"], g["v"], g["gq"], g["gk"], window=p.window, eps=p.eps, ve=g["ve"],
            tok=g["tok"], ve_scale=p.ve_scale)
        o = torch.full_like(g["q"], float("nan"))
        lse = torch.full((p.B, p.Hq, p.T), float("nan"), device=dev)
        ptr = lambda t: None if t is None else t.data_ptr()
        st = lib.swa_attn_fwd_noalloc(ctypes.byref(prm), ptr(g["q"]), ptr(g["k"]), ptr(g["v"]),
                                      ptr(g["gq"]), ptr(g["gk"]), ptr(g["ve"]), ptr(g["tok"]),
                                      None, ptr(o), ptr(lse), stream)
        torch.cuda.synchronize()
        assert st == swa.SWA_OK, swa.swa_strerror(st)
        f = {k: as_f64(t) for k, t in x.items()}
        o_ref, lse_ref = oracle.attention_forward(
            f["q"], f["k"], f["v"], f["gq"], f["gk"], window=p.window, eps=p.eps, ve=f["ve"],
            tok=x["tok"].numpy(), ve_scale=p.ve_scale)
        check("o", o.cpu(), o_ref, tol)
        check("lse", lse.cpu(), lse_ref, tol)
        check("o", o.cpu(), as_f64(o_ws), tol)
        check("lse", lse.cpu(), as_f64(lse_ws), tol)


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_noalloc_forward_rejects_problems_beyond_its_scratch(kind):
    lib = swa.load(kind)
    big = swa.make_params(16, 2048, 6, 3, 128, 1024, True, 0.0, 1e-6, 0.5, 0)
    assert swa.swa_attn_workspace_size(big, 0, kind) > SCRATCH_BYTES
    a = 1 << 20   # never dereferenced: the size check comes before any launch
    st = lib.swa_attn_fwd_noalloc(ctypes.byref(big), a, a, a, None, None, None, None, None, a,
                                  a, None)
    assert st == swa.SWA_ERR_WORKSPACE
