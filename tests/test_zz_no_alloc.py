"""The forward entry point that allocates nothing (swa_attn_fwd_noalloc).

Some callers cannot allocate device memory where they run the attention:
plug-ins whose host framework owns every allocation, services that must not
grow their memory after start-up, latency-critical paths that cannot afford
cudaMalloc's implicit device synchronisation. For them the library keeps the
forward's scratch in one fixed device array instead of a caller-provided
workspace. This test calls
that entry point through the C ABI and checks that its outputs equal those of
the regular swa_attn_fwd (with a workspace) within the parity tolerance, on
two calls in a row with different inputs (the array keeps the previous
call's contents, which must not leak into the next result).

The file is named so that pytest collects it last."""

import ctypes

import numpy as np
import pytest
import torch

import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300 import build as swa_build
from sliding_window_gqa_qk_gb300.inputs import Problem, as_f64, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2   # the bf16 parity tolerance of the other GPU tests


@pytest.fixture(scope="module", autouse=True)
def built():
    swa_build.build()


def rel(a, b):
    a, b = as_f64(a), as_f64(b)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    lib = swa.load("bf16")
    dev = torch.device("cuda:0")
    p = Problem(B=1, T=300, Hq=4, Hkv=2, d=128, window=150, gain_std=0.1, ve=True, vocab=257)
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps,
                          p.ve_scale, p.vocab)
    assert swa.swa_attn_workspace_size(prm, 0) <= 32 * 1024 * 1024
    stream = torch.cuda.current_stream().cuda_stream
    for layer in (1, 2):   # two calls in a row, different inputs
        x = make_inputs(p, layer=layer)
        g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
        o_ref, lse_ref, _ = swa.attention_forward(
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
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert rel(o, o_ref) <= TOL and rel(lse, lse_ref) <= TOL


def test_noalloc_forward_rejects_problems_beyond_its_scratch():
    lib = swa.load("bf16")
    big = swa.make_params(16, 2048, 6, 3, 128, 1024, True, 0.0, 1e-6, 0.5, 0)
    assert swa.swa_attn_workspace_size(big, 0) > 32 * 1024 * 1024
    a = 1 << 20   # never dereferenced: the size check comes before any launch
    st = lib.swa_attn_fwd_noalloc(ctypes.byref(big), a, a, a, None, None, None, None, None, a,
                                  a, None)
    assert st == swa.SWA_ERR_WORKSPACE
