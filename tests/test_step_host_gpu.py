"""The training step with host buffers (swa_attn_step_host): inputs copied in,
forward and backward, outputs copied out, all on one stream through the C
ABI. Checked against the float64 oracle (both libraries), on two calls in a
row with different inputs through the same device buffer, and with pageable
as well as pinned host memory."""

import pytest
import torch

import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300.inputs import Problem
from gpu_helpers import TOL, compare, inputs, run_oracle

pytestmark = pytest.mark.gpu

CASE = Problem(B=2, T=300, Hq=4, Hkv=2, d=128, window=150, gain_std=0.1, ve=True, vocab=257)


def _step(p, x, buf, kind, pinned, stream):
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps, p.ve_scale,
                          p.vocab if p.ve else 0)
    h = {k: (t.contiguous().pin_memory() if pinned else t.contiguous()) if t is not None else None
         for k, t in x.items()}
    alloc = (lambda *s, **kw: torch.empty(*s, **kw).pin_memory()) if pinned else torch.empty
    out = {"o": alloc(h["q"].shape, dtype=h["q"].dtype),
           "lse": alloc((p.B, p.Hq, p.T), dtype=torch.float32),
           "dq": alloc(h["q"].shape, dtype=h["q"].dtype),
           "dk": alloc(h["k"].shape, dtype=h["k"].dtype),
           "dv": alloc(h["v"].shape, dtype=h["v"].dtype),
           "dgq": alloc((p.d,), dtype=torch.float32),
           "dgk": alloc((p.d,), dtype=torch.float32),
           "dve": alloc(h["ve"].shape, dtype=torch.float32) if p.ve else None}
    for t in out.values():
        if t is not None:
            t.fill_(float("nan"))
    st = swa.swa_attn_step_host(prm, None, h["q"], h["k"], h["v"], h["gq"], h["gk"], h["ve"], h["tok"],
                                h["gate"], h["dO"], out["o"], out["lse"], out["dq"], out["dk"],
                                out["dv"], out["dgq"], out["dgk"], out["dve"], buf, stream=stream,
                                kind=kind)
    assert st == swa.SWA_OK, swa.swa_strerror(st)
    torch.cuda.synchronize()
    assert swa.swa_attn_check_status(buf, None, kind) == swa.SWA_OK
    return out


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_step_with_host_buffers_matches_oracle_on_two_calls(kind):
    p = CASE
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps, p.ve_scale,
                          p.vocab)
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream()
    buf = swa.new_step_host_buffer(prm, dev, kind, stream=stream.cuda_stream)
    for layer, pinned in ((1, True), (3, False)):   # different inputs, same buffer
        x = inputs(p, kind, layer=layer, with_gate=True)
        got = _step(p, x, buf, kind, pinned, stream.cuda_stream)
        ref = run_oracle(p, x)
        compare(got, ref, TOL[kind], keys=("o", "lse", "dq", "dk", "dv", "dgq", "dgk", "dve"))
