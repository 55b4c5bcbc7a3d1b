"""GPU parity: the CUDA library against the float64 oracle, element by
element on the same seeded inputs, for both builds (bf16 tensor-core path at
a relative error of 2e-2, fp32 SIMT debug path at 1e-5; relative error =
Frobenius norm of the difference over that of the oracle, per tensor)."""

import numpy as np
import pytest
import torch

from sliding_window_gqa_qk_gb300.inputs import TINY, Problem
import sliding_window_gqa_qk_gb300 as swa
from gpu_helpers import TOL, compare, inputs, run_library, run_oracle, run_staged

pytestmark = pytest.mark.gpu

# Sizes the oracle finishes in seconds, spanning several 128-row tiles and a
# ragged tail, plus the degenerate cases of the method.
CASES = {
    "tiny": TINY,
    "ragged_gqa_ve": Problem(B=2, T=300, Hq=4, Hkv=2, d=128, window=150, gain_std=0.1, ve=True,
                             vocab=257),
    "full_causal_d64": Problem(B=1, T=333, Hq=2, Hkv=2, d=64, window=-1, gain_std=0.1),
    "mha_d128_l": Problem(B=1, T=256, Hq=2, Hkv=2, d=128, window=-1, gain_std=0.2),
    "group4_short": Problem(B=1, T=77, Hq=4, Hkv=1, d=128, window=20, gain_std=0.1, ve=True,
                            vocab=50),
    "window0": Problem(B=1, T=150, Hq=2, Hkv=1, d=64, window=0),
    "window_ge_T": Problem(B=1, T=200, Hq=2, Hkv=1, d=64, window=500, gain_std=0.1),
    "single_token": Problem(B=2, T=1, Hq=2, Hkv=1, d=128, window=-1, gain_std=0.1),
    "noncausal_window": Problem(B=1, T=200, Hq=3, Hkv=1, d=128, window=40, causal=False,
                                gain_std=0.1),
    "noncausal_full_d64": Problem(B=1, T=130, Hq=2, Hkv=1, d=64, window=-1, causal=False),
    "long_window_ragged": Problem(B=1, T=700, Hq=2, Hkv=1, d=128, window=300, gain_std=0.1,
                                  ve=True, vocab=100),
}


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(CASES))
def test_parity_small(kind, name):
    p = CASES[name]
    x = inputs(p, kind, layer=1, with_gate=True)
    got = run_library(p, x)
    assert got["status"] == swa.SWA_OK
    ref = run_oracle(p, x)
    compare(got, ref, TOL[kind])


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_backward_without_prologue_reuse_matches(kind):
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, kind, with_gate=True)
    a = run_library(p, x, reuse_prologue=True)
    b = run_library(p, x, reuse_prologue=False)
    for k in ("dq", "dk", "dv", "dgq", "dgk", "dve"):
        diff = (a[k].double() - b[k].double()).abs().max().item()
        scale = a[k].double().abs().max().item()
        assert diff <= 1e-6 * max(scale, 1.0) or kind == "bf16" and diff <= 1e-2 * scale, k


def test_backward_stages_one_call_at_a_time_equal_one_call():
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, "bf16", with_gate=True)
    dev = torch.device("cuda:0")
    g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
    o, lse, ws = swa.attention_forward(g["q"], g["k"], g["v"], g["gq"], g["gk"], window=p.window,
                                       ve=g["ve"], tok=g["tok"], ve_scale=p.ve_scale)
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps, p.ve_scale,
                          p.vocab)
    outs = []
    for staged in (False, True):
        dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
        dgq = torch.empty(p.d, device=dev)
        dgk = torch.empty(p.d, device=dev)
        dve = torch.empty(g["ve"].shape, device=dev)
        args = (prm, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"], g["tok"], None, o, lse,
                g["dO"], dq, dk, dv, dgq, dgk, dve, ws)
        if staged:
            for st in (swa.SWA_BWD_STAGE_PRE, swa.SWA_BWD_STAGE_MAIN, swa.SWA_BWD_STAGE_POST):
                assert swa.swa_attn_bwd(*args, flags=swa.SWA_REUSE_PROLOGUE | st) == swa.SWA_OK
        else:
            assert swa.swa_attn_bwd(*args, flags=swa.SWA_REUSE_PROLOGUE) == swa.SWA_OK
        torch.cuda.synchronize()
        outs.append([t.float().cpu() for t in (dq, dk, dv, dgq, dgk, dve)])
    for a, b in zip(*outs):
        # dQ is accumulated with float atomics: equal up to summation order
        assert torch.allclose(a, b, rtol=1e-2, atol=1e-3)


def test_out_of_range_token_is_reported_and_skipped():
    p = Problem(B=1, T=64, Hq=2, Hkv=1, d=64, window=-1, ve=True, vocab=10)
    x = inputs(p, "bf16")
    x["tok"][0, 5] = 10          # one past the table
    x["tok"][0, 9] = -1
    got = run_library(p, x)
    assert got["status"] == swa.SWA_ERR_DEVICE_CHECK
    # the two rows contribute nothing from the table: oracle with a zero row
    ve = x["ve"].clone()
    ve2 = torch.cat([ve, torch.zeros(1, ve.shape[1], dtype=ve.dtype)])
    y = dict(x, ve=ve2, tok=x["tok"].clone())
    y["tok"][0, 5] = 10
    y["tok"][0, 9] = 10
    p2 = p.replace(vocab=11)
    ref = run_oracle(p2, y)
    compare(got, ref, TOL["bf16"], keys=("o", "lse", "dq", "dk", "dv"))


def test_empty_problem_backward_zeroes_shared_gradients():
    dev = torch.device("cuda:0")
    p = swa.make_params(0, 16, 2, 1, 64, -1, True, 0.0, 1e-6, 0.5, 8)
    ws = torch.zeros(swa.swa_attn_workspace_size(p, 1), dtype=torch.uint8, device=dev)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    dgq = torch.full((64,), 7.0, device=dev)
    dgk = torch.full((64,), 7.0, device=dev)
    dve = torch.full((8, 64), 7.0, device=dev)
    st = swa.swa_attn_bwd(p, dummy, dummy, dummy, None, None, dummy, dummy, None, dummy, dgq,
                          dummy, dummy, dummy, dummy, dgq, dgk, dve, ws)
    torch.cuda.synchronize()
    assert st == swa.SWA_OK
    assert dgq.abs().sum().item() == 0 and dgk.abs().sum().item() == 0
    assert dve.abs().sum().item() == 0


def _grads_bf16(p, g, o, lse, ws, ws_bytes=None, flags=0):
    dev = torch.device("cuda:0")
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps, p.ve_scale,
                          p.vocab if p.ve else 0)
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
    dgq = torch.empty(p.d, device=dev)
    dgk = torch.empty(p.d, device=dev)
    dve = torch.empty(g["ve"].shape, device=dev) if p.ve else None
    st = swa.swa_attn_bwd(prm, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"], g["tok"], None,
                          o, lse, g["dO"], dq, dk, dv, dgq, dgk, dve, ws, ws_bytes=ws_bytes,
                          flags=flags)
    assert st == swa.SWA_OK, swa.swa_strerror(st)
    torch.cuda.synchronize()
    out = {"dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu(), "dgq": dgq.cpu(), "dgk": dgk.cpu()}
    if dve is not None:
        out["dve"] = dve.cpu()
    return out


def test_second_backward_after_one_forward_clears_the_accumulator_again():
    # The forward leaves the dQ accumulator zeroed for the backward that
    # follows; the backward's main kernel marks it used, so a second backward
    # on the same workspace must clear it itself.
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, "bf16")
    ref = run_oracle(p, x)
    dev = torch.device("cuda:0")
    g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
    o, lse, ws = swa.attention_forward(g["q"], g["k"], g["v"], g["gq"], g["gk"], window=p.window,
                                       ve=g["ve"], tok=g["tok"], ve_scale=p.ve_scale)
    for _ in range(2):
        got = _grads_bf16(p, g, o, lse, ws, flags=swa.SWA_REUSE_PROLOGUE)
        compare(got, ref, TOL["bf16"], keys=("dq", "dk", "dv", "dgq", "dgk", "dve"))


@pytest.mark.parametrize("zeroing", [True, False])
def test_forward_of_another_problem_in_between_keeps_the_backward_right(zeroing):
    # Forward of X, then a forward of a larger problem Y in the same
    # workspace (its prologue outputs land where X's accumulator lies), then
    # the backward of X without prologue reuse. With zeroing=False the second
    # forward gets a forward-only workspace size and must drop the record of
    # X's zeroed accumulator; with zeroing=True it records its own, which
    # does not name X's.
    X = Problem(B=1, T=256, Hq=2, Hkv=1, d=128, window=100, gain_std=0.1)
    Y = Problem(B=2, T=1024, Hq=4, Hkv=2, d=128, window=-1, gain_std=0.1)
    dev = torch.device("cuda:0")
    px = swa.make_params(X.B, X.T, X.Hq, X.Hkv, X.d, X.window, X.causal, 0.0, X.eps, X.ve_scale, 0)
    py = swa.make_params(Y.B, Y.T, Y.Hq, Y.Hkv, Y.d, Y.window, Y.causal, 0.0, Y.eps, Y.ve_scale, 0)
    nbytes = max(swa.swa_attn_workspace_size(px, 1), swa.swa_attn_workspace_size(py, 1))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    xx, xy = inputs(X, "bf16"), inputs(Y, "bf16", layer=2)
    gx = {k: (t.to(dev) if t is not None else None) for k, t in xx.items()}
    gy = {k: (t.to(dev) if t is not None else None) for k, t in xy.items()}

    def fwd(p, prm, g, ws_bytes):
        o = torch.empty_like(g["q"])
        lse = torch.empty(p.B, p.Hq, p.T, dtype=torch.float32, device=dev)
        st = swa.swa_attn_fwd(prm, g["q"], g["k"], g["v"], g["gq"], g["gk"], None, None, None, o,
                              lse, ws, ws_bytes=ws_bytes)
        assert st == swa.SWA_OK, swa.swa_strerror(st)
        return o, lse

    ox, lx = fwd(X, px, gx, nbytes)
    fwd(Y, py, gy, nbytes if zeroing else swa.swa_attn_workspace_size(py, 0))
    got = _grads_bf16(X, gx, ox, lx, ws, ws_bytes=nbytes, flags=0)
    assert swa.swa_attn_check_status(ws) == swa.SWA_OK
    compare(got, run_oracle(X, xx), TOL["bf16"], keys=("dq", "dk", "dv", "dgq", "dgk"))


# Rotary position embedding fused into the prologue (rotation, then the norm)
# and into the backward (norm backward of the rotated rows, then the
# transposed rotation). Tables with more rows than T; positions start at 0.
ROPE_CASES = {
    "ragged_gqa_ve": CASES["ragged_gqa_ve"],
    "full_causal_d64": CASES["full_causal_d64"],
    "noncausal_window": CASES["noncausal_window"],
    "long_window_ragged": CASES["long_window_ragged"],
}


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(ROPE_CASES))
def test_parity_with_rope(kind, name):
    from gpu_helpers import rope_tables
    p = ROPE_CASES[name]
    x = inputs(p, kind, layer=3, with_gate=True)
    rope = rope_tables(p.T + 7, p.d)
    got = run_library(p, x, rope=rope)
    assert got["status"] == swa.SWA_OK
    compare(got, run_oracle(p, x, rope=rope), TOL[kind])


def test_rope_without_prologue_reuse_and_identity_tables():
    from gpu_helpers import rope_tables
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, "bf16", with_gate=True)
    rope = rope_tables(p.T, p.d)
    a = run_library(p, x, reuse_prologue=False, rope=rope)
    compare(a, run_oracle(p, x, rope=rope), TOL["bf16"])
    # identity tables (cos 1, sin 0) give exactly the result without rotary
    ident = (torch.ones(p.T, p.d // 2), torch.zeros(p.T, p.d // 2))
    b = run_library(p, x, rope=ident)
    c = run_library(p, x)
    for k in ("o", "lse"):
        assert torch.equal(b[k], c[k]), k


# Learned value-embedding gate 2 sigmoid(w x[:C]) computed in the prologue,
# with its gradients (dgate_w, dgate_x) from the backward's post stage.
GATE_CASES = {
    "ragged_gqa_ve": CASES["ragged_gqa_ve"],
    "group4_short": CASES["group4_short"],
    "long_window_ragged": CASES["long_window_ragged"],
}


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(GATE_CASES))
def test_parity_with_learned_gate(kind, name):
    from gpu_helpers import gate_weights
    p = GATE_CASES[name]
    x = inputs(p, kind, layer=5)
    gate = gate_weights(p, kind)
    got = run_library(p, x, gate=gate)
    assert got["status"] == swa.SWA_OK
    assert got["dgate_x"] is not None and got["dgate_w"] is not None
    compare(got, run_oracle(p, x, learned=gate), TOL[kind])


def test_learned_gate_with_rope_and_without_prologue_reuse():
    from gpu_helpers import gate_weights, rope_tables
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, "bf16", layer=6)
    gate = gate_weights(p, "bf16", channels=20, width=20)
    rope = rope_tables(p.T, p.d)
    got = run_library(p, x, reuse_prologue=False, rope=rope, gate=gate)
    compare(got, run_oracle(p, x, rope=rope, learned=gate), TOL["bf16"])


def test_learned_gate_at_zero_weights_equals_unit_gate():
    # the Guide: the gate weight starts at zero, 2 sigmoid(0) = 1
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, "bf16", layer=7)
    gx, gw = (torch.randn(p.B, p.T, 32).to(torch.bfloat16), torch.zeros(p.Hkv, 32))
    a = run_library(p, x, gate=(gx, gw))
    b = run_library(p, dict(x, gate=None))
    for k in ("o", "lse"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_cuda_graph_of_forward_and_backward_replays_correctly(kind):
    # The entry points make no synchronous calls, so a caller can capture a
    # whole step; replays recompute every output (they start from NaN) and
    # the second replay finds the workspace as the first left it.
    p = CASES["ragged_gqa_ve"]
    x = inputs(p, kind, layer=1, with_gate=True)
    got = run_staged(p, x, graph=True)
    assert got["status"] == swa.SWA_OK
    compare(got, run_oracle(p, x), TOL[kind])
