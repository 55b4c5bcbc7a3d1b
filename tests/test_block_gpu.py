"""GPU parity of the whole attention block (pre-norm, c_q / c_k / c_v, the
attention, c_proj and the residual) through the C ABI, against the float64
block oracle on the same seeded inputs, for both builds (2e-2 for bf16
tensors and fp32 accumulation, 1e-5 for the fp32 debug build, on the
relative error of every tensor as a whole and of every row of it, and on
every element of the gain gradients, as in gpu_helpers.errors). The output
and the input gradient are also compared without the residual's exact
pass-through (out - x, dx - dout), so the attention branch is held to the
same bounds."""

import numpy as np
import pytest
import torch

import oracle
import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300.inputs import S_LAYER, Problem, as_f64, make_block_inputs
from gpu_helpers import DTYPE, ELEMENTWISE, FLOOR, ROW_FLOOR, TOL, _record, errors, rope_tables

pytestmark = pytest.mark.gpu

# (problem, model width C, learned-gate channels or None, rotary tables)
CASES = {
    "gqa_ve_gate_rope_d64": (Problem(B=2, T=200, Hq=4, Hkv=2, d=64, window=100, gain_std=0.1,
                                     ve=True, vocab=97), 192, 32, True),
    "mha_full_causal_d128": (Problem(B=1, T=300, Hq=2, Hkv=2, d=128, window=-1, gain_std=0.1),
                             256, None, False),
    "group3_ragged_unit_gains": (Problem(B=1, T=131, Hq=3, Hkv=1, d=128, window=40, ve=True,
                                         vocab=50), 136, 8, False),
    # head dim 128 and T a multiple of 32: the bf16 library folds the
    # attention's prologue into the q, k, v projection (rows 288 = 2.25 tiles)
    "fold_gqa_ve_gate_rope": (Problem(B=3, T=96, Hq=4, Hkv=2, d=128, window=40, gain_std=0.1, ve=True,
                                      vocab=61), 200, 32, True),
    "fold_mha_plain": (Problem(B=2, T=64, Hq=2, Hkv=2, d=128, window=-1, gain_std=0.1), 256, None, False),
}


def offset_copy(t, dev, elems):
    """A contiguous device copy of t that starts `elems` elements into a
    larger buffer (a tensor that is 16-byte but not 256-byte aligned)."""
    flat = torch.empty(t.numel() + elems, dtype=t.dtype, device=dev)
    view = flat[elems:].view(t.shape)
    view.copy_(t)
    return view


def run_block_library(p, C, x, rope=False, offset=None):
    dev = torch.device("cuda:0")
    g = {k: (t.to(dev).contiguous() if t is not None else None) for k, t in x.items()}
    if offset is not None:
        for k in ("x", "dout", "wo"):
            g[k] = offset_copy(x[k], dev, offset)
    kind = "fp32" if x["x"].dtype == torch.float32 else "bf16"
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps, p.ve_scale,
                          p.vocab if p.ve else 0)
    rp = None
    if rope:
        rp = tuple(t.to(dev).contiguous() for t in rope_tables(p.T, p.d))
    dgw = torch.zeros_like(g["gate_w"]) if g["gate_w"] is not None else None
    ex = swa.make_block_extras(rope=rp, gate_w=g["gate_w"], d_gate_w=dgw)
    w = swa.make_block_weights(g["wq"], g["wk"], g["wv"], g["wo"])
    n = swa.swa_block_workspace_size(prm, C, 1, kind)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    assert swa.swa_attn_workspace_init(ws, n, kind=kind) == swa.SWA_OK
    out = torch.empty_like(g["x"]) if offset is None else offset_copy(torch.zeros_like(x["x"]), dev, offset)
    assert swa.swa_block_fwd(prm, ex, w, g["x"], g["gq"], g["gk"], g["ve"], g["tok"], out, ws) == swa.SWA_OK
    f32 = dict(dtype=torch.float32, device=dev)
    dx = torch.empty_like(g["x"]) if offset is None else offset_copy(torch.zeros_like(x["x"]), dev, offset)
    dwq, dwk, dwv, dwo = (torch.empty(g[k].shape, **f32) for k in ("wq", "wk", "wv", "wo"))
    dgq = torch.empty(p.d, **f32) if g["gq"] is not None else None
    dgk = torch.empty(p.d, **f32) if g["gk"] is not None else None
    dve = torch.empty(g["ve"].shape, **f32) if g["ve"] is not None else None
    assert swa.swa_block_bwd(prm, ex, w, g["x"], g["gq"], g["gk"], g["ve"], g["tok"], g["dout"], dx,
                             dwq, dwk, dwv, dwo, dgq, dgk, dve, ws) == swa.SWA_OK
    status = swa.swa_attn_check_status(ws, kind=kind)
    torch.cuda.synchronize()
    res = {"out": out, "dx": dx, "dwq": dwq, "dwk": dwk, "dwv": dwv, "dwo": dwo, "dgq": dgq,
           "dgk": dgk, "dve": dve, "dgate_w": dgw}
    res = {k: (v.cpu() if v is not None else None) for k, v in res.items()}
    res["status"] = status
    return res


def run_block_oracle(p, x, rope=False, b_slice=None):
    f = {k: as_f64(t) for k, t in x.items()}
    kw = dict(Hq=p.Hq, Hkv=p.Hkv, window=p.window, causal=p.causal, eps=p.eps, gq=f["gq"],
              gk=f["gk"], ve=f["ve"], tok=x["tok"].numpy() if x["tok"] is not None else None,
              ve_scale=p.ve_scale, gate_w=f["gate_w"])
    if rope:
        kw["rope"] = tuple(t.double().numpy() for t in rope_tables(p.T, p.d))
    xs, dout = f["x"], f["dout"]
    if b_slice is not None:
        xs, dout = xs[b_slice:b_slice + 1], dout[b_slice:b_slice + 1]
        kw["tok"] = None if kw["tok"] is None else kw["tok"][b_slice:b_slice + 1]
    out, _ = oracle.block_forward(xs, f["wq"], f["wk"], f["wv"], f["wo"], **kw)
    g = oracle.block_backward(xs, f["wq"], f["wk"], f["wv"], f["wo"], dout, **kw)
    g["out"] = out
    return g


def compare_block(got, ref, x, tol, keys):
    xs, dout = as_f64(x["x"]), as_f64(x["dout"])
    pairs = []
    for k in keys:
        if ref.get(k) is None:
            assert got.get(k) is None or k == "dgate_w", k
            continue
        pairs.append((k, got[k].double().numpy(), ref[k]))
    pairs.append(("out - x", got["out"].double().numpy() - xs, ref["out"] - xs))
    pairs.append(("dx - dout", got["dx"].double().numpy() - dout, ref["dx"] - dout))
    errs, bad = {}, {}
    for k, a, r in pairs:
        e = errors(a, r, elementwise=k in ELEMENTWISE, floor=FLOOR.get(k, ROW_FLOOR))
        _record(k, *e)
        errs[k] = e
        if not (e[0] <= tol and e[1] <= tol):
            bad[k] = e
    assert not bad, ("(frob, worst row, max abs)", bad, errs)


ALL = ("out", "dx", "dwq", "dwk", "dwv", "dwo", "dgq", "dgk", "dve", "dgate_w")


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(CASES))
def test_block_parity_small(kind, name):
    p, C, gate_ch, rope = CASES[name]
    x = make_block_inputs(p, C, layer=1, dtype=DTYPE[kind], gate_ch=gate_ch)
    got = run_block_library(p, C, x, rope)
    assert got["status"] == swa.SWA_OK
    compare_block(got, run_block_oracle(p, x, rope), x, TOL[kind], ALL)


def test_block_at_zero_output_projection_is_the_identity():
    """The pages' initialisation (c_proj = 0): the block returns its input
    bit for bit and passes dout through to dx."""
    p, C, gate_ch, rope = CASES["gqa_ve_gate_rope_d64"]
    x = make_block_inputs(p, C, dtype=torch.bfloat16, gate_ch=gate_ch)
    x["wo"] = torch.zeros_like(x["wo"])
    got = run_block_library(p, C, x, rope)
    assert torch.equal(got["out"], x["x"])
    assert torch.equal(got["dx"], x["dout"])
    assert not torch.any(got["dwq"]) and not torch.any(got["dgate_w"])


def test_block_full_size_s_layer():
    """The S layer's shapes inside the block at the model width of the pages'
    default (C = 768 = Hq * d), with the value embedding, its learned gate and
    rotary tables: every output and gradient over the whole batch (B = 16,
    T = 2048), the weight gradients summed over all 32768 positions."""
    p = S_LAYER.replace(ve=True, vocab=8192)
    C = 768
    x = make_block_inputs(p, C, layer=1, dtype=torch.bfloat16, gate_ch=32)
    got = run_block_library(p, C, x, rope=True)
    assert got["status"] == swa.SWA_OK
    ref = run_block_oracle(p, x, rope=True)
    compare_block(got, ref, x, TOL["bf16"], ALL)


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_block_ignores_the_gate_without_a_value_embedding(kind):
    """gate_w given on a layer without a VE table: the gate does not apply (as
    in the attention calls), so the block equals the block without a gate."""
    p, C, _, rope = CASES["mha_full_causal_d128"]
    x = make_block_inputs(p, C, layer=2, dtype=DTYPE[kind], gate_ch=16)
    got = run_block_library(p, C, x, rope)
    assert got["status"] == swa.SWA_OK
    ref = run_block_oracle(p, dict(x, gate_w=None), rope)
    keys = tuple(k for k in ALL if k != "dgate_w")
    compare_block(got, ref, x, TOL[kind], keys)


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_block_with_16_byte_aligned_tensors(kind):
    """x, dout, out, dx and wo start 16 bytes past a 256-byte boundary (the
    library asks for 16-byte alignment only)."""
    p, C, gate_ch, rope = CASES["gqa_ve_gate_rope_d64"]
    x = make_block_inputs(p, C, layer=3, dtype=DTYPE[kind], gate_ch=gate_ch)
    elems = 16 // (2 if kind == "bf16" else 4)
    got = run_block_library(p, C, x, rope, offset=elems)
    assert got["status"] == swa.SWA_OK
    compare_block(got, run_block_oracle(p, x, rope), x, TOL[kind], ALL)
