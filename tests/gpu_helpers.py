"""Shared helpers of the GPU parity tests: run the library through its C ABI
and the float64 oracle on the same seeded inputs, and compare."""

import os

import numpy as np
import torch

import oracle
import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300.inputs import as_f64, make_inputs

TOL = {"bf16": 2e-2, "fp32": 1e-5}
DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32}


def gate_for(p, seed=7):
    g = torch.Generator().manual_seed(seed)
    return 2.0 * torch.sigmoid(torch.randn(p.B, p.T, p.Hkv, generator=g))


def inputs(p, kind, layer=0, with_gate=False):
    x = make_inputs(p, layer=layer, dtype=DTYPE[kind])
    x["gate"] = gate_for(p) if (with_gate and p.ve) else None
    return x


def rope_tables(rows, d, base=10000.0):
    """Standard rotary tables (angle t * base^(-2c/d)) as fp32 CPU tensors
    [rows, d/2]; the oracle gets the same fp32 values."""
    half = d // 2
    inv = base ** (-np.arange(half) * 2.0 / d)
    ang = np.arange(rows)[:, None] * inv[None, :]
    return (torch.tensor(np.cos(ang), dtype=torch.float32), torch.tensor(np.sin(ang), dtype=torch.float32))


def gate_weights(p, kind, channels=32, width=48, seed=9):
    """Inputs of the learned VE gate: block-input rows [B, T, width] (the gate
    reads the first ``channels``) in the library's element type, and weights
    [Hkv, channels] fp32 of a size that puts the gate well inside (0, 2)."""
    g = torch.Generator().manual_seed(seed)
    gx = torch.randn(p.B, p.T, width, generator=g).to(DTYPE[kind])
    gw = 0.25 * torch.randn(p.Hkv, channels, generator=g)
    return gx, gw


def run_library(p, x, reuse_prologue=True, rope=None, gate=None):
    """Forward + backward through the C ABI on cuda:0. Returns CPU tensors.
    rope: None or (cos, sin) CPU fp32 tensors; gate: None or (gate_x, gate_w)
    CPU tensors of the learned value-embedding gate."""
    dev = torch.device("cuda:0")
    g = {k: (t.to(dev).contiguous() if t is not None else None) for k, t in x.items()}
    rp = None if rope is None else tuple(t.to(dev).contiguous() for t in rope)
    gx = gw = None
    if gate is not None:
        gx, gw = gate[0].to(dev).contiguous(), gate[1].to(dev).contiguous()
    o, lse, ws = swa.attention_forward(
        g["q"], g["k"], g["v"], g["gq"], g["gk"], window=p.window, causal=p.causal, eps=p.eps,
        ve=g["ve"], tok=g["tok"], ve_gate=None if gate is not None else g["gate"], ve_scale=p.ve_scale,
        rope=rp, gate_x=gx, gate_w=gw)
    grads = swa.attention_backward(
        g["q"], g["k"], g["v"], g["gq"], g["gk"], o, lse, g["dO"], window=p.window,
        causal=p.causal, eps=p.eps, ve=g["ve"], tok=g["tok"],
        ve_gate=None if gate is not None else g["gate"], ve_scale=p.ve_scale, workspace=ws,
        reuse_prologue=reuse_prologue, rope=rp, gate_x=gx, gate_w=gw)
    kind = "fp32" if x["q"].dtype == torch.float32 else "bf16"
    status = swa.swa_attn_check_status(ws, kind=kind)
    torch.cuda.synchronize()
    out = {"o": o.cpu(), "lse": lse.cpu(), "status": status}
    for k in ("dq", "dk", "dv", "dgq", "dgk", "dve", "dgate_x", "dgate_w"):
        out[k] = grads[k].cpu() if grads.get(k) is not None else None
    return out


def run_oracle(p, x, b_slice=None, rope=None, learned=None):
    f = {k: as_f64(t) for k, t in x.items()}
    tok = x["tok"].numpy() if x["tok"] is not None else None
    gate = f.get("gate")
    q, k, v, dO = f["q"], f["k"], f["v"], f["dO"]
    if b_slice is not None:
        sl = slice(b_slice, b_slice + 1)
        q, k, v, dO = q[sl], k[sl], v[sl], dO[sl]
        tok = tok[sl] if tok is not None else None
        gate = gate[sl] if gate is not None else None
    kw = dict(window=p.window, causal=p.causal, eps=p.eps, ve=f["ve"], tok=tok, gate=gate,
              ve_scale=p.ve_scale)
    if rope is not None:
        kw["rope"] = (rope[0].double().numpy(), rope[1].double().numpy())
    if learned is not None:   # (gate_x, gate_w) of the learned VE gate
        C = learned[1].shape[1]
        kw["gate"] = None
        kw["gate_x"] = as_f64(learned[0])[..., :C]
        kw["gate_w"] = learned[1].double().numpy()
    o, lse = oracle.attention_forward(q, k, v, f["gq"], f["gk"], **kw)
    ref = oracle.attention_backward(q, k, v, f["gq"], f["gk"], dO, scales=True, **kw)
    ref["o"], ref["lse"] = o, lse
    return ref


def rel_err(a, r):
    a = as_f64(a) if isinstance(a, torch.Tensor) else np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert a.shape == r.shape, (a.shape, r.shape)
    assert np.all(np.isfinite(a)), "non-finite values"
    den = np.linalg.norm(r)
    return float(np.linalg.norm(a - r) / den) if den > 0 else float(np.linalg.norm(a))


# Keys compared element by element (every element its own "row"); the others
# row by row along their last axis (a head row of d channels, a VE-table row).
ELEMENTWISE = ("lse", "dgq", "dgk")
# Floor of a row's reference norm in the per-row bound, as a multiple of the
# root mean square of all rows' reference norms. The library's rounding
# errors in a row are absolute, at the scale of a typical row, not relative
# to the row's own size. Rows that see only a few keys show it most: there
# dS = P (dP - D) is a difference of nearly equal numbers of size |dO| |v|
# formed from bf16 operands (on value-embedding layers v_eff itself is
# rounded to bf16), so a row whose exact gradient is small keeps an error of
# 2-3 % of a typical row (measured worst: 2.9 %, the second query row of a
# value-embedding layer; 1.9 % on layers without value embeddings); the fp32
# build shows the same at its own precision. So every row is held to tol
# times the larger of its own norm and twice the rows' root mean square norm:
# relative for rows of twice the typical size and above, absolute below. A
# wrong row, or a wrong element of lse or of the gain gradients, is off by
# about its own size and exceeds the bound many times over.
ROW_FLOOR = 2.0
FLOOR = {}
# (test, tensor, Frobenius error, worst row error, max abs error) of every
# comparison of this session, printed at its end by conftest.py.
REPORT = []


def _rows(x, elementwise):
    return x.reshape(-1, 1) if (elementwise or x.ndim < 2) else x.reshape(-1, x.shape[-1])


def errors(a, r, elementwise=False, zero_ref_scale=None, floor=ROW_FLOOR, row_scale=None):
    """Errors of the library's tensor a against the oracle's r (same shape):
      frob   ||a - r|| / ||r|| over the whole tensor;
      row    max over rows of ||a_row - r_row|| / max(||r_row||, floor * rms_row),
             rms_row the root mean square of the reference rows' norms (rows =
             last axis, or single elements when ``elementwise``);
      maxabs max |a - r| over all elements.
    ``row_scale`` (one value per row, e.g. the oracle's
    rms_norm_backward_scale of a dq or dk row) raises a row's reference norm
    to the natural scale of its errors where that is larger.
    Where r is exactly zero (a degenerate case of the method) the scale comes
    from another tensor: ``zero_ref_scale`` = (its norm, the root mean square
    of its rows' norms), giving frob = ||a|| / norm and row = max ||a_row|| /
    rms."""
    a = as_f64(a) if isinstance(a, torch.Tensor) else np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert a.shape == r.shape, (a.shape, r.shape)
    assert np.all(np.isfinite(a)), "non-finite values"
    diff = a - r
    maxabs = float(np.max(np.abs(diff))) if diff.size else 0.0
    dn = np.linalg.norm(_rows(diff, elementwise), axis=1)
    if zero_ref_scale is not None:
        norm, rms = zero_ref_scale
        frob = float(np.linalg.norm(diff) / norm)
        row = float(np.max(dn) / rms) if dn.size else 0.0
        return frob, row, maxabs
    den = np.linalg.norm(r)
    frob = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    sn = np.linalg.norm(_rows(r, elementwise), axis=1)
    rms = float(np.sqrt(np.mean(sn ** 2))) if sn.size else 0.0
    if dn.size == 0:
        row = 0.0
    elif rms > 0:
        den = np.maximum(sn, floor * rms)
        if row_scale is not None:
            den = np.maximum(den, np.asarray(row_scale, dtype=np.float64).reshape(-1))
        row = float(np.max(dn / den))
    else:
        row = 0.0 if np.all(dn == 0) else float("inf")
    return frob, row, maxabs


def _record(key, frob, row, maxabs):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    REPORT.append((test, key, frob, row, maxabs))


def check(key, a, r, tol, row_scale=None):
    """Asserts the Frobenius and the per-row (per-element for ELEMENTWISE keys)
    bounds of ``errors`` at ``tol``; records the errors. Returns (frob, row,
    maxabs)."""
    e = errors(a, r, elementwise=key in ELEMENTWISE, floor=FLOOR.get(key, ROW_FLOOR),
               row_scale=row_scale)
    _record(key, *e)
    frob, row, maxabs = e
    assert frob <= tol and row <= tol, (
        f"{key}: relative error {frob:.3e}, worst row {row:.3e} (tolerance {tol}), "
        f"max abs error {maxabs:.3e}")
    return e


def compare(got, ref, tol, keys=("o", "lse", "dq", "dk", "dv", "dgq", "dgk", "dve", "dgate_x", "dgate_w"),
            sl=None):
    """Errors per tensor (``errors``), each bounded by ``tol`` both over the
    whole tensor and row by row. Where the oracle's tensor is exactly zero (a
    degenerate case of the method, e.g. window 0 makes dS vanish, so dq, dk and
    the gain gradients are 0), the library's values are measured against the
    oracle's dv, the gradient the same terms are built from: its norm for the
    whole tensor, the root mean square of its row norms for each row. Rows of
    dq and dk are the output of the QK-norm's backward, a projection that
    removes the component of the gradient along the normed row: their scale
    is at least the oracle's dq_scale / dk_scale (the row norm before that
    projection), where the errors they carry come from."""
    errs = {}
    bad = {}
    for k in keys:
        if ref.get(k) is None or got.get(k) is None:
            continue
        a = got[k]
        if sl is not None and k not in ("dgq", "dgk", "dve", "dgate_w"):
            a = a[sl]
        zs = None
        if np.linalg.norm(ref[k]) == 0.0 and ref.get("dv") is not None:
            dv = np.asarray(ref["dv"], dtype=np.float64)
            dvn = np.linalg.norm(_rows(dv, False), axis=1)
            zs = (float(np.linalg.norm(dv)), float(np.sqrt(np.mean(dvn ** 2))))
        rs = ref.get(k + "_scale") if k in ("dq", "dk") else None
        if rs is not None and sl is not None:
            rs = rs[sl]
        e = errors(a, ref[k], elementwise=k in ELEMENTWISE, zero_ref_scale=zs,
                   floor=FLOOR.get(k, ROW_FLOOR), row_scale=rs)
        _record(k, *e)
        errs[k] = e[0]
        errs[k + "_row"] = e[1]
        errs[k + "_maxabs"] = e[2]
        if not (e[0] <= tol and e[1] <= tol):
            bad[k] = e
    assert not bad, f"errors above {tol} (frob, worst row, max abs): {bad} (all: {errs})"
    return errs


def run_staged(p, x, dev=None, rope=None, graph=False):
    """Forward + backward through the C ABI exactly as the benchmark calls
    it: swa_attn_fwd with the ve gate left out, then the three backward
    stages one call at a time with the prologue outputs reused. Returns CPU
    tensors (bf16 outputs as stored, fp32 gradients of the shared
    parameters). graph=True captures the four calls in a CUDA graph, fills
    every output with NaN and replays the graph twice."""
    dev = dev or torch.device("cuda:0")
    g = {k: (t.to(dev).contiguous() if t is not None else None) for k, t in x.items()}
    kind = "fp32" if x["q"].dtype == torch.float32 else "bf16"
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps,
                          p.ve_scale, p.vocab if p.ve else 0)
    ws = swa.new_workspace(prm, True, dev, kind)
    o = torch.empty_like(g["q"])
    lse = torch.empty(p.B, p.Hq, p.T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
    dgq = torch.empty(p.d, device=dev) if g["gq"] is not None else None
    dgk = torch.empty(p.d, device=dev) if g["gk"] is not None else None
    dve = torch.empty(g["ve"].shape, device=dev) if p.ve else None
    gate = g.get("gate")
    rt = None if rope is None else tuple(t.to(dev).contiguous() for t in rope)
    rp = None if rope is None else swa.make_extras(rope=rt)
    def calls():
        st = swa.swa_attn_fwd_ex(prm, rp, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"],
                                 g["tok"], gate, o, lse, ws, kind=kind)
        assert st == swa.SWA_OK, swa.swa_strerror(st)
        for stage in (swa.SWA_BWD_STAGE_PRE, swa.SWA_BWD_STAGE_MAIN, swa.SWA_BWD_STAGE_POST):
            st = swa.swa_attn_bwd_ex(prm, rp, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"],
                                     g["tok"], gate, o, lse, g["dO"], dq, dk, dv, dgq, dgk, dve, ws,
                                     flags=swa.SWA_REUSE_PROLOGUE | stage, kind=kind)
            assert st == swa.SWA_OK, swa.swa_strerror(st)

    if graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            calls()
        for t in (o, lse, dq, dk, dv, dgq, dgk, dve):
            if t is not None:
                t.fill_(float("nan"))
        gr.replay()
        gr.replay()
    else:
        calls()
    status = swa.swa_attn_check_status(ws, kind=kind)
    torch.cuda.synchronize()
    out = {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu(),
           "dgq": dgq.cpu() if dgq is not None else None,
           "dgk": dgk.cpu() if dgk is not None else None,
           "dve": dve.cpu() if dve is not None else None, "status": status}
    del ws, g
    return out


def batch_slice(x, b):
    """The inputs of batch element b alone (a B=1 problem); shared tensors kept."""
    out = {}
    for k, t in x.items():
        if t is None or k in ("gq", "gk", "ve"):
            out[k] = t
        else:
            out[k] = t[b:b + 1].contiguous()
    return out
