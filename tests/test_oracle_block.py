"""Pins of the float64 block oracle (pre-norm, projections, residual around
the attention core) against what the pages and the mathematics fix: central
finite differences of every input, the pages' initialisation (a zero output
projection returns the input), a special case that reduces the block to the
attention alone, linearity in the output projection, and an independent
float64 torch autograd run."""

import numpy as np
import pytest

from oracle import attention as orc
from oracle import block as blk


def block_problem(seed, B=1, T=6, C=10, Hq=2, Hkv=1, d=4, vocab=5, gate_ch=3,
                  with_ve=True, with_gate=True, with_gain=True):
    r = np.random.default_rng(seed)
    x = {
        "x": r.standard_normal((B, T, C)),
        "wq": 0.4 * r.standard_normal((Hq * d, C)),
        "wk": 0.4 * r.standard_normal((Hkv * d, C)),
        "wv": 0.4 * r.standard_normal((Hkv * d, C)),
        "wo": 0.4 * r.standard_normal((C, Hq * d)),
        "dout": r.standard_normal((B, T, C)),
        "gq": 1 + 0.3 * r.standard_normal(d) if with_gain else None,
        "gk": 1 + 0.3 * r.standard_normal(d) if with_gain else None,
        "ve": r.standard_normal((vocab, Hkv * d)) if with_ve else None,
        "tok": r.integers(0, vocab, size=(B, T)) if with_ve else None,
        "gate_w": 0.5 * r.standard_normal((Hkv, gate_ch)) if (with_ve and with_gate) else None,
    }
    return x, dict(Hq=Hq, Hkv=Hkv)


def rope_tables(T, d, base=10000.0):
    inv = base ** (-np.arange(d // 2) * 2.0 / d)
    ang = np.arange(T)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def run_fwd(x, shape, **kw):
    out, _ = blk.block_forward(x["x"], x["wq"], x["wk"], x["wv"], x["wo"], gq=x["gq"], gk=x["gk"],
                               ve=x["ve"], tok=x["tok"], gate_w=x["gate_w"], **shape, **kw)
    return out


def run_bwd(x, shape, **kw):
    return blk.block_backward(x["x"], x["wq"], x["wk"], x["wv"], x["wo"], x["dout"], gq=x["gq"],
                              gk=x["gk"], ve=x["ve"], tok=x["tok"], gate_w=x["gate_w"], **shape,
                              **kw)


@pytest.mark.parametrize("window,causal,with_rope", [(2, True, True), (-1, True, False),
                                                     (2, False, False)])
def test_block_backward_matches_central_finite_differences(window, causal, with_rope):
    x, shape = block_problem(101)
    kw = dict(window=window, causal=causal, eps=1e-4, ve_scale=0.7)
    if with_rope:
        kw["rope"] = rope_tables(6, 4)
    g = run_bwd(x, shape, **kw)
    h = 1e-6
    names = {"x": "dx", "wq": "dwq", "wk": "dwk", "wv": "dwv", "wo": "dwo", "gq": "dgq",
             "gk": "dgk", "ve": "dve", "gate_w": "dgate_w"}
    for name, gname in names.items():
        arr = x[name]
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = float(np.sum(run_fwd(x, shape, **kw) * x["dout"]))
            arr[idx] = old - h
            lm = float(np.sum(run_fwd(x, shape, **kw) * x["dout"]))
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(g[gname] - num) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-6, (name, err)


def test_zero_output_projection_returns_the_input():
    """The pages' initialisation zeroes c_proj: the block is then the identity,
    and the gradient of its input is the upstream gradient unchanged."""
    x, shape = block_problem(102)
    x["wo"] = np.zeros_like(x["wo"])
    kw = dict(window=2, causal=True, eps=1e-5)
    assert np.array_equal(run_fwd(x, shape, **kw), x["x"])
    g = run_bwd(x, shape, **kw)
    assert np.array_equal(g["dx"], x["dout"])
    for name in ("dwq", "dwk", "dwv", "dgate_w"):
        assert not np.any(g[name]), name
    assert np.any(g["dwo"])


def test_identity_projections_reduce_the_block_to_the_attention():
    """With C = Hq*d, one kv head per query head and identity projections, the
    block minus its input is the attention of the normed input viewed as
    heads (channel h*d + c is channel c of head h)."""
    B, T, Hq, d = 2, 7, 3, 4
    C = Hq * d
    r = np.random.default_rng(103)
    xin = r.standard_normal((B, T, C))
    eye = np.eye(C)
    kw = dict(window=3, causal=True, eps=1e-5)
    out, _ = blk.block_forward(xin, eye, eye, eye, eye, Hq=Hq, Hkv=Hq, **kw)
    xn = xin / np.sqrt(np.mean(xin * xin, axis=-1, keepdims=True) + 1e-5)
    heads = xn.reshape(B, T, Hq, d)
    o, _ = orc.attention_forward(heads, heads, heads, **kw)
    np.testing.assert_allclose(out - xin, o.reshape(B, T, C), rtol=1e-13, atol=1e-13)


def test_block_is_linear_in_the_output_projection():
    x, shape = block_problem(104)
    kw = dict(window=-1, causal=True, eps=1e-5)
    base = run_fwd(x, shape, **kw) - x["x"]
    x["wo"] = -2.5 * x["wo"]
    np.testing.assert_allclose(run_fwd(x, shape, **kw) - x["x"], -2.5 * base, rtol=1e-12,
                               atol=1e-12)


def test_block_against_float64_torch_autograd():
    """Independent library check: torch float64 autograd through F.rms_norm,
    F.linear and F.scaled_dot_product_attention with an explicit mask."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, T, C, Hq, Hkv, d, window, eps, s_ve = 2, 9, 12, 4, 2, 4, 4, 1e-5, 0.6
    x, shape = block_problem(105, B=B, T=T, C=C, Hq=Hq, Hkv=Hkv, d=d, vocab=7, gate_ch=5)
    kw = dict(window=window, causal=True, eps=eps, ve_scale=s_ve)
    out = run_fwd(x, shape, **kw)
    g = run_bwd(x, shape, **kw)

    names = ("x", "wq", "wk", "wv", "wo", "gq", "gk", "ve", "gate_w")
    t = {k: torch.tensor(x[k], dtype=torch.float64, requires_grad=True) for k in names}
    tok = torch.tensor(x["tok"], dtype=torch.long)
    xn = F.rms_norm(t["x"], (C,), None, eps)
    q = F.linear(xn, t["wq"]).view(B, T, Hq, d)
    k = F.linear(xn, t["wk"]).view(B, T, Hkv, d)
    v = F.linear(xn, t["wv"]).view(B, T, Hkv, d)
    gate = 2 * torch.sigmoid(F.linear(xn[..., :5], t["gate_w"]))
    v = v + s_ve * gate.unsqueeze(-1) * t["ve"][tok].view(B, T, Hkv, d)
    qn = F.rms_norm(q, (d,), t["gq"], eps)
    kn = F.rms_norm(k, (d,), t["gk"], eps)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    mask = (j <= i) & (i - j <= window)
    o = F.scaled_dot_product_attention(qn.transpose(1, 2), kn.transpose(1, 2), v.transpose(1, 2),
                                       attn_mask=mask, enable_gqa=True).transpose(1, 2)
    y = t["x"] + F.linear(o.reshape(B, T, Hq * d), t["wo"])
    np.testing.assert_allclose(y.detach().numpy(), out, rtol=1e-12, atol=1e-12)
    (y * torch.tensor(x["dout"])).sum().backward()
    pairs = {"x": "dx", "wq": "dwq", "wk": "dwk", "wv": "dwv", "wo": "dwo", "gq": "dgq",
             "gk": "dgk", "ve": "dve", "gate_w": "dgate_w"}
    for name, gname in pairs.items():
        np.testing.assert_allclose(t[name].grad.numpy(), g[gname], rtol=1e-10, atol=1e-12,
                                   err_msg=name)


def test_grouped_query_block_equals_the_block_with_repeated_kv_projections():
    """GQA inside the block: query head h reads kv head h // G, so the block
    with Hkv kv heads equals the block with one kv head per query head whose
    k / v projection rows, VE-table columns and gate rows are the group's,
    repeated; the gradients of the shared rows are the sums over the group."""
    B, T, C, Hq, Hkv, d, G = 1, 7, 12, 4, 2, 4, 2
    x, _ = block_problem(106, B=B, T=T, C=C, Hq=Hq, Hkv=Hkv, d=d, vocab=6, gate_ch=3)
    kw = dict(window=3, causal=True, eps=1e-5, ve_scale=0.6)

    def rep_rows(w):       # [Hkv*d, ...] -> [Hq*d, ...], kv head h // G for query head h
        return np.concatenate([w[(h // G) * d:(h // G + 1) * d] for h in range(Hq)], axis=0)

    mha = dict(x)
    mha["wk"], mha["wv"] = rep_rows(x["wk"]), rep_rows(x["wv"])
    mha["ve"] = rep_rows(x["ve"].T).T
    mha["gate_w"] = np.repeat(x["gate_w"], G, axis=0)
    out_g = run_fwd(x, dict(Hq=Hq, Hkv=Hkv), **kw)
    out_m = run_fwd(mha, dict(Hq=Hq, Hkv=Hq), **kw)
    np.testing.assert_allclose(out_g, out_m, rtol=1e-12, atol=1e-12)
    g_g = run_bwd(x, dict(Hq=Hq, Hkv=Hkv), **kw)
    g_m = run_bwd(mha, dict(Hq=Hq, Hkv=Hq), **kw)
    for name in ("dx", "dwq", "dwo", "dgq", "dgk"):
        np.testing.assert_allclose(g_g[name], g_m[name], rtol=1e-10, atol=1e-12, err_msg=name)

    def group_sum(dw):     # [Hq*d, ...] -> [Hkv*d, ...]
        return np.concatenate([sum(dw[h * d:(h + 1) * d] for h in range(k * G, (k + 1) * G))
                               for k in range(Hkv)], axis=0)

    for name in ("dwk", "dwv"):
        np.testing.assert_allclose(g_g[name], group_sum(g_m[name]), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g_g["dve"], group_sum(g_m["dve"].T).T, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g_g["dgate_w"], g_m["dgate_w"].reshape(Hkv, G, -1).sum(axis=1),
                               rtol=1e-10, atol=1e-12)
