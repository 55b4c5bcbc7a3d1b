"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these re-type the oracle's formulas: each compares it with a worked
example printed on the pages, a closed form, an invariant, a special case that
reduces to something simpler, pure-Python brute force, central finite
differences, or an independent float64 autograd run (torch SDPA).
"""

import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def rand_problem(seed, B=1, T=12, Hq=2, Hkv=1, d=8, with_gain=True, with_ve=False,
                 with_gate=False, vocab=11):
    r = rng(seed)
    x = {
        "q": r.standard_normal((B, T, Hq, d)),
        "k": r.standard_normal((B, T, Hkv, d)),
        "v": r.standard_normal((B, T, Hkv, d)),
        "dO": r.standard_normal((B, T, Hq, d)),
        "gq": 1 + 0.3 * r.standard_normal(d) if with_gain else None,
        "gk": 1 + 0.3 * r.standard_normal(d) if with_gain else None,
        "ve": None, "tok": None, "gate": None,
    }
    if with_ve:
        x["ve"] = r.standard_normal((vocab, Hkv * d))
        x["tok"] = r.integers(0, vocab, size=(B, T))
        if with_gate:
            x["gate"] = 2.0 / (1.0 + np.exp(-r.standard_normal((B, T, Hkv))))
    return x


def fwd(x, **kw):
    return orc.attention_forward(x["q"], x["k"], x["v"], x["gq"], x["gk"], ve=x["ve"],
                                 tok=x["tok"], gate=x["gate"], **kw)


def bwd(x, **kw):
    return orc.attention_backward(x["q"], x["k"], x["v"], x["gq"], x["gk"], x["dO"],
                                  ve=x["ve"], tok=x["tok"], gate=x["gate"], **kw)


# ---------------------------------------------------------------------------
# The pages' worked examples
# ---------------------------------------------------------------------------

def load_golden_schedule():
    rows = []
    with open(os.path.join(GOLDEN, "sssl_8_layers.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            layer, kind, window, ve = line.split()
            rows.append((int(layer), kind, int(window), bool(int(ve))))
    return rows


def test_sssl_schedule_matches_pages_example():
    rows = load_golden_schedule()
    assert len(rows) == 8
    for layer, kind, window, _ in rows:
        assert orc.sssl_window(layer, 8, "SSSL", 2048) == window
        assert (window == -1) == (kind == "L")
    local = [l for l, kind, _, _ in rows if kind == "S"]
    assert local == [0, 1, 2, 4, 5, 6]


def test_last_layer_forced_global():
    # The pattern "SSSS" would make every layer local; the last is still global.
    assert [orc.sssl_window(i, 6, "SSSS", 100) for i in range(6)] == [50] * 5 + [-1]
    assert orc.sssl_window(4, 5, "S", 64) == -1


def test_has_ve_matches_pages_example():
    rows = load_golden_schedule()
    for layer, _, _, ve in rows:
        assert orc.has_ve(layer, 8) == ve
    assert [i for i in range(8) if orc.has_ve(i, 8)] == [1, 3, 5, 7]
    # odd depth: alternating, last included
    assert [i for i in range(7) if orc.has_ve(i, 7)] == [0, 2, 4, 6]


# ---------------------------------------------------------------------------
# Brute force: pure-Python loops on tiny inputs
# ---------------------------------------------------------------------------

def brute_force(x, window, causal, scale, eps, ve_scale):
    """Attention by scalar loops and math.exp, written independently."""
    q, k, v = x["q"], x["k"], x["v"]
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv

    def norm(vec, g):
        ms = sum(c * c for c in vec) / len(vec)
        r = 1.0 / math.sqrt(ms + eps)
        return [vec[c] * r * (1.0 if g is None else g[c]) for c in range(len(vec))]

    o = np.zeros(q.shape)
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i in range(T):
                qi = norm(list(q[b, i, h]), x["gq"])
                logits, vals = [], []
                for j in range(T):
                    if causal:
                        ok = j <= i and (window < 0 or i - j <= window)
                    else:
                        ok = window < 0 or abs(i - j) <= window
                    if not ok:
                        continue
                    kj = norm(list(k[b, j, hk]), x["gk"])
                    logits.append(scale * sum(a * c for a, c in zip(qi, kj)))
                    vj = list(v[b, j, hk])
                    if x["ve"] is not None:
                        g = 1.0 if x["gate"] is None else x["gate"][b, j, hk]
                        row = x["ve"][x["tok"][b, j]]
                        vj = [vj[c] + ve_scale * g * row[hk * d + c] for c in range(d)]
                    vals.append(vj)
                m = max(logits)
                w = [math.exp(s - m) for s in logits]
                tot = sum(w)
                for c in range(d):
                    o[b, i, h, c] = sum(wj * vj[c] for wj, vj in zip(w, vals)) / tot
                lse[b, h, i] = m + math.log(tot)
    return o, lse


@pytest.mark.parametrize("window,causal", [(-1, True), (0, True), (3, True), (7, True),
                                           (2, False), (-1, False)])
@pytest.mark.parametrize("ve", [False, True])
def test_forward_matches_brute_force(window, causal, ve):
    x = rand_problem(1, B=2, T=10, Hq=4, Hkv=2, d=6, with_ve=ve, with_gate=ve)
    scale, eps = 0.37, 1e-3
    o, lse = fwd(x, window=window, causal=causal, scale=scale, eps=eps, ve_scale=0.7)
    o2, lse2 = brute_force(x, window, causal, scale, eps, 0.7)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Special cases and closed forms
# ---------------------------------------------------------------------------

def test_window_at_least_T_minus_1_is_full_causal():
    x = rand_problem(2, B=1, T=40, Hq=2, Hkv=1, d=8)
    o_full, l_full = fwd(x, window=-1)
    for w in (39, 40, 1000):
        o, l = fwd(x, window=w)
        assert np.array_equal(o, o_full) and np.array_equal(l, l_full)
    o, _ = fwd(x, window=38)
    assert not np.array_equal(o, o_full)


def test_window_zero_returns_v_eff():
    x = rand_problem(3, B=2, T=16, Hq=4, Hkv=2, d=8, with_ve=True, with_gate=True)
    o, lse = fwd(x, window=0, ve_scale=0.5)
    v_eff = orc.ve_mix(x["v"], x["ve"], x["tok"], x["gate"], 0.5)
    np.testing.assert_allclose(o, np.repeat(v_eff, 2, axis=2), rtol=0, atol=1e-14)
    # one visible key: LSE is that key's logit
    qn, _ = orc.rms_norm(x["q"], x["gq"], 1e-6)
    kn, _ = orc.rms_norm(x["k"], x["gk"], 1e-6)
    diag = np.einsum("bthc,bthc->bht", qn, np.repeat(kn, 2, axis=2)) / math.sqrt(8)
    np.testing.assert_allclose(lse, diag, rtol=1e-13, atol=1e-13)


def test_single_token_sequence():
    x = rand_problem(4, B=3, T=1, Hq=2, Hkv=2, d=8)
    o, _ = fwd(x, window=-1)
    np.testing.assert_allclose(o, x["v"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("window", [-1, 5])
def test_zero_queries_average_the_band(window):
    """q = 0 gives qn = 0 (eps > 0): all logits vanish, so every visible key
    gets the same weight: O_i is the mean of v over the band, LSE_i = ln(band)."""
    x = rand_problem(5, B=1, T=20, Hq=2, Hkv=1, d=8)
    x["q"][:] = 0.0
    o, lse = fwd(x, window=window)
    for i in range(20):
        lo = 0 if window < 0 else max(0, i - window)
        mean = x["v"][0, lo:i + 1, 0, :].mean(axis=0)
        for h in range(2):
            np.testing.assert_allclose(o[0, i, h], mean, rtol=1e-13, atol=1e-14)
            assert abs(lse[0, h, i] - math.log(i - lo + 1)) < 1e-13


def test_softmax_rows_sum_to_one_and_ignore_off_band_keys():
    x = rand_problem(6, B=1, T=24, Hq=2, Hkv=1, d=8)
    x["v"][:] = 1.0
    o, _ = fwd(x, window=4)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)      # sum_j A_ij = 1
    # a value vector outside every band of row i has no effect on row i
    x2 = rand_problem(6, B=1, T=24, Hq=2, Hkv=1, d=8)
    o_a, _ = fwd(x2, window=4)
    x2["v"][0, 3, 0, :] += 100.0           # key 3 is visible to rows 3..7 only
    o_b, _ = fwd(x2, window=4)
    changed = np.where(np.abs(o_a - o_b).max(axis=(0, 2, 3)) > 0)[0]
    assert list(changed) == [3, 4, 5, 6, 7]


def test_lse_bounds_and_shift_invariance():
    x = rand_problem(7, B=1, T=30, Hq=2, Hkv=1, d=8)
    o, lse = fwd(x, window=6)
    qn, _ = orc.rms_norm(x["q"], x["gq"], 1e-6)
    kn, _ = orc.rms_norm(x["k"], x["gk"], 1e-6)
    for h in range(2):
        S = orc.attention_logits(qn, kn, 0, h, np.arange(30), 1 / math.sqrt(8))
        M = orc.band_mask(np.arange(30), 30, 6, True)
        mx = np.where(M, S, -np.inf).max(axis=1)
        band = M.sum(axis=1)
        assert np.all(lse[0, h] >= mx - 1e-13)
        assert np.all(lse[0, h] <= mx + np.log(band) + 1e-13)
    # Adding a constant to every logit of a row cannot change O: scaling the
    # key gains by c changes logits multiplicatively, so use the v-side instead:
    # softmax weights do not depend on v, hence O is linear in v.
    x2 = dict(x)
    x2["v"] = 2.0 * x["v"] + 0.5
    o2, lse2 = fwd(x2, window=6)
    np.testing.assert_allclose(o2, 2.0 * o + 0.5, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(lse2, lse)


# ---------------------------------------------------------------------------
# QK-norm
# ---------------------------------------------------------------------------

def test_rms_norm_unit_rms_and_scale_invariance():
    r = rng(8)
    x = r.standard_normal((5, 7, 16)) * 3.0
    y, rstd = orc.rms_norm(x, None, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    y2, _ = orc.rms_norm(7.5 * x, None, 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-14, atol=1e-14)
    # gains are per channel
    g = r.standard_normal(16)
    yg, _ = orc.rms_norm(x, g, 0.0)
    np.testing.assert_allclose(yg, y * g, rtol=1e-14, atol=1e-14)
    # eps enters under the square root: a constant row c*1 gives c/sqrt(c^2+eps)
    c, eps = 0.3, 0.05
    yc, _ = orc.rms_norm(np.full((1, 4), c), None, eps)
    np.testing.assert_allclose(yc, c / math.sqrt(c * c + eps), rtol=1e-15)


def test_attention_is_invariant_to_q_and_k_scale():
    x = rand_problem(9, B=1, T=16, Hq=2, Hkv=1, d=8)
    o, lse = fwd(x, window=5, eps=0.0)
    x2 = dict(x)
    x2["q"] = 13.0 * x["q"]
    x2["k"] = 0.01 * x["k"]
    o2, lse2 = fwd(x2, window=5, eps=0.0)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-12)


def test_logit_bound_of_qk_norm():
    """|logit| <= scale * ||gq*qh|| ||gk*kh|| <= sqrt(d) * max|gq| * max|gk| with
    scale = 1/sqrt(d); with unit gains |logit| <= sqrt(d), reached when qn || kn."""
    d = 16
    x = rand_problem(10, B=1, T=64, Hq=2, Hkv=1, d=d)
    qn, _ = orc.rms_norm(x["q"], x["gq"], 1e-6)
    kn, _ = orc.rms_norm(x["k"], x["gk"], 1e-6)
    bound = math.sqrt(d) * np.abs(x["gq"]).max() * np.abs(x["gk"]).max()
    for h in range(2):
        S = orc.attention_logits(qn, kn, 0, h, np.arange(64), 1 / math.sqrt(d))
        assert np.abs(S).max() <= bound
    # unit gains, eps = 0, q == k: the diagonal reaches sqrt(d) exactly
    y = rand_problem(11, B=1, T=8, Hq=1, Hkv=1, d=d, with_gain=False)
    qn, _ = orc.rms_norm(y["q"], None, 0.0)
    S = orc.attention_logits(qn, qn, 0, 0, np.arange(8), 1 / math.sqrt(d))
    assert np.abs(S).max() <= math.sqrt(d) * (1 + 1e-14)
    np.testing.assert_allclose(np.diag(S), math.sqrt(d), rtol=1e-14)


def test_product_of_gain_norms_over_sqrt_d_is_not_a_bound():
    """The stated bound 'product of the two gain norms over sqrt(d)' fails for
    general gains: d = 2, q = k = (1, 0), g = (1, 0) gives logit sqrt(2) > 1/sqrt(2)."""
    q = np.array([[[[1.0, 0.0]]]])
    g = np.array([1.0, 0.0])
    qn, _ = orc.rms_norm(q, g, 0.0)
    S = orc.attention_logits(qn, qn, 0, 0, np.arange(1), 1 / math.sqrt(2))
    assert abs(S[0, 0] - math.sqrt(2)) < 1e-15
    assert S[0, 0] > np.linalg.norm(g) ** 2 / math.sqrt(2)
    assert S[0, 0] <= math.sqrt(2) * 1.0 * 1.0 + 1e-15


# ---------------------------------------------------------------------------
# GQA and value embeddings
# ---------------------------------------------------------------------------

def test_gqa_equals_mha_with_repeated_kv():
    x = rand_problem(12, B=2, T=14, Hq=6, Hkv=2, d=8)
    o, lse = fwd(x, window=4)
    g = bwd(x, window=4)
    y = dict(x)
    y["k"] = np.repeat(x["k"], 3, axis=2)
    y["v"] = np.repeat(x["v"], 3, axis=2)
    o2, lse2 = fwd(y, window=4)
    g2 = bwd(y, window=4)
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(g["dq"], g2["dq"], rtol=1e-12, atol=1e-12)
    for key in ("dk", "dv"):
        summed = g2[key].reshape(2, 14, 2, 3, 8).sum(axis=3)
        np.testing.assert_allclose(g[key], summed, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dgk"], g2["dgk"], rtol=1e-12, atol=1e-12)


def test_value_embedding_special_cases():
    x = rand_problem(13, B=2, T=12, Hq=4, Hkv=2, d=8, with_ve=True, with_gate=True)
    o_plain, _ = fwd(dict(x, ve=None, tok=None, gate=None), window=3)
    o_zero, _ = fwd(dict(x, ve=np.zeros_like(x["ve"])), window=3)
    o_s0, _ = fwd(x, window=3, ve_scale=0.0)
    np.testing.assert_array_equal(o_zero, o_plain)
    np.testing.assert_array_equal(o_s0, o_plain)
    # v = 0 and window 0: the output is the gated, scaled table row of the token
    y = dict(x, v=np.zeros_like(x["v"]))
    o, _ = fwd(y, window=0, ve_scale=0.5)
    for b in range(2):
        for t in range(12):
            for h in range(4):
                hk = h // 2
                want = 0.5 * x["gate"][b, t, hk] * x["ve"][x["tok"][b, t], hk * 8:(hk + 1) * 8]
                np.testing.assert_allclose(o[b, t, h], want, rtol=1e-14, atol=1e-15)
    # the pages' gate at initialisation: 2 * sigmoid(0) = 1 -> same as gate None
    o_g1, _ = fwd(dict(x, gate=np.full((2, 12, 2), 2.0 / (1.0 + math.exp(0.0)))), window=3)
    o_gn, _ = fwd(dict(x, gate=None), window=3)
    np.testing.assert_array_equal(o_g1, o_gn)


# ---------------------------------------------------------------------------
# Backward: finite differences, identities, independent autograd
# ---------------------------------------------------------------------------

def loss(x, **kw):
    o, _ = fwd(x, **kw)
    return float(np.sum(o * x["dO"]))


@pytest.mark.parametrize("window,causal", [(-1, True), (3, True), (2, False)])
def test_backward_matches_central_finite_differences(window, causal):
    x = rand_problem(14, B=1, T=9, Hq=2, Hkv=1, d=4, with_ve=True, with_gate=True, vocab=5)
    kw = dict(window=window, causal=causal, eps=1e-4, ve_scale=0.7)
    g = bwd(x, **kw)
    h = 1e-6
    names = {"q": "dq", "k": "dk", "v": "dv", "gq": "dgq", "gk": "dgk", "ve": "dve"}
    for name, gname in names.items():
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = base[idx]
            base[idx] = old + h
            lp = loss(x, **kw)
            base[idx] = old - h
            lm = loss(x, **kw)
            base[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(g[gname] - num) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-6, (name, err)


def test_rms_norm_backward_identities():
    r = rng(15)
    x = r.standard_normal((6, 10))
    dy = r.standard_normal((6, 10))
    dx, _ = orc.rms_norm_backward(x, None, 0.0, dy)
    # eps = 0: y is scale invariant, so its gradient is orthogonal to x per row
    np.testing.assert_allclose(np.sum(dx * x, axis=1), 0.0, atol=1e-12)
    # with gains, dg = sum_rows dy * xhat
    g = r.standard_normal(10)
    _, dg = orc.rms_norm_backward(x, g, 0.1, dy)
    xh = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 0.1)
    np.testing.assert_allclose(dg, np.sum(dy * xh, axis=0), rtol=1e-13)


def test_rms_norm_backward_scale_bounds_the_gradient_and_is_reached_orthogonally():
    """The row scale of the RMSNorm backward: |dx_row| <= r |g * dy_row| (the
    last step is an orthogonal projection), with equality when g * dy is
    orthogonal to the normed row, and a ratio near zero when g * dy lies
    along it (the cancellation the scale is for)."""
    r = rng(41)
    x = r.standard_normal((7, 12))
    g = 1.0 + 0.3 * r.standard_normal(12)
    eps = 0.05
    dy = r.standard_normal((7, 12))
    dx, _ = orc.rms_norm_backward(x, g, eps, dy)
    sc = orc.rms_norm_backward_scale(x, g, eps, dy)
    assert sc.shape == (7,)
    assert np.all(np.linalg.norm(dx, axis=1) <= sc * (1 + 1e-12))
    xh = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)
    # g * dy orthogonal to xh row by row: no cancellation, equality
    w = r.standard_normal((7, 12))
    w -= xh * (np.sum(w * xh, axis=1, keepdims=True) / np.sum(xh * xh, axis=1, keepdims=True))
    dy_perp = w / g
    dx, _ = orc.rms_norm_backward(x, g, eps, dy_perp)
    np.testing.assert_allclose(np.linalg.norm(dx, axis=1), orc.rms_norm_backward_scale(x, g, eps, dy_perp),
                               rtol=1e-12)
    # g * dy along xh (eps = 0): dx vanishes while the scale does not
    dy_par = 3.0 * xh / g
    dx, _ = orc.rms_norm_backward(x, g, 0.0, dy_par)
    assert np.max(np.linalg.norm(dx, axis=1)) < 1e-12 * np.min(orc.rms_norm_backward_scale(x, g, 0.0, dy_par))
    # the scales the attention backward returns belong to its dq and dk rows
    p = rand_problem(42, B=1, T=9, Hq=2, Hkv=1, d=8, with_ve=False, with_gate=False)
    out = bwd(p, window=3, eps=1e-6, scales=True)
    for key in ("dq", "dk"):
        rows = np.linalg.norm(out[key], axis=-1)
        assert out[key + "_scale"].shape == rows.shape
        assert np.all(rows <= out[key + "_scale"] * (1 + 1e-12))


def test_against_float64_torch_autograd():
    """Independent library check: torch float64 autograd through
    F.scaled_dot_product_attention with an explicit boolean mask."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    x = rand_problem(16, B=2, T=20, Hq=4, Hkv=2, d=8, with_ve=True, with_gate=True)
    window, eps, s_ve = 5, 1e-5, 0.5
    o, lse = fwd(x, window=window, eps=eps, ve_scale=s_ve)
    g = bwd(x, window=window, eps=eps, ve_scale=s_ve)

    t = {k: (torch.tensor(v, dtype=torch.float64, requires_grad=k in
                          ("q", "k", "v", "gq", "gk", "ve"))
             if v is not None and k != "tok" else v) for k, v in x.items()}
    tok = torch.tensor(x["tok"], dtype=torch.long)
    qn = F.rms_norm(t["q"], (8,), t["gq"], eps)
    kn = F.rms_norm(t["k"], (8,), t["gk"], eps)
    ve_rows = t["ve"][tok].view(2, 20, 2, 8)
    v = t["v"] + s_ve * t["gate"].unsqueeze(-1) * ve_rows
    i = torch.arange(20)[:, None]
    j = torch.arange(20)[None, :]
    mask = (j <= i) & (i - j <= window)
    out = F.scaled_dot_product_attention(
        qn.transpose(1, 2), kn.transpose(1, 2), v.transpose(1, 2), attn_mask=mask,
        enable_gqa=True).transpose(1, 2)
    np.testing.assert_allclose(out.detach().numpy(), o, rtol=1e-12, atol=1e-12)
    (out * t["dO"]).sum().backward()
    pairs = {"q": "dq", "k": "dk", "v": "dv", "gq": "dgq", "gk": "dgk", "ve": "dve"}
    for name, gname in pairs.items():
        np.testing.assert_allclose(t[name].grad.numpy(), g[gname], rtol=1e-10, atol=1e-12)
    # LSE against logsumexp of the masked logits
    S = (qn.transpose(1, 2) @ torch.repeat_interleave(kn.transpose(1, 2), 2, dim=1)
         .transpose(-1, -2)) / math.sqrt(8)
    S = S.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(torch.logsumexp(S, -1).detach().numpy(), lse, rtol=1e-12)


def test_forward_rows_sampler_agrees_with_full_forward():
    x = rand_problem(17, B=2, T=30, Hq=4, Hkv=2, d=8, with_ve=True, with_gate=True)
    o, lse = fwd(x, window=7)
    rows = [0, 5, 29]
    for b, h in [(0, 0), (1, 3)]:
        o_r, l_r = orc.attention_forward_rows(
            x["q"], x["k"], x["v"], x["gq"], x["gk"], b=b, h=h, rows=rows, window=7,
            ve=x["ve"], tok=x["tok"], gate=x["gate"])
        np.testing.assert_allclose(o_r, o[b, rows, h], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(l_r, lse[b, h, rows], rtol=1e-13)


def test_row_chunking_does_not_change_results():
    x = rand_problem(18, B=1, T=33, Hq=2, Hkv=1, d=8)
    o1, l1 = fwd(x, window=9, row_chunk=1024)
    o2, l2 = fwd(x, window=9, row_chunk=7)
    np.testing.assert_allclose(o1, o2, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)
    g1 = bwd(x, window=9, row_chunk=1024)
    g2 = bwd(x, window=9, row_chunk=5)
    for k in ("dq", "dk", "dv", "dgq", "dgk"):
        np.testing.assert_allclose(g1[k], g2[k], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("window,causal", [(6, True), (-1, True), (4, False)])
def test_backward_samplers_against_float64_torch_autograd(window, causal):
    """The row (dq) and column (dk, dv) samplers of the backward, checked
    against torch float64 autograd through SDPA with an explicit mask, and
    against the full oracle backward."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, T, Hq, Hkv, d = 2, 23, 4, 2, 8
    x = rand_problem(19, B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, with_ve=True, with_gate=True)
    eps, s_ve = 1e-6, 0.5
    t = {k: (torch.tensor(v, dtype=torch.float64, requires_grad=k in ("q", "k", "v"))
             if v is not None and k != "tok" else v) for k, v in x.items()}
    tok = torch.tensor(x["tok"], dtype=torch.long)
    qn = F.rms_norm(t["q"], (d,), t["gq"], eps)
    kn = F.rms_norm(t["k"], (d,), t["gk"], eps)
    v = t["v"] + s_ve * t["gate"].unsqueeze(-1) * t["ve"][tok].view(B, T, Hkv, d)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    if causal:
        mask = (j <= i) & ((i - j <= window) if window >= 0 else True)
    else:
        mask = (i - j).abs() <= window
    out = F.scaled_dot_product_attention(qn.transpose(1, 2), kn.transpose(1, 2),
                                         v.transpose(1, 2), attn_mask=mask,
                                         enable_gqa=True).transpose(1, 2)
    (out * t["dO"]).sum().backward()
    full = bwd(x, window=window, causal=causal, eps=eps, ve_scale=s_ve)
    kw = dict(window=window, causal=causal, eps=eps, ve=x["ve"], tok=x["tok"], gate=x["gate"],
              ve_scale=s_ve)
    args = (x["q"], x["k"], x["v"], x["gq"], x["gk"], x["dO"])
    rows = [0, 3, 11, 22]
    for b, h in [(0, 0), (1, 3), (1, 2)]:
        dq = orc.attention_backward_rows(*args, b=b, h=h, rows=rows, **kw)
        np.testing.assert_allclose(dq, t["q"].grad[b, rows, h].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dq, full["dq"][b, rows, h], rtol=1e-10, atol=1e-12)
    cols = [0, 1, 9, 21, 22]
    for b, hk in [(0, 0), (1, 1)]:
        dk, dv = orc.attention_backward_cols(*args, b=b, hk=hk, cols=cols, row_chunk=5, **kw)
        np.testing.assert_allclose(dk, t["k"].grad[b, cols, hk].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv, t["v"].grad[b, cols, hk].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv, full["dv"][b, cols, hk], rtol=1e-10, atol=1e-12)


def test_backward_column_sampler_skips_only_rows_that_add_zero():
    """A key seen by no row of a chunk: the sampler's result does not depend
    on the chunking (rows outside every band are skipped, not dropped)."""
    x = rand_problem(20, B=1, T=40, Hq=2, Hkv=1, d=8)
    args = (x["q"], x["k"], x["v"], x["gq"], x["gk"], x["dO"])
    a = orc.attention_backward_cols(*args, b=0, hk=0, cols=[2, 30, 39], window=3, row_chunk=4)
    c = orc.attention_backward_cols(*args, b=0, hk=0, cols=[2, 30, 39], window=3, row_chunk=64)
    full = bwd(x, window=3)
    for got, ref in ((a[0], full["dk"]), (c[0], full["dk"]), (a[1], full["dv"])):
        np.testing.assert_allclose(got, ref[0, [2, 30, 39], 0], rtol=1e-11, atol=1e-13)


def test_band_mask_on_chosen_keys_is_a_column_selection():
    rows = np.arange(0, 50, 3)
    cols = [0, 7, 8, 33, 49]
    for window, causal in [(5, True), (-1, True), (4, False), (-1, False), (0, True)]:
        full = orc.band_mask(rows, 50, window, causal)
        np.testing.assert_array_equal(orc.band_mask(rows, 50, window, causal, keys=cols),
                                      full[:, cols])


# ---------------------------------------------------------------------------
# Rotary position embedding (applied to q and k before the QK-norm)
# ---------------------------------------------------------------------------

def rope_tables(T, d, base=10000.0, offset=0):
    """Standard rotary tables: angle t * base^(-2c/d) for pair c at position t."""
    half = d // 2
    inv = base ** (-np.arange(half) * 2.0 / d)
    ang = (np.arange(T) + offset)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def test_rotary_keeps_norms_and_zero_angle_is_identity():
    r = rng(40)
    x = r.standard_normal((2, 7, 3, 8))
    ang = r.uniform(-10, 10, size=(7, 4))
    y = orc.rotary(x, np.cos(ang), np.sin(ang))
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    z = orc.rotary(x, np.ones((7, 4)), np.zeros((7, 4)))
    assert np.array_equal(z, x)


def test_rotary_quarter_turn_closed_form():
    # angle pi/2 everywhere: y_c = x_{c+d/2}, y_{c+d/2} = -x_c (the reading's sign)
    r = rng(41)
    x = r.standard_normal((1, 5, 2, 6))
    y = orc.rotary(x, np.zeros((5, 3)), np.ones((5, 3)))
    np.testing.assert_array_equal(y[..., :3], x[..., 3:])
    np.testing.assert_array_equal(y[..., 3:], -x[..., :3])


def test_rotary_angles_add_and_backward_is_the_inverse_and_adjoint():
    r = rng(42)
    x = r.standard_normal((2, 6, 2, 8))
    a = r.uniform(-3, 3, size=(6, 4))
    b = r.uniform(-3, 3, size=(6, 4))
    two = orc.rotary(orc.rotary(x, np.cos(a), np.sin(a)), np.cos(b), np.sin(b))
    np.testing.assert_allclose(two, orc.rotary(x, np.cos(a + b), np.sin(a + b)), atol=1e-13)
    y = orc.rotary(x, np.cos(a), np.sin(a))
    np.testing.assert_allclose(orc.rotary_backward(y, np.cos(a), np.sin(a)), x, atol=1e-13)
    w = r.standard_normal(x.shape)
    np.testing.assert_allclose(np.sum(y * w), np.sum(x * orc.rotary_backward(w, np.cos(a), np.sin(a))),
                               rtol=1e-12)


def test_rotary_dot_products_depend_only_on_the_offset():
    # the property rotary embeddings are built for: <R_t q, R_s k> is a
    # function of t - s (standard tables), whatever the absolute positions
    r = rng(43)
    d = 16
    qv, kv = r.standard_normal(d), r.standard_normal(d)
    cos, sin = rope_tables(64, d)
    x = np.zeros((64, 1, d))
    x[:] = qv
    y = np.zeros((64, 1, d))
    y[:] = kv
    rq = orc.rotary(x, cos, sin)[:, 0]
    rk = orc.rotary(y, cos, sin)[:, 0]
    for off in (0, 3, 17):
        dots = [rq[t] @ rk[t - off] for t in range(off, 64)]
        np.testing.assert_allclose(dots, dots[0], rtol=1e-11, atol=1e-11)


def test_rotary_sampler_positions_select_table_rows():
    r = rng(44)
    x = r.standard_normal((1, 10, 2, 8))
    cos, sin = rope_tables(10, 8)
    full = orc.rotary(x, cos, sin)
    rows = np.array([7, 2, 9])
    part = orc.rotary(x[0, rows][None], cos, sin, positions=rows)
    np.testing.assert_allclose(part[0], full[0, rows], atol=1e-15)


def test_identity_rope_tables_change_nothing():
    x = rand_problem(45, B=1, T=10, Hq=2, Hkv=1, d=8, with_ve=True)
    ident = (np.ones((10, 4)), np.zeros((10, 4)))
    o0, l0 = fwd(x, window=4)
    o1, l1 = fwd(x, window=4, rope=ident)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0, g1 = bwd(x, window=4), bwd(x, window=4, rope=ident)
    for k in ("dq", "dk", "dv", "dgq", "dgk", "dve"):
        np.testing.assert_allclose(g1[k], g0[k], rtol=0, atol=1e-15)


def test_rope_is_undone_by_scale_free_rotation_of_both_sides():
    # the same rotation at every position leaves all q.k products, hence the
    # whole attention, unchanged (a global rotation is an isometry)
    x = rand_problem(46, B=1, T=9, Hq=2, Hkv=1, d=8, with_gain=False)
    ang = np.tile(np.array([[0.3, -1.1, 2.0, 0.7]]), (9, 1))
    o0, _ = fwd(x, window=-1)
    o1, _ = fwd(x, window=-1, rope=(np.cos(ang), np.sin(ang)))
    np.testing.assert_allclose(o1, o0, atol=1e-12)


@pytest.mark.parametrize("window,causal", [(-1, True), (3, True)])
def test_backward_with_rope_matches_central_finite_differences(window, causal):
    x = rand_problem(47, B=1, T=8, Hq=2, Hkv=1, d=6, with_ve=True, with_gate=True, vocab=5)
    cos, sin = rope_tables(8, 6, base=3.0)
    kw = dict(window=window, causal=causal, eps=1e-4, ve_scale=0.7, rope=(cos, sin))
    g = bwd(x, **kw)
    h = 1e-6
    for name, gname in {"q": "dq", "k": "dk", "gq": "dgq", "gk": "dgk"}.items():
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = base[idx]
            base[idx] = old + h
            lp = loss(x, **kw)
            base[idx] = old - h
            lm = loss(x, **kw)
            base[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(g[gname] - num) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-6, (name, err)


def test_rope_samplers_agree_with_full_backward():
    x = rand_problem(48, B=2, T=16, Hq=4, Hkv=2, d=8, with_ve=True, with_gate=True)
    cos, sin = rope_tables(16, 8)
    kw = dict(window=5, eps=1e-5, ve_scale=0.5, rope=(cos, sin))
    o, lse = fwd(x, **kw)
    g = bwd(x, **kw)
    rows = np.array([0, 6, 15])
    for b in range(2):
        for h in range(4):
            ro, rl = orc.attention_forward_rows(x["q"], x["k"], x["v"], x["gq"], x["gk"], b=b, h=h,
                                                rows=rows, ve=x["ve"], tok=x["tok"], gate=x["gate"],
                                                **kw)
            np.testing.assert_allclose(ro, o[b, rows, h], atol=1e-12)
            dq = orc.attention_backward_rows(x["q"], x["k"], x["v"], x["gq"], x["gk"], x["dO"], b=b, h=h,
                                             rows=rows, ve=x["ve"], tok=x["tok"], gate=x["gate"], **kw)
            np.testing.assert_allclose(dq, g["dq"][b, rows, h], atol=1e-12)
        for hk in range(2):
            dk, dv = orc.attention_backward_cols(x["q"], x["k"], x["v"], x["gq"], x["gk"], x["dO"], b=b,
                                                 hk=hk, cols=rows, ve=x["ve"], tok=x["tok"],
                                                 gate=x["gate"], **kw)
            np.testing.assert_allclose(dk, g["dk"][b, rows, hk], atol=1e-12)
            np.testing.assert_allclose(dv, g["dv"][b, rows, hk], atol=1e-12)


# ---------------------------------------------------------------------------
# Learned value-embedding gate: gate = 2 sigmoid(W x[:C]) per kv head
# ---------------------------------------------------------------------------

def gate_inputs(seed, B, T, Hkv, C=5, scale=0.7):
    r = rng(seed)
    return r.standard_normal((B, T, C)), scale * r.standard_normal((Hkv, C))


def test_learned_gate_at_initialisation_is_one():
    # the Guide: the gate weight starts at zero, so 2 * sigmoid(0) = 1 and the
    # value-embedding path starts as the identity mix
    x = rand_problem(50, B=2, T=7, Hq=2, Hkv=1, d=8, with_ve=True)
    gx, _ = gate_inputs(51, 2, 7, 1)
    w0 = np.zeros((1, gx.shape[-1]))
    assert np.array_equal(orc.learned_gate(gx, w0), np.ones((2, 7, 1)))
    o0, l0 = fwd(x, window=3)
    o1, l1 = fwd(x, window=3, gate_x=gx, gate_w=w0)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_learned_gate_range_and_saturation():
    gx, w = gate_inputs(52, 1, 9, 2, scale=3.0)
    g = orc.learned_gate(gx, w)
    assert np.all(g > 0) and np.all(g < 2)
    # symmetry of the sigmoid: gate(-z) = 2 - gate(z)
    np.testing.assert_allclose(orc.learned_gate(-gx, w), 2.0 - g, rtol=0, atol=1e-15)
    # far in the tails the gate is 0 or 2 and its gradient vanishes
    big = np.array([[[200.0]]]), np.array([[1.0]])
    assert orc.learned_gate(*big)[0, 0, 0] == 2.0
    dx, dw = orc.learned_gate_backward(big[0], big[1], np.ones((1, 1, 1)))
    assert dx[0, 0, 0] == 0.0 and dw[0, 0] == 0.0
    # at z = 0 the slope of 2 sigmoid is 1/2
    dx, dw = orc.learned_gate_backward(np.array([[[0.0]]]), np.array([[0.3]]), np.ones((1, 1, 1)))
    assert dx[0, 0, 0] == 0.5 * 0.3 and dw[0, 0] == 0.0


def test_learned_gate_equals_the_same_gate_given_as_input():
    x = rand_problem(53, B=2, T=8, Hq=4, Hkv=2, d=8, with_ve=True)
    gx, w = gate_inputs(54, 2, 8, 2)
    kw = dict(window=4, eps=1e-5, ve_scale=0.6)
    o0, _ = orc.attention_forward(x["q"], x["k"], x["v"], x["gq"], x["gk"], ve=x["ve"], tok=x["tok"],
                                  gate=orc.learned_gate(gx, w), **kw)
    o1, _ = fwd(x, gate_x=gx, gate_w=w, **kw)
    assert np.array_equal(o0, o1)


def test_backward_with_learned_gate_matches_central_finite_differences():
    x = rand_problem(55, B=1, T=7, Hq=2, Hkv=2, d=4, with_ve=True, vocab=5)
    gx, w = gate_inputs(56, 1, 7, 2, C=3)
    kw = dict(window=3, causal=True, eps=1e-4, ve_scale=0.8)
    g = bwd(x, gate_x=gx, gate_w=w, **kw)
    h = 1e-6

    def lossf():
        o, _ = fwd(x, gate_x=gx, gate_w=w, **kw)
        return float(np.sum(o * x["dO"]))

    for arr, gname in ((gx, "dgate_x"), (w, "dgate_w"), (x["v"], "dv"), (x["ve"], "dve")):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = lossf()
            arr[idx] = old - h
            lm = lossf()
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(g[gname] - num) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-6, (gname, err)
