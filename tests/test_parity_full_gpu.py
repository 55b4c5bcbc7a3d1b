"""GPU parity at the full sizes of the benchmark configurations, through the
same C-ABI calls the benchmark makes (forward, then the three backward stages
one call at a time, prologue outputs reused).

Per-sequence tensors (o, lse, dq, dk, dv) are compared element by element
with the float64 oracle on whole batch elements where the oracle finishes in
seconds (T = 2048), and on sampled query rows and key columns at T = 16384
and at the largest T the library accepts. The shared-parameter gradients
(dgq, dgk, dVE) sum over the batch: they are compared with the oracle summed
over every batch element for the S layer, and elsewhere with the oracle on
single batch elements plus the identity "gradient of the batch = sum of the
gradients of its elements", which holds at any size.

Tolerance, 2e-2 for the bf16 library, on three measures of every compared
tensor (gpu_helpers.errors): the Frobenius norm of the difference over that
of the oracle over the compared set; the same ratio for every row (a head row
of d channels of o, dq, dk, dv, against the larger of its own norm and twice
the rows' root mean square norm, gpu_helpers.ROW_FLOOR); and every element of
lse and of the gain gradients, in the same way. The largest absolute error of each tensor is
recorded and printed at the end of the session.
"""

import numpy as np
import pytest
import torch

import oracle
import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300.inputs import (L_LAYER, LONG_L, LONG_S, S_LAYER, Problem,
                                                as_f64, make_inputs)
from gpu_helpers import (TOL, batch_slice, check, compare, rel_err, rope_tables, run_oracle,
                         run_staged)

pytestmark = pytest.mark.gpu

TOL_BF16 = TOL["bf16"]
# batch-additivity of fp32 gradient sums: equal up to the order of fp32 additions
TOL_SUM = 1e-4

# (problem, layer index whose seeded inputs are drawn) of the T=2048 configurations:
# the S and L layers, and the two kinds of value-embedding layers of the 8-layer
# SSSL stack (layer 1: window 1024 + VE; layer 3: full causal + VE).
T2048 = {
    "s_layer": (S_LAYER, 0),
    "l_layer": (L_LAYER, 0),
    "stack_layer1_s_ve": (S_LAYER.replace(ve=True), 1),
    "stack_layer3_l_ve": (L_LAYER.replace(ve=True), 3),
    # the Guide's default n_kv_head = n_head (plain multi-head attention),
    # window 1024 with value embeddings, on 4 sequences
    "mha_s_layer_ve": (S_LAYER.replace(B=4, Hkv=6, ve=True), 1),
}


def _slice_checks(p, x, got, slices, rope=None):
    for b in slices:
        ref = run_oracle(p.replace(B=1), batch_slice(x, b), rope=rope)
        compare({k: got[k][b:b + 1] for k in ("o", "dq", "dk", "dv")} | {"lse": got["lse"][b:b + 1]},
                ref, TOL_BF16, keys=("o", "lse", "dq", "dk", "dv"))


def _additivity(p, x, got):
    """Shared-parameter gradients of the batch against the sum of the
    library's per-element results; returns the per-element results."""
    per = [run_staged(p.replace(B=1), batch_slice(x, b)) for b in range(p.B)]
    for r in per:
        assert r["status"] == swa.SWA_OK
    for k in ("dgq", "dgk", "dve"):
        if got[k] is None:
            continue
        total = sum(r[k].double() for r in per)
        assert rel_err(got[k], as_f64(total)) <= TOL_SUM, k
    return per


@pytest.mark.parametrize("name", list(T2048))
def test_full_size_t2048(name):
    p, layer = T2048[name]
    x = make_inputs(p, layer=layer)
    got = run_staged(p, x)
    assert got["status"] == swa.SWA_OK
    _slice_checks(p, x, got, slices=(0, p.B - 1))
    per = _additivity(p, x, got)
    # the per-element shared gradients of the checked elements against the oracle
    for b in (0, p.B - 1):
        ref = run_oracle(p.replace(B=1), batch_slice(x, b))
        compare(per[b], ref, TOL_BF16, keys=("dgq", "dgk", "dve"))


def test_full_size_s_layer_gain_gradients_over_the_whole_batch():
    """dgq and dgk of the S layer against the oracle summed over all 16
    batch elements (the benchmark's headline configuration, no sampling)."""
    p = S_LAYER
    x = make_inputs(p, layer=0)
    got = run_staged(p, x)
    sums = {"dgq": 0.0, "dgk": 0.0}
    for b in range(p.B):
        ref = run_oracle(p.replace(B=1), batch_slice(x, b))
        for k in sums:
            sums[k] = sums[k] + ref[k]
    for k, r in sums.items():
        check(k, got[k], r, TOL_BF16)


def _rows(T, seed):
    r = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, T // 2 - 1, T // 2, T // 2 + 1, T - 129, T - 128, T - 1]
    return np.unique(np.concatenate([fixed, r.integers(0, T, 21)]))


def _sampled(p, x, got, heads, kv_heads, cols, row_chunk=512):
    f = {k: as_f64(t) for k, t in x.items()}
    tok = x["tok"].numpy() if x["tok"] is not None else None
    kw = dict(window=p.window, causal=p.causal, eps=p.eps, ve=f["ve"], tok=tok,
              gate=f.get("gate"), ve_scale=p.ve_scale)
    args = (f["q"], f["k"], f["v"], f["gq"], f["gk"], f["dO"])
    rows = _rows(p.T, 5)
    acc = {k: ([], []) for k in ("o", "lse", "dq", "dk", "dv")}
    scale = {"dq": [], "dk": []}
    for b in range(p.B):
        for h in heads:
            o_r, l_r = oracle.attention_forward_rows(*args[:5], b=b, h=h, rows=rows, **kw)
            dq_r, dq_s = oracle.attention_backward_rows(*args, b=b, h=h, rows=rows, with_scale=True,
                                                        **kw)
            scale["dq"].append(dq_s)
            for k, mine, ref in (("o", got["o"][b, rows, h], o_r),
                                 ("lse", got["lse"][b, h, rows], l_r),
                                 ("dq", got["dq"][b, rows, h], dq_r)):
                assert tuple(mine.shape) == np.shape(ref), (k, tuple(mine.shape), np.shape(ref))
                acc[k][0].append(as_f64(mine))
                acc[k][1].append(np.asarray(ref))
        for hk in kv_heads:
            dk_c, dv_c, dk_s = oracle.attention_backward_cols(*args, b=b, hk=hk, cols=cols,
                                                              row_chunk=row_chunk, with_scale=True,
                                                              **kw)
            scale["dk"].append(dk_s)
            for k, mine, ref in (("dk", got["dk"][b, cols, hk], dk_c),
                                 ("dv", got["dv"][b, cols, hk], dv_c)):
                assert tuple(mine.shape) == np.shape(ref), (k, tuple(mine.shape), np.shape(ref))
                acc[k][0].append(as_f64(mine))
                acc[k][1].append(np.asarray(ref))
    for k, (a, r) in acc.items():
        rs = np.concatenate(scale[k]) if k in scale else None
        check(k, np.concatenate(a), np.concatenate(r), TOL_BF16, row_scale=rs)


LONG = {"long_context_s": (LONG_S, 0), "long_context_l": (LONG_L, 3)}


@pytest.mark.parametrize("name", list(LONG))
def test_full_size_long_context_sampled(name):
    """B=2, T=16384, Hq=16, Hkv=4: sampled query rows (o, lse, dq) of three
    heads of each sequence, sampled key columns (dk, dv) of two kv heads, and
    the gain gradients by batch additivity."""
    p, layer = LONG[name]
    x = make_inputs(p, layer=layer)
    got = run_staged(p, x)
    assert got["status"] == swa.SWA_OK
    T = p.T
    _sampled(p, x, got, heads=(0, 5, 15), kv_heads=(0, 3),
             cols=np.array([T - 513, T - 200, T - 129, T - 128, T - 2, T - 1]))
    _additivity(p, x, got)


def test_maximum_batch_times_heads():
    """B * Hq = 65534, the largest the row-wise kernels' grids take (the ABI
    refuses more), on short sequences: whole-problem oracle comparison."""
    p = Problem(B=32767, T=8, Hq=2, Hkv=1, d=64, window=-1, gain_std=0.1)
    x = make_inputs(p, layer=0)
    x["gate"] = None
    ref = run_oracle(p, x)
    # the fp32 build gets the same (bf16-representable) values in fp32 tensors
    x32 = {k: (t.float() if t is not None and t.is_floating_point() else t) for k, t in x.items()}
    for kind, xi in (("bf16", x), ("fp32", x32)):
        got = run_staged(p, xi)
        assert got["status"] == swa.SWA_OK
        compare(got, ref, TOL[kind])


def test_maximum_sequence_length_sampled():
    """T = 2^22, the longest sequence the ABI accepts, with a 64-key causal
    window. Row i of the output (and of dq) depends only on positions
    [i - 64, i], and key column j (dk, dv) only on rows [j, j + 64] and hence
    on positions [j - 64, j + 64]; so the oracle run on a 512-position slice
    of the inputs gives the exact values at the rows and columns whose whole
    dependence lies in the slice. Three slices: the start, the middle and the
    end of the sequence. (The gain gradients sum over all 4M rows and are not
    sampled at this size.)"""
    T, W, L = 1 << 22, 64, 512
    p = Problem(B=1, T=T, Hq=2, Hkv=1, d=64, window=W, gain_std=0.1)
    dev = torch.device("cuda:0")
    x = make_inputs(p, layer=0, device=dev)
    got = run_staged(p, x, dev)
    assert got["status"] == swa.SWA_OK
    acc = {k: ([], []) for k in ("o", "lse", "dq", "dk", "dv")}
    scale = {"dq": [], "dk": []}
    for s0 in (0, T // 2 - L // 2, T - L):
        sl = slice(s0, s0 + L)
        xs = {k: (None if t is None else (t[:, sl] if k in ("q", "k", "v", "dO") else t).cpu())
              for k, t in x.items()}
        ref = run_oracle(p.replace(T=L), xs)
        ref["dq_scale"] = ref["dq_scale"][0]        # [L, Hq]
        ref["dk_scale"] = ref["dk_scale"][0]        # [L, Hkv]
        lo = 0 if s0 == 0 else W                       # rows with their whole band inside
        rows = np.arange(lo, L)
        c_hi = L if s0 + L == T else L - W             # columns with all their rows inside
        cols = np.arange(lo, c_hi)
        for k, mine, r in (("o", got["o"][0, s0 + rows], ref["o"][0, rows]),
                           ("lse", got["lse"][0][:, s0 + rows], ref["lse"][0][:, rows]),
                           ("dq", got["dq"][0, s0 + rows], ref["dq"][0, rows]),
                           ("dk", got["dk"][0, s0 + cols], ref["dk"][0, cols]),
                           ("dv", got["dv"][0, s0 + cols], ref["dv"][0, cols])):
            assert tuple(mine.shape) == np.shape(r), (k, tuple(mine.shape), np.shape(r))
            # rows of d channels (o, dq: [rows, Hq, d]; dk, dv: [cols, Hkv, d]);
            # lse [Hq, rows] element by element
            acc[k][0].append(as_f64(mine).reshape(-1) if k == "lse" else as_f64(mine).reshape(-1, p.d))
            acc[k][1].append(np.reshape(r, -1) if k == "lse" else np.reshape(r, (-1, p.d)))
        scale["dq"].append(ref["dq_scale"][rows].reshape(-1))
        scale["dk"].append(ref["dk_scale"][cols].reshape(-1))
    for k, (a, r) in acc.items():
        rs = np.concatenate(scale[k]) if k in scale else None
        check(k, np.concatenate(a), np.concatenate(r), TOL_BF16, row_scale=rs)


def test_full_size_value_embedding_s_layer_with_rope():
    """Layer 1 of the stack (window 1024, value embedding) at B=16, T=2048
    with standard rotary tables through the _rope calls: two whole batch
    elements against the oracle, shared gradients by batch additivity."""
    p, layer = T2048["stack_layer1_s_ve"]
    x = make_inputs(p, layer=layer)
    rope = rope_tables(p.T, p.d)
    got = run_staged(p, x, rope=rope)
    assert got["status"] == swa.SWA_OK
    _slice_checks(p, x, got, (0, p.B - 1), rope=rope)
    per = [run_staged(p.replace(B=1), batch_slice(x, b), rope=rope) for b in range(p.B)]
    for k in ("dgq", "dgk", "dve"):
        total = sum(r[k].double() for r in per)
        assert rel_err(got[k], as_f64(total)) <= TOL_SUM, k
