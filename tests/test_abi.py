"""Host-side checks of the C ABI: both libraries load, export every function
the header declares, and reject bad arguments with the documented status
before touching the GPU. No test here launches a kernel."""

import ctypes
import os
import re

import pytest

import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300 import build as swa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swa_attn.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "sssl_8_layers.txt")

KINDS = ["bf16", "fp32"]


@pytest.fixture(scope="session", autouse=True)
def built_libraries():
    swa_build.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_[a-z_0-9]+)\s*\(", text)))


@pytest.mark.parametrize("kind", KINDS)
def test_library_loads_and_exports_every_declared_symbol(kind):
    lib = swa.load(kind)
    names = declared_functions()
    assert "swa_attn_fwd" in names and "swa_attn_bwd" in names
    for name in names:
        assert hasattr(lib, name), name
    info = swa.swa_build_info(kind)
    assert ("bf16" in info) == (kind == "bf16")


@pytest.mark.parametrize("kind", KINDS)
def test_layer_schedule_matches_pages_example(kind):
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    for layer, _, window, ve in rows:
        assert swa.swa_sssl_window(int(layer), 8, "SSSL", 2048, kind) == int(window)
        assert swa.swa_has_ve(int(layer), 8, kind) == int(ve)


def test_layer_schedule_helpers_reject_bad_arguments():
    assert swa.swa_sssl_window(0, 8, "SXSL", 2048) == -2
    assert swa.swa_sssl_window(8, 8, "SSSL", 2048) == -2
    assert swa.swa_sssl_window(-1, 8, "SSSL", 2048) == -2
    assert swa.load("bf16").swa_sssl_window(0, 8, None, 2048) == -2
    assert swa.swa_sssl_window(0, 8, "", 2048) == -2
    assert swa.swa_has_ve(3, 0) == -1
    assert swa.swa_has_ve(-1, 4) == -1
    # last layer forced global even for an all-local pattern
    assert swa.swa_sssl_window(5, 6, "S", 100) == -1
    assert swa.swa_sssl_window(4, 6, "S", 101) == 50


@pytest.mark.parametrize("pattern", ["L", "S", "SL", "SSL", "SSSL", "SSSSL", "LSSS", "SLSL"])
@pytest.mark.parametrize("n_layer", [1, 2, 5, 8, 12])
def test_layer_schedule_agrees_with_the_oracle_for_other_window_patterns(pattern, n_layer):
    # WINDOW_PATTERN is the script's main tuning lever (the Guide, §3.4 and the
    # techniques table): the library's schedule helpers and the oracle's,
    # written independently, agree on every layer of every pattern
    import oracle
    for T in (2048, 777):
        for layer in range(n_layer):
            assert swa.swa_sssl_window(layer, n_layer, pattern, T) == oracle.sssl_window(layer, n_layer, pattern, T)
            assert swa.swa_has_ve(layer, n_layer) == int(oracle.has_ve(layer, n_layer))


def test_strerror_covers_every_status():
    texts = {swa.swa_strerror(s) for s in range(7)}
    assert len(texts) == 7
    assert "unknown" in swa.swa_strerror(99)


def params(**kw):
    base = dict(B=2, T=300, Hq=4, Hkv=2, d=128, window=150, causal=True, softmax_scale=0.0,
                eps=1e-6, ve_scale=0.5, vocab=0)
    base.update(kw)
    return swa.make_params(**base)


@pytest.mark.parametrize("kind", KINDS)
def test_workspace_size(kind):
    p = params()
    fwd = swa.swa_attn_workspace_size(p, 0, kind)
    bwd = swa.swa_attn_workspace_size(p, 1, kind)
    es = 2 if kind == "bf16" else 4
    B, T, Hq, Hkv, d = 2, 300, 4, 2, 128
    assert fwd >= 256 + B * T * d * (Hq + 2 * Hkv) * es + 4 * B * T * (Hq + Hkv)
    assert bwd >= fwd + 4 * B * T * d * (Hq + 2 * Hkv)
    assert fwd % 256 == 0 and bwd % 256 == 0
    assert swa.swa_attn_workspace_size(params(d=96), 0, kind) == 0
    assert swa.swa_attn_workspace_size(params(Hq=3), 0, kind) == 0


# Fake, never-dereferenced device addresses: argument checks run before any
# CUDA call, so these are safe on a machine without a GPU.
A = 1 << 20          # 16-byte aligned
MIS = A + 8          # not 16-byte aligned


def fwd_call(p, kind="bf16", ws_bytes=1 << 40, **over):
    args = dict(q=A, k=A, v=A, gq=None, gk=None, ve=None, tok=None, gate=None, o=A, lse=A,
                ws=A, flags=0)
    args.update(over)
    lib = swa.load(kind)
    return lib.swa_attn_fwd(ctypes.byref(p), args["q"], args["k"], args["v"], args["gq"],
                            args["gk"], args["ve"], args["tok"], args["gate"], args["o"],
                            args["lse"], args["ws"], ws_bytes, args["flags"], None)


def bwd_call(p, kind="bf16", ws_bytes=1 << 40, **over):
    args = dict(q=A, k=A, v=A, gq=None, gk=None, ve=None, tok=None, gate=None, o=A, lse=A,
                dO=A, dq=A, dk=A, dv=A, dgq=None, dgk=None, dve=None, ws=A, flags=0)
    args.update(over)
    lib = swa.load(kind)
    return lib.swa_attn_bwd(ctypes.byref(p), *[args[k] for k in (
        "q", "k", "v", "gq", "gk", "ve", "tok", "gate", "o", "lse", "dO", "dq", "dk", "dv", "dgq",
        "dgk", "dve", "ws")], ws_bytes, args["flags"], None)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("bad,expect", [
    (dict(Hq=3, Hkv=2), swa.SWA_ERR_INVALID_ARG),
    (dict(Hkv=0), swa.SWA_ERR_INVALID_ARG),
    (dict(B=-1), swa.SWA_ERR_INVALID_ARG),
    (dict(T=-5), swa.SWA_ERR_INVALID_ARG),
    (dict(window=-2), swa.SWA_ERR_INVALID_ARG),
    (dict(d=96), swa.SWA_ERR_UNSUPPORTED),
    (dict(d=256), swa.SWA_ERR_UNSUPPORTED),
    (dict(eps=-1.0), swa.SWA_ERR_INVALID_ARG),
    (dict(softmax_scale=-0.1), swa.SWA_ERR_INVALID_ARG),
    (dict(softmax_scale=float("nan")), swa.SWA_ERR_INVALID_ARG),
    (dict(ve_scale=float("inf")), swa.SWA_ERR_INVALID_ARG),
    (dict(T=(1 << 22) + 1), swa.SWA_ERR_UNSUPPORTED),
])
def test_bad_params_are_rejected(kind, bad, expect):
    p = params(**bad)
    assert fwd_call(p, kind) == expect
    assert bwd_call(p, kind) == expect


@pytest.mark.parametrize("kind", KINDS)
def test_bad_pointers_flags_and_workspace_are_rejected(kind):
    p = params()
    lib = swa.load(kind)
    assert lib.swa_attn_fwd(None, A, A, A, None, None, None, None, None, A, A, A, 1 << 40, 0,
                            None) == swa.SWA_ERR_INVALID_ARG
    for name in ("q", "k", "v", "o", "lse", "ws"):
        assert fwd_call(p, kind, **{name: None}) == swa.SWA_ERR_INVALID_ARG, name
    for name in ("q", "k", "v", "o"):
        assert fwd_call(p, kind, **{name: MIS}) == swa.SWA_ERR_INVALID_ARG, name
    assert fwd_call(p, kind, ws=A + 16) == swa.SWA_ERR_INVALID_ARG       # workspace 256-aligned
    assert fwd_call(p, kind, flags=2) == swa.SWA_ERR_INVALID_ARG
    need = swa.swa_attn_workspace_size(p, 0, kind)
    assert fwd_call(p, kind, ws_bytes=need - 1) == swa.SWA_ERR_WORKSPACE
    # value embeddings need token ids and a vocabulary size
    assert fwd_call(params(vocab=8), kind, ve=A) == swa.SWA_ERR_INVALID_ARG
    assert fwd_call(params(vocab=0), kind, ve=A, tok=A) == swa.SWA_ERR_INVALID_ARG
    assert fwd_call(params(vocab=8), kind, ve=MIS, tok=A) == swa.SWA_ERR_INVALID_ARG
    # backward
    for name in ("q", "k", "v", "o", "lse", "dO", "dq", "dk", "dv", "ws"):
        assert bwd_call(p, kind, **{name: None}) == swa.SWA_ERR_INVALID_ARG, name
    for name in ("dO", "dq", "dk", "dv"):
        assert bwd_call(p, kind, **{name: MIS}) == swa.SWA_ERR_INVALID_ARG, name
    assert bwd_call(p, kind, flags=16) == swa.SWA_ERR_INVALID_ARG
    need_b = swa.swa_attn_workspace_size(p, 1, kind)
    assert bwd_call(p, kind, ws_bytes=need_b - 1) == swa.SWA_ERR_WORKSPACE
    assert bwd_call(p, kind, ws_bytes=need) == swa.SWA_ERR_WORKSPACE  # forward-sized only


@pytest.mark.parametrize("kind", KINDS)
def test_empty_forward_is_a_no_op(kind):
    # B == 0 or T == 0: valid, nothing launched (so it runs without a GPU)
    assert fwd_call(params(B=0), kind) == swa.SWA_OK
    assert fwd_call(params(T=0), kind) == swa.SWA_OK


def test_binding_names_mirror_the_c_abi():
    for name in declared_functions():
        assert hasattr(swa, name), name


def fwd_ex_call(p, ex, kind="bf16", **over):
    args = dict(q=A, k=A, v=A, gq=None, gk=None, ve=None, tok=None, gate=None, o=A, lse=A, ws=A)
    args.update(over)
    lib = swa.load(kind)
    ep = None if ex is None else ctypes.byref(ex)
    return lib.swa_attn_fwd_ex(ctypes.byref(p), ep, args["q"], args["k"], args["v"], args["gq"],
                               args["gk"], args["ve"], args["tok"], args["gate"], args["o"],
                               args["lse"], args["ws"], 1 << 40, 0, None)


def bwd_ex_call(p, ex, kind="bf16", **over):
    args = dict(q=A, k=A, v=A, gq=None, gk=None, ve=None, tok=None, gate=None, o=A, lse=A,
                dO=A, dq=A, dk=A, dv=A, dgq=None, dgk=None, dve=None, ws=A)
    args.update(over)
    lib = swa.load(kind)
    ep = None if ex is None else ctypes.byref(ex)
    return lib.swa_attn_bwd_ex(ctypes.byref(p), ep, args["q"], args["k"], args["v"], args["gq"],
                               args["gk"], args["ve"], args["tok"], args["gate"], args["o"],
                               args["lse"], args["dO"], args["dq"], args["dk"], args["dv"],
                               args["dgq"], args["dgk"], args["dve"], args["ws"], 1 << 40, 0, None)


def extras(**kw):
    e = swa.swa_extras()
    for k, v in kw.items():
        setattr(e, k, v)
    return e


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("bad", [
    dict(rope_cos=A, rope_rows=1 << 20),                       # one table only
    dict(rope_cos=A, rope_sin=A, rope_rows=63),                # fewer rows than T
    dict(rope_cos=MIS, rope_sin=A, rope_rows=1 << 20),         # not 16-byte aligned
    dict(gate_w=A, gate_x=None, gate_ch=32, gate_x_stride=32), # no gate input
    dict(gate_w=A, gate_x=A, gate_ch=0, gate_x_stride=32),
    dict(gate_w=A, gate_x=A, gate_ch=33, gate_x_stride=33),
    dict(gate_w=A, gate_x=A, gate_ch=32, gate_x_stride=16),    # rows shorter than the channels
])
def test_bad_extras_are_rejected(kind, bad):
    p = params(T=64)
    assert fwd_ex_call(p, extras(**bad), kind) == swa.SWA_ERR_INVALID_ARG
    assert bwd_ex_call(p, extras(**bad), kind) == swa.SWA_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", KINDS)
def test_learned_gate_excludes_a_given_gate_and_large_head_counts(kind):
    gate = dict(gate_w=A, gate_x=A, gate_ch=32, gate_x_stride=32)
    assert fwd_ex_call(params(T=64), extras(**gate), kind, gate=A) == swa.SWA_ERR_INVALID_ARG
    assert fwd_ex_call(params(T=64, Hq=33, Hkv=33), extras(**gate), kind) == swa.SWA_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", KINDS)
def test_null_extras_behave_like_the_plain_calls(kind):
    assert fwd_ex_call(params(B=0), None, kind) == swa.SWA_OK
    assert fwd_ex_call(params(B=0), extras(), kind) == swa.SWA_OK
    assert fwd_ex_call(params(), None, kind, q=None) == swa.SWA_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# Block calls (pre-norm, projections, residual around the attention)
# ---------------------------------------------------------------------------

def block_weights(C=512, wq=A, wk=A, wv=A, wo=A):
    return swa.swa_block_weights(C, wq, wk, wv, wo)


def block_fwd_call(p, w, ex=None, kind="bf16", ws_bytes=1 << 40, x=A, out=A, ws=A, ve=None,
                   tok=None):
    lib = swa.load(kind)
    ep = None if ex is None else ctypes.byref(ex)
    wp = None if w is None else ctypes.byref(w)
    return lib.swa_block_fwd(ctypes.byref(p), ep, wp, x, None, None, ve, tok, out, ws, ws_bytes,
                             None)


def block_bwd_call(p, w, ex=None, kind="bf16", ws_bytes=1 << 40, x=A, dout=A, dx=A, ws=A, ve=None,
                   tok=None):
    lib = swa.load(kind)
    ep = None if ex is None else ctypes.byref(ex)
    wp = None if w is None else ctypes.byref(w)
    return lib.swa_block_bwd(ctypes.byref(p), ep, wp, x, None, None, ve, tok, dout, dx, None,
                             None, None, None, None, None, None, ws, ws_bytes, None)


@pytest.mark.parametrize("kind", KINDS)
def test_block_workspace_size(kind):
    p = params()
    attn = swa.swa_attn_workspace_size(p, 1, kind)
    fwd = swa.swa_block_workspace_size(p, 512, 0, kind)
    bwd = swa.swa_block_workspace_size(p, 512, 1, kind)
    es = 2 if kind == "bf16" else 4
    B, T, Hq, Hkv, d, C = 2, 300, 4, 2, 128, 512
    # the attention's backward workspace, xn, q, k, v, o, lse, rstd and the
    # rotary tables transposed (fp32 [2][d/2][T]); no GEMM scratch
    fixed = B * T * (C + 2 * Hq * d + 2 * Hkv * d) * es + 4 * B * T * (Hq + 1) + 4 * T * d
    assert attn + fixed <= fwd < attn + fixed + 9 * 256
    # + dO, dq, dk, dv, dxn (fp32), the gate's channel gradients (fp32)
    assert bwd >= fwd + B * T * (2 * Hq * d + 2 * Hkv * d) * es + 4 * B * T * (C + 32)
    for C_bad in (0, 4, 12, 1 << 17):
        assert swa.swa_block_workspace_size(p, C_bad, 0, kind) == 0
    assert swa.swa_block_workspace_size(params(d=96), 512, 0, kind) == 0


@pytest.mark.parametrize("kind", KINDS)
def test_block_calls_reject_bad_arguments(kind):
    p = params()
    for call in (block_fwd_call, block_bwd_call):
        assert call(p, None, kind=kind) == swa.SWA_ERR_INVALID_ARG
        assert call(p, block_weights(C=12), kind=kind) == swa.SWA_ERR_INVALID_ARG
        for name in ("wq", "wk", "wv", "wo"):
            assert call(p, block_weights(**{name: None}), kind=kind) == swa.SWA_ERR_INVALID_ARG
            assert call(p, block_weights(**{name: MIS}), kind=kind) == swa.SWA_ERR_INVALID_ARG
        assert call(p, block_weights(), kind=kind, x=MIS) == swa.SWA_ERR_INVALID_ARG
        assert call(p, block_weights(), kind=kind, ws=A + 16) == swa.SWA_ERR_INVALID_ARG
        assert call(params(d=96), block_weights(), kind=kind) == swa.SWA_ERR_UNSUPPORTED
        # the block gives the gate its input itself
        assert call(p, block_weights(), extras(gate_w=A, gate_x=A, gate_ch=8, gate_x_stride=8),
                    kind=kind) == swa.SWA_ERR_INVALID_ARG
        assert call(p, block_weights(C=16), extras(gate_w=A, gate_ch=32), kind=kind) == \
            swa.SWA_ERR_INVALID_ARG
    # the attention's own argument checks run before the block launches anything
    for call in (block_fwd_call, block_bwd_call):
        assert call(params(T=64), block_weights(), extras(rope_cos=A, rope_sin=A, rope_rows=63),
                    kind=kind) == swa.SWA_ERR_INVALID_ARG
        assert call(params(T=64), block_weights(), extras(rope_cos=A, rope_rows=64),
                    kind=kind) == swa.SWA_ERR_INVALID_ARG
        assert call(params(vocab=8), block_weights(), kind=kind, ve=A) == swa.SWA_ERR_INVALID_ARG
        assert call(params(vocab=0), block_weights(), kind=kind, ve=A, tok=A) == \
            swa.SWA_ERR_INVALID_ARG
        assert call(params(Hq=66, Hkv=33), block_weights(), extras(gate_w=A, gate_ch=8),
                    kind=kind) == swa.SWA_ERR_INVALID_ARG
    assert block_fwd_call(p, block_weights(), kind=kind, out=None) == swa.SWA_ERR_INVALID_ARG
    assert block_bwd_call(p, block_weights(), kind=kind, dx=MIS) == swa.SWA_ERR_INVALID_ARG
    assert block_bwd_call(p, block_weights(), extras(d_gate_x=A), kind=kind) == swa.SWA_ERR_INVALID_ARG
    need = swa.swa_block_workspace_size(p, 512, 0, kind)
    need_b = swa.swa_block_workspace_size(p, 512, 1, kind)
    assert block_fwd_call(p, block_weights(), kind=kind, ws_bytes=need - 1) == swa.SWA_ERR_WORKSPACE
    assert block_bwd_call(p, block_weights(), kind=kind, ws_bytes=need) == swa.SWA_ERR_WORKSPACE
    assert block_bwd_call(p, block_weights(), kind=kind, ws_bytes=need_b - 1) == swa.SWA_ERR_WORKSPACE


@pytest.mark.parametrize("kind", KINDS)
def test_empty_block_forward_is_a_no_op(kind):
    assert block_fwd_call(params(B=0), block_weights(), kind=kind) == swa.SWA_OK
    assert block_fwd_call(params(T=0), block_weights(), kind=kind) == swa.SWA_OK
    # nothing to zero when every gradient output is NULL
    assert block_bwd_call(params(B=0), block_weights(), kind=kind) == swa.SWA_OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the compiled library the binding raises: there is no fallback
    path that would compute anything elsewhere."""
    import torch
    monkeypatch.setattr(swa, "_LIBS", {})
    monkeypatch.setattr(swa._build, "lib_path", lambda kind: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        swa.load("bf16")
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError, match="not built"):
        swa.attention_forward(q, k, k, window=4)


@pytest.mark.parametrize("kind", KINDS)
def test_step_host_size_and_argument_checks(kind):
    """The host-buffer training step: its device buffer holds the backward
    workspace plus device copies of every input and output; bad arguments are
    refused before anything is enqueued (no GPU is touched here)."""
    p = params()
    es = 2 if kind == "bf16" else 4
    B, T, Hq, Hkv, d = 2, 300, 4, 2, 128
    ws = swa.swa_attn_workspace_size(p, 1, kind)
    need = swa.swa_attn_step_host_size(p, kind)
    tensors = B * T * d * es * (4 * Hq + 4 * Hkv) + B * T * Hq * 4 + 4 * d * 4 + B * T * (4 + 4 * Hkv)
    assert ws + tensors <= need <= ws + tensors + 20 * 256
    assert swa.swa_attn_step_host_size(params(d=96), kind) == 0
    lib = swa.load(kind)

    def call(buf=A, nbytes=1 << 40, **over):
        a = dict(q=A, k=A, v=A, gq=None, gk=None, ve=None, tok=None, gate=None, dO=A, o=A, lse=A,
                 dq=A, dk=A, dv=A, dgq=None, dgk=None, dve=None)
        a.update(over)
        return lib.swa_attn_step_host(ctypes.byref(p), None, a["q"], a["k"], a["v"], a["gq"], a["gk"],
                                      a["ve"], a["tok"], a["gate"], a["dO"], a["o"], a["lse"], a["dq"],
                                      a["dk"], a["dv"], a["dgq"], a["dgk"], a["dve"], buf, nbytes, None)

    for name in ("q", "k", "v", "dO", "o", "lse", "dq", "dk", "dv"):
        assert call(**{name: None}) == swa.SWA_ERR_INVALID_ARG, name
    assert call(buf=None) == swa.SWA_ERR_INVALID_ARG
    assert call(buf=A + 16) == swa.SWA_ERR_INVALID_ARG          # not 256-byte aligned
    assert call(ve=A) == swa.SWA_ERR_INVALID_ARG                # a VE table needs token ids
    assert call(nbytes=need - 1) == swa.SWA_ERR_WORKSPACE
