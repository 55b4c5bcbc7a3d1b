"""Plain float64 CPU oracle of the SSSL / GQA / QK-norm attention block.

TEST INFRASTRUCTURE ONLY. This module is the checker that the CUDA library is
compared against. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the library itself never does, and
this module imports nothing from the library.

Everything is computed the slow, obvious way in float64 NumPy: the full T x T
logit matrix of every head (row-chunked only to bound memory), an explicit
boolean band mask, a max-subtracted softmax, and the analytic backward written
out from the chain rule. No tiling, no online softmax, no fused steps.

Sources (the pages this follows):
  [Post]  the autoresearch ``train.py`` walkthrough post (cnoyu.systems
          "discover" post, Spanish/French/German/Czech copies), model paragraph:
          QK-norm "right before the attention dot product"; the "SSSL" pattern
          with window = half the sequence, last layer forced global; value
          embeddings mixed into v on every other layer.
  [Guide] "autoresearch Administrator & Developer Guide":
          §3.4 (``WINDOW_PATTERN``, last layer overridden to L),
          §6.3 techniques table (sliding-window attention, GQA),
          §8.2.1 Model - GPT (``F.rms_norm``; GQA ``n_kv_head <= n_head``;
          value embeddings ``Embedding(vocab_size, kv_dim)`` and the gated mix
          ``v = v + gate * ve``; ``has_ve``: alternating layers, last included).

Readings where the pages are silent (the CUDA library takes the same ones):
  * window: key j is visible to query i iff 0 <= i - j <= W (W + 1 keys,
    self included); W < 0 means no window. Non-causal: |i - j| <= W.
  * softmax scale 1/sqrt(d) unless given; RMSNorm epsilon is a parameter.
  * RMSNorm gains are per-channel vectors [d] shared by all heads (None = 1).
  * GQA: query head h reads kv head h // (Hq / Hkv).
  * VE mix: v_eff = v + ve_scale * gate[b, t, hkv] * VE[tok[b, t], hkv*d:(hkv+1)*d]
    (gate None = 1). The pages' learned gate is an input of this function.
  * Layout: q [B, T, Hq, d], k/v [B, T, Hkv, d], LSE [B, Hq, T] in natural log.
  * Rotary (optional, ``rope=(cos, sin)`` tables [>= T, d/2] given by the
    caller): applied to q and k before the norm, pairing channel c with
    c + d/2 and turning the pair by the angle of table entry [t, c]:
    y_c = x_c cos + x_{c+d/2} sin, y_{c+d/2} = -x_c sin + x_{c+d/2} cos.
  * Learned VE gate (optional, ``gate_x`` [B, T, C] and ``gate_w`` [Hkv, C]):
    gate[b, t, h] = 2 * sigmoid(<gate_w[h], gate_x[b, t]>), in place of a
    given ``gate``; the backward then also returns its gradients.

parity pinned: every function here is checked in ``tests/test_oracle.py``
against the pages' worked examples, closed forms, invariants, brute force,
central finite differences and an independent float64 autograd run.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "sssl_window",
    "has_ve",
    "rotary",
    "rotary_backward",
    "rms_norm",
    "rms_norm_backward",
    "rms_norm_backward_scale",
    "ve_mix",
    "learned_gate",
    "band_mask",
    "attention_logits",
    "attention_forward",
    "attention_backward",
    "attention_forward_rows",
    "attention_backward_rows",
    "attention_backward_cols",
]


# ----------------------------------------------------------------------------
# Layer schedule helpers
# ----------------------------------------------------------------------------

def sssl_window(layer: int, n_layer: int, pattern: str, T: int) -> int:
    """Window of one layer under a window pattern such as "SSSL".

    [Post] model paragraph: "SSSL" = three sliding-window layers (window = half
    the sequence length) then one full causal layer, repeating; the last layer
    is forced global whatever the pattern says. [Guide] §3.4 ``WINDOW_PATTERN``
    row: the pattern character of layer i is ``pattern[i % len(pattern)]``.

    Returns the window W (keys i-W..i visible) for an 'S' layer, -1 (no
    window, full causal) for an 'L' layer or the last layer.
    """
    if layer == n_layer - 1:
        return -1
    ch = pattern[layer % len(pattern)]
    if ch == "S":
        return T // 2
    if ch == "L":
        return -1
    raise ValueError(f"window pattern character {ch!r} is neither 'S' nor 'L'")


def has_ve(layer: int, n_layer: int) -> bool:
    """Whether a layer mixes value embeddings into v.

    [Guide] §8.2.1, ``has_ve``: alternating layers carry value embeddings and
    the last layer always does; with 8 layers that is 1, 3, 5, 7. Reading:
    the layers with the same parity as the last one.
    """
    return (layer % 2) == ((n_layer - 1) % 2)


# ----------------------------------------------------------------------------
# QK-norm and the value-embedding mix
# ----------------------------------------------------------------------------

def rotary(x: np.ndarray, cos, sin, positions=None) -> np.ndarray:
    """Rotary position embedding over the last axis of x [..., T or len(positions), H, d].

    [Guide] §8.2.1, model table, "Rotary embeddings" row: the cos / sin tables
    are precomputed once for a length beyond the sequence and applied to q and
    k; [Post] model paragraph: the QK-norm comes right before the dot product,
    so the rotation comes first. The pages print neither the pairing nor the
    sign; the reading taken here pairs channel c with c + d/2 and turns each
    pair by the table's angle for its position:
      y_c       =  x_c cos[t, c] + x_{c+d/2} sin[t, c]
      y_{c+d/2} = -x_c sin[t, c] + x_{c+d/2} cos[t, c]
    The position axis is axis -3 (rows t of the tables, or the rows
    ``positions``).
    """
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    n = x.shape[-3]
    pos = np.arange(n) if positions is None else np.asarray(positions, dtype=np.int64)
    c = np.asarray(cos, dtype=np.float64)[pos][:, None, :]    # [n, 1, d/2]
    sn = np.asarray(sin, dtype=np.float64)[pos][:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c + x2 * sn, -x1 * sn + x2 * c], axis=-1)


def rotary_backward(dy: np.ndarray, cos, sin, positions=None) -> np.ndarray:
    """Gradient of ``rotary``: the transposed rotation of every pair,
      dx_c = dy_c cos - dy_{c+d/2} sin,  dx_{c+d/2} = dy_c sin + dy_{c+d/2} cos,
    i.e. the rotation by the opposite angle."""
    return rotary(dy, cos, -np.asarray(sin, dtype=np.float64), positions)


def rms_norm(x: np.ndarray, g, eps: float):
    """RMSNorm over the last axis: y = g * x / sqrt(mean(x^2) + eps).

    [Guide] §8.2.1 "RMSNorm via F.rms_norm"; [Post] QK-norm applies it to q and
    k right before the dot product. ``g`` is a [d] gain vector or None (= 1).
    Returns (y, rstd) with rstd = 1/sqrt(mean(x^2) + eps) of shape x.shape[:-1].
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1)
    rstd = 1.0 / np.sqrt(ms + eps)
    y = x * rstd[..., None]
    if g is not None:
        y = y * np.asarray(g, dtype=np.float64)
    return y, rstd


def rms_norm_backward(x: np.ndarray, g, eps: float, dy: np.ndarray):
    """Gradient of ``rms_norm`` by the chain rule.

    With r = (mean(x^2)+eps)^(-1/2), xh = x r and y = g * xh:
      dxh = g * dy
      dx  = r * (dxh - xh * mean(dxh * xh))      (mean over the last axis)
      dg  = sum over all rows of dy * xh
    Returns (dx, dg); dg is None when g is None.
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    _, r = rms_norm(x, None, eps)
    xh = x * r[..., None]
    dxh = dy if g is None else dy * np.asarray(g, dtype=np.float64)
    dx = r[..., None] * (dxh - xh * np.mean(dxh * xh, axis=-1, keepdims=True))
    dg = None
    if g is not None:
        dg = (dy * xh).reshape(-1, x.shape[-1]).sum(axis=0)
    return dx, dg


def rms_norm_backward_scale(x: np.ndarray, g, eps: float, dy: np.ndarray) -> np.ndarray:
    """Row norms of r * (g * dy): the gradient of ``rms_norm_backward`` before
    its last step removes the component along xh (dx = r * (dxh - xh *
    mean(dxh * xh)) with dxh = g * dy, and that step is an orthogonal
    projection, so |dx_row| <= this norm, with equality when dxh is
    orthogonal to xh). Returns an array of shape x.shape[:-1]. It is the
    scale of a row of dx that carries errors of dy through the projection:
    where most of dxh lies along xh, dx is small and the error is not."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    _, r = rms_norm(x, None, eps)
    dxh = dy if g is None else dy * np.asarray(g, dtype=np.float64)
    return r * np.linalg.norm(dxh, axis=-1)


def ve_mix(v: np.ndarray, ve, tok, gate, ve_scale: float) -> np.ndarray:
    """v_eff = v + ve_scale * gate * VE[tok], per kv head.

    [Guide] §8.2.1 value-embedding row and the printed gate snippet: a table
    ``Embedding(vocab_size, kv_dim)`` looked up by token id is added into v
    through a per-head gate. v is [B, T, Hkv, d]; ve is [vocab, Hkv*d];
    tok is [B, T]; gate is [B, T, Hkv] or None (= 1). ve None returns v.
    """
    v = np.asarray(v, dtype=np.float64)
    if ve is None:
        return v.copy()
    B, T, Hkv, d = v.shape
    table = np.asarray(ve, dtype=np.float64).reshape(-1, Hkv, d)
    rows = table[np.asarray(tok, dtype=np.int64)]          # [B, T, Hkv, d]
    g = np.ones((B, T, Hkv)) if gate is None else np.asarray(gate, dtype=np.float64)
    return v + ve_scale * g[..., None] * rows


def learned_gate(gate_x, gate_w) -> np.ndarray:
    """The value-embedding gate of [Guide] §8.2.1 (the printed gate snippet):
    2 * sigmoid of a bias-free linear map of the first C channels of the
    block input, one output per kv head:
      gate[b, t, h] = 2 / (1 + exp(-sum_c gate_w[h, c] * gate_x[b, t, c])).
    With gate_w = 0 (its initialisation) the gate is 1 everywhere."""
    z = np.asarray(gate_x, dtype=np.float64) @ np.asarray(gate_w, dtype=np.float64).T
    return 2.0 / (1.0 + np.exp(-z))


def learned_gate_backward(gate_x, gate_w, dgate):
    """Gradients of ``learned_gate`` for an upstream dgate [B, T, Hkv]:
    with s = sigmoid(z), d gate / dz = 2 s (1 - s), so
      dz = dgate * 2 s (1 - s);  dgate_x = dz gate_w;  dgate_w = sum_{b,t} dz^T gate_x.
    Returns (dgate_x [B, T, C], dgate_w [Hkv, C])."""
    x = np.asarray(gate_x, dtype=np.float64)
    w = np.asarray(gate_w, dtype=np.float64)
    sg = 1.0 / (1.0 + np.exp(-(x @ w.T)))
    dz = np.asarray(dgate, dtype=np.float64) * 2.0 * sg * (1.0 - sg)
    dx = dz @ w
    dw = dz.reshape(-1, w.shape[0]).T @ x.reshape(-1, x.shape[-1])
    return dx, dw


# ----------------------------------------------------------------------------
# Mask and attention
# ----------------------------------------------------------------------------

def band_mask(rows, T: int, window: int, causal: bool, keys=None) -> np.ndarray:
    """Boolean visibility matrix for query rows ``rows`` against keys 0..T-1
    (or against the key positions ``keys`` only, when given).

    Causal: key j visible to query i iff j <= i and (window < 0 or i - j <= window).
    Non-causal: iff window < 0 or |i - j| <= window.
    [Post] sliding-window layers see a band of width half the sequence;
    [Guide] §6.3 "Sliding-window attention".
    """
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = (np.arange(T, dtype=np.int64) if keys is None else np.asarray(keys, dtype=np.int64))[None, :]
    if causal:
        m = j <= i
        if window >= 0:
            m &= (i - j) <= window
    else:
        m = np.ones((i.shape[0], j.shape[1]), dtype=bool)
        if window >= 0:
            m &= np.abs(i - j) <= window
    return m


def _rot(x, rope, positions=None):
    return x if rope is None else rotary(x, rope[0], rope[1], positions)


def _unrot(dx, rope, positions=None):
    return dx if rope is None else rotary_backward(dx, rope[0], rope[1], positions)


def _prep(q, k, v, gq, gk, eps, ve, tok, gate, ve_scale, rope=None):
    qn, rq = rms_norm(_rot(q, rope), gq, eps)
    kn, rk = rms_norm(_rot(k, rope), gk, eps)
    v_eff = ve_mix(v, ve, tok, gate, ve_scale)
    return qn, kn, v_eff


def _scale(d, scale):
    return 1.0 / math.sqrt(d) if (scale is None or scale == 0) else float(scale)


def attention_logits(qn, kn, b: int, h: int, rows, scale: float) -> np.ndarray:
    """Scaled logits S[i, j] = scale * <qn[b, i, h], kn[b, j, h // G]> for i in rows."""
    G = qn.shape[2] // kn.shape[2]
    return scale * (qn[b, rows, h, :] @ kn[b, :, h // G, :].T)


def _softmax_rows(S: np.ndarray, M: np.ndarray):
    """Masked softmax of each row; returns (A, lse). A row with no visible
    key gives A = 0 and lse = -inf."""
    Sm = np.where(M, S, -np.inf)
    mx = Sm.max(axis=1)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    E = np.where(M, np.exp(Sm - mx_safe[:, None]), 0.0)
    l = E.sum(axis=1)
    A = E / np.where(empty, 1.0, l)[:, None]
    lse = np.where(empty, -np.inf, mx_safe + np.log(np.where(empty, 1.0, l)))
    return A, lse


def attention_forward(q, k, v, gq=None, gk=None, *, window: int, causal: bool = True,
                      scale=None, eps: float = 1e-6, ve=None, tok=None, gate=None,
                      ve_scale: float = 0.5, row_chunk: int = 1024, rope=None,
                      gate_x=None, gate_w=None):
    """Forward of the attention block: returns (o [B,T,Hq,d], lse [B,Hq,T]).

    Steps in the pages' order: rotary of q and k when ``rope`` is given
    ([Guide] §8.2.1 rotary row), QK-norm of q and k ([Post]; [Guide] §8.2.1),
    value-embedding mix into v on VE layers ([Guide] §8.2.1), then for every
    batch b and query head h (kv head h // G, [Guide] §8.2.1 GQA row):
    S = scale * qn kn^T, masked to the causal / sliding band, A = softmax(S),
    O = A v_eff, LSE = log sum exp S over the visible keys.
    """
    q = np.asarray(q, dtype=np.float64)
    B, T, Hq, d = q.shape
    Hkv = np.asarray(k).shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    sc = _scale(d, scale)
    if gate_w is not None:
        gate = learned_gate(gate_x, gate_w)
    qn, kn, v_eff = _prep(q, k, v, gq, gk, eps, ve, tok, gate, ve_scale, rope)
    o = np.zeros((B, T, Hq, d))
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for r0 in range(0, T, row_chunk):
                rows = np.arange(r0, min(T, r0 + row_chunk))
                S = attention_logits(qn, kn, b, h, rows, sc)
                A, l = _softmax_rows(S, band_mask(rows, T, window, causal))
                o[b, rows, h, :] = A @ v_eff[b, :, hk, :]
                lse[b, h, rows] = l
    return o, lse


def attention_forward_rows(q, k, v, gq=None, gk=None, *, b: int, h: int, rows,
                           window: int, causal: bool = True, scale=None,
                           eps: float = 1e-6, ve=None, tok=None, gate=None,
                           ve_scale: float = 0.5, rope=None):
    """Same as ``attention_forward`` for the query rows ``rows`` of one (b, h)
    only; returns (o [len(rows), d], lse [len(rows)]). Used to sample outputs
    of full-size problems one by one."""
    q = np.asarray(q[b:b + 1], dtype=np.float64)
    k = np.asarray(k[b:b + 1], dtype=np.float64)
    v = np.asarray(v[b:b + 1], dtype=np.float64)
    T, d = q.shape[1], q.shape[3]
    G = q.shape[2] // k.shape[2]
    sc = _scale(d, scale)
    tk = None if tok is None else np.asarray(tok)[b:b + 1]
    gt = None if gate is None else np.asarray(gate)[b:b + 1]
    qn, _ = rms_norm(_rot(q[:, :, h:h + 1, :], rope), gq, eps)
    kn, _ = rms_norm(_rot(k[:, :, h // G:h // G + 1, :], rope), gk, eps)
    v_eff = ve_mix(v, ve, tk, gt, ve_scale)[:, :, h // G, :]
    rows = np.asarray(rows, dtype=np.int64)
    S = sc * (qn[0, rows, 0, :] @ kn[0, :, 0, :].T)
    A, l = _softmax_rows(S, band_mask(rows, T, window, causal))
    return A @ v_eff[0], l


def attention_backward(q, k, v, gq=None, gk=None, dO=None, *, window: int,
                       causal: bool = True, scale=None, eps: float = 1e-6, ve=None,
                       tok=None, gate=None, ve_scale: float = 0.5,
                       row_chunk: int = 1024, rope=None, gate_x=None, gate_w=None,
                       scales: bool = False):
    """Analytic backward of ``attention_forward`` for the loss <O, dO>.

    Per (b, h), with A the masked softmax and kv head hk = h // G:
      dA  = dO v_eff^T
      dS  = A * (dA - rowsum(dA * A))              (softmax backward)
      dqn = scale * dS kn
      dkn[hk] += scale * dS^T qn                   (summed over the G heads of a group)
      dv_eff[hk] += A^T dO
    then the RMSNorm backward of q and k (dq, dgq, dk, dgk; of the rotated q
    and k, followed by the transposed rotation, when ``rope`` is given),
    dv = dv_eff and dVE[tok] += ve_scale * gate * dv_eff ([Guide] §8.2.1 VE
    mix, differentiated).

    With the learned gate (``gate_w``), dgate[b, t, h] = ve_scale *
    <dv_eff[b, t, h], VE[tok[b, t], h]> goes through ``learned_gate_backward``.

    Returns a dict with dq, dk, dv, dgq, dgk (None when the gain is None),
    dve ([vocab, Hkv*d], None without VE) and, with the learned gate,
    dgate_x and dgate_w. With ``scales``, also dq_scale [B, T, Hq] and
    dk_scale [B, T, Hkv]: ``rms_norm_backward_scale`` of each row of dq and dk.
    """
    q = np.asarray(q, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, T, Hq, d = q.shape
    Hkv = np.asarray(k).shape[2]
    G = Hq // Hkv
    sc = _scale(d, scale)
    if gate_w is not None:
        gate = learned_gate(gate_x, gate_w)
    qn, kn, v_eff = _prep(q, k, v, gq, gk, eps, ve, tok, gate, ve_scale, rope)
    dqn = np.zeros_like(qn)
    dkn = np.zeros_like(kn)
    dveff = np.zeros_like(v_eff)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for r0 in range(0, T, row_chunk):
                rows = np.arange(r0, min(T, r0 + row_chunk))
                S = attention_logits(qn, kn, b, h, rows, sc)
                A, _ = _softmax_rows(S, band_mask(rows, T, window, causal))
                dOr = dO[b, rows, h, :]
                dA = dOr @ v_eff[b, :, hk, :].T
                dS = A * (dA - np.sum(dA * A, axis=1, keepdims=True))
                dqn[b, rows, h, :] += sc * (dS @ kn[b, :, hk, :])
                dkn[b, :, hk, :] += sc * (dS.T @ qn[b, rows, h, :])
                dveff[b, :, hk, :] += A.T @ dOr
    qr, kr = _rot(q, rope), _rot(np.asarray(k, dtype=np.float64), rope)
    dq, dgq = rms_norm_backward(qr, gq, eps, dqn)
    dk, dgk = rms_norm_backward(kr, gk, eps, dkn)
    dq, dk = _unrot(dq, rope), _unrot(dk, rope)
    dve = None
    if ve is not None:
        Hd = Hkv * d
        g = np.ones((B, T, Hkv)) if gate is None else np.asarray(gate, dtype=np.float64)
        contrib = (ve_scale * g[..., None] * dveff).reshape(B * T, Hd)
        dve = np.zeros((np.asarray(ve).shape[0], Hd))
        np.add.at(dve, np.asarray(tok, dtype=np.int64).reshape(-1), contrib)
    out = {"dq": dq, "dk": dk, "dv": dveff, "dgq": dgq, "dgk": dgk, "dve": dve}
    if scales:
        out["dq_scale"] = rms_norm_backward_scale(qr, gq, eps, dqn)
        out["dk_scale"] = rms_norm_backward_scale(kr, gk, eps, dkn)
    if gate_w is not None:
        rows = np.asarray(ve, dtype=np.float64).reshape(-1, Hkv, d)[np.asarray(tok, dtype=np.int64)]
        dgate = ve_scale * np.sum(dveff * rows, axis=-1)          # [B, T, Hkv]
        out["dgate_x"], out["dgate_w"] = learned_gate_backward(gate_x, gate_w, dgate)
    return out


def _one_batch(q, k, v, dO, tok, gate, b):
    """Batch element b of the inputs, kept 4-D (leading axis of size 1)."""
    sl = slice(b, b + 1)
    f = lambda x: None if x is None else np.asarray(x[sl], dtype=np.float64)
    tk = None if tok is None else np.asarray(tok)[sl]
    return f(q), f(k), f(v), f(dO), tk, f(gate)


def attention_backward_rows(q, k, v, gq=None, gk=None, dO=None, *, b: int, h: int, rows,
                            window: int, causal: bool = True, scale=None, eps: float = 1e-6,
                            ve=None, tok=None, gate=None, ve_scale: float = 0.5, rope=None,
                            with_scale: bool = False):
    """dq of ``attention_backward`` at the query rows ``rows`` of one (b, h).

    Row i of dq depends only on row i of the softmax: dA_i = dO_i v_eff^T,
    dS_i = A_i * (dA_i - <dA_i, A_i>), dqn_i = scale * dS_i kn, then the
    RMSNorm backward of that row. Returns dq [len(rows), d] (and, with
    ``with_scale``, its rows' ``rms_norm_backward_scale``). Used to sample the
    gradient of full-size problems one row at a time.
    """
    q, k, v, dO, tk, gt = _one_batch(q, k, v, dO, tok, gate, b)
    T, d = q.shape[1], q.shape[3]
    G = q.shape[2] // k.shape[2]
    hk = h // G
    sc = _scale(d, scale)
    rows = np.asarray(rows, dtype=np.int64)
    qr = _rot(q[0, rows, h:h + 1, :], rope, rows)[:, 0, :]
    qn, _ = rms_norm(qr, gq, eps)
    kn, _ = rms_norm(_rot(k[0, :, hk:hk + 1, :], rope)[:, 0, :], gk, eps)
    v_eff = ve_mix(v, ve, tk, gt, ve_scale)[0, :, hk, :]
    A, _ = _softmax_rows(sc * (qn @ kn.T), band_mask(rows, T, window, causal))
    dA = dO[0, rows, h, :] @ v_eff.T
    dS = A * (dA - np.sum(dA * A, axis=1, keepdims=True))
    dqn = sc * (dS @ kn)
    dq, _ = rms_norm_backward(qr, gq, eps, dqn)
    dq = _unrot(dq[:, None, :], rope, rows)[:, 0, :]
    return (dq, rms_norm_backward_scale(qr, gq, eps, dqn)) if with_scale else dq


def attention_backward_cols(q, k, v, gq=None, gk=None, dO=None, *, b: int, hk: int, cols,
                            window: int, causal: bool = True, scale=None, eps: float = 1e-6,
                            ve=None, tok=None, gate=None, ve_scale: float = 0.5,
                            row_chunk: int = 512, rope=None, with_scale: bool = False):
    """dk and dv of ``attention_backward`` at the key positions ``cols`` of one
    (b, kv head hk).

    Column j collects, over the G query heads of the group and every query
    row i: dv_j += A_ij dO_i and dkn_j += scale * dS_ij qn_i, with A and dS
    the full rows of the softmax and its backward (a row must be seen whole
    to be normalised). Only rows whose band holds one of ``cols`` are
    visited; the others add exact zeros. Then the RMSNorm backward of the k
    rows. Returns (dk [len(cols), d], dv [len(cols), d]), and with
    ``with_scale`` the dk rows' ``rms_norm_backward_scale`` third.
    """
    q, k, v, dO, tk, gt = _one_batch(q, k, v, dO, tok, gate, b)
    T, Hq, d = q.shape[1], q.shape[2], q.shape[3]
    G = Hq // k.shape[2]
    sc = _scale(d, scale)
    cols = np.asarray(cols, dtype=np.int64)
    kr = _rot(k[0, :, hk:hk + 1, :], rope)[:, 0, :]
    kn, _ = rms_norm(kr, gk, eps)
    v_eff = ve_mix(v, ve, tk, gt, ve_scale)[0, :, hk, :]
    dkn = np.zeros((cols.size, d))
    dv = np.zeros((cols.size, d))
    for r0 in range(0, T, row_chunk):
        rows = np.arange(r0, min(T, r0 + row_chunk))
        keep = band_mask(rows, T, window, causal, keys=cols).any(axis=1)
        if not keep.any():
            continue
        rows = rows[keep]
        M = band_mask(rows, T, window, causal)
        for h in range(hk * G, (hk + 1) * G):
            qn, _ = rms_norm(_rot(q[0, rows, h:h + 1, :], rope, rows)[:, 0, :], gq, eps)
            A, _ = _softmax_rows(sc * (qn @ kn.T), M)
            dOr = dO[0, rows, h, :]
            dA = dOr @ v_eff.T
            dS = A * (dA - np.sum(dA * A, axis=1, keepdims=True))
            dv += A[:, cols].T @ dOr
            dkn += sc * (dS[:, cols].T @ qn)
    dk, _ = rms_norm_backward(kr[cols], gk, eps, dkn)
    dk = _unrot(dk[:, None, :], rope, cols)[:, 0, :]
    if with_scale:
        return dk, dv, rms_norm_backward_scale(kr[cols], gk, eps, dkn)
    return dk, dv
