"""Float64 CPU oracle of the whole attention block around the attention core:
pre-norm, the four projections and the residual.

TEST INFRASTRUCTURE ONLY, like ``oracle.attention``: imported by ``tests/``,
never by the library, and sharing no code with the CUDA path.

Sources:
  [Guide] "autoresearch Administrator & Developer Guide" §8.2.1 model table:
          "Pre-norm + residual", the block adds the attention of the RMS-normed
          input back onto its input (x = x + attn(norm(x))); RMSNorm is
          ``F.rms_norm`` (no gain on the block's pre-norm).
  [Post]  the autoresearch ``train.py`` walkthrough post, model paragraph:
          RMSNorm on the block inputs (pre-norm) as well as on q and k; the
          gate reads the first 32 channels of the hidden state, which inside
          the block is the normed x ([Guide] §8.2.1 gate snippet); optimizer
          paragraph: the attention projections are 2-D weight matrices.
  [Guide] §1.4 process flow: ``init_weights()`` initialises the attention
          matrices and zeroes ``c_proj`` (the output projection), so at
          initialisation the block returns its input.

Readings where the pages are silent (the CUDA library takes the same ones):
  * weights in the ``nn.Linear`` layout [out_features, in_features]:
    wq [Hq*d, C], wk and wv [Hkv*d, C], wo [C, Hq*d]; a projection is
    y = x @ w^T; no biases.
  * the projections' outputs are viewed as [B, T, H, d] heads (head-major
    channel order h*d + c), and the attention output [B, T, Hq, d] is viewed
    back as [B, T, Hq*d] before the output projection.
  * the pre-norm uses the same epsilon as the QK-norm.

parity pinned in ``tests/test_oracle_block.py`` (central finite differences
of every input, special cases that reduce the block to its input or to the
attention alone, linearity in the output projection, and an independent
float64 torch autograd run).
"""

from __future__ import annotations

import numpy as np

from .attention import attention_backward, attention_forward, rms_norm, rms_norm_backward

__all__ = ["block_forward", "block_backward"]


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _project(xn, w, H):
    """Bias-free projection of the normed rows, viewed as heads: [B, T, H, d]."""
    B, T, _ = xn.shape
    y = xn @ np.asarray(w, dtype=np.float64).T
    return y.reshape(B, T, H, -1)


def block_forward(x, wq, wk, wv, wo, *, Hq: int, Hkv: int, window: int, causal: bool = True,
                  scale=None, eps: float = 1e-6, gq=None, gk=None, ve=None, tok=None,
                  ve_scale: float = 0.5, rope=None, gate_w=None):
    """out = x + (attn(xn wq^T, xn wk^T, xn wv^T) viewed [B, T, Hq*d]) wo^T,
    with xn = rms_norm(x) and the attention of ``attention_forward`` (QK-norm
    with gains gq / gk, rotary tables, VE mix, learned gate reading
    xn[..., :C] with C = gate_w.shape[1]).

    Returns (out [B, T, C], saved) where ``saved`` holds the intermediates
    xn, q, k, v, o, lse (o and lse are the attention's outputs)."""
    x = _f64(x)
    B, T, _ = x.shape
    xn, _ = rms_norm(x, None, eps)
    q, k, v = _project(xn, wq, Hq), _project(xn, wk, Hkv), _project(xn, wv, Hkv)
    gate_x = None if gate_w is None else xn[..., :np.asarray(gate_w).shape[1]]
    o, lse = attention_forward(q, k, v, gq, gk, window=window, causal=causal, scale=scale,
                               eps=eps, ve=ve, tok=tok, ve_scale=ve_scale, rope=rope,
                               gate_x=gate_x, gate_w=gate_w)
    y = o.reshape(B, T, -1) @ np.asarray(wo, dtype=np.float64).T
    return x + y, {"xn": xn, "q": q, "k": k, "v": v, "o": o, "lse": lse}


def block_backward(x, wq, wk, wv, wo, dout, *, Hq: int, Hkv: int, window: int,
                   causal: bool = True, scale=None, eps: float = 1e-6, gq=None, gk=None,
                   ve=None, tok=None, ve_scale: float = 0.5, rope=None, gate_w=None):
    """Analytic backward of ``block_forward`` for the loss <out, dout>, by the
    chain rule through each step in reverse:
      residual:          dx gets dout directly
      output projection: dwo = sum_rows dout^T o;  do = dout wo
      attention:         ``attention_backward`` with dO = do gives dq, dk, dv
                         (and dgq, dgk, dve, the gate's dgate_x, dgate_w)
      projections:       dwq = sum_rows dq^T xn (likewise dwk, dwv);
                         dxn = dq wq + dk wk + dv wv, plus dgate_x on the
                         gate's channels
      pre-norm:          dx += rms_norm_backward(x, dxn)
    Returns a dict with dx, dwq, dwk, dwv, dwo, dgq, dgk, dve and dgate_w
    (None where the input is absent)."""
    x = _f64(x)
    dout = _f64(dout)
    B, T, C = x.shape
    _, s = block_forward(x, wq, wk, wv, wo, Hq=Hq, Hkv=Hkv, window=window, causal=causal,
                         scale=scale, eps=eps, gq=gq, gk=gk, ve=ve, tok=tok, ve_scale=ve_scale,
                         rope=rope, gate_w=gate_w)
    xn, o = s["xn"], s["o"]
    rows_out = dout.reshape(B * T, C)
    dwo = rows_out.T @ o.reshape(B * T, -1)
    do = (dout @ np.asarray(wo, dtype=np.float64)).reshape(o.shape)
    gate_x = None if gate_w is None else xn[..., :np.asarray(gate_w).shape[1]]
    g = attention_backward(s["q"], s["k"], s["v"], gq, gk, do, window=window, causal=causal,
                           scale=scale, eps=eps, ve=ve, tok=tok, ve_scale=ve_scale, rope=rope,
                           gate_x=gate_x, gate_w=gate_w)
    rows_xn = xn.reshape(B * T, C)
    grads = {}
    dxn = np.zeros_like(xn)
    for name, w, dh in (("dwq", wq, g["dq"]), ("dwk", wk, g["dk"]), ("dwv", wv, g["dv"])):
        dh = dh.reshape(B * T, -1)
        grads[name] = dh.T @ rows_xn
        dxn += (dh @ np.asarray(w, dtype=np.float64)).reshape(B, T, C)
    if gate_w is not None:
        dxn[..., :np.asarray(gate_w).shape[1]] += g["dgate_x"]
    dx_norm, _ = rms_norm_backward(x, None, eps, dxn)
    grads.update({"dx": dout + dx_norm, "dwo": dwo, "dgq": g["dgq"], "dgk": g["dgk"],
                  "dve": g["dve"], "dgate_w": g.get("dgate_w")})
    return grads
