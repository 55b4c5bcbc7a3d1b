"""The bounded pipeline waits of the tensor-core kernels, run out on purpose.

Every wait of the forward and backward kernels on a shared-memory barrier has
a time limit (swa_extras.wait_limit_ns; 2 s by default). A wait that runs out
makes its CTA give up: it records SWA_ERR_TIMEOUT in the workspace status
word, lets the copies and MMAs it issued land (those waits keep their own
fixed limit) and returns, so the context stays usable. Here the S-layer
forward and backward run with a limit of 1 ns, far below the time one tile
copy takes, so that waits run out; swa_attn_check_status must report the
timeout, and the same workspace must then give oracle-exact results on a
normal call in the same process. Nothing here waits on a flag that nothing
sets: the waited-for copies and products all complete, only later than the
limit allows.
"""

import pytest
import torch

import sliding_window_gqa_qk_gb300 as swa
from sliding_window_gqa_qk_gb300.inputs import S_LAYER, make_inputs
from gpu_helpers import TOL, batch_slice, compare, run_oracle

pytestmark = pytest.mark.gpu


def _call(prm, ex, g, o, lse, grads, ws, flags=0):
    st = swa.swa_attn_fwd_ex(prm, ex, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"], g["tok"],
                             None, o, lse, ws, flags=flags)
    assert st == swa.SWA_OK, swa.swa_strerror(st)
    st = swa.swa_attn_bwd_ex(prm, ex, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"], g["tok"],
                             None, o, lse, g["dO"], grads["dq"], grads["dk"], grads["dv"],
                             grads["dgq"], grads["dgk"], grads["dve"], ws, flags=flags)
    assert st == swa.SWA_OK, swa.swa_strerror(st)


@pytest.mark.parametrize("ve", [False, True])
def test_waits_that_run_out_are_reported_and_the_workspace_stays_usable(ve):
    p = S_LAYER.replace(ve=ve)
    dev = torch.device("cuda:0")
    x = make_inputs(p, layer=1 if ve else 0)
    g = {k: (t.to(dev) if t is not None else None) for k, t in x.items()}
    prm = swa.make_params(p.B, p.T, p.Hq, p.Hkv, p.d, p.window, p.causal, 0.0, p.eps,
                          p.ve_scale, p.vocab if ve else 0)
    ws = swa.new_workspace(prm, True, dev, "bf16")
    o = torch.empty_like(g["q"])
    lse = torch.empty(p.B, p.Hq, p.T, dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    grads = {"dq": torch.empty_like(g["q"]), "dk": torch.empty_like(g["k"]),
             "dv": torch.empty_like(g["v"]), "dgq": torch.empty(p.d, **f32),
             "dgk": torch.empty(p.d, **f32),
             "dve": torch.empty(g["ve"].shape, **f32) if ve else None}

    # forward alone with the short limit
    short = swa.make_extras(wait_limit_ns=1)
    st = swa.swa_attn_fwd_ex(prm, short, g["q"], g["k"], g["v"], g["gq"], g["gk"], g["ve"],
                             g["tok"], None, o, lse, ws)
    assert st == swa.SWA_OK
    assert swa.swa_attn_check_status(ws) == swa.SWA_ERR_TIMEOUT
    assert swa.swa_attn_check_status(ws) == swa.SWA_OK   # read and cleared

    # forward and backward with the short limit
    _call(prm, short, g, o, lse, grads, ws)
    assert swa.swa_attn_check_status(ws) == swa.SWA_ERR_TIMEOUT

    # the same workspace, default limit: oracle-exact on two batch elements
    for t in (o, lse, *[t for t in grads.values() if t is not None]):
        t.fill_(float("nan"))
    _call(prm, None, g, o, lse, grads, ws)
    assert swa.swa_attn_check_status(ws) == swa.SWA_OK
    torch.cuda.synchronize()
    for b in (0, p.B - 1):
        ref = run_oracle(p.replace(B=1), batch_slice(x, b))
        got = {"o": o[b:b + 1].cpu(), "lse": lse[b:b + 1].cpu(), "dq": grads["dq"][b:b + 1].cpu(),
               "dk": grads["dk"][b:b + 1].cpu(), "dv": grads["dv"][b:b + 1].cpu()}
        compare(got, ref, TOL["bf16"], keys=("o", "lse", "dq", "dk", "dv"))
