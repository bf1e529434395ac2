"""Seeded random shapes against the oracle: the whole path (lookup, loss
forward and backward, embedding backward, greedy argmax) on problem sizes drawn
from a fixed generator; every other case runs the embedding backward as a plan
made beside the lookup and its application.

T, H, V_real, the padding to Vp, S and the ignored fraction are drawn so that
shard bounds, forward units, token blocks and vocabulary tiles fall at
unrelated places. A few cases take H large enough to split the tensor-core
items into token-block groups. The tolerances are those of the fixed cases:
bit-exact for the lookup and the replayed embedding backward; bf16 loss and lse
1e-3 relative; dH and dW 2e-2 max-abs relative; fp32 1e-5.
"""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": dict(loss=1e-5, grad=1e-5), "bf16": dict(loss=1e-3, grad=2e-2)}
CHUNK = 32


def _draw(i):
    g = np.random.default_rng(1000 + i)
    dtype = "f32" if i % 5 == 4 else "bf16"
    step = 8 if dtype == "bf16" else 4
    if i % 6 == 5:   # wide rows: token-block groups below all of T
        H = int(g.choice([6144, 8192]))
        T = int(g.integers(2600, 4000))
        V = int(g.integers(300, 1500))
    else:
        H = step * int(g.integers(1, 96))
        T = int(g.integers(1, 900))
        V = int(g.integers(2, 6000))
    Vp = -(-V // 64) * 64 + 64 * int(g.integers(0, 3))
    S = int(g.integers(1, min(Vp, 12) + 1))
    return dict(T=T, H=H, V_real=V, Vp=Vp, S=S, dtype=dtype, seed=2000 + i,
                ignore_frac=float(g.choice([0.0, 0.05, 0.3])), pad_id_frac=0.05, oor_id_frac=0.05,
                pad_fill=8.0)


CASES = [_draw(i) for i in range(40)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{T}_H{H}_V{V_real}_Vp{Vp}_S{S}_{dtype}".format(**c))
def test_random_shape(case):
    wl = I.custom("random", **case)
    tol = TOL[wl.dtype]
    d = I.make_all(wl, ("W", "h", "targets", "ids", "dE"))
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    # lookup, bit for bit; every other case makes the embedding backward's plan
    # beside it and applies the plan below, the others use the one-call backward
    split = case["seed"] % 2 == 1
    p = R.prob(wl)
    if split:
        ws_e = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
        E = torch.empty((wl.T, wl.H), dtype=W_d.dtype, device="cuda")
        R.vce.vce_embed_fwd_plan(p, torch.from_numpy(d["ids"]).cuda(), W_d, E, ws_e)
        torch.cuda.synchronize()
        got = {"E": D.to_host_bits(E)}
    else:
        got = R.embed_fwd(wl, W_d, d["ids"])
    assert np.array_equal(got["E"], O.embed_forward(d["ids"], d["W"], wl.V_real))
    # loss forward
    out = R.loss_fwd(wl, h_d, W_d, d["targets"], maps=False)
    ref = O.cross_entropy_forward(d["h"], d["W"], d["targets"], wl.V_real)
    assert out["status"] == 0
    assert R.rel(out["loss"], ref["loss"]) <= tol["loss"] or (ref["loss"] == 0 and out["loss"] == 0)
    assert np.all(np.abs(out["lse"] - ref["lse"]) <= tol["loss"] * np.maximum(np.abs(ref["lse"]), 1.0))
    # loss backward
    dH, dW, st = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"])
    assert st == 0
    rdH, rdW = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    assert R.max_abs_rel(dH.cpu().numpy(), rdH) <= tol["grad"]
    dWn = dW.cpu().numpy()
    assert R.max_abs_rel(dWn, rdW) <= tol["grad"]
    assert np.all(dWn[wl.V_real:] == 0)
    # embedding backward into that dW, bit for bit against the fp32 replay
    dE32 = I.bf16_to_f32(d["dE"]) if wl.dtype == "bf16" else d["dE"]
    if split:
        st_e = R.status_word()
        R.vce.vce_embed_bwd_apply(p, D.to_device(d["dE"]), dW, ws_e, dev_status=st_e)
        torch.cuda.synchronize()
        assert int(st_e.item()) == 0
    else:
        assert R.embed_bwd(wl, d["ids"], D.to_device(d["dE"]), dW) == 0
    want = O.embed_backward_replay_f32(d["ids"], dE32, wl.V_real, CHUNK, dWn)
    assert np.array_equal(dW.cpu().numpy().view(np.uint32), want.view(np.uint32))
    # greedy argmax: a valid class whose logit is the maximum within the logits' rounding
    arg = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    ws = D.workspace(max(R.vce.vce_workspace_size(p, R.vce.VCE_OP_GREEDY_ARGMAX), 256))
    R.vce.vce_greedy_argmax(p, h_d, W_d, arg, ws=ws)
    torch.cuda.synchronize()
    z = O.logits(d["h"], d["W"], wl.V_real)
    a = arg.cpu().numpy()
    zmax = z.max(axis=1)
    assert np.all((a >= 0) & (a < wl.V_real))
    slack = (1e-3 if wl.dtype == "bf16" else 1e-5) * np.maximum(np.abs(zmax), 1.0)
    assert np.all(z[np.arange(wl.T), a] >= zmax - slack)
