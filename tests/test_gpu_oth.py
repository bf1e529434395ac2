"""GPU parity of the OT-H auxiliary head ("Sampled Softmax with Over-Tokenized
Transformer", Setup and its loss listing): a second head W2 on h[:-1] scored on
tokens[2:] at weight 0.1, its dH added into the main head's dH through
VCE_FLAG_ACCUMULATE_DH. Compared with the oracle's `oth_loss`.

Tolerances as for the cross-entropy: fp32 1e-5 relative; bf16 loss 1e-3
relative, dH/dW 2e-2 max-abs relative.
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
WEIGHT = 0.1


def _inputs(wl):
    """h, W, W2 and tokens[T+1] (targets of head one are tokens[1:], of head two tokens[2:])."""
    d = I.make_all(wl, ("W", "h", "targets"))
    W2 = I.make_W(I.custom("oth_head2", T=wl.T, H=wl.H, V_real=wl.V_real, Vp=wl.Vp, S=wl.S, dtype=wl.dtype,
                           seed=wl.seed + 1000, pad_fill=wl.pad_fill))
    y = d["targets"]
    extra = np.random.default_rng(wl.seed + 7).integers(0, wl.V_real, 1)
    tokens = np.concatenate([extra, y]).astype(np.int64)   # tokens[1:] == targets of head one
    return d["h"], d["W"], W2, tokens


def _run(wl, h, W, W2, tokens, bwd_ws_bytes=None):
    T = wl.T
    h_d, W_d, W2_d = D.to_device(h), D.to_device(W), D.to_device(W2)
    y1 = torch.from_numpy(tokens[1:].copy()).cuda()
    y2 = torch.from_numpy(tokens[2:].copy()).cuda()
    p1 = R.prob(wl, T=T, tied=False)
    p2 = R.prob(wl, T=T - 1, tied=False)
    p2_acc = R.prob(wl, T=T - 1, tied=False, flags=R.vce.VCE_FLAG_ACCUMULATE_DH)
    st = R.status_word()
    loss1 = torch.full((1,), float("nan"), device="cuda")
    loss2 = torch.full((1,), float("nan"), device="cuda")
    lse1 = torch.empty(T, device="cuda")
    lse2 = torch.empty(max(T - 1, 1), device="cuda")
    dH = torch.full((T, wl.H), float("nan"), device="cuda")
    dW = torch.full((wl.Vp, wl.H), float("nan"), device="cuda")
    dW2 = torch.full((wl.Vp, wl.H), float("nan"), device="cuda")
    ws_f = D.workspace(max(R.vce.vce_workspace_size(p1, R.vce.VCE_OP_LOSS_FWD), 256))
    nb = R.vce.vce_workspace_size(p1, R.vce.VCE_OP_LOSS_BWD) if bwd_ws_bytes is None else bwd_ws_bytes
    ws_b = D.workspace(nb)
    R.vce.vce_loss_fwd(p1, h_d, W_d, y1, loss1, lse1, ws=ws_f, dev_status=st)
    R.vce.vce_loss_fwd(p2, h_d, W2_d, y2, loss2, lse2, ws=ws_f, dev_status=st)
    R.vce.vce_loss_bwd(p1, h_d, W_d, y1, lse1, 1.0, dH, dW, ws_b, ws_bytes=nb, dev_status=st)
    R.vce.vce_loss_bwd(p2_acc, h_d, W2_d, y2, lse2, WEIGHT, dH, dW2, ws_b, ws_bytes=nb, dev_status=st)
    torch.cuda.synchronize()
    return dict(loss=float(loss1.item()) + WEIGHT * float(loss2.item()), main=float(loss1.item()),
                aux=float(loss2.item()), dH=dH.cpu().numpy(), dW=dW.cpu().numpy(), dW2=dW2.cpu().numpy(),
                status=int(st.item()))


def _check(wl, bwd_ws_bytes=None):
    h, W, W2, tokens = _inputs(wl)
    out = _run(wl, h, W, W2, tokens, bwd_ws_bytes)
    ref = O.oth_loss(h, W, W2, tokens, wl.V_real, wl.Vp, weight=WEIGHT)
    tol = TOL[wl.dtype]
    assert out["status"] == 0
    assert R.rel(out["main"], ref["main"]) <= tol["loss"]
    assert R.rel(out["aux"], ref["aux"]) <= tol["loss"]
    assert R.rel(out["loss"], ref["loss"]) <= tol["loss"]
    assert R.max_abs_rel(out["dH"], ref["dH"]) <= tol["grad"]
    # the last row is head one's alone
    assert R.max_abs_rel(out["dH"][-1], ref["dH"][-1]) <= tol["grad"] * 4
    assert R.max_abs_rel(out["dW"], ref["dW"]) <= tol["grad"]
    assert R.max_abs_rel(out["dW2"], ref["dW2"]) <= tol["grad"]


def test_oth_f32_tiny():
    _check(I.custom("oth_f32", T=64, H=64, V_real=1000, Vp=1024, S=4, dtype="f32", seed=40, ignore_frac=0.1,
                    pad_fill=8.0))


def test_oth_bf16_small():
    """T=300, H=128, V_real=1000 -> 1024, S=4: one K part (dH added by TMA reduce-add)."""
    _check(I.custom("oth_bf16", T=300, H=128, V_real=1000, Vp=1024, S=4, dtype="bf16", seed=41, ignore_frac=0.1,
                    pad_fill=8.0))


def test_oth_bf16_dh_parts_and_chunks():
    """V_real=20000 -> 20032, H=256: the dH GEMM splits K into parts (their sum is
    added into dH); a small workspace also cuts the vocabulary into chunks."""
    wl = I.custom("oth_parts", T=520, H=256, V_real=20000, Vp=20032, S=8, dtype="bf16", seed=42, ignore_frac=0.05,
                  pad_fill=8.0)
    _check(wl)
    p = R.prob(wl, T=wl.T)
    small = R.vce.vce_workspace_size_min(p, R.vce.VCE_OP_LOSS_BWD) + wl.T * 2 * 4096
    _check(wl, bwd_ws_bytes=small)


def test_accumulate_flag_adds_exactly():
    """dH with the flag equals dH without it plus the initial contents (fp32 sum
    of two terms, one rounding), row for row; rows of ignored tokens keep the
    initial value."""
    wl = I.custom("oth_acc", T=200, H=128, V_real=1000, Vp=1024, S=4, dtype="bf16", seed=43, ignore_frac=0.2,
                  pad_fill=8.0)
    d = I.make_all(wl, ("W", "h", "targets"))
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    out = R.loss_fwd(wl, h_d, W_d, d["targets"], maps=False)
    dH0, _, st0 = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], g=0.3)
    init = torch.randn((wl.T, wl.H), device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    dH = init.clone()
    p = R.prob(wl, flags=R.vce.VCE_FLAG_ACCUMULATE_DH)
    dW = torch.empty((wl.Vp, wl.H), device="cuda")
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_LOSS_BWD))
    st = R.status_word()
    R.vce.vce_loss_bwd(p, h_d, W_d, out["targets_d"], out["lse_d"], 0.3, dH, dW, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st0 == 0 and int(st.item()) == 0
    assert torch.equal(dH, init + dH0)
    ign = torch.from_numpy(~((d["targets"] >= 0) & (d["targets"] < wl.V_real))).cuda()
    assert torch.equal(dH[ign], init[ign])
