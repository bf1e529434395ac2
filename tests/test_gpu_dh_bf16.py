"""bf16 dH output of the loss backward (VCE_FLAG_DH_BF16).

The library sums dH over the vocabulary in fp32 exactly as the fp32-dH call
does, then rounds once. So, bit for bit:

- the bf16 dH is the fp32-dH call's result rounded to nearest even;
- with VCE_FLAG_ACCUMULATE_DH, it is the rounding of (the bf16 value already
  there + that fp32 sum).

Against the fp64 oracle the bf16 dH stays within the bf16 gradient tolerance,
2e-2 max-abs relative.
"""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

BF16, ACC = R.vce.VCE_FLAG_DH_BF16, R.vce.VCE_FLAG_ACCUMULATE_DH


def _case(dtype, T=1000, H=256, V=5000, seed=90):
    wl = I.custom("dh_bf16", T=T, H=H, V_real=V, Vp=-(-V // 64) * 64, S=4, dtype=dtype, seed=seed,
                  ignore_frac=0.05)
    d = I.make_all(wl, ("W", "h", "targets"))
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    out = R.loss_fwd(wl, h_d, W_d, d["targets"], maps=False)
    assert out["status"] == 0
    return wl, d, h_d, W_d, out["targets_d"], out["lse_d"]


def _bwd(wl, h_d, W_d, y_d, lse_d, dH, flags, ws_bytes=None, minimal=False):
    p = R.prob(wl, flags=flags)
    if ws_bytes is None:
        op = R.vce.VCE_OP_LOSS_BWD
        ws_bytes = R.vce.vce_workspace_size_min(p, op) if minimal else R.vce.vce_workspace_size(p, op)
    dW = torch.zeros((wl.Vp, wl.H), device="cuda")
    ws = D.workspace(ws_bytes)
    st = R.status_word()
    R.vce.vce_loss_bwd(p, h_d, W_d, y_d, lse_d, 1.0, dH, dW, ws, ws_bytes=ws_bytes, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return dW


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("minimal", [False, True], ids=["recommended_ws", "minimal_ws_256_col_chunks"])
def test_bf16_dh_is_the_rounded_fp32_sum(dtype, minimal):
    wl, d, h_d, W_d, y_d, lse_d = _case(dtype)
    dH32 = torch.full((wl.T, wl.H), float("nan"), device="cuda")
    dW32 = _bwd(wl, h_d, W_d, y_d, lse_d, dH32, 0, minimal=minimal)
    dHb = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dWb = _bwd(wl, h_d, W_d, y_d, lse_d, dHb, BF16, minimal=minimal)
    assert np.array_equal(_bits(dHb), O._round_bf16_bits(dH32.cpu().numpy()))
    assert torch.equal(dWb.view(torch.int32), dW32.view(torch.int32))   # dW is untouched by the flag
    rdH, _ = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    got = I.bf16_to_f32(_bits(dHb))
    assert R.max_abs_rel(got, rdH) <= 2e-2


def test_bf16_dh_accumulates_before_rounding():
    wl, d, h_d, W_d, y_d, lse_d = _case("bf16", seed=91)
    dH32 = torch.zeros((wl.T, wl.H), device="cuda")
    _bwd(wl, h_d, W_d, y_d, lse_d, dH32, 0)
    init = torch.randn((wl.T, wl.H), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    dHb = init.clone()
    _bwd(wl, h_d, W_d, y_d, lse_d, dHb, BF16 | ACC)
    want = O._round_bf16_bits(I.bf16_to_f32(_bits(init)) + dH32.cpu().numpy())
    assert np.array_equal(_bits(dHb), want)


def test_bf16_dh_sampled_loss():
    wl = I.custom("dh_bf16_sampled", T=512, H=128, V_real=3000, Vp=3008, S=4, dtype="bf16", seed=92,
                  ignore_frac=0.05)
    d = I.make_all(wl, ("W", "h", "targets"))
    draws = torch.from_numpy(I.make_negative_draws(wl, wl.V_real)).cuda()
    h_d, W_d, y_d = D.to_device(d["h"]), D.to_device(d["W"]), torch.from_numpy(d["targets"]).cuda()
    P = 700
    res = {}
    for flags, dt in ((0, torch.float32), (BF16, torch.bfloat16)):
        p = R.prob(wl, flags=flags)
        dH = torch.full((wl.T, wl.H), float("nan"), dtype=dt, device="cuda")
        dW = torch.zeros((wl.Vp, wl.H), device="cuda")
        loss = torch.empty(1, device="cuda")
        cand = torch.empty(P, dtype=torch.int64, device="cuda")
        pos = torch.empty(wl.T, dtype=torch.int64, device="cuda")
        nu = torch.empty(1, dtype=torch.int32, device="cuda")
        ws = D.workspace(R.vce.vce_sampled_workspace_size(p, P))
        st = R.status_word()
        R.vce.vce_sampled_loss(p, h_d, W_d, y_d, draws, P, 1.0, loss, None, dH, dW, cand, pos, nu, ws,
                               dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res[flags] = (dH, dW)
    assert np.array_equal(_bits(res[BF16][0]), O._round_bf16_bits(res[0][0].cpu().numpy()))
    assert torch.equal(res[BF16][1].view(torch.int32), res[0][1].view(torch.int32))
