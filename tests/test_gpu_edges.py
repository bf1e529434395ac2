"""Edge cases on the GPU, against the oracle:

- an empty batch (T = 0) through every entry point: nothing is read, the loss
  is 0, an untied dW is zeroed, a tied or accumulated dW is left alone;
- hidden sizes that are not multiples of the 64-wide K block of the
  tensor-core tiles (H = 72, 200), a wide one (H = 8192, 16 KB rows), and an
  fp32 width that is not a multiple of 64 (H = 100);
- token-block item groups of unequal size with a ragged last block.
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


@pytest.mark.parametrize("tied", [False, True])
def test_empty_batch_every_entry(tied):
    wl = I.custom("empty", T=0, H=64, V_real=1000, Vp=1024, S=4, dtype="bf16", seed=80, tied=tied)
    vce = R.vce
    p = R.prob(wl)
    W = D.to_device(I.make_W(wl))
    empty_i = torch.zeros(0, dtype=torch.int64, device="cuda")
    empty_h = torch.zeros((0, wl.H), dtype=torch.bfloat16, device="cuda")
    st = R.status_word()
    E = torch.zeros((0, wl.H), dtype=torch.bfloat16, device="cuda")
    vce.vce_embed_fwd(p, empty_i, W, E, dev_status=st)
    init = torch.randn((wl.Vp, wl.H), device="cuda", generator=torch.Generator("cuda").manual_seed(1))
    dW = init.clone()
    ws = D.workspace(max(vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD), 256))
    vce.vce_embed_bwd(p, empty_i, empty_h, dW, ws, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(dW, init)                      # the embedding backward accumulates nothing
    loss = torch.full((1,), float("nan"), device="cuda")
    lse = torch.zeros(0, device="cuda")
    wsf = D.workspace(max(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD), 256))
    vce.vce_loss_fwd(p, empty_h, W, empty_i, loss, lse, ws=wsf, dev_status=st)
    dH = torch.zeros((0, wl.H), device="cuda")
    wsb = D.workspace(max(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD), 256))
    vce.vce_loss_bwd(p, empty_h, W, empty_i, lse, 1.0, dH, dW, wsb, dev_status=st)
    torch.cuda.synchronize()
    assert loss.item() == 0.0
    if tied:
        assert torch.equal(dW, init)                  # accumulated into: nothing added
    else:
        assert not dW.any().item()                    # overwritten: the gradient of nothing is zero
    arg = torch.zeros(0, dtype=torch.int64, device="cuda")
    vce.vce_greedy_argmax(p, empty_h, W, arg, ws=wsf, dev_status=st)
    E2 = torch.zeros((0, wl.H), dtype=torch.bfloat16, device="cuda")
    vce.vce_ngram_embed_fwd(p, empty_i, W, W, 512, W, 512, E2, dev_status=st)
    dW2 = init.clone()
    d2 = torch.zeros((512, wl.H), device="cuda")
    wsn = D.workspace(max(vce.vce_ngram_workspace_size(p), 256))
    vce.vce_ngram_embed_bwd(p, empty_i, empty_h, dW2, d2, 512, d2, 512, wsn, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(dW2, init) and not d2.any().item()
    assert int(st.item()) == 0


def test_uneven_token_block_groups():
    """H = 8192 puts 4 MB of h in each 256-token block, so the tensor-core items
    come in groups of at most 10 token blocks. T = 5500 gives 22 blocks, the
    last one ragged, in groups of 8, 8 and 6; the backward runs in several
    column chunks (minimal workspace)."""
    wl = I.custom("groups", T=5500, H=8192, V_real=3000, Vp=3008, S=3, dtype="bf16", seed=85,
                  ignore_frac=0.05, pad_fill=8.0)
    d = I.make_all(wl, ("W", "h", "targets"))
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    out = R.loss_fwd(wl, h_d, W_d, d["targets"], maps=False)
    ref = O.cross_entropy_forward(d["h"], d["W"], d["targets"], wl.V_real)
    assert out["status"] == 0
    assert R.rel(out["loss"], ref["loss"]) <= 1e-3
    assert np.all(np.abs(out["lse"] - ref["lse"]) <= 1e-3 * np.maximum(np.abs(ref["lse"]), 1.0))
    ws_min = R.vce.vce_workspace_size_min(R.prob(wl), R.vce.VCE_OP_LOSS_BWD)
    dH, dW, st = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], ws_bytes=ws_min)
    assert st == 0
    rdH, rdW = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    assert R.max_abs_rel(dH.cpu().numpy(), rdH) <= 2e-2
    assert R.max_abs_rel(dW.cpu().numpy(), rdW) <= 2e-2
    # greedy argmax walks the same item groups
    p = R.prob(wl)
    arg = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_GREEDY_ARGMAX))
    R.vce.vce_greedy_argmax(p, h_d, W_d, arg, ws=ws)
    torch.cuda.synchronize()
    z = O.logits(d["h"], d["W"], wl.V_real)
    got = arg.cpu().numpy()
    zmax = z.max(axis=1)
    assert np.all((got >= 0) & (got < wl.V_real))
    assert np.all(z[np.arange(wl.T), got] >= zmax - 1e-3 * np.maximum(np.abs(zmax), 1.0))


@pytest.mark.parametrize("dtype,H", [("bf16", 72), ("bf16", 200), ("bf16", 8192), ("f32", 100)])
def test_hidden_sizes_off_the_tile(dtype, H):
    T, V = (256, 3000) if H < 8192 else (512, 4000)
    wl = I.custom("odd_h", T=T, H=H, V_real=V, Vp=-(-V // 64) * 64, S=3, dtype=dtype, seed=81 + H,
                  ignore_frac=0.05, pad_id_frac=0.05, oor_id_frac=0.05, pad_fill=8.0)
    d = I.make_all(wl, ("W", "h", "targets", "ids", "dE"))
    tol = TOL[dtype]
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    out = R.loss_fwd(wl, h_d, W_d, d["targets"], maps=False)
    ref = O.cross_entropy_forward(d["h"], d["W"], d["targets"], wl.V_real)
    assert out["status"] == 0
    assert R.rel(out["loss"], ref["loss"]) <= tol["loss"]
    dH, dW, st = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"])
    assert st == 0
    rdH, rdW = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    assert R.max_abs_rel(dH.cpu().numpy(), rdH) <= tol["grad"]
    assert R.max_abs_rel(dW.cpu().numpy(), rdW) <= tol["grad"]
    # the embedding at this width: lookup exact, backward exact against the fp32 replay
    got = R.embed_fwd(wl, W_d, d["ids"], maps=False)
    assert np.array_equal(got["E"], O.embed_forward(d["ids"], d["W"], wl.V_real))
    dW0 = np.random.default_rng(H).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    assert R.embed_bwd(wl, d["ids"], D.to_device(d["dE"]), dW_d) == 0
    dE32 = I.bf16_to_f32(d["dE"]) if dtype == "bf16" else d["dE"]
    want = O.embed_backward_replay_f32(d["ids"], dE32, wl.V_real, R.vce.vce_embed_bwd_chunk(), dW0)
    assert np.array_equal(dW_d.cpu().numpy().view(np.uint32), want.view(np.uint32))
