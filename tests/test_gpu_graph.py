"""The library's calls are stream-ordered and allocate nothing, so a whole
training step can be captured in a CUDA graph and replayed. Replays must give
the same bits as the eager calls (every kernel on the path is deterministic)."""
import numpy as np
import pytest
import torch

import vce_run as R
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_step_in_a_cuda_graph(dtype):
    wl = I.custom("graph_step", T=1000, H=256, V_real=5000, Vp=5056, S=8, dtype=dtype, seed=90, tied=True,
                  ignore_frac=0.05, pad_id_frac=0.02, oor_id_frac=0.02)
    d = I.make_all(wl)
    vce = R.vce
    p = R.prob(wl)
    W, h, dE = D.to_device(d["W"]), D.to_device(d["h"]), D.to_device(d["dE"])
    ids = torch.from_numpy(d["ids"]).cuda()
    y = torch.from_numpy(d["targets"]).cuda()
    E = torch.empty((wl.T, wl.H), dtype=W.dtype, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(wl.T, device="cuda")
    dH = torch.empty((wl.T, wl.H), device="cuda")
    dW = torch.empty((wl.Vp, wl.H), device="cuda")
    st = R.status_word()
    ws_f = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD))
    ws_b = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD))
    ws_e = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD))

    def step():
        dW.zero_()
        vce.vce_embed_fwd(p, ids, W, E, dev_status=st)
        vce.vce_loss_fwd(p, h, W, y, loss, lse, ws=ws_f, dev_status=st)
        vce.vce_loss_bwd(p, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st)
        vce.vce_embed_bwd(p, ids, dE, dW, ws_e, dev_status=st)

    step()
    torch.cuda.synchronize()
    ref = [x.clone() for x in (E, loss, lse, dH, dW)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        for x in (E, loss, lse, dH, dW):
            x.fill_(float("nan")) if x.is_floating_point() else x.zero_()
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip((E, loss, lse, dH, dW), ref):
            assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))
    assert int(st.item()) == 0
