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


@pytest.mark.parametrize("dtype,split", [("bf16", None), ("f32", None), ("bf16", "plan"), ("f32", "plan"),
                                         ("bf16", "lookup_plan"), ("f32", "lookup_plan")])
def test_step_in_a_cuda_graph(dtype, split):
    """split: the embedding backward as its plan (made after the lookup, or
    beside it by vce_embed_fwd_plan, the order bench.py runs) and the plan's
    application."""
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
        if split == "lookup_plan":
            vce.vce_embed_fwd_plan(p, ids, W, E, ws_e, dev_status=st)
        else:
            vce.vce_embed_fwd(p, ids, W, E, dev_status=st)
        if split == "plan":
            vce.vce_embed_bwd_plan(p, ids, ws_e, dev_status=st)
        vce.vce_loss_fwd(p, h, W, y, loss, lse, ws=ws_f, dev_status=st)
        vce.vce_loss_bwd(p, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st)
        if split:
            vce.vce_embed_bwd_apply(p, dE, dW, ws_e, dev_status=st)
        else:
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


def test_wider_entries_in_a_cuda_graph_and_on_a_side_stream():
    """The sampled loss, the greedy argmax, the n-gram embeddings (three tables
    reduced in one launch) and a bf16-dH backward: captured in one graph and
    replayed, and run eagerly on a second stream; every result bit-identical to
    the eager run on the current stream."""
    wl = I.custom("graph_wide", T=600, H=128, V_real=3000, Vp=3008, S=4, dtype="bf16", seed=91,
                  ignore_frac=0.05, pad_id_frac=0.02, oor_id_frac=0.02)
    d = I.make_all(wl)
    vce = R.vce
    p = R.prob(wl, tied=False)
    pb = R.prob(wl, tied=False, flags=vce.VCE_FLAG_DH_BF16)
    W, h, dE = D.to_device(d["W"]), D.to_device(d["h"]), D.to_device(d["dE"])
    ids = torch.from_numpy(d["ids"]).cuda()
    y = torch.from_numpy(d["targets"]).cuda()
    draws = torch.from_numpy(I.make_negative_draws(wl, wl.V_real)).cuda()
    P, M2, M3 = 700, 613, 1024
    T2 = D.to_device(I.make_ngram_table(wl, 2, M2))
    T3 = D.to_device(I.make_ngram_table(wl, 3, M3))
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(wl.T, device="cuda")
    dHs = torch.empty((wl.T, wl.H), device="cuda")
    dWs = torch.empty((wl.Vp, wl.H), device="cuda")
    cand = torch.empty(P, dtype=torch.int64, device="cuda")
    pos = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    nu = torch.empty(1, dtype=torch.int32, device="cuda")
    arg = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    En = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    dWn = torch.empty((wl.Vp, wl.H), device="cuda")
    dT2 = torch.empty((M2, wl.H), device="cuda")
    dT3 = torch.empty((M3, wl.H), device="cuda")
    dHb = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    dWb = torch.empty((wl.Vp, wl.H), device="cuda")
    lse_b = torch.empty(wl.T, device="cuda")
    loss_b = torch.empty(1, device="cuda")
    st = R.status_word()
    ws_s = D.workspace(vce.vce_sampled_workspace_size(p, P))
    ws_a = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_GREEDY_ARGMAX))
    ws_n = D.workspace(vce.vce_ngram_workspace_size(p))
    ws_f = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD))
    ws_b = D.workspace(vce.vce_workspace_size(pb, vce.VCE_OP_LOSS_BWD))
    outs = (loss, dHs, dWs, cand, pos, nu, arg, En, dWn, dT2, dT3, dHb, dWb)

    def run():
        for x in (dWs, dWn, dT2, dT3):
            x.zero_()
        vce.vce_sampled_loss(p, h, W, y, draws, P, 1.0, loss, None, dHs, dWs, cand, pos, nu, ws_s, dev_status=st)
        vce.vce_greedy_argmax(p, h, W, arg, ws=ws_a, dev_status=st)
        vce.vce_ngram_embed_fwd(p, ids, W, T2, M2, T3, M3, En, seq_len=150, dev_status=st)
        vce.vce_ngram_embed_bwd(p, ids, dE, dWn, dT2, M2, dT3, M3, ws_n, seq_len=150, dev_status=st)
        vce.vce_loss_fwd(p, h, W, y, loss_b, lse_b, ws=ws_f, dev_status=st)
        vce.vce_loss_bwd(pb, h, W, y, lse_b, 1.0, dHb, dWb, ws_b, dev_status=st)

    run()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    ref = [x.clone() for x in outs]

    def check():
        for got, want in zip(outs, ref):
            assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))

    def poison():
        for x in outs:
            x.fill_(float("nan")) if x.is_floating_point() else x.fill_(-7)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    poison()
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    check()
    g = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            run()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        poison()
        g.replay()
        torch.cuda.synchronize()
        check()
    assert int(st.item()) == 0
