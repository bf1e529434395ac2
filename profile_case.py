"""Small, self-contained invocations of the library for a profiler.

    python profile_case.py loss    [--workload NAME] [--tokens T] [--iters N]
    python profile_case.py embed   [--workload NAME] [--iters N] [--split]
    python profile_case.py sampled [--tokens T] [--iters N]
    python profile_case.py ngram   [--rows M] [--iters N]

`loss` runs the loss forward and backward on a named workload's shapes
(default the Qwen3-like H=2048, V=151936, S=8, tied dW), with T tokens or the
workload's own; `embed` runs the embedding lookup and its backward on a named
workload (with --split: the lookup with the backward's plan made beside it,
then the plan's application); `sampled` runs vce_sampled_loss (P=8192) with T tokens (default
2048); `ngram` runs the hashed n-gram lookup and its one-call backward on the
Qwen3-like ids (T=8192 in sequences of 2048, H=2048) with two tables of M rows
(default 2^16). Inputs are the seeded synthetic ones of `inputs.py`. Each case checks
the device status word and exits non-zero on any error, so that a profiler is
only pointed at a command that has already run cleanly.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from vocab_embedding_cross_gb300 import _lib as vce  # noqa: E402
from vocab_embedding_cross_gb300 import device as D  # noqa: E402
from vocab_embedding_cross_gb300 import inputs as I  # noqa: E402


def _loss(args):
    wl = I.WORKLOADS[args.workload]
    if args.tokens:
        wl = I.with_T(wl, args.tokens)
    d = I.make_all(wl, ("W", "h", "targets"))
    p = vce.problem(wl.T, wl.H, wl.Vp, wl.V_real, wl.S, vce.VCE_BF16, tied=wl.tied)
    W, h = D.to_device(d["W"]), D.to_device(d["h"])
    y = torch.from_numpy(d["targets"]).cuda()
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(wl.T, device="cuda")
    dH = torch.empty((wl.T, wl.H), device="cuda")
    dW = torch.zeros((wl.Vp, wl.H), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_f = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD))
    ws_b = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD))
    for _ in range(args.iters):
        vce.vce_loss_fwd(p, h, W, y, loss, lse, ws=ws_f, dev_status=st)
        vce.vce_loss_bwd(p, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st)
    torch.cuda.synchronize()
    return int(st.item()), f"loss {loss.item():.6f}"


def _embed(args):
    wl = I.WORKLOADS[args.workload]
    d = I.make_all(wl, ("W", "ids", "dE"))
    p = vce.problem(wl.T, wl.H, wl.Vp, wl.V_real, wl.S, vce.VCE_BF16 if wl.dtype == "bf16" else vce.VCE_F32,
                    tied=wl.tied)
    W = D.to_device(d["W"])
    ids = torch.from_numpy(d["ids"]).cuda()
    dE = D.to_device(d["dE"])
    E = torch.empty((wl.T, wl.H), dtype=W.dtype, device="cuda")
    dW = torch.zeros((wl.Vp, wl.H), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD))
    for _ in range(args.iters):
        if args.split:   # the lookup with the backward's plan beside it, then the plan's application
            vce.vce_embed_fwd_plan(p, ids, W, E, ws, dev_status=st)
            vce.vce_embed_bwd_apply(p, dE, dW, ws, dev_status=st)
        else:
            vce.vce_embed_fwd(p, ids, W, E, dev_status=st)
            vce.vce_embed_bwd(p, ids, dE, dW, ws, dev_status=st)
    torch.cuda.synchronize()
    return int(st.item()), "embedding ok"


def _sampled(args):
    wl = I.with_T(I.WORKLOADS["sampled"], args.tokens or 2048)
    P = I.SAMPLED_P
    d = I.make_all(wl, ("W", "h", "targets"))
    p = vce.problem(wl.T, wl.H, wl.Vp, wl.V_real, wl.S, vce.VCE_BF16)
    W, h = D.to_device(d["W"]), D.to_device(d["h"])
    y = torch.from_numpy(d["targets"]).cuda()
    draws = torch.from_numpy(I.make_negative_draws(wl, P)).cuda()
    loss = torch.empty(1, device="cuda")
    dH = torch.empty((wl.T, wl.H), device="cuda")
    dW = torch.zeros((wl.Vp, wl.H), device="cuda")
    cand = torch.empty(P, dtype=torch.int64, device="cuda")
    pos = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    nu = torch.empty(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = D.workspace(vce.vce_sampled_workspace_size(p, P))
    for _ in range(args.iters):
        vce.vce_sampled_loss(p, h, W, y, draws, P, 1.0, loss, None, dH, dW, cand, pos, nu, ws, dev_status=st)
    torch.cuda.synchronize()
    return int(st.item()), f"loss {loss.item():.6f}, {int(nu.item())} distinct targets"


def _ngram(args):
    wl = I.WORKLOADS["qwen3_tied"]
    M, L = args.rows, I.NGRAM_SEQ_LEN
    d = I.make_all(wl, ("W", "ids", "dE"))
    p = vce.problem(wl.T, wl.H, wl.Vp, wl.V_real, wl.S, vce.VCE_BF16)
    W, dE = D.to_device(d["W"]), D.to_device(d["dE"])
    T2, T3 = D.to_device(I.make_ngram_table(wl, 2, M)), D.to_device(I.make_ngram_table(wl, 3, M))
    ids = torch.from_numpy(d["ids"]).cuda()
    E = torch.empty((wl.T, wl.H), dtype=W.dtype, device="cuda")
    dW = torch.zeros((wl.Vp, wl.H), device="cuda")
    dT2 = torch.zeros((M, wl.H), device="cuda")
    dT3 = torch.zeros((M, wl.H), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = D.workspace(vce.vce_ngram_workspace_size(p))
    for _ in range(args.iters):
        vce.vce_ngram_embed_fwd(p, ids, W, T2, M, T3, M, E, seq_len=L, dev_status=st)
        vce.vce_ngram_embed_bwd(p, ids, dE, dW, dT2, M, dT3, M, ws, seq_len=L, dev_status=st)
    torch.cuda.synchronize()
    return int(st.item()), f"n-gram tables of {M} rows ok"


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("case", choices=["loss", "embed", "sampled", "ngram"])
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--workload", default="qwen3_tied")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--rows", type=int, default=1 << 16, help="ngram: rows of each hashed table")
    ap.add_argument("--split", action="store_true",
                    help="embed: vce_embed_fwd_plan and vce_embed_bwd_apply instead of the lookup and the one-call backward")
    args = ap.parse_args(argv)
    status, msg = {"loss": _loss, "embed": _embed, "sampled": _sampled, "ngram": _ngram}[args.case](args)
    print(f"{args.case}: status {status} ({vce.status_str(status)}); {msg}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
