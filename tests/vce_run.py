"""Test helpers: run the library through its C ABI on seeded inputs and
bring the results back as numpy arrays. No method arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

from vocab_embedding_cross_gb300 import _lib as vce
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I


def code(wl) -> int:
    return vce.VCE_BF16 if wl.dtype == "bf16" else vce.VCE_F32


def prob(wl, **over):
    kw = dict(T=wl.T, H=wl.H, Vp=wl.Vp, V_real=wl.V_real, S=wl.S, dtype=code(wl), tied=wl.tied)
    kw.update(over)
    return vce.problem(**kw)


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def embed_fwd(wl, W_d, ids_np, maps=True):
    p = prob(wl, T=len(ids_np))
    ids = torch.from_numpy(ids_np).cuda()
    T = len(ids_np)
    E = torch.full((T, wl.H), 7, dtype=W_d.dtype, device="cuda")   # poisoned: every row must be written
    owner = torch.full((T,), -7, dtype=torch.int32, device="cuda") if maps else None
    local = torch.full((T,), -7, dtype=torch.int32, device="cuda") if maps else None
    vce.vce_embed_fwd(p, ids, W_d, E, owner, local)
    torch.cuda.synchronize()
    out = dict(E=D.to_host_bits(E))
    if maps:
        out.update(owner=owner.cpu().numpy(), local=local.cpu().numpy())
    return out


def embed_bwd(wl, ids_np, dE_d, dW_init: torch.Tensor):
    p = prob(wl, T=len(ids_np))
    ids = torch.from_numpy(ids_np).cuda()
    ws = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD))
    st = status_word()
    vce.vce_embed_bwd(p, ids, dE_d, dW_init, ws, dev_status=st)
    torch.cuda.synchronize()
    return int(st.item())


def loss_fwd(wl, h_d, W_d, targets_np, maps=True):
    p = prob(wl, T=len(targets_np))
    T = len(targets_np)
    y = torch.from_numpy(targets_np).cuda()
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
    tl = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
    to = torch.full((T,), -7, dtype=torch.int32, device="cuda") if maps else None
    mo = torch.full((T,), -7, dtype=torch.int32, device="cuda") if maps else None
    ws = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD))
    st = status_word()
    vce.vce_loss_fwd(p, h_d, W_d, y, loss, lse, tl, to, mo, ws, dev_status=st)
    torch.cuda.synchronize()
    out = dict(loss=float(loss.item()), lse=lse.cpu().numpy(), token_loss=tl.cpu().numpy(),
               status=int(st.item()), lse_d=lse, targets_d=y)
    if maps:
        out.update(target_owner=to.cpu().numpy(), max_owner=mo.cpu().numpy())
    return out


def loss_bwd(wl, h_d, W_d, targets_d, lse_d, g=1.0, dW: torch.Tensor = None, ws_bytes=None, tied=None):
    T = targets_d.shape[0]
    p = prob(wl, T=T, **({} if tied is None else {"tied": tied}))
    dH = torch.full((T, wl.H), float("nan"), dtype=torch.float32, device="cuda")
    if dW is None:
        dW = torch.full((wl.Vp, wl.H), float("nan"), dtype=torch.float32, device="cuda")
    nb = vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD) if ws_bytes is None else ws_bytes
    ws = D.workspace(nb)
    st = status_word()
    vce.vce_loss_bwd(p, h_d, W_d, targets_d, lse_d, g, dH, dW, ws, ws_bytes=nb, dev_status=st)
    torch.cuda.synchronize()
    return dH, dW, int(st.item())


def rel(a, b):
    return abs(a - b) / max(abs(b), 1e-30)


def max_abs_rel(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(gpu - ref).max() / (den if den > 0 else 1.0))


def upload(wl, d):
    return {k: (D.to_device(v) if k in ("W", "h", "dE") else v) for k, v in d.items()}


__all__ = ["I", "D", "vce"]
