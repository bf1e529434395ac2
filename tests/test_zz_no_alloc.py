"""The loss forward for callers that cannot allocate device memory.

vce_loss_fwd_noalloc must give what vce_loss_fwd gives (same kernels, its
scratch in the library's fixed device array instead of a caller workspace),
call after call, and must refuse problems that do not fit the fixed scratch
before enqueuing anything. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import vce_run as R
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-3}   # the loss tolerances of the parity tests


def _outputs(T):
    z = lambda dt=torch.float32: torch.full((T,), float("nan") if dt == torch.float32 else -7, dtype=dt,
                                            device="cuda")
    return dict(loss=torch.full((1,), float("nan"), device="cuda"), lse=z(), tl=z(),
                to=z(torch.int32), mo=z(torch.int32), st=torch.zeros(1, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_workspace_call_twice(dtype):
    wl = I.custom(T=300, H=192, V_real=1000, Vp=1024, S=3, dtype=dtype, seed=41, ignore_frac=0.1)
    d = I.make_all(wl, ("W", "h", "targets"))
    p = R.prob(wl)
    h, W = D.to_device(d["h"]), D.to_device(d["W"])
    y = torch.from_numpy(d["targets"]).cuda()
    ref = _outputs(wl.T)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_LOSS_FWD))
    R.vce.vce_loss_fwd(p, h, W, y, ref["loss"], ref["lse"], ref["tl"], ref["to"], ref["mo"], ws,
                       dev_status=ref["st"])
    for _ in range(2):                       # two calls in a row share the one scratch array
        got = _outputs(wl.T)
        R.vce.vce_loss_fwd_noalloc(p, h, W, y, got["loss"], got["lse"], got["tl"], got["to"], got["mo"],
                                   dev_status=got["st"])
        torch.cuda.synchronize()
        assert int(got["st"].item()) == int(ref["st"].item()) == 0
        tol = TOL[dtype]
        assert abs(got["loss"].item() - ref["loss"].item()) <= tol * abs(ref["loss"].item())
        assert torch.all((got["lse"] - ref["lse"]).abs() <= tol * ref["lse"].abs().clamp(min=1.0)).item()
        assert (got["tl"] - ref["tl"]).abs().max().item() <= tol * ref["tl"].abs().max().item()
        assert torch.equal(got["to"], ref["to"]) and torch.equal(got["mo"], ref["mo"])


def test_noalloc_without_status_word():
    wl = I.custom(T=64, H=64, V_real=500, Vp=512, S=2, dtype="bf16", seed=42)
    d = I.make_all(wl, ("W", "h", "targets"))
    p = R.prob(wl)
    h, W = D.to_device(d["h"]), D.to_device(d["W"])
    y = torch.from_numpy(d["targets"]).cuda()
    a, b = _outputs(wl.T), _outputs(wl.T)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_LOSS_FWD))
    R.vce.vce_loss_fwd(p, h, W, y, a["loss"], a["lse"], ws=ws)
    R.vce.vce_loss_fwd_noalloc(p, h, W, y, b["loss"], b["lse"])
    torch.cuda.synchronize()
    assert abs(a["loss"].item() - b["loss"].item()) <= 1e-3 * abs(a["loss"].item())


def test_noalloc_rejects_problems_larger_than_its_scratch():
    cap = R.vce.vce_loss_fwd_noalloc_max_scratch()
    assert cap == 16 << 20
    wl = I.custom(T=40000, H=64, V_real=100000, Vp=100032, S=8, dtype="bf16", seed=43)
    p = R.prob(wl)
    assert R.vce.vce_workspace_size(p, R.vce.VCE_OP_LOSS_FWD) > cap
    h = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((wl.Vp, wl.H), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(wl.T, dtype=torch.int64, device="cuda")
    out = _outputs(wl.T)
    with pytest.raises(R.vce.VceError) as e:
        R.vce.vce_loss_fwd_noalloc(p, h, W, y, out["loss"], out["lse"])
    assert e.value.status == R.vce.VCE_ERR_WORKSPACE
    # the refusal says why: the scratch this problem needs and the array's size
    why = R.vce.lib().vce_last_error().decode()
    need = R.vce.vce_workspace_size(p, R.vce.VCE_OP_LOSS_FWD)
    assert "vce_loss_fwd_noalloc" in why and str(need) in why and str(cap) in why, why
    torch.cuda.synchronize()
    assert torch.isnan(out["loss"]).all().item()     # nothing was enqueued


def test_noalloc_accepts_the_bf16_dh_flag():
    """A problem that carries VCE_FLAG_DH_BF16 for its backward runs through
    both forwards unchanged (the flag concerns the backward only)."""
    wl = I.custom(T=200, H=128, V_real=900, Vp=960, S=4, dtype="bf16", seed=44)
    d = I.make_all(wl, ("W", "h", "targets"))
    p = R.prob(wl, flags=R.vce.VCE_FLAG_DH_BF16)
    h, W = D.to_device(d["h"]), D.to_device(d["W"])
    y = torch.from_numpy(d["targets"]).cuda()
    a, b = _outputs(wl.T), _outputs(wl.T)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_LOSS_FWD))
    R.vce.vce_loss_fwd(p, h, W, y, a["loss"], a["lse"], ws=ws, dev_status=a["st"])
    R.vce.vce_loss_fwd_noalloc(p, h, W, y, b["loss"], b["lse"], dev_status=b["st"])
    torch.cuda.synchronize()
    assert int(a["st"].item()) == int(b["st"].item()) == 0
    assert torch.equal(a["loss"], b["loss"]) and torch.equal(a["lse"], b["lse"])
