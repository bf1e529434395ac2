"""GPU parity of the sharded greedy argmax ("Tensor Parallelism (TP)",
on-device sampling) against the fp64 oracle.

The argmax is an integer decided by floating point: where the oracle's two
largest logits of a token are further apart than the logit error bound, the
GPU's class must equal the oracle's exactly; elsewhere (a near tie) the GPU's
class must hold a logit within the bound of the maximum. The owner map is
always the shard of the returned class. Exact ties (duplicate rows) must go to
the lowest class. max_logit: fp32 1e-5, bf16 1e-3 relative (floor 1).
"""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-3}


def _argmax(wl, h, W):
    T = h.shape[0]
    p = R.prob(wl, T=T)
    arg = torch.full((T,), -7, dtype=torch.int64, device="cuda")
    mx = torch.full((T,), float("nan"), device="cuda")
    own = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_GREEDY_ARGMAX))
    st = R.status_word()
    R.vce.vce_greedy_argmax(p, D.to_device(h), D.to_device(W), arg, mx, own, ws, dev_status=st)
    torch.cuda.synchronize()
    return arg.cpu().numpy(), mx.cpu().numpy(), own.cpu().numpy(), int(st.item())


def _check(wl, h, W, rows=None):
    arg, mx, own, st = _argmax(wl, h, W)
    assert st == 0
    if rows is None:
        rows = np.arange(h.shape[0])
    z = O.logits(h[rows], W, wl.V_real)
    ref_arg, ref_m = O.greedy_argmax(h[rows], W, wl.V_real)
    tol = TOL[wl.dtype] * np.maximum(np.abs(ref_m), 1.0)
    top2 = np.sort(z, axis=1)[:, -2:] if z.shape[1] > 1 else np.concatenate([z, z], 1)
    clear = (top2[:, 1] - top2[:, 0]) > 4 * tol
    got = arg[rows]
    assert np.all((got >= 0) & (got < wl.V_real))
    assert np.array_equal(got[clear], ref_arg[clear])
    assert np.all(z[np.arange(len(rows)), got] >= ref_m - 4 * tol)
    assert np.all(np.abs(mx[rows] - ref_m) <= tol)
    assert np.array_equal(own, O.ownership(arg, wl.V_real, wl.Vp, wl.S)[1].astype(np.int32))
    return clear.mean()


def test_argmax_tiny_f32():
    """fp32, T=64, V_real=1000 -> 1024, S=4, padded rows 8.0 (they must never
    win), maxima injected into shards that do not own the target."""
    wl = I.WORKLOADS["tiny_f32"]
    d = I.make_all(wl, ("W", "h"))
    assert _check(wl, d["h"], d["W"]) > 0.9


@pytest.mark.parametrize("T,V_real,Vp,S", [(300, 1000, 1024, 4), (129, 4000, 4032, 7), (520, 20000, 20032, 8)])
def test_argmax_bf16_ragged(T, V_real, Vp, S):
    wl = I.custom("argmax_bf16", T=T, H=256, V_real=V_real, Vp=Vp, S=S, dtype="bf16", seed=50 + S, pad_fill=8.0,
                  w_std=0.05)
    d = I.make_all(wl, ("W", "h"))
    assert _check(wl, d["h"], d["W"]) > 0.9


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_exact_ties_go_to_the_lowest_class(dtype):
    """Row 700 (shard 2 of 4) duplicated at rows 100 (shard 0) and 900
    (shard 3), and rows 5 and 6 equal inside one shard: h along those rows must
    return 100 and 5."""
    wl = I.custom("argmax_ties", T=64, H=64, V_real=1000, Vp=1024, S=4, dtype=dtype, seed=60, pad_fill=8.0)
    W = I.make_W(wl)
    W[100] = W[700]
    W[900] = W[700]
    W[6] = W[5]
    Wf = I.to_f64(W, wl.dtype)
    h32 = np.zeros((wl.T, wl.H), dtype=np.float32)
    h32[0::2] = (20.0 * Wf[700] / np.linalg.norm(Wf[700])).astype(np.float32)
    h32[1::2] = (20.0 * Wf[5] / np.linalg.norm(Wf[5])).astype(np.float32)
    h = I.bf16_bits(h32) if dtype == "bf16" else h32
    arg, _, own, st = _argmax(wl, h, W)
    assert st == 0
    assert np.all(arg[0::2] == 100) and np.all(own[0::2] == 0)
    assert np.all(arg[1::2] == 5)


def test_argmax_qwen3_full_size():
    """T=8192, H=2048, V=151936, S=8 (the tied workload's inputs): sampled
    tokens against the oracle, every class in range, owners consistent."""
    wl = I.WORKLOADS["qwen3_tied"]
    d = I.make_all(wl, ("W", "h"))
    rows = np.unique(np.concatenate([np.random.default_rng(3).choice(wl.T, 64, replace=False), [0, wl.T - 1]]))
    assert _check(wl, d["h"], d["W"], rows=rows) > 0.5
