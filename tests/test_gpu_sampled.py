"""GPU parity of the sampled softmax ("Sampled Softmax with Over-Tokenized
Transformer", Setup and its loss listing) against the fp64 oracle.

The candidate list and the target positions are index work: compared exactly.
The loss over the candidates has the tolerances of the full cross-entropy
(fp32 1e-5 relative; bf16 loss and lse 1e-3 relative, dH and dW 2e-2 max-abs
relative). dW is accumulated into: rows that are not candidates must come
back bit-identical to what the caller passed in.
"""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": dict(loss=1e-5, lse=1e-5, grad=1e-5), "bf16": dict(loss=1e-3, lse=1e-3, grad=2e-2)}


def _candidates(wl, y, draws, P):
    p = R.prob(wl, T=len(y))
    cand = torch.full((P,), -7, dtype=torch.int64, device="cuda")
    pos = torch.full((len(y),), -7, dtype=torch.int64, device="cuda")
    nu = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_SAMPLED_CANDIDATES))
    st = R.status_word()
    R.vce.vce_sampled_candidates(p, torch.from_numpy(y).cuda(), torch.from_numpy(draws).cuda(), P, cand, pos, nu,
                                 ws, dev_status=st)
    torch.cuda.synchronize()
    return cand.cpu().numpy(), pos.cpu().numpy(), int(nu.item()), int(st.item())


def _sampled_loss(wl, h, W, y, draws, P, g=1.0, dW_init=None):
    T = len(y)
    p = R.prob(wl, T=T)
    dW = (torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda") if dW_init is None
          else torch.from_numpy(dW_init).cuda())
    out = dict(loss=torch.full((1,), float("nan"), device="cuda"),
               lse=torch.full((T,), float("nan"), device="cuda"),
               dH=torch.full((T, wl.H), float("nan"), device="cuda"),
               cand=torch.full((P,), -7, dtype=torch.int64, device="cuda"),
               pos=torch.full((T,), -7, dtype=torch.int64, device="cuda"),
               nu=torch.full((1,), -7, dtype=torch.int32, device="cuda"))
    ws = D.workspace(R.vce.vce_sampled_workspace_size(p, P))
    st = R.status_word()
    R.vce.vce_sampled_loss(p, D.to_device(h), D.to_device(W), torch.from_numpy(y).cuda(),
                           torch.from_numpy(draws).cuda(), P, g, out["loss"], out["lse"], out["dH"], dW,
                           out["cand"], out["pos"], out["nu"], ws, dev_status=st)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["loss"] = float(res["loss"][0])
    res["nu"] = int(res["nu"][0])
    res["dW"] = dW.cpu().numpy()
    res["status"] = int(st.item())
    return res


def _small(dtype="bf16", T=300, H=128, V_real=1000, Vp=1024, S=4, seed=21, ignore_frac=0.1):
    return I.custom("sampled_small", T=T, H=H, V_real=V_real, Vp=Vp, S=S, dtype=dtype, seed=seed,
                    ignore_frac=ignore_frac, pad_fill=8.0)


@pytest.mark.parametrize("P", [256, 300, 1000])
def test_candidates_exact(P):
    """Distinct targets ascending, then draws in order skipping targets; P up
    to the whole vocabulary (every class a candidate)."""
    wl = _small()
    y = I.make_targets(wl)
    draws = I.make_negative_draws(wl, wl.V_real)
    cand, pos, nu, st = _candidates(wl, y, draws, P)
    rc, rp, rnu = O.sampled_candidates(y, wl.V_real, P, draws)
    assert st == 0
    assert nu == rnu
    assert np.array_equal(cand, rc)
    assert np.array_equal(pos, rp)


def test_candidates_skip_out_of_range_draws_and_flag_bad_targets():
    wl = _small()
    y = I.make_targets(wl)
    y[5] = 1000           # = V_real: neither valid nor ignore_index
    y[6] = -3
    draws = I.make_negative_draws(wl, wl.V_real)
    noisy = np.insert(draws, [0, 10, 10, 500], [-1, 1000, 5000, -100]).astype(np.int64)
    cand, pos, nu, st = _candidates(wl, y, noisy, 256)
    rc, rp, rnu = O.sampled_candidates(y, wl.V_real, 256, noisy)
    assert st == R.vce.VCE_ERR_BAD_INDEX
    assert nu == rnu and np.array_equal(cand, rc) and np.array_equal(pos, rp)
    assert np.array_equal(rc, O.sampled_candidates(y, wl.V_real, 256, draws)[0])
    assert pos[5] == -100 and pos[6] == -100


@pytest.mark.parametrize("P", [400, 900])
def test_candidates_repeated_draws(P):
    """Draws with replacement (repeats inside one round of 1024 draws and
    across rounds): each class is taken once, at its first draw."""
    wl = _small()
    y = I.make_targets(wl)
    rng = np.random.default_rng(31)
    draws = rng.integers(0, wl.V_real, size=6000).astype(np.int64)
    draws[1500:1600] = draws[100:200]              # repeats of an earlier round
    draws[2100:2110] = 17                          # one value ten times in a round
    cand, pos, nu, st = _candidates(wl, y, draws, P)
    rc, rp, rnu = O.sampled_candidates(y, wl.V_real, P, draws)
    assert st == 0
    assert nu == rnu and np.array_equal(cand, rc) and np.array_equal(pos, rp)
    assert np.unique(cand).size == P


def test_candidates_data_errors():
    wl = _small(T=300, ignore_frac=0.0)
    # more distinct targets than candidates: empty list, every target ignored
    y = np.arange(300, dtype=np.int64)
    draws = I.make_negative_draws(wl, wl.V_real)
    cand, pos, nu, st = _candidates(wl, y, draws, 256)
    assert st == R.vce.VCE_ERR_ARG and nu == 300
    assert np.all(cand == -1) and np.all(pos == -100)
    # too few usable draws: the list is filled as far as they go, then -1
    y = (np.arange(300) % 100).astype(np.int64) * 7
    short = draws[:50]
    cand, pos, nu, st = _candidates(wl, y, short, 256)
    assert st == R.vce.VCE_ERR_ARG and nu == 100
    uniq = np.unique(y)
    negs = [d for d in short if d not in set(uniq.tolist())]
    assert np.array_equal(cand[:100], uniq)
    assert np.array_equal(cand[100:100 + len(negs)], negs)
    assert np.all(cand[100 + len(negs):] == -1)
    assert np.array_equal(pos, np.searchsorted(uniq, y))


def _loss_check(wl, P, g=1.0, init_scale=1e-4):
    d = I.make_all(wl, ("W", "h", "targets"))
    h, W, y = d["h"], d["W"], d["targets"]
    draws = I.make_negative_draws(wl, wl.V_real)
    rng = np.random.default_rng(77)
    dW_init = (rng.standard_normal((wl.Vp, wl.H)) * init_scale).astype(np.float32)
    out = _sampled_loss(wl, h, W, y, draws, P, g=g, dW_init=dW_init)
    cand, pos, nu = O.sampled_candidates(y, wl.V_real, P, draws)
    ref = O.sampled_cross_entropy(h, W, y, wl.V_real, wl.Vp, cand, pos, g=g)
    tol = TOL[wl.dtype]
    assert out["status"] == 0
    assert out["nu"] == nu and np.array_equal(out["cand"], cand) and np.array_equal(out["pos"], pos)
    # the library reports the plain mean; the oracle's loss carries the weight g
    assert R.rel(g * out["loss"], ref["loss"]) <= tol["loss"]
    valid = (y >= 0) & (y < wl.V_real)
    assert np.all(np.abs(out["lse"][valid] - ref["lse"][valid])
                  <= tol["lse"] * np.maximum(np.abs(ref["lse"][valid]), 1.0))
    assert R.max_abs_rel(out["dH"], ref["dH"]) <= tol["grad"]
    assert np.all(out["dH"][~valid] == 0)
    # candidate rows: dW_init + dWc (one rounding); every other row untouched
    got = out["dW"][cand].astype(np.float64) - dW_init[cand].astype(np.float64)
    assert R.max_abs_rel(got, ref["dW_cand"]) <= tol["grad"]
    others = np.ones(wl.Vp, dtype=bool)
    others[cand] = False
    assert np.array_equal(out["dW"][others].view(np.uint32), dW_init[others].view(np.uint32))
    return out, ref


@pytest.mark.parametrize("P", [256, 300])
def test_sampled_loss_bf16_small(P):
    """T=300 (231 distinct targets), H=128, V_real=1000 -> 1024, S=4, 10%
    ignored; P a multiple of 64 and not (the candidate table then has zero
    padding rows)."""
    _loss_check(_small(), P, g=0.7)


def test_sampled_loss_f32_tiny():
    _loss_check(_small(dtype="f32", T=64, H=64, seed=22), 128, init_scale=0.0)


def test_sampled_loss_whole_vocabulary_equals_full_loss():
    """P = V_real: every class is a candidate, so the sampled loss is the full
    loss (same lse per token) up to the order of the columns."""
    wl = _small(T=256, H=64, V_real=640, Vp=640, S=2, seed=23)
    d = I.make_all(wl, ("W", "h", "targets"))
    out = _sampled_loss(wl, d["h"], d["W"], d["targets"], I.make_negative_draws(wl, wl.V_real), wl.V_real)
    full = O.cross_entropy_forward(d["h"], d["W"], d["targets"], wl.V_real)
    assert R.rel(out["loss"], full["loss"]) <= 1e-3


def test_sampled_loss_empty_batch():
    wl = _small(T=0)
    W = I.make_W(wl)
    draws = I.make_negative_draws(wl, wl.V_real)
    dW_init = np.random.default_rng(5).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    out = _sampled_loss(wl, np.zeros((0, wl.H), np.uint16), W, np.zeros(0, np.int64), draws, 64, dW_init=dW_init)
    assert out["status"] == 0 and out["nu"] == 0
    assert np.array_equal(out["cand"], draws[:64])
    assert out["loss"] == 0.0
    assert np.array_equal(out["dW"].view(np.uint32), dW_init.view(np.uint32))


def test_sampled_loss_full_size():
    """T=16384, H=2048, V=151936, P=8192, Zipf next-token targets: the exact
    candidate list, and the loss, every lse, all of dH and the candidate rows
    of dW against the oracle over the whole batch."""
    wl = I.WORKLOADS["sampled"]
    P = I.SAMPLED_P
    d = I.make_all(wl, ("W", "h", "targets"))
    h, W, y = d["h"], d["W"], d["targets"]
    draws = I.make_negative_draws(wl, P)
    out = _sampled_loss(wl, h, W, y, draws, P)
    cand, pos, nu = O.sampled_candidates(y, wl.V_real, P, draws)
    assert out["status"] == 0
    assert out["nu"] == nu and np.array_equal(out["cand"], cand) and np.array_equal(out["pos"], pos)
    ref = O.sampled_cross_entropy(h, W, y, wl.V_real, wl.Vp, cand, pos)
    tol = TOL["bf16"]
    assert R.rel(out["loss"], ref["loss"]) <= tol["loss"]
    assert np.all(np.abs(out["lse"] - ref["lse"]) <= tol["lse"] * np.abs(ref["lse"]))
    assert R.max_abs_rel(out["dH"], ref["dH"]) <= tol["grad"]
    assert R.max_abs_rel(out["dW"][cand], ref["dW_cand"]) <= tol["grad"]
    others = np.ones(wl.Vp, dtype=bool)
    others[cand] = False
    assert not out["dW"][others].any()
