"""GPU parity of the globally normalised cross-entropy (forward and backward)
against the fp64 oracle on the same seeded (bf16-rounded) inputs.

Tolerances: fp32 problems 1e-5 relative for everything; bf16 problems (fp32
accumulation on the tensor cores, G in bf16) loss and lse 1e-3 relative, dH
and dW 2e-2 max-abs relative (max|gpu - ref| / max|ref| per tensor). Owner
maps are compared exactly.
"""
import time

import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": dict(loss=1e-5, lse=1e-5, grad=1e-5), "bf16": dict(loss=1e-3, lse=1e-3, grad=2e-2)}


def _fwd_check(wl, d, tol, out=None):
    h, W, y = d["h"], d["W"], d["targets"]
    if out is None:
        out = R.loss_fwd(wl, D.to_device(h), D.to_device(W), y)
    ref = O.cross_entropy_forward(h, W, y, wl.V_real)
    assert out["status"] == (R.vce.VCE_ERR_BAD_INDEX if ref["bad"].any() else 0)
    assert R.rel(out["loss"], ref["loss"]) <= tol["loss"] or (ref["loss"] == 0 and out["loss"] == 0)
    assert np.all(np.abs(out["lse"] - ref["lse"]) <= tol["lse"] * np.maximum(np.abs(ref["lse"]), 1.0))
    assert R.max_abs_rel(out["token_loss"], ref["token_loss"]) <= tol["loss"]
    assert np.array_equal(out["target_owner"], O.target_owner(y, wl.V_real, wl.Vp, wl.S).astype(np.int32))
    own, gap = O.max_owner(h, W, wl.V_real, wl.Vp, wl.S)
    clear = gap > 4 * tol["lse"] * np.maximum(1.0, np.abs(ref["lse"]))
    assert np.array_equal(out["max_owner"][clear], own[clear].astype(np.int32))
    return out, ref


def _bwd_check(wl, d, out, tol, g=1.0):
    h, W, y = d["h"], d["W"], d["targets"]
    dH, dW, st = R.loss_bwd(wl, D.to_device(h), D.to_device(W), out["targets_d"], out["lse_d"], g=g,
                            dW=torch.full((wl.Vp, wl.H), 0.0 if wl.tied else float("nan"),
                                          dtype=torch.float32, device="cuda"))
    rdH, rdW = O.cross_entropy_backward(h, W, y, wl.V_real, wl.Vp, g=g)
    dH, dW = dH.cpu().numpy(), dW.cpu().numpy()
    assert R.max_abs_rel(dH, rdH) <= tol["grad"]
    assert R.max_abs_rel(dW, rdW) <= tol["grad"]
    assert np.all(dW[wl.V_real:] == 0)
    ign = ~((y >= 0) & (y < wl.V_real))
    assert np.all(dH[ign] == 0)
    return dH, dW


def test_loss_tiny_f32():
    """fp32, T=64, H=64, V_real=1000 -> 1024, S=4: boundary targets 255, 256,
    511, 512, 999, maxima injected in other shards, garbage padded rows 8.0."""
    wl = I.WORKLOADS["tiny_f32"]
    d = I.make_all(wl, ("W", "h", "targets"))
    out, ref = _fwd_check(wl, d, TOL["f32"])
    # the injected maxima really sit in another shard than the target
    assert np.all(out["max_owner"][5:9] != out["target_owner"][5:9])
    _bwd_check(wl, d, out, TOL["f32"])
    _bwd_check(wl, d, out, TOL["f32"], g=0.37)


BF16_CASES = [
    dict(T=300, H=192, V_real=1000, Vp=1024, S=3),     # ragged T, K and vocab
    dict(T=1, H=64, V_real=50, Vp=64, S=1),
    dict(T=129, H=256, V_real=4000, Vp=4032, S=7),
    dict(T=64, H=128, V_real=700, Vp=1024, S=4),       # last shard only padding
    dict(T=16, H=64, V_real=60, Vp=64, S=64),          # one row per shard
    dict(T=520, H=1024, V_real=9000, Vp=9024, S=8, ignore_frac=0.3),
]


@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: "T{T}_H{H}_V{V_real}_S{S}".format(**c))
def test_loss_bf16_cases(case):
    wl = I.custom(dtype="bf16", seed=21, ignore_frac=case.pop("ignore_frac", 0.05), **case)
    d = I.make_all(wl, ("W", "h", "targets"))
    out, _ = _fwd_check(wl, d, TOL["bf16"])
    _bwd_check(wl, d, out, TOL["bf16"])


def test_loss_bf16_boundaries_and_injected_max():
    """The tiny case's forced targets and injected maxima, in bf16 through the
    tensor-core kernels."""
    base = I.WORKLOADS["tiny_f32"]
    wl = I.custom(T=64, H=64, V_real=1000, Vp=1024, S=4, dtype="bf16", seed=0, ignore_frac=0.1,
                  forced_targets=base.forced_targets, injected=base.injected)
    d = I.make_all(wl, ("W", "h", "targets"))
    out, _ = _fwd_check(wl, d, TOL["bf16"])
    assert np.all(out["max_owner"][5:9] != out["target_owner"][5:9])
    _bwd_check(wl, d, out, TOL["bf16"])


def test_loss_all_ignored():
    wl = I.custom(T=200, H=64, V_real=500, Vp=512, S=2, dtype="bf16", seed=22)
    d = I.make_all(wl, ("W", "h"))
    d["targets"] = np.full(wl.T, -100, dtype=np.int64)
    out = R.loss_fwd(wl, D.to_device(d["h"]), D.to_device(d["W"]), d["targets"])
    assert out["loss"] == 0.0 and out["status"] == 0
    assert np.all(out["token_loss"] == 0) and np.all(out["target_owner"] == -1)
    dH, dW, st = R.loss_bwd(wl, D.to_device(d["h"]), D.to_device(d["W"]), out["targets_d"], out["lse_d"])
    assert st == 0
    assert not dH.any().item() and not dW.any().item()


def test_loss_bad_target_flagged_and_ignored():
    wl = I.custom(T=100, H=64, V_real=500, Vp=512, S=2, dtype="bf16", seed=23)
    d = I.make_all(wl, ("W", "h", "targets"))
    d["targets"][[3, 40]] = [505, -7]       # a padded class and a negative non-ignore value
    out, ref = _fwd_check(wl, d, TOL["bf16"])
    assert out["status"] == R.vce.VCE_ERR_BAD_INDEX
    assert out["token_loss"][3] == 0 and out["target_owner"][40] == -1
    # the backward on its own flags them too, and gives them no gradient
    dH, dW, st = R.loss_bwd(wl, D.to_device(d["h"]), D.to_device(d["W"]), out["targets_d"], out["lse_d"])
    assert st == R.vce.VCE_ERR_BAD_INDEX
    assert not dH[3].any().item() and not dH[40].any().item()
    rdH, rdW = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    assert R.max_abs_rel(dH.cpu().numpy(), rdH) <= TOL["bf16"]["grad"]
    assert R.max_abs_rel(dW.cpu().numpy(), rdW) <= TOL["bf16"]["grad"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_loss_bwd_small_workspace_chunks(dtype):
    """The smallest workspace (256 vocabulary columns per pass) gives the same
    gradients as one large pass, within tolerance, and is run to run exact."""
    wl = I.custom(T=200, H=128, V_real=3000, Vp=3008, S=5, dtype=dtype, seed=24, ignore_frac=0.1)
    d = I.make_all(wl, ("W", "h", "targets"))
    out, _ = _fwd_check(wl, d, TOL[dtype])
    p = R.prob(wl)
    nmin = R.vce.vce_workspace_size_min(p, R.vce.VCE_OP_LOSS_BWD)
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    dH1, dW1, _ = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], ws_bytes=nmin)
    dH2, dW2, _ = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], ws_bytes=nmin)
    assert torch.equal(dH1, dH2) and torch.equal(dW1, dW2)
    rdH, rdW = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    assert R.max_abs_rel(dH1.cpu().numpy(), rdH) <= TOL[dtype]["grad"]
    assert R.max_abs_rel(dW1.cpu().numpy(), rdW) <= TOL[dtype]["grad"]
    with pytest.raises(R.vce.VceError) as e:
        R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], ws_bytes=nmin - 256)
    assert e.value.status == R.vce.VCE_ERR_WORKSPACE


def test_tied_embedding_and_head_gradients_combine():
    """Tied W: the head gradient is accumulated into dW and the embedding
    backward adds its rows on top: dW = dW_head + dW_embed."""
    wl = I.custom(T=256, H=128, V_real=1000, Vp=1024, S=4, dtype="bf16", seed=25, tied=True,
                  ignore_frac=0.05)
    d = I.make_all(wl, ("W", "h", "targets", "ids", "dE"))
    dE = I.bf16_bits(I.bf16_to_f32(d["dE"]) * np.float32(1e-3))   # comparable magnitudes
    out, _ = _fwd_check(wl, d, TOL["bf16"])
    dW = torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda")
    R.loss_bwd(wl, D.to_device(d["h"]), D.to_device(d["W"]), out["targets_d"], out["lse_d"], dW=dW)
    assert R.embed_bwd(wl, d["ids"], D.to_device(dE), dW) == 0
    _, rdW_head = O.cross_entropy_backward(d["h"], d["W"], d["targets"], wl.V_real, wl.Vp)
    ref = rdW_head + O.embed_backward(d["ids"], dE, wl.V_real, wl.Vp)
    assert R.max_abs_rel(dW.cpu().numpy(), ref) <= TOL["bf16"]["grad"]
    # tied accumulation: a second head backward adds the same amount again
    before = dW.clone()
    R.loss_bwd(wl, D.to_device(d["h"]), D.to_device(d["W"]), out["targets_d"], out["lse_d"], dW=dW)
    assert R.max_abs_rel((dW - before).cpu().numpy(), rdW_head) <= TOL["bf16"]["grad"]


def test_loss_gpt2_head_full():
    """T=4096, H=1024, V_real=50000 -> 50048, S=8 (6256 rows per shard), 5%
    ignored, untied: every lse, every token loss, all of dH and dW."""
    wl = I.WORKLOADS["gpt2_head"]
    d = I.make_all(wl, ("W", "h", "targets"))
    out, _ = _fwd_check(wl, d, TOL["bf16"])
    _bwd_check(wl, d, out, TOL["bf16"])


def _oracle_rows_all(h, W, y, V_real, rows=1024):
    """The oracle's per-token quantities for every token, a block of rows at a
    time (h and W widened to fp64 once)."""
    hf, Wf = O._as_f64(h), O._as_f64(W)
    lse = np.empty(h.shape[0])
    tl = np.empty(h.shape[0])
    for i in range(0, h.shape[0], rows):
        r = O.cross_entropy_rows(hf[i:i + rows], Wf, y[i:i + rows], V_real)
        lse[i:i + rows] = r["lse"]
        tl[i:i + rows] = r["token_loss"]
    return lse, tl


def _check_sampled_rows(wl, d, out, dH, tol, rng):
    """lse, token losses and dH on a sample of tokens (first and last included)."""
    h, W, y = d["h"], d["W"], d["targets"]
    sample = np.unique(np.concatenate([rng.choice(wl.T, 48, replace=False), [0, wl.T - 1]]))
    r = O.cross_entropy_rows(h[sample], W, y[sample], wl.V_real)
    assert np.all(np.abs(out["lse"][sample] - r["lse"]) <= tol["lse"] * np.abs(r["lse"]))
    assert R.max_abs_rel(out["token_loss"][sample], r["token_loss"]) <= tol["loss"]
    nv = O.n_valid(y, wl.V_real)
    ref_dH = O.hidden_gradient_rows(h[sample], W, y[sample], wl.V_real, 1.0 / nv)
    assert R.max_abs_rel(dH.cpu().numpy()[sample], ref_dH) <= tol["grad"]


def _head_rows(wl, y, rng, n_top=16, n_rand=8):
    """Rows of dW to compare: the most frequent target classes (the Zipf head),
    random classes and the last real class."""
    valid = (y >= 0) & (y < wl.V_real)
    counts = np.bincount(y[valid], minlength=wl.V_real)
    return np.unique(np.concatenate([np.argsort(-counts, kind="stable")[:n_top],
                                     rng.choice(wl.V_real, n_rand, replace=False), [wl.V_real - 1]]))


def _check_full_batch(wl, d, out, dW_head_rows, vs, tol):
    """The exact loss scalar, every lse, and the head's dW rows vs from the
    oracle's full-batch lse. Returns the oracle's head rows."""
    h, W, y = d["h"], d["W"], d["targets"]
    t0 = time.time()
    lse_all, tl_all = _oracle_rows_all(h, W, y, wl.V_real)
    nv = O.n_valid(y, wl.V_real)
    assert R.rel(out["loss"], tl_all.sum() / nv) <= tol["loss"]
    assert np.all(np.abs(out["lse"] - lse_all) <= tol["lse"] * np.abs(lse_all))
    assert R.max_abs_rel(out["token_loss"], tl_all) <= tol["loss"]
    ref_rows = O.head_gradient_rows(O._as_f64(h), O._as_f64(W), y, wl.V_real, lse_all, 1.0 / nv, vs)
    assert R.max_abs_rel(dW_head_rows, ref_rows) <= tol["grad"]
    print(f"oracle over the full batch: {time.time() - t0:.1f}s")
    return ref_rows


def test_loss_gptoss_full():
    """T=16384, H=3072, V_real=201088, S=8, Zipf next-token targets, untied:
    sampled lse, token losses and dH rows; then the loss scalar, every lse and
    every token loss, and dW rows of the most frequent, random and last
    classes, all from the oracle's full-batch lse."""
    wl = I.WORKLOADS["gptoss_embed"]
    d = I.make_all(wl, ("W", "h", "targets"))
    h_d, W_d = D.to_device(d["h"]), D.to_device(d["W"])
    out = R.loss_fwd(wl, h_d, W_d, d["targets"])
    assert out["status"] == 0
    tol = TOL["bf16"]
    rng = np.random.default_rng(0)
    dW = torch.full((wl.Vp, wl.H), float("nan"), dtype=torch.float32, device="cuda")
    dH, dW, st = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], dW=dW)
    assert st == 0
    _check_sampled_rows(wl, d, out, dH, tol, rng)
    vs = _head_rows(wl, d["targets"], rng)
    got = dW.index_select(0, torch.from_numpy(vs).cuda()).cpu().numpy()
    _check_full_batch(wl, d, out, got, vs, tol)
    # properties at any size: finite everywhere
    assert torch.isfinite(dW).all().item() and torch.isfinite(dH).all().item()


def test_qwen3_tied_pipeline_full():
    """The Qwen3-like tied step at full size (T=8192, H=2048, V=151936, S=8),
    run as one pipeline on one W and one fp32 dW, with the tied flag set and
    in the order the benchmark runs it: embedding lookup of the input ids with
    the embedding backward's plan made beside it, loss forward, loss backward adding the
    head's gradient into dW, and the plan's application adding the input
    gradient into the same dW ("Vocabulary shards", paragraph 2: one logical
    parameter, all contributions combined). Checked against the oracle: the lookup bit for
    bit; the loss scalar, every lse and every token loss; the head's dW rows of
    the most frequent (Zipf head) ids, random ids and the last id; the
    embedding's contribution to every touched row; and the combined rows."""
    wl = I.WORKLOADS["qwen3_tied"]
    assert wl.tied
    d = I.make_all(wl)
    h, W, y, ids, dE = d["h"], d["W"], d["targets"], d["ids"], d["dE"]
    tol = TOL["bf16"]
    rng = np.random.default_rng(1)
    W_d, h_d, dE_d = D.to_device(W), D.to_device(h), D.to_device(dE)
    # 1. lookup, with the embedding backward's plan made beside it
    p = R.prob(wl)
    ws_e = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    E_d = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    R.vce.vce_embed_fwd_plan(p, torch.from_numpy(ids).cuda(), W_d, E_d, ws_e)
    torch.cuda.synchronize()
    assert np.array_equal(D.to_host_bits(E_d), O.embed_forward(ids, W, wl.V_real))
    # 2. loss forward
    out = R.loss_fwd(wl, h_d, W_d, y)
    assert out["status"] == 0
    # 3. loss backward with tied_weights = 1: dW += G^T h into a zeroed gradient
    dW = torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda")
    dH, dW, st = R.loss_bwd(wl, h_d, W_d, out["targets_d"], out["lse_d"], dW=dW)
    assert st == 0
    vs = np.unique(np.concatenate([_head_rows(wl, y, rng), _head_rows(wl, ids, rng, n_rand=0)]))
    vs_d = torch.from_numpy(vs).cuda()
    head_rows = dW.index_select(0, vs_d).cpu().numpy()
    touched = np.unique(ids[(ids >= 0) & (ids < wl.V_real)])
    touched_d = torch.from_numpy(touched).cuda()
    head_touched = dW.index_select(0, touched_d).double()
    # 4. the embedding backward (the plan applied to dE) into the same dW
    st_e = R.status_word()
    R.vce.vce_embed_bwd_apply(p, dE_d, dW, ws_e, dev_status=st_e)
    torch.cuda.synchronize()
    assert int(st_e.item()) == 0
    _check_sampled_rows(wl, d, out, dH, tol, rng)
    ref_head = _check_full_batch(wl, d, out, head_rows, vs, tol)
    ref_embed = O.embed_backward(ids, dE, wl.V_real, wl.Vp)
    # the embedding's contribution on every touched row: fp32 run sums against fp64
    got_embed = (dW.index_select(0, touched_d).double() - head_touched).cpu().numpy()
    assert R.max_abs_rel(got_embed, ref_embed[touched]) <= 1e-5
    # the combined tied gradient on the compared rows
    final_rows = dW.index_select(0, vs_d).cpu().numpy()
    assert R.max_abs_rel(final_rows, ref_head + ref_embed[vs]) <= tol["grad"]
    assert torch.isfinite(dW).all().item() and torch.isfinite(dH).all().item()
