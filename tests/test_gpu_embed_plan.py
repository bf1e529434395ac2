"""The embedding backward in two parts: vce_embed_bwd_plan (the sort of the
ids into runs) and vce_embed_bwd_apply (the addition of dE into dW by that
plan). Each application must give the bits of the one-call backward, which
the oracle's fp32 replay of the fixed summation order fixes; a plan must be
reusable, and a workspace without a matching plan must add nothing."""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CHUNK = 32
ERR_ARG = 1

# One shape per sort: the bucketed counting sort with per-CTA id loads, the
# same with clusters of eight CTAs (above 8192 tokens), the bucketed radix sort
# (a vocabulary too large for the counting sort's counters) and the one-CTA
# sort of 64-bit keys in the workspace (above 16384 tokens).
SHAPES = [dict(T=2049, H=136, V_real=151936, Vp=151936, S=8),
          dict(T=16384, H=264, V_real=201088, Vp=201088, S=8),
          dict(T=5000, H=64, V_real=1048000, Vp=1048064, S=8),
          dict(T=20000, H=72, V_real=1000, Vp=1024, S=4)]


def _bits(a):
    return a.view(np.uint32)


def _inputs(case, seed):
    wl = I.custom(dtype="bf16", pad_id_frac=0.03, oor_id_frac=0.02, seed=seed, **case)
    d = I.make_all(wl, ("ids", "dE"))
    ids = d["ids"].copy()
    ids[: wl.T // 6] = 5                       # one id over many runs
    ids = np.random.default_rng(seed).permutation(ids)
    dE2 = I.make_dE(I.custom(dtype="bf16", seed=seed + 1000, **case))
    return wl, ids, d["dE"], dE2


@pytest.mark.parametrize("case", SHAPES, ids=lambda c: "T{T}_H{H}_V{V_real}".format(**c))
def test_plan_then_apply_twice(case):
    """Plan before dE exists; apply to dE1, then the same plan to dE2: both
    results bit-exact against the replay (the second on top of the first)."""
    wl, ids, dE1, dE2 = _inputs(case, 41)
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    ids_d = torch.from_numpy(ids).cuda()
    R.vce.vce_embed_bwd_plan(p, ids_d, ws, dev_status=st)
    dW0 = np.random.default_rng(42).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    R.vce.vce_embed_bwd_apply(p, D.to_device(dE1), dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref1 = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE1), wl.V_real, CHUNK, dW0)
    got1 = dW_d.cpu().numpy()
    assert np.array_equal(_bits(got1), _bits(ref1))
    R.vce.vce_embed_bwd_apply(p, D.to_device(dE2), dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref2 = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE2), wl.V_real, CHUNK, ref1)
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref2))


def test_one_call_leaves_its_plan():
    """vce_embed_bwd leaves the plan of its ids in the workspace: an apply
    after it adds the next dE in the same order."""
    wl, ids, dE1, dE2 = _inputs(dict(T=3000, H=200, V_real=50000, Vp=50048, S=8), 43)
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    dW_d = torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda")
    R.vce.vce_embed_bwd(p, torch.from_numpy(ids).cuda(), D.to_device(dE1), dW_d, ws, dev_status=st)
    R.vce.vce_embed_bwd_apply(p, D.to_device(dE2), dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    zero = np.zeros((wl.Vp, wl.H), np.float32)
    ref = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE1), wl.V_real, CHUNK, zero)
    ref = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE2), wl.V_real, CHUNK, ref)
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref))


def test_apply_without_plan_adds_nothing():
    """A zeroed workspace holds no plan, and a plan made for another batch size
    does not fit: either way dW is left as it was and VCE_ERR_ARG is reported."""
    case = dict(T=700, H=64, V_real=1000, Vp=1024, S=4)
    wl, ids, dE1, _ = _inputs(case, 44)
    p = R.prob(wl)
    nbytes = R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD)
    dW0 = np.random.default_rng(45).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    dE_d = D.to_device(dE1)

    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    st = R.status_word()
    R.vce.vce_embed_bwd_apply(p, dE_d, dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == ERR_ARG
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(dW0))

    # a plan of 699 tokens in a workspace large enough for 700
    p_short = R.prob(wl, T=wl.T - 1)
    R.vce.vce_embed_bwd_plan(p_short, torch.from_numpy(ids[:-1].copy()).cuda(), ws)
    st = R.status_word()
    R.vce.vce_embed_bwd_apply(p, dE_d, dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == ERR_ARG
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(dW0))

    # the matching plan then applies normally
    st = R.status_word()
    R.vce.vce_embed_bwd_plan(p, torch.from_numpy(ids).cuda(), ws)
    R.vce.vce_embed_bwd_apply(p, dE_d, dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE1), wl.V_real, CHUNK, dW0)
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref))


def test_apply_repeated_in_a_graph():
    """Plan once, then a CUDA graph of one application replayed three times:
    the plan's counters are restored by every application, so each replay
    adds the same bits."""
    wl, ids, dE1, _ = _inputs(dict(T=8192, H=512, V_real=151936, Vp=151936, S=8), 46)
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    R.vce.vce_embed_bwd_plan(p, torch.from_numpy(ids).cuda(), ws, dev_status=st)
    dE_d = D.to_device(dE1)
    dW_d = torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            R.vce.vce_embed_bwd_apply(p, dE_d, dW_d, ws, dev_status=st, stream=side.cuda_stream)
    torch.cuda.synchronize()
    ref = np.zeros((wl.Vp, wl.H), np.float32)
    valid = (ids >= 0) & (ids < wl.V_real)
    uniq = np.unique(ids[valid])
    uniq_d = torch.from_numpy(uniq).cuda()
    dE32 = I.bf16_to_f32(dE1)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = O.embed_backward_replay_f32(ids, dE32, wl.V_real, CHUNK, ref)
        rows = dW_d.index_select(0, uniq_d).cpu().numpy()
        assert np.array_equal(_bits(rows), _bits(ref[uniq]))


def test_plan_then_apply_f32():
    """The fp32 reduce by a plan: the tiny fp32 case (T=64, H=64, ids mixing
    real, padded-row, padding and out-of-range values), bit-exact against the
    replay, twice on the same plan."""
    wl = I.WORKLOADS["tiny_f32"]
    d = I.make_all(wl, ("ids", "dE"))
    ids, dE = d["ids"], d["dE"]
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    R.vce.vce_embed_bwd_plan(p, torch.from_numpy(ids).cuda(), ws, dev_status=st)
    dW0 = np.random.default_rng(47).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    dE_d = torch.from_numpy(dE).cuda()
    ref = dW0
    for _ in range(2):
        R.vce.vce_embed_bwd_apply(p, dE_d, dW_d, ws, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = O.embed_backward_replay_f32(ids, dE, wl.V_real, CHUNK, ref)
        assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref))


@pytest.mark.parametrize("case", SHAPES, ids=lambda c: "T{T}_H{H}_V{V_real}".format(**c))
def test_lookup_with_plan(case):
    """vce_embed_fwd_plan: the lookup bit-exact (with the ownership maps), and
    the plan it leaves applied to dE bit-exact against the replay, on every
    sort path; the call ordered before later work on its stream."""
    wl, ids, dE1, _ = _inputs(case, 48)
    W = I.make_W(wl)
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    E = torch.full((wl.T, wl.H), 7, dtype=torch.bfloat16, device="cuda")
    owner = torch.full((wl.T,), -7, dtype=torch.int32, device="cuda")
    local = torch.full((wl.T,), -7, dtype=torch.int32, device="cuda")
    W_d = D.to_device(W)
    dW_d = torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda")
    # the apply is queued right behind the lookup: it must find the plan complete
    R.vce.vce_embed_fwd_plan(p, torch.from_numpy(ids).cuda(), W_d, E, ws, owner=owner, local=local, dev_status=st)
    R.vce.vce_embed_bwd_apply(p, D.to_device(dE1), dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(D.to_host_bits(E), O.embed_forward(ids, W, wl.V_real))
    _, own, loc = O.ownership(ids, wl.V_real, wl.Vp, wl.S)
    assert np.array_equal(owner.cpu().numpy(), own.astype(np.int32))
    assert np.array_equal(local.cpu().numpy(), loc.astype(np.int32))
    ref = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE1), wl.V_real, CHUNK,
                                      np.zeros((wl.Vp, wl.H), np.float32))
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref))


# Multi-run ids' items in narrow column slices (half a wide slice) or wide
# ones: both give the replay's bits, on each sort path, with slices that end
# inside a row (H = 1288 bf16: 2 wide and 3 narrow slices; H = 520: 1 and 2).
NARROW_CASES = [dict(T=2049, H=1288, V_real=151936, Vp=151936, S=8, dtype="bf16"),
                dict(T=16384, H=1288, V_real=201088, Vp=201088, S=8, dtype="bf16"),
                dict(T=5000, H=64, V_real=1048000, Vp=1048064, S=8, dtype="bf16"),
                dict(T=20000, H=520, V_real=1000, Vp=1024, S=4, dtype="bf16"),
                dict(T=3000, H=260, V_real=5000, Vp=5056, S=4, dtype="f32")]


@pytest.mark.parametrize("narrow", ["0", "1"])
@pytest.mark.parametrize("case", NARROW_CASES, ids=lambda c: "T{T}_H{H}_V{V_real}_{dtype}".format(**c))
def test_narrow_and_wide_slices(case, narrow, monkeypatch):
    """VCE_EMBED_NARROW forces the multi-run ids' column slices: the one-call
    backward and a plan applied once are bit-exact against the replay either
    way."""
    monkeypatch.setenv("VCE_EMBED_NARROW", narrow)
    c = dict(case)
    dtype = c.pop("dtype")
    wl = I.custom(dtype=dtype, pad_id_frac=0.03, oor_id_frac=0.02, seed=60, **c)
    d = I.make_all(wl, ("ids", "dE"))
    ids = d["ids"].copy()
    ids[: wl.T // 5] = 7                       # one id over many runs
    ids[wl.T // 5: wl.T // 5 + 40] = 9         # an id of two runs
    ids = np.random.default_rng(61).permutation(ids)
    dE = d["dE"]
    dE32 = I.bf16_to_f32(dE) if dtype == "bf16" else dE
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    ids_d, dE_d = torch.from_numpy(ids).cuda(), D.to_device(dE)
    dW0 = np.random.default_rng(62).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    ref = O.embed_backward_replay_f32(ids, dE32, wl.V_real, CHUNK, dW0)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    R.vce.vce_embed_bwd(p, ids_d, dE_d, dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref))
    dW_d.copy_(torch.from_numpy(dW0))
    R.vce.vce_embed_bwd_plan(p, ids_d, ws, dev_status=st)
    R.vce.vce_embed_bwd_apply(p, dE_d, dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(ref))


def test_plan_of_other_slices_refused(monkeypatch):
    """A plan records its multi-run ids' slice count: one made with narrow
    slices (3 at H = 1288) is refused by an application with wide ones (2),
    which adds nothing and reports VCE_ERR_ARG."""
    wl = I.custom(T=2049, H=1288, V_real=151936, Vp=151936, S=8, dtype="bf16", seed=63)
    d = I.make_all(wl, ("ids", "dE"))
    ids = d["ids"].copy()
    ids[:300] = 11
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    st = R.status_word()
    ids_d = torch.from_numpy(ids).cuda()
    monkeypatch.setenv("VCE_EMBED_NARROW", "1")
    R.vce.vce_embed_bwd_plan(p, ids_d, ws, dev_status=st)
    monkeypatch.setenv("VCE_EMBED_NARROW", "0")
    dW0 = np.random.default_rng(64).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    R.vce.vce_embed_bwd_apply(p, D.to_device(d["dE"]), dW_d, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == ERR_ARG
    assert np.array_equal(_bits(dW_d.cpu().numpy()), _bits(dW0))
