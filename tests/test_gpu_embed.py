"""GPU parity of the embedding lookup and its backward against the oracle.

Forward, ownership and local-index maps: bit-exact. Backward: bit-exact
against the oracle's fp32 replay of the library's fixed summation order.
"""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CHUNK = 32   # the library's published run length (include/vce.h, vce_embed_bwd_chunk)


def test_chunk_constant():
    assert R.vce.vce_embed_bwd_chunk() == CHUNK


def _check_fwd(wl, W, ids):
    out = R.embed_fwd(wl, D.to_device(W), ids)
    ref = O.embed_forward(ids, W, wl.V_real)
    assert np.array_equal(out["E"], ref)
    _, owner, local = O.ownership(ids, wl.V_real, wl.Vp, wl.S)
    assert np.array_equal(out["owner"], owner.astype(np.int32))
    assert np.array_equal(out["local"], local.astype(np.int32))


def test_embed_fwd_tiny_f32():
    wl = I.WORKLOADS["tiny_f32"]
    d = I.make_all(wl, ("W", "ids"))
    _check_fwd(wl, d["W"], d["ids"])


CASES = [
    dict(T=1, H=8, V_real=50, Vp=64, S=1),
    dict(T=63, H=64, V_real=1000, Vp=1024, S=3),
    dict(T=129, H=200, V_real=700, Vp=1024, S=4),     # last shard entirely padding
    dict(T=300, H=1032, V_real=4000, Vp=4032, S=7),
    dict(T=77, H=16, V_real=64, Vp=64, S=64),         # one row per shard
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{T}_H{H}_V{V_real}_S{S}".format(**c))
def test_embed_fwd_bf16_cases(case):
    wl = I.custom(dtype="bf16", pad_id_frac=0.1, oor_id_frac=0.1, seed=11, **case)
    d = I.make_all(wl, ("W", "ids"))
    _check_fwd(wl, d["W"], d["ids"])


def test_embed_fwd_gptoss_full():
    """W[201088, 3072] bf16, S = 8 x 25136, T = 16384 Zipf ids with padding and
    out-of-range ids: every output row bit-exact."""
    wl = I.WORKLOADS["gptoss_embed"]
    d = I.make_all(wl, ("W", "ids"))
    _check_fwd(wl, d["W"], d["ids"])


def _check_bwd(wl, ids, dE, dW0):
    dE_d = D.to_device(dE)
    dW_d = torch.from_numpy(dW0.copy()).cuda()
    st = R.embed_bwd(wl, ids, dE_d, dW_d)
    assert st == 0
    dE32 = I.bf16_to_f32(dE) if wl.dtype == "bf16" else dE
    ref = O.embed_backward_replay_f32(ids, dE32, wl.V_real, CHUNK, dW0)
    got = dW_d.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    return got


def test_embed_bwd_tiny_f32():
    wl = I.WORKLOADS["tiny_f32"]
    d = I.make_all(wl, ("ids", "dE"))
    _check_bwd(wl, d["ids"], d["dE"], np.zeros((wl.Vp, wl.H), np.float32))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{T}_H{H}_V{V_real}_S{S}".format(**c))
def test_embed_bwd_bf16_cases(case):
    wl = I.custom(dtype="bf16", pad_id_frac=0.1, oor_id_frac=0.1, seed=12, **case)
    d = I.make_all(wl, ("ids", "dE"))
    rng = np.random.default_rng(3)
    dW0 = rng.standard_normal((wl.Vp, wl.H)).astype(np.float32)   # accumulates into existing values
    _check_bwd(wl, d["ids"], d["dE"], dW0)


def test_embed_bwd_heavy_repeats():
    """One id repeated over many runs (the left-to-right combine of run sums),
    another over exactly one run, H spanning several column slices."""
    wl = I.custom(T=5000, H=1544, V_real=1000, Vp=1024, S=4, dtype="bf16", seed=13)
    d = I.make_all(wl, ("ids", "dE"))
    ids = d["ids"].copy()
    ids[:3000] = 3            # 94 runs of one id, scattered positions below
    ids[3000:3032] = 999      # exactly one full run
    ids = np.random.default_rng(4).permutation(ids)
    rng = np.random.default_rng(5)
    dW0 = rng.standard_normal((wl.Vp, wl.H)).astype(np.float32)
    _check_bwd(wl, ids, d["dE"], dW0)


def test_embed_bwd_single_segment():
    wl = I.custom(T=4099, H=64, V_real=1000, Vp=1024, S=2, dtype="bf16", seed=14)
    d = I.make_all(wl, ("dE",))
    ids = np.full(wl.T, 511, dtype=np.int64)
    _check_bwd(wl, ids, d["dE"], np.zeros((wl.Vp, wl.H), np.float32))


def test_embed_bwd_nothing_valid():
    wl = I.custom(T=100, H=64, dtype="bf16", seed=15)
    d = I.make_all(wl, ("dE",))
    ids = np.array([-100, -1, 1000, 1023, 1024, 2 ** 40] * 16 + [-100] * 4, dtype=np.int64)
    dW0 = np.random.default_rng(6).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    got = _check_bwd(wl, ids, d["dE"], dW0)
    assert np.array_equal(got, dW0)


def test_embed_bwd_gptoss_full_deterministic():
    """Full GPT-OSS-shaped backward: bit-exact against the fp32 replay, and
    bit-identical over 20 runs."""
    wl = I.WORKLOADS["gptoss_embed"]
    d = I.make_all(wl, ("ids", "dE"))
    ids, dE = d["ids"], d["dE"]
    dE_d = D.to_device(dE)
    ids_d = torch.from_numpy(ids).cuda()
    valid = (ids >= 0) & (ids < wl.V_real)
    uniq = np.unique(ids[valid])
    uniq_d = torch.from_numpy(uniq).cuda()
    dW_d = torch.zeros((wl.Vp, wl.H), dtype=torch.float32, device="cuda")
    p = R.prob(wl)
    ws = D.workspace(R.vce.vce_workspace_size(p, R.vce.VCE_OP_EMBED_BWD))
    R.vce.vce_embed_bwd(p, ids_d, dE_d, dW_d, ws)
    torch.cuda.synchronize()
    rows = dW_d.index_select(0, uniq_d).cpu().numpy()
    untouched = dW_d.abs().sum().item() - np.abs(rows).sum(dtype=np.float64)
    assert abs(untouched) <= 1e-3 * max(1.0, np.abs(rows).sum())
    ref = O.embed_backward_replay_f32(ids, I.bf16_to_f32(dE), wl.V_real, CHUNK,
                                      np.zeros((wl.Vp, wl.H), np.float32))
    assert np.array_equal(rows.view(np.uint32), ref[uniq].view(np.uint32))
    # untouched rows are exactly zero
    mask = torch.ones(wl.Vp, dtype=torch.bool, device="cuda")
    mask[uniq_d] = False
    assert int((dW_d[mask] != 0).sum().item()) == 0
    first = dW_d.clone()
    for _ in range(20):
        dW_d.zero_()
        R.vce.vce_embed_bwd(p, ids_d, dE_d, dW_d, ws)
        torch.cuda.synchronize()
        assert torch.equal(dW_d.view(torch.int32), first.view(torch.int32))


@pytest.mark.parametrize("T,V_real,Vp", [(20000, 1000, 1024),      # more tokens than the shared-memory sorts hold
                                         (5000, 1048000, 1048064),   # too many id / NB values for the counting sort
                                         (12000, 1048000, 1048064)])  # the same above 8192 tokens: no clustered sort
def test_embed_bwd_workspace_sort_path(T, V_real, Vp):
    """The sorts other than the bucketed counting sort: the 64-bit workspace
    sort (T above 16384) and the bucketed radix sort (about 6900 values of
    id / NB, more per-warp counters than the counting sort's shared memory)."""
    wl = I.custom(T=T, H=64, V_real=V_real, Vp=Vp, S=8, dtype="bf16", seed=16, pad_id_frac=0.05, oor_id_frac=0.05)
    d = I.make_all(wl, ("ids", "dE"))
    ids = d["ids"].copy()
    ids[: T // 4] = V_real - 1                 # one heavy id across many runs
    rng = np.random.default_rng(8)
    ids = rng.permutation(ids)
    dW0 = np.zeros((wl.Vp, wl.H), np.float32)
    _check_bwd(wl, ids, d["dE"], dW0)


def _sort_kinds(wl, ids, dE, dW0):
    R.vce.vce_profile_begin(16)
    got = _check_bwd(wl, ids, dE, dW0)
    kinds = [k for k, _ in R.vce.vce_profile_end(16)]
    return got, kinds


@pytest.mark.parametrize("T,V_real", [(1, 1000), (33, 1000), (2049, 151936), (8192, 151936), (8193, 5000),
                                      (16384, 201088)])
def test_embed_bwd_clustered_and_per_cta_id_loads(T, V_real, monkeypatch):
    """The counting sort's two id loads: clusters of eight CTAs sharing the
    loads through distributed shared memory (VCE_EMBED_SORT_CLUSTER=1), and
    every CTA loading all ids (=0). T spans one and two load rounds per warp,
    and a batch so small that most ranks load nothing. Both are bit-exact
    against the replay, with one heavy id over many runs; without the variable
    the clusters run above 8192 tokens only."""
    wl = I.custom(T=T, H=136, V_real=V_real, Vp=-(-V_real // 64) * 64, S=8, dtype="bf16", seed=17,
                  pad_id_frac=0.03, oor_id_frac=0.02)
    d = I.make_all(wl, ("ids", "dE"))
    ids = d["ids"].copy()
    ids[: T // 5] = 7
    ids = np.random.default_rng(9).permutation(ids)
    dW0 = np.random.default_rng(10).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    res = {}
    for env, kind in (("1", "embed_sort_cluster"), ("0", "embed_sort"), (None, None)):
        if env is None:
            monkeypatch.delenv("VCE_EMBED_SORT_CLUSTER", raising=False)
            kind = "embed_sort_cluster" if T > 8192 else "embed_sort"
        else:
            monkeypatch.setenv("VCE_EMBED_SORT_CLUSTER", env)
        got, kinds = _sort_kinds(wl, ids, d["dE"], dW0)
        other = "embed_sort" if kind == "embed_sort_cluster" else "embed_sort_cluster"
        assert kind in kinds and other not in kinds
        res[env] = got
    assert np.array_equal(res["1"].view(np.uint32), res["0"].view(np.uint32))


def _draw_large(i):
    g = np.random.default_rng(300 + i)
    V = int(g.integers(2, 300000))
    return dict(T=int(g.integers(8193, 16385)), H=8 * int(g.integers(1, 40)), V_real=V,
                Vp=-(-V // 64) * 64 + 64 * int(g.integers(0, 2)), S=int(g.integers(1, 9)))


@pytest.mark.parametrize("case", [_draw_large(i) for i in range(6)],
                         ids=lambda c: "T{T}_H{H}_V{V_real}".format(**c))
def test_embed_bwd_random_large_batches(case):
    """Seeded batches between 8192 and 16384 tokens (the clustered counting
    sort, or the radix buckets where the vocabulary is too large for its
    counters), random H and V: bit-exact against the replay."""
    wl = I.custom(dtype="bf16", pad_id_frac=0.02, oor_id_frac=0.02, seed=19, **case)
    d = I.make_all(wl, ("ids", "dE"))
    dW0 = np.random.default_rng(11).standard_normal((wl.Vp, wl.H)).astype(np.float32)
    _check_bwd(wl, d["ids"], d["dE"], dW0)
