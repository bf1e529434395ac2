"""GPU parity of the hashed n-gram input embeddings ("Sampled Softmax with
Over-Tokenized Transformer", Setup and its loss listing) against the oracle.

Everything here is exact: the row indices are integers, the forward is one
fp32 sum of three stored rows rounded once (replayed in fp32 by the oracle),
and each table's backward follows the library's fixed summation order
(replayed in fp32 by the oracle). Comparisons are bit for bit.
"""
import numpy as np
import pytest
import torch

import vce_run as R
from oracle import vce_oracle as O
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CHUNK = 32


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("n,V,M,seq_len", [(2, 1000, 613, 0), (3, 1000, 1024, 50), (3, 151936, 1 << 18, 2048),
                                           (2, 151936, (1 << 31) - 1, 7), (1, 1000, 97, 0)])
def test_hash_exact(n, V, M, seq_len):
    wl = I.custom("ngram_ids", T=4099, H=64, V_real=V, Vp=-(-V // 64) * 64, S=4, dtype="bf16", seed=70,
                  pad_id_frac=0.02, oor_id_frac=0.02)
    ids = I.make_ids(wl)
    out = torch.full((wl.T,), -7, dtype=torch.int64, device="cuda")
    R.vce.vce_ngram_hash(torch.from_numpy(ids).cuda(), n, V, M, out, seq_len=seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), O.ngram_index(ids, n, V, M, seq_len))


def _case(dtype, T, H, V_real, Vp, M2, M3, seed):
    wl = I.custom("ngram_case", T=T, H=H, V_real=V_real, Vp=Vp, S=4, dtype=dtype, seed=seed, pad_id_frac=0.03,
                  oor_id_frac=0.03, pad_fill=8.0)
    d = I.make_all(wl, ("W", "ids", "dE"))
    T2 = I.make_ngram_table(wl, 2, M2) if M2 else None
    T3 = I.make_ngram_table(wl, 3, M3) if M3 else None
    return wl, d, T2, T3


def _fwd(wl, ids, W, T2, M2, T3, M3, seq_len):
    E = torch.full((len(ids), wl.H), 7, dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32, device="cuda")
    st = R.status_word()
    R.vce.vce_ngram_embed_fwd(R.prob(wl, T=len(ids)), torch.from_numpy(ids).cuda(), D.to_device(W),
                              D.to_device(T2) if M2 else None, M2, D.to_device(T3) if M3 else None, M3, E,
                              seq_len=seq_len, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return D.to_host_bits(E)


def _bwd(wl, ids, dE, M2, M3, seq_len, inits):
    p = R.prob(wl, T=len(ids))
    dW = torch.from_numpy(inits[0].copy()).cuda()
    dT2 = torch.from_numpy(inits[1].copy()).cuda() if M2 else None
    dT3 = torch.from_numpy(inits[2].copy()).cuda() if M3 else None
    ws = D.workspace(R.vce.vce_ngram_workspace_size(p))
    st = R.status_word()
    R.vce.vce_ngram_embed_bwd(p, torch.from_numpy(ids).cuda(), D.to_device(dE), dW, dT2, M2, dT3, M3, ws,
                              seq_len=seq_len, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return [x.cpu().numpy() if x is not None else None for x in (dW, dT2, dT3)]


def _replays(wl, ids, dE, M2, M3, seq_len, inits):
    dE32 = I.bf16_to_f32(dE) if wl.dtype == "bf16" else dE
    out = [O.embed_backward_replay_f32(ids, dE32, wl.V_real, CHUNK, inits[0])]
    for n, M, init in ((2, M2, inits[1]), (3, M3, inits[2])):
        out.append(O.embed_backward_replay_f32(O.ngram_index(ids, n, wl.V_real, M, seq_len), dE32, M, CHUNK, init)
                   if M else None)
    return out


@pytest.mark.parametrize("dtype,T,H,V_real,Vp,M2,M3,seq_len", [
    ("f32", 64, 64, 1000, 1024, 613, 1024, 0),
    ("bf16", 300, 128, 1000, 1024, 613, 1024, 50),
    ("bf16", 520, 256, 5000, 5056, 4096, 0, 0),        # 3-gram table left out
    ("bf16", 129, 64, 1000, 1024, 0, 97, 16),           # 2-gram table left out
    ("bf16", 700, 8, 1000, 1024, 613, 1 << 21, 0),     # the 3-gram table sorted by radix buckets, the others counted
    ("bf16", 20000, 8, 1000, 1024, 613, 1024, 0),      # T above the shared-memory sorts: every table in the workspace
    ("bf16", 12000, 16, 5000, 5056, 613, 1 << 18, 3000),  # 8192 < T <= 16384: three clustered counting sorts
    ("bf16", 12000, 16, 5000, 5056, 613, 1024, 3000),     # the same, small enough to run side by side in one launch
    ("f32", 3000, 12, 700, 704, 97, 131, 0),              # fp32, the three counting sorts side by side
])
def test_ngram_fwd_bwd_exact(dtype, T, H, V_real, Vp, M2, M3, seq_len):
    wl, d, T2, T3 = _case(dtype, T, H, V_real, Vp, M2, M3, seed=71 + T)
    ids = d["ids"].copy()
    ids[10:40] = ids[9]                      # a run of one id: repeated n-grams too
    E = _fwd(wl, ids, d["W"], T2, M2, T3, M3, seq_len)
    ref = O.ngram_embed_forward(ids, d["W"], T2, T3, wl.V_real, M2, M3, seq_len)
    assert np.array_equal(_bits(E), _bits(ref))
    rng = np.random.default_rng(9)
    inits = [rng.standard_normal((wl.Vp, wl.H)).astype(np.float32),
             rng.standard_normal((max(M2, 1), wl.H)).astype(np.float32),
             rng.standard_normal((max(M3, 1), wl.H)).astype(np.float32)]
    got = _bwd(wl, ids, d["dE"], M2, M3, seq_len, inits)
    want = _replays(wl, ids, d["dE"], M2, M3, seq_len, inits)
    for g, w in zip(got, want):
        if w is not None:
            assert np.array_equal(g.view(np.uint32), w.view(np.uint32))


def test_ngram_qwen3_full_size():
    """T=8192 Zipf ids (4 sequences of 2048), H=2048, V=151936, two tables of
    2^18 rows: the forward bit-exact on every row, the three backward tables
    bit-exact on every touched row and zero elsewhere."""
    wl = I.WORKLOADS["qwen3_tied"]
    M, L = I.NGRAM_ROWS, I.NGRAM_SEQ_LEN
    d = I.make_all(wl, ("W", "ids", "dE"))
    T2, T3 = I.make_ngram_table(wl, 2, M), I.make_ngram_table(wl, 3, M)
    ids = d["ids"]
    E = _fwd(wl, ids, d["W"], T2, M, T3, M, L)
    assert np.array_equal(E, O.ngram_embed_forward(ids, d["W"], T2, T3, wl.V_real, M, M, L))
    zeros = [np.zeros((wl.Vp, wl.H), np.float32), np.zeros((M, wl.H), np.float32), np.zeros((M, wl.H), np.float32)]
    got = _bwd(wl, ids, d["dE"], M, M, L, zeros)
    want = _replays(wl, ids, d["dE"], M, M, L, zeros)
    for g, w in zip(got, want):
        assert np.array_equal(g.view(np.uint32), w.view(np.uint32))


@pytest.mark.parametrize("T,H,V_real,Vp,M2,M3,seq_len", [
    (300, 128, 1000, 1024, 613, 1024, 50),
    (129, 64, 1000, 1024, 0, 97, 16),                 # 2-gram table left out
    (12000, 16, 5000, 5056, 613, 1 << 18, 3000),     # three clustered counting sorts
])
def test_ngram_plan_then_apply(T, H, V_real, Vp, M2, M3, seq_len):
    """The backward split at its plan: the tables' row indices and sorts made
    from the ids alone, then applied to dE twice (each time the bits of the
    replay, the second on top of the first); a plan of another batch size
    adds nothing to any table and reports VCE_ERR_ARG."""
    wl, d, _, _ = _case("bf16", T, H, V_real, Vp, M2, M3, seed=90 + T)
    ids = d["ids"]
    p = R.prob(wl)
    rng = np.random.default_rng(10)
    inits = [rng.standard_normal((wl.Vp, wl.H)).astype(np.float32),
             rng.standard_normal((max(M2, 1), wl.H)).astype(np.float32),
             rng.standard_normal((max(M3, 1), wl.H)).astype(np.float32)]
    dW = torch.from_numpy(inits[0].copy()).cuda()
    dT2 = torch.from_numpy(inits[1].copy()).cuda() if M2 else None
    dT3 = torch.from_numpy(inits[2].copy()).cuda() if M3 else None
    ws = D.workspace(R.vce.vce_ngram_workspace_size(p))
    st = R.status_word()
    R.vce.vce_ngram_embed_bwd_plan(p, torch.from_numpy(ids).cuda(), M2, M3, ws, seq_len=seq_len, dev_status=st)
    dE_d = D.to_device(d["dE"])
    want = inits
    for _ in range(2):
        R.vce.vce_ngram_embed_bwd_apply(p, dE_d, dW, dT2, M2, dT3, M3, ws, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        want = _replays(wl, ids, d["dE"], M2, M3, seq_len, [w if w is not None else inits[i]
                                                               for i, w in enumerate(want)])
        got = [x.cpu().numpy() if x is not None else None for x in (dW, dT2, dT3)]
        for g, w in zip(got, want):
            if g is not None:
                assert np.array_equal(g.view(np.uint32), w.view(np.uint32))
    # a plan of one token fewer in the same (cleared) workspace: refused, nothing
    # added (its tables' parts of the workspace sit at other offsets, so the
    # apply finds either no plan or the short one)
    before = [x.clone() if x is not None else None for x in (dW, dT2, dT3)]
    ws.zero_()
    p_short = R.prob(wl, T=wl.T - 1)
    R.vce.vce_ngram_embed_bwd_plan(p_short, torch.from_numpy(ids[:-1].copy()).cuda(), M2, M3, ws, seq_len=seq_len)
    st = R.status_word()
    R.vce.vce_ngram_embed_bwd_apply(p, dE_d, dW, dT2, M2, dT3, M3, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1   # VCE_ERR_ARG
    for a, b in zip((dW, dT2, dT3), before):
        if a is not None:
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("narrow", ["0", "1"])
def test_ngram_bwd_narrow_and_wide_slices(narrow, monkeypatch):
    """The three tables' reduce with the multi-run ids' column slices forced
    narrow or wide (VCE_EMBED_NARROW; by default the three-table reduce keeps
    them wide): bit-exact against the replays either way, with slices that end
    inside a row (H = 1288)."""
    monkeypatch.setenv("VCE_EMBED_NARROW", narrow)
    T, H, V_real, Vp, M2, M3, seq_len = 3000, 1288, 5000, 5056, 613, 1024, 0
    wl, d, _, _ = _case("bf16", T, H, V_real, Vp, M2, M3, seed=95)
    ids = d["ids"].copy()
    ids[100:700] = ids[99]                   # a long run of one id: multi-run rows in every table
    rng = np.random.default_rng(11)
    inits = [rng.standard_normal((wl.Vp, wl.H)).astype(np.float32),
             rng.standard_normal((M2, wl.H)).astype(np.float32),
             rng.standard_normal((M3, wl.H)).astype(np.float32)]
    got = _bwd(wl, ids, d["dE"], M2, M3, seq_len, inits)
    want = _replays(wl, ids, d["dE"], M2, M3, seq_len, inits)
    for g, w in zip(got, want):
        assert np.array_equal(g.view(np.uint32), w.view(np.uint32))
