"""Pins for the oracle: checks against what the pages and the mathematics fix.

Each pin is a function of the oracle module ``O`` so that the same pin can be
run against a copy of the oracle with a planted mistake (test_oracle_pins.py
asserts that every planted mistake is caught by at least one pin).

Nothing here retypes an oracle formula: pins use closed forms, hand-derived
values, values printed on the pages (tests/golden), exact brute force in
decimal arithmetic, finite differences, and independent library routines
(torch fp64 autograd, scipy, numpy ufunc.at).
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext

import numpy as np
import torch
import torch.nn.functional as F

from conftest import read_golden

IGN = -100


def _rand_case(seed, T, H, V_real, Vp, ignore=(), bad=(), pad=8.0, scale=1.0):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((T, H)) * scale
    W = rng.standard_normal((Vp, H)) * 0.5
    if Vp > V_real:
        W[V_real:] = pad
    y = rng.integers(0, V_real, size=T)
    for t in ignore:
        y[t] = IGN
    for t in bad:
        y[t] = V_real + 3
    return h, W, y


# --------------------------------------------------------------------------
# Padding and shard layout
# --------------------------------------------------------------------------

def pin_pad_vocab(O):
    g = read_golden("padded_head_demo.txt")
    assert O.pad_vocab_size(g["head_vocab"]) == g["head_vocab_padded"]
    assert O.pad_vocab_size(g["vocab_real"]) == g["vocab_padded"]
    # closed form: the least multiple of 64 that is >= v
    for v in list(range(1, 300)) + [50000, 151936, 201088]:
        p = O.pad_vocab_size(v)
        assert p % 64 == 0 and v <= p < v + 64
    assert O.vocab_aligned(64) and not O.vocab_aligned(g["vocab_real"])


def pin_shards_tp_page(O):
    g = read_golden("tp_embedding_shards.txt")
    lo = O.shard_bounds(g["V"], g["ranks"])
    assert np.all(np.diff(lo) == g["rows_per_rank"])
    for k in (0, 1, 7):
        a, b = g[f"rank{k}"]
        assert lo[k] == a and lo[k + 1] - 1 == b
    ids = np.array([0, 25135, 25136, 50271, 175952, 201087, 201088, -100])
    valid, owner, local = O.ownership(ids, g["V"], g["V"], g["ranks"])
    assert list(owner) == [0, 0, 1, 1, 7, 7, -1, -1]
    assert list(local) == [0, 25135, 0, 25135, 0, 25135, -1, -1]


def pin_shards_cover(O):
    """Shards tile [0, Vp) contiguously; sizes are floor or ceil of Vp/S; an
    even split agrees with numpy's array_split; every valid id has exactly one
    owner and invalid ids none."""
    for Vp in (64, 1024, 50048, 151936):
        for S in (1, 2, 3, 4, 7, 8, 64):
            lo = O.shard_bounds(Vp, S)
            assert lo[0] == 0 and lo[-1] == Vp
            sz = np.diff(lo)
            assert set(sz.tolist()) <= {Vp // S, -(-Vp // S)}
            if Vp % S == 0:
                ref = [a[0] for a in np.array_split(np.arange(Vp), S)]
                assert list(lo[:-1]) == ref
    Vp, V_real = 1024, 1000
    ids = np.concatenate([np.arange(-3, Vp + 3), [IGN, -(2 ** 31), 2 ** 40]])
    for S in (1, 3, 4, 7, Vp):
        valid, owner, local = O.ownership(ids, V_real, Vp, S)
        lo = O.shard_bounds(Vp, S)
        for i, v in enumerate(ids):
            inside = [k for k in range(S) if lo[k] <= v < lo[k + 1]]
            if 0 <= v < V_real:
                assert valid[i] and owner[i] == inside[0] and local[i] == v - lo[inside[0]]
            else:
                assert not valid[i] and owner[i] == -1 and local[i] == -1


# --------------------------------------------------------------------------
# Embedding
# --------------------------------------------------------------------------

def pin_embedding_forward(O):
    rng = np.random.default_rng(5)
    Vp, V_real, H = 1024, 1000, 24
    W = rng.standard_normal((Vp, H)).astype(np.float32)
    W[V_real:] = 8.0
    ids = np.concatenate([rng.integers(0, Vp, 200), [IGN, -1, Vp, Vp + 10, 999, 1000, 0]])
    E = O.embed_forward(ids, W, V_real)
    valid = (ids >= 0) & (ids < V_real)
    # torch's own lookup on the valid ids; padded rows, padding and
    # out-of-range ids give zero rows
    ref = F.embedding(torch.from_numpy(np.where(valid, ids, 0)), torch.from_numpy(W)).numpy()
    assert np.array_equal(E[valid], ref[valid])
    assert np.all(E[~valid] == 0)
    for S in (1, 2, 3, 4, 7, 8):
        Es = O.embed_forward_by_shards(ids, W, V_real, Vp, S)
        assert np.array_equal(Es, E.astype(np.float64))
    # bf16 bit patterns are copied exactly
    Wb = rng.integers(0, 2 ** 16, size=(Vp, H), dtype=np.uint16)
    Eb = O.embed_forward(ids, Wb, V_real)
    assert np.array_equal(Eb[valid], Wb[ids[valid]])


def pin_embedding_backward(O):
    rng = np.random.default_rng(6)
    Vp, V_real, H, T = 256, 250, 16, 500
    ids = rng.integers(-5, Vp + 5, size=T)
    ids[:40] = 3                                   # a long run of one id
    ids[40:45] = IGN
    dE = rng.standard_normal((T, H))
    dW = O.embed_backward(ids, dE, V_real, Vp)
    ref = np.zeros((Vp, H))
    keep = (ids >= 0) & (ids < V_real)
    np.add.at(ref, ids[keep], dE[keep])
    assert np.allclose(dW, ref, rtol=0, atol=1e-12)
    ref_t = torch.zeros(Vp, H, dtype=torch.float64).index_add_(
        0, torch.from_numpy(ids[keep]), torch.from_numpy(dE[keep]))
    assert np.allclose(dW, ref_t.numpy(), rtol=0, atol=1e-12)
    assert np.all(dW[V_real:] == 0)


def pin_embedding_replay_order(O):
    """Hand-derived fp32 results that fix the summation order.

    1e8 has an fp32 spacing of 8, so adding 1.0 to it is lost while eight
    ones summed first give 8.0, which is kept.
    """
    H = 1
    big = np.float32(1e8)
    vals = [big] + [np.float32(1.0)] * 15                  # t = 0..15, one id
    dE = np.array(vals, dtype=np.float32).reshape(-1, 1)
    ids = np.full(16, 5)
    init = np.zeros((8, H), dtype=np.float32)
    # one run of 16: every +1 is absorbed -> 1e8
    r16 = O.embed_backward_replay_f32(ids, dE, 8, 16, init)
    assert r16[5, 0] == np.float32(100000000.0)
    # runs of 8: (1e8 + seven ones -> 1e8) + (eight ones -> 8) = 100000008
    r8 = O.embed_backward_replay_f32(ids, dE, 8, 8, init)
    assert r8[5, 0] == np.float32(100000008.0)
    # runs of 4: 1e8, 4, 4, 4 added left to right; 1e8 + 4 is a tie that rounds
    # to the even neighbour 1e8 each time (right to left would give 100000016)
    r4 = O.embed_backward_replay_f32(ids, dE, 8, 4, init)
    assert r4[5, 0] == np.float32(100000000.0)
    # tokens ascending in t: the same values in reverse t order sum the ones first
    r_rev = O.embed_backward_replay_f32(ids, dE[::-1].copy(), 8, 16, init)
    assert r_rev[5, 0] == np.float32(100000016.0)          # 1e8 + 15 rounds to +16
    # the total is added once to the existing row
    init2 = init.copy(); init2[5, 0] = np.float32(3.0)
    r = O.embed_backward_replay_f32(np.array([5]), np.array([[np.float32(2.0)]]), 8, 4, init2)
    assert r[5, 0] == np.float32(5.0)
    # other rows and invalid ids leave dW unchanged
    r = O.embed_backward_replay_f32(np.array([IGN, 9, -1]), np.ones((3, 1), np.float32), 8, 4, init2)
    assert np.array_equal(r, init2)


def pin_embedding_replay_bound(O):
    """The fp32 replay equals the exact sum within the sequential-summation
    error bound n*u*sum|x|, and single-token rows are exact."""
    rng = np.random.default_rng(7)
    Vp, V_real, H, T = 300, 300, 8, 2000
    ids = np.minimum(rng.zipf(1.3, size=T) - 1, V_real - 1)
    dE = rng.standard_normal((T, H)).astype(np.float32)
    init = rng.standard_normal((Vp, H)).astype(np.float32)
    for chunk in (1, 4, 32, 4096):
        got = O.embed_backward_replay_f32(ids, dE, V_real, chunk, init).astype(np.float64)
        exact = init.astype(np.float64)
        np.add.at(exact, ids, dE.astype(np.float64))
        n = np.bincount(ids, minlength=Vp)[:, None] + 1
        absum = np.abs(init.astype(np.float64)).copy()
        np.add.at(absum, ids, np.abs(dE.astype(np.float64)))
        u = 2.0 ** -24
        assert np.all(np.abs(got - exact) <= n * u * absum * 1.01 + 1e-30)
        single = np.bincount(ids, minlength=Vp) == 1
        for v in np.nonzero(single)[0]:
            t = int(np.nonzero(ids == v)[0][0])
            assert np.array_equal(got[v].astype(np.float32), (init[v] + dE[t]).astype(np.float32))


# --------------------------------------------------------------------------
# Cross-entropy forward
# --------------------------------------------------------------------------

def pin_equal_logits(O):
    """All-equal logits give loss = ln(V_real) exactly (up to rounding)."""
    T, H, V_real, Vp = 64, 64, 1000, 1024
    h = np.zeros((T, H))
    rng = np.random.default_rng(1)
    W = rng.standard_normal((Vp, H)) * 0.02
    W[V_real:] = 8.0
    y = rng.integers(0, V_real, T)
    r = O.cross_entropy_forward(h, W, y, V_real)
    assert abs(r["loss"] - math.log(1000)) < 1e-12
    assert abs(math.log(1000) - 6.907755278982137) < 1e-15
    # identical rows of W with any h: every logit of a row is the same value
    W2 = np.tile(rng.standard_normal(H), (Vp, 1))
    W2[V_real:] = 8.0
    r2 = O.cross_entropy_forward(rng.standard_normal((T, H)), W2, y, V_real)
    assert np.allclose(r2["token_loss"], math.log(V_real), rtol=0, atol=1e-11)


def pin_normalisation(O):
    h, W, y = _rand_case(2, 20, 16, 77, 128)
    p = O.probabilities(h, W, 77, 128)
    assert np.allclose(p[:, :77].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p[:, 77:] == 0.0)
    # the assertion of section 7: padded mass below 1e-6
    assert np.abs(p[:, 77:]).sum() < 1e-6


def pin_padded_head_demo(O):
    """Section 4 of the padding write-up: real-class mass 1.000 once masked."""
    g = read_golden("padded_head_demo.txt")
    V, Vp = g["vocab_real"], g["vocab_padded"]
    rng = np.random.default_rng(0)
    z = rng.standard_normal(Vp)
    z[V:] = g["pad_logit"]
    # logits chosen directly: H = Vp, W = identity, h = the logit row
    h = z[None, :]
    W = np.eye(Vp)
    p = O.probabilities(h, W, V, Vp)
    assert round(float(p[0, :V].sum()), 3) == g["masked_real_mass"]
    assert p[0, V:].sum() == 0.0
    # unmasked, the garbage would hold most of the mass (closed form)
    unmasked_real = np.exp(z[:V]).sum() / np.exp(z).sum()
    assert unmasked_real < 0.01


def pin_bruteforce_decimal(O):
    """Tiny problems: logits summed exactly and log-sum-exp evaluated in
    60-digit decimal arithmetic."""
    getcontext().prec = 60
    for seed in range(4):
        T, H, V_real, Vp = 3, 4, 7, 64
        h, W, y = _rand_case(10 + seed, T, H, V_real, Vp, ignore=(2,) if seed % 2 else ())
        r = O.cross_entropy_forward(h, W, y, V_real)
        total, nv = Decimal(0), 0
        for t in range(T):
            zs = [sum(Decimal(float(h[t, j])) * Decimal(float(W[v, j])) for j in range(H))
                  for v in range(V_real)]
            lse = sum(z.exp() for z in zs).ln()
            assert abs(float(lse) - r["lse"][t]) < 1e-13 * max(1.0, abs(float(lse)))
            if y[t] != IGN:
                total += lse - zs[y[t]]
                nv += 1
        assert abs(float(total / nv) - r["loss"]) < 1e-13


def pin_torch_cross_entropy(O):
    """torch's fp64 cross_entropy (padded logits at -inf, ignore_index=-100,
    mean) and its autograd gradients, the library form of the padded head."""
    for seed, (T, H, V_real, Vp, g) in enumerate([(16, 8, 50, 64, 1.0), (33, 12, 200, 256, 0.37),
                                                   (5, 3, 64, 64, 2.0)]):
        h, W, y = _rand_case(20 + seed, T, H, V_real, Vp, ignore=(1, 4))
        ht = torch.tensor(h, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        z = ht @ Wt.T
        mask = torch.zeros(Vp, dtype=torch.float64)
        mask[V_real:] = float("-inf")
        loss = g * F.cross_entropy(z + mask, torch.tensor(y), ignore_index=IGN)
        loss.backward()
        r = O.cross_entropy_forward(h, W, y, V_real, g=g)
        assert abs(r["loss"] - loss.item()) < 1e-12 * max(1, abs(loss.item()))
        dH, dW = O.cross_entropy_backward(h, W, y, V_real, Vp, g=g)
        assert np.allclose(dH, ht.grad.numpy(), rtol=0, atol=1e-12)
        assert np.allclose(dW, Wt.grad.numpy(), rtol=0, atol=1e-12)
        lse_ref = torch.logsumexp(z.detach()[:, :V_real], dim=1).numpy()
        assert np.allclose(r["lse"], lse_ref, rtol=1e-14, atol=1e-14)


def pin_shard_invariance(O):
    """The sharded schedule equals the unsharded definition for any S, with
    targets at shard edges, the maximum in another shard, and the padded tail."""
    T, H, V_real, Vp = 24, 16, 1000, 1024
    h, W, y = _rand_case(30, T, H, V_real, Vp, ignore=(3,))
    y[:6] = [255, 256, 511, 512, 999, 0]
    # rows 6..9 get a dominant logit at a column in another shard than y
    for i, (yt, vs) in enumerate([(10, 519), (261, 779), (515, 17), (999, 0)]):
        y[6 + i] = yt
        h[6 + i] = 50 * W[vs] / np.linalg.norm(W[vs])
    plain = O.cross_entropy_forward(h, W, y, V_real)
    for S in (1, 2, 3, 4, 5, 6, 7, 8, Vp):
        sh = O.cross_entropy_forward_sharded(h, W, y, V_real, Vp, S)
        assert abs(sh["loss"] - plain["loss"]) <= 1e-12 * abs(plain["loss"])
        assert np.allclose(sh["lse"], plain["lse"], rtol=1e-13, atol=0)
        assert np.allclose(sh["z_target"], plain["z_target"], rtol=1e-13, atol=1e-13)
    own, _gap = O.max_owner(h, W, V_real, Vp, 4)
    tgt = O.target_owner(y, V_real, Vp, 4)
    assert all(own[6 + i] != tgt[6 + i] for i in range(4))
    z = h @ W[:V_real].T
    assert list(z[6:10].argmax(axis=1)) == [519, 779, 17, 0]
    sh4 = O.cross_entropy_forward_sharded(h, W, y, V_real, Vp, 4)
    assert list(np.argmax(sh4["shard_max"], axis=1)[6:10]) == [2, 3, 0, 0]


def pin_ignored_and_bad(O):
    h, W, y = _rand_case(40, 12, 8, 90, 128, ignore=(0, 5), bad=(7,))
    r = O.cross_entropy_forward(h, W, y, 90)
    assert r["n_valid"] == 9
    assert r["token_loss"][0] == 0 and r["token_loss"][5] == 0 and r["token_loss"][7] == 0
    assert list(np.nonzero(r["bad"])[0]) == [7]
    dH, dW = O.cross_entropy_backward(h, W, y, 90, 128)
    assert np.all(dH[[0, 5, 7]] == 0)
    # a bad target behaves exactly like an ignored one
    y2 = y.copy(); y2[7] = IGN
    dH2, dW2 = O.cross_entropy_backward(h, W, y2, 90, 128)
    assert np.array_equal(dH, dH2) and np.array_equal(dW, dW2)
    # no valid token at all: loss 0 and no gradient (reading R4)
    yn = np.full(12, IGN)
    assert O.cross_entropy_forward(h, W, yn, 90)["loss"] == 0.0
    dHn, dWn = O.cross_entropy_backward(h, W, yn, 90, 128)
    assert not dHn.any() and not dWn.any()
    # an ignore value naming a real class is refused; one past the real classes is not
    for ig in (0, 89):
        try:
            O.cross_entropy_forward(h, W, y, 90, ignore_index=ig)
        except ValueError:
            pass
        else:
            raise AssertionError(f"ignore_index {ig} accepted")
    y3 = y2.copy(); y3[5] = 90                      # 90 is the ignore value now; -100 is bad
    r90 = O.cross_entropy_forward(h, W, y3, 90, ignore_index=90)
    assert r90["n_valid"] == 9 and list(np.nonzero(r90["bad"])[0]) == [0, 7]


# --------------------------------------------------------------------------
# Cross-entropy backward
# --------------------------------------------------------------------------

def pin_finite_differences(O):
    """Central differences of the fp64 loss against dH and dW."""
    T, H, V_real, Vp, g = 3, 4, 7, 16, 1.7
    h, W, y = _rand_case(50, T, H, V_real, Vp, ignore=(1,))
    dH, dW = O.cross_entropy_backward(h, W, y, V_real, Vp, g=g)
    eps = 1e-6

    def L(hh, WW):
        return O.cross_entropy_forward(hh, WW, y, V_real, g=g)["loss"]

    for t in range(T):
        for j in range(H):
            e = np.zeros_like(h); e[t, j] = eps
            fd = (L(h + e, W) - L(h - e, W)) / (2 * eps)
            assert abs(fd - dH[t, j]) < 1e-7
    for v in range(Vp):
        for j in range(H):
            e = np.zeros_like(W); e[v, j] = eps
            fd = (L(h, W + e) - L(h, W - e)) / (2 * eps)
            assert abs(fd - dW[v, j]) < 1e-7


def pin_gradient_invariants(O):
    T, H, V_real, Vp = 40, 16, 300, 320
    h, W, y = _rand_case(60, T, H, V_real, Vp, ignore=(2, 9))
    nv = O.n_valid(y, V_real)
    G = O.logit_gradient(h, W, y, V_real, Vp, 1.0 / nv)
    valid = y != IGN
    assert np.allclose(G[valid].sum(axis=1), 0.0, atol=1e-15)
    assert np.all(G[~valid] == 0) and np.all(G[:, V_real:] == 0)
    dH, dW = O.cross_entropy_backward(h, W, y, V_real, Vp)
    # sum over classes of dW_head = sum_t (sum_v G_tv) h_t = 0
    assert np.allclose(dW.sum(axis=0), 0.0, atol=1e-13)
    assert np.all(dW[V_real:] == 0)
    # rows of dH computed alone agree with the full computation
    part = O.hidden_gradient_rows(h[5:9], W, y[5:9], V_real, 1.0 / nv)
    assert np.allclose(part, dH[5:9], rtol=0, atol=1e-15)
    # rows of dW_head from the batch lse agree with the full computation
    lse = O.cross_entropy_forward(h, W, y, V_real)["lse"]
    rows = [0, y[0], y[1], V_real - 1]
    part = O.head_gradient_rows(h, W, y, V_real, lse, 1.0 / nv, rows)
    assert np.allclose(part, dW[rows], rtol=0, atol=1e-15)


def pin_sampled_candidates(O):
    """Candidate list: sorted distinct targets (numpy's unique), then draws in
    order that are not targets; positions point back at each target."""
    rng = np.random.default_rng(70)
    V, P, T = 500, 160, 120
    y = rng.integers(0, V, T)
    y[:5] = IGN
    y[5:40] = 7                               # repeats
    draws = rng.permutation(V)
    cand, pos, nu = O.sampled_candidates(y, V, P, draws)
    uniq = np.unique(y[y != IGN])
    assert nu == uniq.size and np.array_equal(cand[:nu], uniq)
    assert cand.size == P and np.unique(cand).size == P
    negs = cand[nu:]
    assert not np.isin(negs, uniq).any()
    order = [int(np.nonzero(draws == v)[0][0]) for v in negs]
    assert order == sorted(order)
    expected_first = [d for d in draws if d not in set(uniq.tolist())][:P - nu]
    assert list(negs) == expected_first
    valid = y != IGN
    assert np.array_equal(cand[pos[valid]], y[valid]) and np.all(pos[~valid] == IGN)
    # draws with repeats and values outside the vocabulary, worked by hand:
    # targets {2, 5}; draws 5 (a target), 9, -1 (outside), 9 (repeat), 500
    # (outside), 3, 2 (a target), 7 -> negatives 9, 3, 7
    cand, pos, nu = O.sampled_candidates([5, 2, IGN, 5], V, 5, [5, 9, -1, 9, 500, 3, 2, 7, 8])
    assert list(cand) == [2, 5, 9, 3, 7] and nu == 2 and list(pos) == [1, 0, IGN, 1]


def pin_sampled_full_set_is_full_softmax(O):
    """With every class a candidate (P = V_real), the sampled loss is the full
    loss and its gradients the full gradients (the candidate order only
    permutes the classes)."""
    T, H, V = 30, 8, 40
    h, W, y = _rand_case(71, T, H, V, 64, ignore=(3,))
    draws = np.random.default_rng(72).permutation(V)
    cand, pos, _ = O.sampled_candidates(y, V, V, draws)
    r = O.sampled_cross_entropy(h, W, y, V, 64, cand, pos)
    full = O.cross_entropy_forward(h, W, y, V)
    dH, dW = O.cross_entropy_backward(h, W, y, V, 64)
    assert abs(r["loss"] - full["loss"]) < 1e-12
    assert np.allclose(r["dH"], dH, atol=1e-14) and np.allclose(r["dW"], dW, atol=1e-14)
    # a smaller candidate list: torch's cross-entropy on the gathered logits
    y2 = np.where(y == IGN, IGN, y % 10)      # at most 10 distinct targets
    cand, pos, nu = O.sampled_candidates(y2, V, 16, draws)
    assert nu <= 10
    z = torch.tensor(h) @ torch.tensor(W)[torch.tensor(cand)].T
    ref = F.cross_entropy(z, torch.tensor(pos), ignore_index=IGN).item()
    assert abs(O.sampled_cross_entropy(h, W, y2, V, 64, cand, pos)["loss"] - ref) < 1e-12


def pin_oth_head(O):
    """OT-H: the second head is scored on the token two positions ahead of each
    input position, at weight 0.1."""
    V, H = 8, 8
    tokens = np.array([0, 1, 2, 3, 4, 5, 6, 7], dtype=np.int64)   # T + 1 = 8
    T = tokens.size - 1
    h = 50.0 * np.eye(H)[tokens[:-1]]               # h[t] encodes the input token at t
    W = np.zeros((V, H))                             # head one: equal logits, loss ln V
    W2 = np.zeros((V, H))
    for v in range(2, V):
        W2[v, v - 2] = 1.0                           # head two: logit 50 for class tokens[t] + 2
    r = O.oth_loss(h, W, W2, tokens, V, V)
    assert abs(r["main"] - np.log(V)) < 1e-12
    # aligned on tokens[2:], head two is right at every position (loss ~ 7 e^-50)
    assert r["aux"] < 1e-18
    assert abs(r["loss"] - (np.log(V) + 0.1 * r["aux"])) < 1e-15
    # with equal logits in head two as well, the total is 1.1 ln V
    r0 = O.oth_loss(h, W, np.zeros((V, H)), tokens, V, V)
    assert abs(r0["loss"] - 1.1 * np.log(V)) < 1e-12
    # gradients: finite differences of the total loss in h, which also sees the
    # row T-1 that head two never reads
    rng = np.random.default_rng(80)
    h = rng.standard_normal((T, H))
    W = rng.standard_normal((V, H)) * 0.3
    W2 = rng.standard_normal((V, H)) * 0.3
    tokens = rng.integers(0, V, T + 1)
    tokens[3] = IGN
    r = O.oth_loss(h, W, W2, tokens, V, V)
    eps = 1e-6
    for (i, j) in [(0, 0), (2, 5), (T - 2, 1), (T - 1, 3)]:
        hp, hm = h.copy(), h.copy()
        hp[i, j] += eps
        hm[i, j] -= eps
        fd = (O.oth_loss(hp, W, W2, tokens, V, V)["loss"] - O.oth_loss(hm, W, W2, tokens, V, V)["loss"]) / (2 * eps)
        assert abs(fd - r["dH"][i, j]) < 1e-8
    # head two's weight gradient: torch autograd of 0.1 * CE(h[:-1] W2^T, tokens[2:])
    W2t = torch.tensor(W2, requires_grad=True)
    (0.1 * F.cross_entropy(torch.tensor(h[:-1]) @ W2t.T, torch.tensor(tokens[2:]), ignore_index=IGN)).backward()
    assert np.allclose(r["dW2"], W2t.grad.numpy(), atol=1e-14)


def pin_greedy_argmax(O):
    """Greedy argmax: a constructed head whose answer is known, ties to the
    lowest class, padded rows never chosen, the sharded schedule equal to the
    plain one for every S, and brute force by plain loops."""
    rng = np.random.default_rng(90)
    V, H, Vp = 40, 48, 64
    Q, _ = np.linalg.qr(rng.standard_normal((H, H)))
    W = np.zeros((Vp, H))
    W[:V] = Q[:V]                                    # orthonormal rows: z_v = 10 * [v == v*]
    W[V:] = 8.0                                      # padding rows with large logits
    want = np.array([0, 7, 39, 16, 23, 31], dtype=np.int64)
    h = 10.0 * W[want]
    arg, m = O.greedy_argmax(h, W, V)
    assert np.array_equal(arg, want) and np.allclose(m, 10.0, atol=1e-12)
    # a duplicate of row 23 at row 35 (another shard for S = 4): the lower class wins
    W2 = W.copy()
    W2[35] = W2[23]
    arg, _ = O.greedy_argmax(10.0 * W2[[23, 35]], W2, V)
    assert list(arg) == [23, 23]
    for S in (1, 2, 3, 4, 5, 8, Vp):
        a_s, m_s = O.greedy_argmax_sharded(10.0 * W2[[23, 35, 7]], W2, V, Vp, S)
        assert list(a_s) == [23, 23, 7] and np.allclose(m_s, 10.0, atol=1e-12)
    # random heads: plain loops over classes (strict >, so the first maximum stays)
    h = rng.standard_normal((9, H))
    Wr = rng.standard_normal((Vp, H))
    arg, m = O.greedy_argmax(h, Wr, V)
    for t in range(9):
        bv, bc = -np.inf, -1
        for v in range(V):
            zv = sum(float(h[t, j]) * float(Wr[v, j]) for j in range(H))
            if zv > bv:
                bv, bc = zv, v
        assert bc == arg[t] and abs(bv - m[t]) < 1e-12
    for S in (1, 3, 7, 64):
        a_s, _ = O.greedy_argmax_sharded(h, Wr, V, Vp, S)
        assert np.array_equal(a_s, arg)


def pin_max_owner(O):
    """max_owner against a head whose logits are known in closed form: with
    orthonormal rows Q_v and h = sum_v a_v Q_v, the logit of class v is a_v, so
    the owner of the largest one and the gap to the second largest are fixed
    by the chosen a. Ties (two identical rows) go to the lowest column, hence
    the lowest shard, with a gap of exactly 0; padded rows never count."""
    rng = np.random.default_rng(95)
    V, H, Vp, S = 48, 64, 64, 4                      # shards of 16 rows: [0,16), [16,32), [32,48), [48,64)
    Q, _ = np.linalg.qr(rng.standard_normal((H, H)))
    W = np.zeros((Vp, H))
    W[:V] = Q[:V]
    W[V:] = 8.0 * Q[V:]                              # padding rows: orthonormal directions with large logits
    # (largest class, its logit, second class, its logit) per token
    cases = [(3, 5.0, 40, 4.25), (20, 2.5, 21, 2.0), (47, 1.0, 0, -0.5), (33, 7.0, 17, 6.875)]
    a = np.full((len(cases), Vp), -3.0)
    a[:, V:] = 9.0                                   # padded classes hold the largest coefficients
    for t, (c1, v1, c2, v2) in enumerate(cases):
        a[t, c1], a[t, c2] = v1, v2
    h = a @ Q                                        # z_tv = a_tv for every v
    own, gap = O.max_owner(h, W, V, Vp, S)
    assert list(own) == [0, 1, 2, 2]
    want = [v1 - v2 for (_, v1, _, v2) in cases]
    assert np.allclose(gap, want, rtol=0, atol=1e-12), (gap, want)
    # identical rows 5 and 37 (shards 0 and 2): the lowest column's shard, gap 0
    W2 = W.copy()
    W2[37] = W2[5]
    h2 = 6.0 * W2[5][None, :]
    own2, gap2 = O.max_owner(h2, W2, V, Vp, S)
    assert list(own2) == [0] and gap2[0] == 0.0
    # the same rows moved so that the tie spans shards 1 and 3's real part
    W3 = W.copy()
    W3[45] = W3[18]
    own3, gap3 = O.max_owner(4.0 * W3[18][None, :], W3, V, Vp, S)
    assert list(own3) == [1] and gap3[0] == 0.0


def pin_ngram_hash(O):
    """The n-gram row index: hand-worked in base 10, sequence starts, invalid
    ids, and base-V digits recovered exactly when M = V^n."""
    x = [1, 2, 3, 4]
    assert list(O.ngram_index(x, 2, 10, 1000)) == [-1, 12, 23, 34]
    assert list(O.ngram_index(x, 3, 10, 1000)) == [-1, -1, 123, 234]
    assert list(O.ngram_index(x, 2, 10, 7)) == [-1, 5, 2, 6]        # 12, 23, 34 mod 7
    assert list(O.ngram_index(x, 3, 10, 7)) == [-1, -1, 4, 3]       # 123, 234 mod 7
    assert list(O.ngram_index(x, 1, 10, 1000)) == [1, 2, 3, 4]
    # two sequences of 2 tokens: no n-gram crosses the boundary
    assert list(O.ngram_index(x, 2, 10, 1000, seq_len=2)) == [-1, 12, -1, 34]
    assert list(O.ngram_index(x, 3, 10, 1000, seq_len=2)) == [-1, -1, -1, -1]
    # an invalid id removes every n-gram that contains it
    assert list(O.ngram_index([1, IGN, 3, 4], 2, 10, 1000)) == [-1, -1, -1, 34]
    assert list(O.ngram_index([1, 2, 10, 4, 5], 3, 10, 1000)) == [-1, -1, -1, -1, -1]
    # M = V^3: the index is the n-gram itself, written in base V
    V = 151936
    rng = np.random.default_rng(95)
    y = rng.integers(0, V, 50)
    idx = O.ngram_index(y, 3, V, V ** 3)
    for t in range(2, 50):
        a, r = divmod(int(idx[t]), V * V)
        b, c = divmod(r, V)
        assert (a, b, c) == (y[t - 2], y[t - 1], y[t])
    # reduced mod M exactly (Python integers, no overflow)
    big = O.ngram_index([V - 1] * 3, 3, V, 1 << 19)
    assert big[2] == (V ** 3 - 1) % (1 << 19)


def pin_ngram_embedding(O):
    """E = W[x] + T2[idx_2] + T3[idx_3]: exact on integer-valued fp32 tables,
    one round-to-nearest-even to bf16 (hand-worked ties), and the tables'
    gradients against np.add.at."""
    V, H, M2, M3 = 10, 4, 7, 11
    W = (100.0 * np.arange(V)[:, None] * np.ones((1, H))).astype(np.float32)
    T2 = (10.0 * np.arange(M2)[:, None] * np.ones((1, H))).astype(np.float32)
    T3 = (1.0 * np.arange(M3)[:, None] * np.ones((1, H))).astype(np.float32)
    x = np.array([1, 2, 3, IGN, 4, 5, 6], dtype=np.int64)
    E = O.ngram_embed_forward(x, W, T2, T3, V, M2, M3)
    i2 = O.ngram_index(x, 2, V, M2)
    i3 = O.ngram_index(x, 3, V, M3)
    want = (100.0 * np.where((x >= 0) & (x < V), x, 0) + 10.0 * np.maximum(i2, 0) + np.maximum(i3, 0))
    assert np.array_equal(E[:, 0], want.astype(np.float32))
    assert list(i2) == [-1, 12 % 7, 23 % 7, -1, -1, 45 % 7, 56 % 7]
    # bf16: 1 + 2^-8 rounds to 1 (a tie, to the even neighbour); 1 + 2^-8 + 2^-7
    # = 1 + 1.5 * 2^-7 rounds up to 1 + 2^-6 (the even neighbour of 1 + 2^-7)
    Wb = np.full((V, 2), 0x3F80, dtype=np.uint16)          # 1.0
    T2b = np.full((M2, 2), 0x3B80, dtype=np.uint16)        # 2^-8
    T3b = np.full((M3, 2), 0x3C00, dtype=np.uint16)        # 2^-7
    Eb = O.ngram_embed_forward(np.array([1, 2, 3]), Wb, T2b, T3b, V, M2, M3)
    assert list(Eb[:, 0]) == [0x3F80, 0x3F80, 0x3F82]
    # gradients: the three tables against np.add.at
    rng = np.random.default_rng(96)
    x = rng.integers(0, V, 40)
    x[[5, 17]] = IGN
    dE = rng.standard_normal((40, H))
    dW, dT2, dT3 = O.ngram_embed_backward(x, dE, V, 16, M2, M3, seq_len=8)
    for table, idx, rows in ((dW, np.where((x >= 0) & (x < V), x, -1), 16),
                             (dT2, O.ngram_index(x, 2, V, M2, 8), M2), (dT3, O.ngram_index(x, 3, V, M3, 8), M3)):
        ref = np.zeros((rows, H))
        ok = idx >= 0
        np.add.at(ref, idx[ok], dE[ok])
        assert np.allclose(table, ref, rtol=0, atol=1e-12)


ALL_PINS = [
    pin_pad_vocab, pin_shards_tp_page, pin_shards_cover, pin_embedding_forward,
    pin_embedding_backward, pin_embedding_replay_order, pin_embedding_replay_bound,
    pin_equal_logits, pin_normalisation, pin_padded_head_demo, pin_bruteforce_decimal,
    pin_torch_cross_entropy, pin_shard_invariance, pin_ignored_and_bad,
    pin_finite_differences, pin_gradient_invariants, pin_sampled_candidates,
    pin_sampled_full_set_is_full_softmax, pin_oth_head, pin_greedy_argmax, pin_max_owner, pin_ngram_hash,
    pin_ngram_embedding,
]
