"""Oracle for the vocabulary-sharded embedding and the globally normalised
cross-entropy: plain, slow, fp64 CPU definitions written from the method's
description.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg may import or call this module. The CUDA path never does, and this
module never imports the CUDA path: the two share nothing but the seeded input
arrays the callers pass in.

Sources (cited by page title and section):

* "Vocabulary shards: look up locally and normalize globally" (the method
  page; its paragraphs are cited as P1..P5):
  P1 ownership test, local index, masked lookup whose shard sum rebuilds the
     embedding; P2 explicit rules for padding / out-of-range ids, repeated
     tokens accumulate into one row, tied weights combine contributions;
  P3 global max over valid entries, local sums of exp against it combined
     globally, target logit from its unique owner, one global denominator;
  P4 padded classes excluded, ignored targets follow the loss mask, gradient
     = probability - target indicator times the loss scale;
  P5 no full-logit materialisation is required (the oracle does materialise:
     it is the definition, not the fast path).
* "Training collapses when token embeddings are not padded to a multiple of 64"
  (sections 4-7): pad_vocab_size, logits of padded classes set to -inf before
  softmax, cross-entropy with ignore_index=-100, the two assertions.
* "Sequence-parallel normalization" (paragraph 3): loss averaged once over the
  global valid tokens.
* "Tensor Parallelism (TP)", Embedding (VocabDimShardedEmbedding) and LM Head
  (ColumnParallelLinear): rank k holds rows [k*V/8, (k+1)*V/8).

Readings where the pages leave a step open (each is listed in the design notes):
  R1 shard k covers [floor(k*Vp/S), floor((k+1)*Vp/S)); uneven S is allowed.
  R2 a class is valid iff 0 <= v < V_real; padded rows may hold anything.
  R3 a target outside [0, V_real) that is not ignore_index is a data error; the
     token is then treated as ignored (flagged in ``bad``). The ignore value
     itself lies outside [0, V_real): one naming a real class is refused.
  R4 loss = g * sum of per-token losses / N_valid; with N_valid == 0 the loss
     and every gradient are 0 (the pages are silent; torch would give NaN).
  R5 the upstream scale g multiplies the loss and the gradient.
  R6 an embedding id outside [0, V_real) (the padding id ignore_index,
     negatives, padded rows, >= Vp) yields a zero row and no gradient.
  R7 tied weights: dW = dW_head + dW_embed.
  R8 max_owner ties go to the lowest global column.

Parity status: every function here is pinned by tests/test_oracle_pins.py
against closed forms, brute force, library routines or values the pages print.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


# ---------------------------------------------------------------------------
# Hashed n-gram input embeddings ("Sampled Softmax with Over-Tokenized
# Transformer", Setup and its loss listing)
# ---------------------------------------------------------------------------

def ngram_index(ids, n: int, V: int, M: int, seq_len: int = 0) -> np.ndarray:
    """Row of the hashed n-gram that ends at each token, -1 where there is none.

    Reading (the pages name hashed 2-gram and 3-gram tables but no hash): the
    n-gram (x[t-n+1], ..., x[t]) is read as a number in base V with x[t] the
    lowest digit, and reduced mod the table's M rows. A token with fewer than
    n-1 earlier tokens in its sequence (sequences of seq_len tokens laid end to
    end; 0 means one sequence), or whose n-gram holds an id outside [0, V),
    has no n-gram. Exact Python integers, one token at a time.
    """
    x = [int(v) for v in np.asarray(ids, dtype=np.int64)]
    out = np.full(len(x), -1, dtype=np.int64)
    if M <= 0:
        return out
    for t in range(len(x)):
        pos = t % seq_len if seq_len > 0 else t
        if pos < n - 1:
            continue
        gram = x[t - n + 1:t + 1]
        if any(v < 0 or v >= V for v in gram):
            continue
        value = sum(v * V ** j for j, v in enumerate(reversed(gram)))
        out[t] = value % M
    return out


def _rows_f32(table, idx: np.ndarray, H: int) -> np.ndarray:
    """fp32 values of the rows idx of a stored table; +0 rows where idx < 0."""
    out = np.zeros((idx.shape[0], H), dtype=np.float32)
    ok = idx >= 0
    if table is not None and ok.any():
        rows = np.asarray(table)[idx[ok]]
        if rows.dtype == np.uint16:
            rows = (rows.astype(np.uint32) << np.uint32(16)).view(np.float32)
        out[ok] = rows.astype(np.float32)
    return out


def _round_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even (finite values)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)


def ngram_embed_forward(ids, W, T2, T3, V_real: int, M2: int, M3: int, seq_len: int = 0) -> np.ndarray:
    """E[t] = W[x_t] + T2[idx_2(t)] + T3[idx_3(t)] (the listing's embed plus the
    two n-gram embeddings), summed in fp32 in that order from +0 with a missing
    term read as +0, then rounded once to the tables' storage type (bf16 bit
    patterns when W is stored as uint16). Reading: one fp32 sum and one
    rounding, the plainest way to add three stored rows."""
    x = np.asarray(ids, dtype=np.int64)
    H = np.asarray(W).shape[1]
    i1 = np.where((x >= 0) & (x < V_real), x, -1)
    i2 = ngram_index(x, 2, V_real, M2, seq_len)
    i3 = ngram_index(x, 3, V_real, M3, seq_len)
    acc = np.zeros((x.shape[0], H), dtype=np.float32)
    acc = acc + _rows_f32(W, i1, H)
    acc = acc + _rows_f32(T2, i2, H)
    acc = acc + _rows_f32(T3, i3, H)
    return _round_bf16_bits(acc) if np.asarray(W).dtype == np.uint16 else acc


def ngram_embed_backward(ids, dE, V_real: int, Vp: int, M2: int, M3: int, seq_len: int = 0):
    """fp64 gradients of the three tables: dW[x_t], dT2[idx_2(t)] and
    dT3[idx_3(t)] each receive dE[t] (P2's accumulation, table by table)."""
    x = np.asarray(ids, dtype=np.int64)
    dW = embed_backward(x, dE, V_real, Vp)
    dT2 = embed_backward(ngram_index(x, 2, V_real, M2, seq_len), dE, M2, M2) if M2 > 0 else None
    dT3 = embed_backward(ngram_index(x, 3, V_real, M3, seq_len), dE, M3, M3) if M3 > 0 else None
    return dW, dT2, dT3


# ---------------------------------------------------------------------------
# Vocabulary padding and shard layout
# ---------------------------------------------------------------------------

def pad_vocab_size(vocab_size: int, multiple: int = 64) -> int:
    """Round the vocabulary up to a multiple of 64 ("Training collapses ...",
    section 5, pad_vocab_size)."""
    return ((vocab_size + multiple - 1) // multiple) * multiple


def vocab_aligned(Vp: int, multiple: int = 64) -> bool:
    """The build-time check of section 7 (assert_vocab_aligned) as a predicate."""
    return Vp % multiple == 0


def shard_bounds(Vp: int, S: int) -> np.ndarray:
    """Row bounds lo[0..S] of S contiguous shards (reading R1; "Tensor
    Parallelism (TP)", Embedding: rank k holds rows [k*V/8, (k+1)*V/8))."""
    return np.array([(k * Vp) // S for k in range(S + 1)], dtype=np.int64)


def ownership(ids: np.ndarray, V_real: int, Vp: int, S: int):
    """Ownership test and local index of each global id ("Vocabulary shards",
    P1, P2; readings R1, R2, R6).

    Returns (valid, owner, local): owner is the shard whose range holds a valid
    id (-1 otherwise) and local = id - lo[owner] (-1 otherwise). The test is
    done shard by shard, as each rank would do it, before any index is formed.
    """
    ids = np.asarray(ids, dtype=np.int64)
    lo = shard_bounds(Vp, S)
    valid = (ids >= 0) & (ids < V_real)
    owner = np.full(ids.shape, -1, dtype=np.int64)
    local = np.full(ids.shape, -1, dtype=np.int64)
    for k in range(S):
        mine = valid & (ids >= lo[k]) & (ids < lo[k + 1])
        owner[mine] = k
        local[mine] = ids[mine] - lo[k]
    return valid, owner, local


def target_status(targets: np.ndarray, V_real: int, ignore_index: int = IGNORE_INDEX):
    """(valid, bad) masks of the loss targets (P4 and readings R3)."""
    if 0 <= ignore_index < V_real:
        raise ValueError("ignore_index names a real class")
    y = np.asarray(targets, dtype=np.int64)
    valid = (y >= 0) & (y < V_real)
    bad = ~valid & (y != ignore_index)
    return valid, bad


# ---------------------------------------------------------------------------
# Embedding lookup and its gradient
# ---------------------------------------------------------------------------

def embed_forward(ids: np.ndarray, W: np.ndarray, V_real: int) -> np.ndarray:
    """E[t] = W[id_t] for a valid id, else a zero row (P1, reading R6).

    W is taken as stored (fp32 values or bf16 bit patterns); rows are copied,
    so the result is exact.
    """
    ids = np.asarray(ids, dtype=np.int64)
    E = np.zeros((ids.shape[0], W.shape[1]), dtype=W.dtype)
    valid = (ids >= 0) & (ids < V_real)
    E[valid] = W[ids[valid]]
    return E


def embed_forward_by_shards(ids: np.ndarray, W: np.ndarray, V_real: int,
                            Vp: int, S: int) -> np.ndarray:
    """The sharded form of P1 and "Tensor Parallelism (TP)", Embedding, prefill:
    each shard looks up only the ids it owns through its local table, gives a
    zero vector for the rest, and the S partial embeddings are summed.

    Values are carried in fp64 (rows of zeros add exactly)."""
    ids = np.asarray(ids, dtype=np.int64)
    lo = shard_bounds(Vp, S)
    Wf = _as_f64(W)
    total = np.zeros((ids.shape[0], W.shape[1]), dtype=np.float64)
    for k in range(S):
        table_k = Wf[lo[k]:lo[k + 1]]                    # the shard's own rows
        owned = (ids >= lo[k]) & (ids < lo[k + 1]) & (ids >= 0) & (ids < V_real)
        part = np.zeros_like(total)
        part[owned] = table_k[ids[owned] - lo[k]]        # local index only
        total += part
    return total


def embed_backward(ids: np.ndarray, dE: np.ndarray, V_real: int, Vp: int) -> np.ndarray:
    """dW[v] = sum of dE[t] over tokens with id_t == v, in fp64 (P2: repeated
    tokens accumulate into the same owned row; invalid ids contribute nothing)."""
    ids = np.asarray(ids, dtype=np.int64)
    dEf = _as_f64(dE)
    dW = np.zeros((Vp, dEf.shape[1]), dtype=np.float64)
    for t in range(ids.shape[0]):
        v = ids[t]
        if 0 <= v < V_real:
            dW[v] += dEf[t]
    return dW


def embed_backward_replay_f32(ids: np.ndarray, dE32: np.ndarray, V_real: int,
                              chunk: int, dW_init: np.ndarray) -> np.ndarray:
    """The same sum as ``embed_backward`` carried out in fp32 in one fixed order,
    so that a deterministic implementation can be compared bit for bit.

    Order: valid ids ascending; the tokens of one id ascending in t, cut into
    runs of ``chunk`` consecutive tokens; each run is summed in fp32 from 0.0,
    token after token; the run sums are added left to right in fp32; the total
    is added once to the fp32 row dW_init[id]. Rows without a valid id keep
    dW_init unchanged.
    """
    ids = np.asarray(ids, dtype=np.int64)
    dE32 = np.asarray(dE32, dtype=np.float32)
    dW = np.array(dW_init, dtype=np.float32, copy=True)
    valid_t = [t for t in range(ids.shape[0]) if 0 <= ids[t] < V_real]
    by_id = {}
    for t in valid_t:
        by_id.setdefault(int(ids[t]), []).append(t)
    for v in sorted(by_id):
        ts = by_id[v]
        total = None
        for c0 in range(0, len(ts), chunk):
            run = np.zeros(dE32.shape[1], dtype=np.float32)
            for t in ts[c0:c0 + chunk]:
                run = run + dE32[t]
            total = run if total is None else total + run
        dW[v] = dW[v] + total
    return dW


# ---------------------------------------------------------------------------
# Cross-entropy over the padded vocabulary
# ---------------------------------------------------------------------------

def logits(h: np.ndarray, W: np.ndarray, V_real: int) -> np.ndarray:
    """z[t, v] = <h_t, W_v> in fp64 over the real classes v < V_real only; the
    padded classes are never formed, which is the -inf mask of "Training
    collapses ...", section 5 (PaddedLMHead.forward)."""
    return _as_f64(h) @ _as_f64(W)[:V_real].T


def probabilities(h: np.ndarray, W: np.ndarray, V_real: int, Vp: int) -> np.ndarray:
    """p[t, v] over all Vp columns: softmax of the real logits, exactly 0 on the
    padded columns (section 5: padded logits set to -inf)."""
    z = logits(h, W, V_real)
    lse = log_sum_exp(z)
    p = np.zeros((z.shape[0], Vp), dtype=np.float64)
    p[:, :V_real] = np.exp(z - lse[:, None])
    return p


def log_sum_exp(z: np.ndarray) -> np.ndarray:
    """lse_t = M_t + log sum_v exp(z_tv - M_t), M_t the row maximum (P3, P4:
    subtracting the maximum changes no probability)."""
    M = z.max(axis=1)
    return M + np.log(np.exp(z - M[:, None]).sum(axis=1))


def n_valid(targets: np.ndarray, V_real: int, ignore_index: int = IGNORE_INDEX) -> int:
    valid, _ = target_status(targets, V_real, ignore_index)
    return int(valid.sum())


def cross_entropy_rows(h: np.ndarray, W: np.ndarray, targets: np.ndarray,
                       V_real: int, ignore_index: int = IGNORE_INDEX):
    """Per-token quantities for the given rows: lse, the target logit and the
    per-token loss lse - z_target (0 for ignored or bad targets)."""
    y = np.asarray(targets, dtype=np.int64)
    z = logits(h, W, V_real)
    lse = log_sum_exp(z)
    valid, bad = target_status(y, V_real, ignore_index)
    z_tgt = np.zeros(y.shape[0], dtype=np.float64)
    z_tgt[valid] = z[np.nonzero(valid)[0], y[valid]]
    token_loss = np.where(valid, lse - z_tgt, 0.0)
    return dict(lse=lse, z_target=z_tgt, token_loss=token_loss, valid=valid, bad=bad)


def cross_entropy_forward(h, W, targets, V_real: int, ignore_index: int = IGNORE_INDEX,
                          g: float = 1.0):
    """Globally normalised cross-entropy (P3, P4), averaged once over the valid
    tokens ("Sequence-parallel normalization", paragraph 3; readings R3-R5)."""
    r = cross_entropy_rows(h, W, targets, V_real, ignore_index)
    nv = int(r["valid"].sum())
    loss = g * r["token_loss"].sum() / nv if nv > 0 else 0.0
    r.update(loss=loss, n_valid=nv)
    return r


def cross_entropy_forward_sharded(h, W, targets, V_real: int, Vp: int, S: int,
                                  ignore_index: int = IGNORE_INDEX, g: float = 1.0):
    """The method's own schedule over S vocabulary shards (P3):

    1. each shard forms the logits of the rows it owns (its [T, Vp/S] block);
    2. the global maximum M over valid entries of all shards;
    3. each shard sums exp(z - M) over its valid columns; the sums are added;
    4. the target logit is read from the one shard that owns the target;
    5. loss_t = M + log(sum) - z_target, averaged once over valid tokens.

    Also returns each shard's local maximum and its sum against M.
    """
    hf, Wf = _as_f64(h), _as_f64(W)
    y = np.asarray(targets, dtype=np.int64)
    T = hf.shape[0]
    lo = shard_bounds(Vp, S)
    blocks = []
    for k in range(S):
        rows = Wf[lo[k]:lo[k + 1]]
        zk = hf @ rows.T                                     # [T, rows of shard k]
        cols = np.arange(lo[k], lo[k + 1])
        zk = np.where(cols[None, :] < V_real, zk, -np.inf)   # padded classes out
        blocks.append(zk)
    m_k = np.stack([b.max(axis=1) if b.shape[1] else np.full(T, -np.inf) for b in blocks], axis=1)
    M = m_k.max(axis=1)
    s_k = np.stack([np.exp(b - M[:, None]).sum(axis=1) for b in blocks], axis=1)
    L = s_k.sum(axis=1)
    valid, bad = target_status(y, V_real, ignore_index)
    _, owner, local = ownership(np.where(valid, y, -1), V_real, Vp, S)
    z_tgt = np.zeros(T)
    for t in range(T):
        if valid[t]:
            z_tgt[t] = blocks[owner[t]][t, local[t]]
    lse = M + np.log(L)
    token_loss = np.where(valid, lse - z_tgt, 0.0)
    nv = int(valid.sum())
    loss = g * token_loss.sum() / nv if nv > 0 else 0.0
    return dict(loss=loss, lse=lse, z_target=z_tgt, token_loss=token_loss,
                shard_max=m_k, shard_sum=s_k, global_max=M, n_valid=nv,
                valid=valid, bad=bad)


def logit_gradient(h, W, targets, V_real: int, Vp: int, scale: float,
                   ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """G[t, v] = (p_tv - 1[v = y_t]) * scale on valid tokens and real classes,
    0 elsewhere (P4)."""
    y = np.asarray(targets, dtype=np.int64)
    G = probabilities(h, W, V_real, Vp)
    valid, _ = target_status(y, V_real, ignore_index)
    G[~valid] = 0.0
    rows = np.nonzero(valid)[0]
    G[rows, y[rows]] -= 1.0
    return G * scale


def cross_entropy_backward(h, W, targets, V_real: int, Vp: int,
                           ignore_index: int = IGNORE_INDEX, g: float = 1.0):
    """dH = G W and dW_head = G^T h, with scale = g / N_valid (P4; "Sequence-
    parallel normalization", paragraph 3; R4, R5). Rows [V_real, Vp) of dW_head
    are zero: padded classes carry no probability and no gradient."""
    nv = n_valid(targets, V_real, ignore_index)
    scale = g / nv if nv > 0 else 0.0
    G = logit_gradient(h, W, targets, V_real, Vp, scale, ignore_index)
    hf, Wf = _as_f64(h), _as_f64(W)
    dH = G[:, :V_real] @ Wf[:V_real]
    dW = np.zeros((Vp, hf.shape[1]), dtype=np.float64)
    dW[:V_real] = G[:, :V_real].T @ hf
    return dH, dW


def hidden_gradient_rows(h_rows, W, targets_rows, V_real: int, scale: float,
                         ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """dH for a subset of tokens, given the scale g / N_valid of the whole batch
    (each row of dH depends only on its own token)."""
    y = np.asarray(targets_rows, dtype=np.int64)
    z = logits(h_rows, W, V_real)
    p = np.exp(z - log_sum_exp(z)[:, None])
    valid, _ = target_status(y, V_real, ignore_index)
    p[~valid] = 0.0
    rows = np.nonzero(valid)[0]
    p[rows, y[rows]] -= 1.0
    return (p * scale) @ _as_f64(W)[:V_real]


def head_gradient_rows(h, W, targets, V_real: int, lse: np.ndarray, scale: float, rows,
                       ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """dW_head[v] = sum_t G[t, v] h_t for the given real classes v, from the
    batch's lse (computed by this oracle) and scale = g / N_valid (P4)."""
    y = np.asarray(targets, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    hf = _as_f64(h)
    z = hf @ _as_f64(W)[rows].T
    p = np.exp(z - np.asarray(lse, dtype=np.float64)[:, None])
    valid, _ = target_status(y, V_real, ignore_index)
    p[~valid] = 0.0
    for j, v in enumerate(rows):
        p[valid & (y == v), j] -= 1.0
    return (p * scale).T @ hf


# ---------------------------------------------------------------------------
# Sampled softmax ("Sampled Softmax with Over-Tokenized Transformer", Setup:
# the loss_fn listing scores this GPU's targets plus random negatives, P
# tokens in all, and takes the cross-entropy at each target's position in
# that candidate list; no correction for the sampling is applied)
# ---------------------------------------------------------------------------

def sampled_candidates(targets, V_real: int, P: int, draws, ignore_index: int = IGNORE_INDEX):
    """The candidate list and each target's position in it.

    Reading: the distinct valid targets in ascending order, then negatives
    taken in draw order from `draws` (uniform draws from [0, V_real), the
    random numbers of the method) until P entries. Negatives are drawn
    without replacement, so a draw is skipped when it is a target, when it
    repeats an earlier negative, or when it lies outside [0, V_real); every
    class then appears at most once and a target's position is well defined.
    Ignored or bad targets keep ignore_index as position.
    """
    y = np.asarray(targets, dtype=np.int64)
    valid, _ = target_status(y, V_real, ignore_index)
    uniq = np.unique(y[valid])
    if uniq.size > P:
        raise ValueError("more distinct targets than candidates")
    taken = set(uniq.tolist())
    negs = []
    for d in np.asarray(draws, dtype=np.int64):
        if len(negs) == P - uniq.size:
            break
        d = int(d)
        if 0 <= d < V_real and d not in taken:
            negs.append(d)
            taken.add(d)
    if len(negs) < P - uniq.size:
        raise ValueError("not enough draws to fill the candidate list")
    cand = np.concatenate([uniq, np.array(negs, dtype=np.int64)])
    pos = np.full(y.shape, ignore_index, dtype=np.int64)
    pos[valid] = np.searchsorted(uniq, y[valid])
    return cand, pos, int(uniq.size)


def sampled_cross_entropy(h, W, targets, V_real: int, Vp: int, cand, pos, g: float = 1.0,
                          ignore_index: int = IGNORE_INDEX):
    """Cross-entropy over the P candidate classes only (logits h W[cand]^T),
    its gradient with respect to h, and the gradient of the full W, which is
    non-zero only on the candidate rows."""
    cand = np.asarray(cand, dtype=np.int64)
    P = cand.size
    Wc = _as_f64(W)[cand]
    fwd = cross_entropy_forward(h, Wc, pos, P, ignore_index, g=g)
    dH, dWc = cross_entropy_backward(h, Wc, pos, P, P, ignore_index, g=g)
    dW = np.zeros((Vp, Wc.shape[1]), dtype=np.float64)
    dW[cand] += dWc
    fwd.update(dH=dH, dW=dW, dW_cand=dWc)
    return fwd


def oth_loss(h, W, W2, tokens, V_real: int, Vp: int, weight: float = 0.1,
             ignore_index: int = IGNORE_INDEX):
    """OT-H: the next-token cross-entropy of the head W plus `weight` times the
    cross-entropy of a second head W2 that predicts the token two positions
    ahead ("Sampled Softmax with Over-Tokenized Transformer", Setup and its
    loss listing: the second head reads h[:-1] and is scored on tokens[2:]).

    tokens holds T+1 ids; h[t] is the hidden state at input position t (the
    input is tokens[:-1]), so head one is scored on tokens[1:]. Each term is
    averaged over its own valid tokens. Returns the total loss, both terms, dH
    (head two's gradient lands on rows [0, T-1)), dW and dW2.
    """
    tok = np.asarray(tokens, dtype=np.int64)
    T = np.asarray(h).shape[0]
    if tok.size != T + 1:
        raise ValueError("tokens must hold T+1 ids")
    y1, y2 = tok[1:], tok[2:]
    main = cross_entropy_forward(h, W, y1, V_real, ignore_index)
    dH, dW = cross_entropy_backward(h, W, y1, V_real, Vp, ignore_index)
    if T > 1:
        aux = cross_entropy_forward(h[:T - 1], W2, y2, V_real, ignore_index)["loss"]
        dH2, dW2 = cross_entropy_backward(h[:T - 1], W2, y2, V_real, Vp, ignore_index, g=weight)
        dH[:T - 1] += dH2
    else:
        aux, dW2 = 0.0, np.zeros((Vp, np.asarray(h).shape[1]))
    return dict(loss=main["loss"] + weight * aux, main=main["loss"], aux=aux, dH=dH, dW=dW, dW2=dW2)


def greedy_argmax(h, W, V_real: int):
    """Greedy decoding over the head: for each token the lowest class holding
    the largest real logit, and that logit ("Tensor Parallelism (TP)",
    on-device sampling; padded classes take no part, P3)."""
    z = logits(h, W, V_real)
    arg = z.argmax(axis=1).astype(np.int64)           # first occurrence: the lowest class
    return arg, z[np.arange(z.shape[0]), arg]


def greedy_argmax_sharded(h, W, V_real: int, Vp: int, S: int):
    """The sharded schedule: every shard reports the largest logit over its
    valid rows and the lowest row holding it; the shards' pairs are then
    merged (largest value, lowest class on a tie) without gathering logits."""
    hf, Wf = _as_f64(h), _as_f64(W)
    T = hf.shape[0]
    lo = shard_bounds(Vp, S)
    best = np.full(T, -np.inf)
    arg = np.full(T, -1, dtype=np.int64)
    for k in range(S):
        hi = min(lo[k + 1], V_real)
        if hi <= lo[k]:
            continue                                   # a shard of padding only
        zk = hf @ Wf[lo[k]:hi].T
        a_k = zk.argmax(axis=1)
        m_k = zk[np.arange(T), a_k]
        take = m_k > best                              # shards ascend: ties keep the lower one
        best[take] = m_k[take]
        arg[take] = lo[k] + a_k[take]
    return arg, best


def target_owner(targets, V_real: int, Vp: int, S: int,
                 ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Shard that owns each valid target, -1 for ignored or bad ones (P3)."""
    y = np.asarray(targets, dtype=np.int64)
    _, owner, _ = ownership(y, V_real, Vp, S)
    return owner


def max_owner(h, W, V_real: int, Vp: int, S: int):
    """Shard holding each token's largest real logit (lowest column on ties,
    R8) and the gap between the two largest logits of the row."""
    z = logits(h, W, V_real)
    arg = z.argmax(axis=1)
    top2 = np.sort(z, axis=1)[:, -2:] if z.shape[1] > 1 else np.concatenate([z, z], 1)
    _, owner, _ = ownership(arg, V_real, Vp, S)
    return owner, top2[:, 1] - top2[:, 0]


# ---------------------------------------------------------------------------

def _as_f64(x: np.ndarray) -> np.ndarray:
    """fp64 values of a tensor stored as fp32/fp64, or as bf16 bit patterns
    (uint16), widened exactly."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64, copy=False)
