"""Seeded synthetic inputs for the vocabulary-sharded embedding and cross-entropy.

This module only draws numbers. It holds none of the method's arithmetic (no
ownership test, no softmax, no gradient): the oracle and the CUDA path both
receive the arrays made here and nothing else is shared between them.

Every tensor is drawn from its own numpy PCG64 stream, keyed by
``(seed, tensor tag)``, so drawing one tensor never shifts another one.
bf16 tensors are drawn in fp32 and rounded to bf16 with round-to-nearest-even
on the host; they are returned as raw ``uint16`` bit patterns together with
helpers to widen them exactly.

Workloads are stand-ins for the shapes on the pages: a GPT-2-sized LM head, the
Qwen3 vocabulary (151936 classes) and the GPT-OSS-20B embedding table
``[201088, 3072]`` ("Tensor Parallelism (TP)", Problem Statement). No public
dataset is read.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional, Tuple

import numpy as np

IGNORE_INDEX = -100

# Stream tags: one independent PCG64 stream per tensor.
_TAG = {"W": 1, "h": 2, "targets": 3, "ids": 4, "dE": 5, "tokens": 6,
        "corrupt": 7, "forced": 8, "cand": 9, "T2": 10, "T3": 11}


@dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic case."""
    name: str
    T: int
    H: int
    V_real: int
    Vp: int
    S: int
    dtype: str            # "f32" or "bf16"
    tied: bool
    seed: int
    w_std: float = 0.02   # W ~ N(0, w_std^2)
    pad_fill: Optional[float] = 8.0   # value written into rows [V_real, Vp)
    ignore_frac: float = 0.0          # fraction of targets set to IGNORE_INDEX
    token_dist: str = "uniform"       # "uniform" targets, or "zipf" next-token
    zipf_s: float = 1.1
    h_kind: str = "normal"            # "normal" or "rmsnorm"
    pad_id_frac: float = 0.0          # embedding ids replaced by IGNORE_INDEX
    oor_id_frac: float = 0.0          # embedding ids replaced by out-of-range
    # Targets forced onto given classes (first tokens), and (target, column)
    # pairs whose token gets an injected maximum logit at that column.
    forced_targets: Tuple[int, ...] = ()
    injected: Tuple[Tuple[int, int], ...] = ()


# The five cases. Sizes are the ones the method is exercised on; seeds are fixed.
WORKLOADS: Dict[str, Workload] = {
    # Tiny fp32 case: boundary targets, injected maxima, garbage padded rows.
    "tiny_f32": Workload("tiny_f32", T=64, H=64, V_real=1000, Vp=1024, S=4,
                         dtype="f32", tied=False, seed=0, ignore_frac=0.10,
                         pad_id_frac=0.05, oor_id_frac=0.05,
                         # shard edges of 4 x 256 rows, and the last real class
                         forced_targets=(255, 256, 511, 512, 999),
                         # target shard != shard holding the injected maximum
                         injected=((10, 519), (261, 779), (515, 17), (999, 0))),
    # GPT-2-like LM head, untied, loss only.
    "gpt2_head": Workload("gpt2_head", T=4096, H=1024, V_real=50000, Vp=50048,
                          S=8, dtype="bf16", tied=False, seed=1,
                          ignore_frac=0.05),
    # Qwen3-like tied step: Zipf tokens, next-token targets, RMS-normalised h.
    "qwen3_tied": Workload("qwen3_tied", T=8192, H=2048, V_real=151936,
                           Vp=151936, S=8, dtype="bf16", tied=True, seed=2,
                           pad_fill=None, token_dist="zipf", h_kind="rmsnorm"),
    # GPT-OSS-shaped embedding table; the same tokens feed the loss.
    "gptoss_embed": Workload("gptoss_embed", T=16384, H=3072, V_real=201088,
                             Vp=201088, S=8, dtype="bf16", tied=False, seed=3,
                             pad_fill=None, token_dist="zipf", h_kind="rmsnorm",
                             pad_id_frac=0.02, oor_id_frac=0.01),
    # Sampled softmax over P = 8192 candidates of the Qwen3 vocabulary.
    "sampled": Workload("sampled", T=16384, H=2048, V_real=151936, Vp=151936, S=8,
                        dtype="bf16", tied=False, seed=4, pad_fill=None,
                        token_dist="zipf", h_kind="rmsnorm"),
}

SAMPLED_P = 8192   # candidates of the sampled-softmax workload


# Hashed n-gram tables of the n-gram embedding case: 2^18 rows each (the
# pages' OT-H tables hold billions of parameters; their ten-times-smaller
# variant is of this order per table at H=2048), over sequences of 2048 tokens
# (the Qwen3-like batch is 4 x 2048).
NGRAM_ROWS = 1 << 18
NGRAM_SEQ_LEN = 2048


def make_ngram_table(wl: Workload, n: int, rows: int, chunk_rows: int = 1 << 15) -> np.ndarray:
    """Table of the hashed n-grams (n = 2 or 3): [rows, H] ~ N(0, w_std^2), in the workload's dtype."""
    rng = _rng(wl, "T2" if n == 2 else "T3")
    out = np.empty((rows, wl.H), dtype=np.uint16 if wl.dtype == "bf16" else np.float32)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, wl.H), dtype=np.float32) * np.float32(wl.w_std)
        out[r0:r1] = _store(x, wl.dtype)
    return out


def make_negative_draws(wl: Workload, n: int) -> np.ndarray:
    """Uniform draws without replacement from [0, V_real), in draw order: the
    random numbers the sampled softmax consumes for its negatives."""
    rng = _rng(wl, "cand")
    return rng.permutation(wl.V_real)[:n].astype(np.int64)


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit fields (tests use this for ragged shapes)."""
    base = dict(T=64, H=64, V_real=1000, Vp=1024, S=4, dtype="bf16",
                tied=False, seed=123)
    base.update(kw)
    return Workload(name, **base)


def with_T(wl: Workload, T: int) -> Workload:
    return replace(wl, T=T)


# ----------------------------------------------------------------------------
# bf16 bit helpers (input preparation, not the method)
# ----------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32/fp64 values to bf16 (round to nearest, ties to even).

    Returns the uint16 bit patterns. Inputs are finite by construction.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 view of an input tensor as stored (bf16 bits or fp32)."""
    if dtype == "bf16":
        return bf16_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def _rng(wl: Workload, tag: str) -> np.random.Generator:
    return np.random.default_rng([wl.seed, _TAG[tag]])


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(x32) if dtype == "bf16" else np.ascontiguousarray(x32, np.float32)


def zipf_draw(rng: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Truncated Zipf(s) over ranks 1..V by inverse CDF; token id = rank - 1."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    r = np.searchsorted(cdf, u, side="right")
    return np.minimum(r, V - 1).astype(np.int64)


# ----------------------------------------------------------------------------
# Tensors
# ----------------------------------------------------------------------------

def make_W(wl: Workload, chunk_rows: int = 1 << 15) -> np.ndarray:
    """W[Vp, H]: N(0, w_std^2) rows; rows [V_real, Vp) hold pad_fill if set."""
    rng = _rng(wl, "W")
    out = np.empty((wl.Vp, wl.H), dtype=np.uint16 if wl.dtype == "bf16" else np.float32)
    for r0 in range(0, wl.Vp, chunk_rows):
        r1 = min(wl.Vp, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, wl.H), dtype=np.float32) * np.float32(wl.w_std)
        out[r0:r1] = _store(x, wl.dtype)
    if wl.pad_fill is not None and wl.Vp > wl.V_real:
        out[wl.V_real:] = _store(np.full((wl.Vp - wl.V_real, wl.H), wl.pad_fill, np.float32), wl.dtype)
    return out


def _tokens(wl: Workload) -> np.ndarray:
    """T+1 clean tokens (Zipf next-token workloads)."""
    return zipf_draw(_rng(wl, "tokens"), wl.T + 1, wl.V_real, wl.zipf_s)


def _corrupted_tokens(wl: Workload) -> np.ndarray:
    """T+1 tokens with a fraction replaced by the padding id and by out-of-range ids.

    Out-of-range ids are half drawn from [V_real, 2*V_real) and half from
    [-2^31, -101].
    """
    tok = _tokens(wl).copy()
    n = tok.shape[0]
    rng = _rng(wl, "corrupt")
    n_pad = int(round(wl.pad_id_frac * n))
    n_oor = int(round(wl.oor_id_frac * n))
    pos = rng.permutation(n)
    pad_pos = pos[:n_pad]
    oor_pos = pos[n_pad:n_pad + n_oor]
    tok[pad_pos] = IGNORE_INDEX
    half = n_oor // 2
    tok[oor_pos[:half]] = rng.integers(wl.V_real, 2 * wl.V_real, size=half)
    tok[oor_pos[half:]] = rng.integers(-(2 ** 31), -101 + 1, size=n_oor - half)
    return tok


def make_ids(wl: Workload) -> np.ndarray:
    """Embedding input ids [T] int64."""
    if wl.token_dist == "zipf":
        return np.ascontiguousarray(_corrupted_tokens(wl)[:-1])
    rng = _rng(wl, "ids")
    T = wl.T
    ids = rng.integers(0, wl.V_real, size=T)
    # Some ids fall on padded rows, some are the padding id, some out of range;
    # a run of repeats exercises accumulation into one row.
    pos = rng.permutation(T)
    n_pad = int(round(wl.pad_id_frac * T))
    n_oor = int(round(wl.oor_id_frac * T))
    n_padrow = n_oor if wl.Vp > wl.V_real else 0
    ids[pos[:n_pad]] = IGNORE_INDEX
    oor = pos[n_pad:n_pad + n_oor]
    ids[oor[: len(oor) // 2]] = rng.integers(wl.Vp, wl.Vp + 1000, size=len(oor) // 2)
    ids[oor[len(oor) // 2:]] = rng.integers(-1000, -1, size=len(oor) - len(oor) // 2)
    padrow_pos = pos[n_pad + n_oor:n_pad + n_oor + n_padrow]
    if len(padrow_pos):
        ids[padrow_pos] = rng.integers(wl.V_real, wl.Vp, size=len(padrow_pos))
    if T >= 16:
        rep = pos[-min(8, T // 8):]
        ids[rep] = 7
    return ids.astype(np.int64)


def make_targets(wl: Workload) -> np.ndarray:
    """Loss targets [T] int64; IGNORE_INDEX marks ignored tokens."""
    if wl.token_dist == "zipf":
        tok = _corrupted_tokens(wl)[1:].copy()
        bad = (tok < 0) | (tok >= wl.V_real)
        tok[bad] = IGNORE_INDEX
        return np.ascontiguousarray(tok)
    rng = _rng(wl, "targets")
    y = rng.integers(0, wl.V_real, size=wl.T).astype(np.int64)
    n_ign = int(round(wl.ignore_frac * wl.T))
    if n_ign:
        y[rng.permutation(wl.T)[:n_ign]] = IGNORE_INDEX
    for i, v in enumerate(wl.forced_targets):
        y[i] = v
    for i, (yt, _vstar) in enumerate(wl.injected):
        y[len(wl.forced_targets) + i] = yt
    return y


def make_h(wl: Workload, W: Optional[np.ndarray] = None) -> np.ndarray:
    """Hidden states h[T, H].

    "normal": N(0,1). "rmsnorm": N(0,1) rows scaled by 1/sqrt(mean(x^2)+1e-6)
    (unit gain). The tiny case overwrites a few rows with h_t = 50 W[v*]/|W[v*]|
    so that the largest logit of that token lands in a shard that does not own
    its target.
    """
    rng = _rng(wl, "h")
    x = rng.standard_normal((wl.T, wl.H), dtype=np.float32)
    if wl.h_kind == "rmsnorm":
        ms = np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True)
        x = (x / np.sqrt(ms + 1e-6)).astype(np.float32)
    if wl.injected:
        if W is None:
            W = make_W(wl)
        Wf = to_f64(W, wl.dtype)
        base = len(wl.forced_targets)
        for i, (_yt, vstar) in enumerate(wl.injected):
            r = Wf[vstar]
            x[base + i] = (50.0 * r / np.linalg.norm(r)).astype(np.float32)
    return _store(x, wl.dtype)


def make_dE(wl: Workload) -> np.ndarray:
    """Upstream gradient of the embedding output, dE[T, H] ~ N(0,1)."""
    rng = _rng(wl, "dE")
    x = rng.standard_normal((wl.T, wl.H), dtype=np.float32)
    return _store(x, wl.dtype)


def make_all(wl: Workload, parts=("W", "h", "targets", "ids", "dE")) -> Dict[str, np.ndarray]:
    out: Dict[str, np.ndarray] = {}
    if "W" in parts or ("h" in parts and wl.injected):
        out["W"] = make_W(wl)
    if "h" in parts:
        out["h"] = make_h(wl, out.get("W"))
    if "targets" in parts:
        out["targets"] = make_targets(wl)
    if "ids" in parts:
        out["ids"] = make_ids(wl)
    if "dE" in parts:
        out["dE"] = make_dE(wl)
    return out
