"""The oracle against its pins, and planted mistakes that the pins must catch.

CPU only. The mutation tests plant a mistake in a fresh copy of the oracle's
source (never in the CUDA path) and check that at least one pin fails.
"""
import os
import types

import pytest

import oracle_pins as P
from oracle import vce_oracle

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "vce_oracle.py")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(vce_oracle)


def _mutant(old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("vce_oracle_mutant")
    exec(compile(src.replace(old, new), "vce_oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = {
    # the max term dropped from log-sum-exp
    "lse_drops_max": ("return M + np.log(np.exp(z - M[:, None]).sum(axis=1))",
                      "return np.log(np.exp(z - M[:, None]).sum(axis=1))"),
    # padded classes not excluded: the softmax runs over all Vp columns
    "padded_classes_kept": ("z = logits(h, W, V_real)\n    lse = log_sum_exp(z)\n    valid, bad",
                            "z = logits(h, W, W.shape[0])\n    lse = log_sum_exp(z)\n    valid, bad"),
    # wrong sign of the target indicator
    "onehot_sign": ("G[rows, y[rows]] -= 1.0", "G[rows, y[rows]] += 1.0"),
    # the target indicator forgotten
    "onehot_dropped": ("G[rows, y[rows]] -= 1.0", "pass"),
    # averaged over all tokens instead of the valid ones
    "mean_over_all": ("scale = g / nv if nv > 0 else 0.0",
                      "scale = g / len(targets) if nv > 0 else 0.0"),
    # transposed operand in dW_head
    "dw_uses_W": ("dW[:V_real] = G[:, :V_real].T @ hf",
                  "dW[:V_real] = G[:, :V_real].T @ Wf[:V_real][:, :hf.shape[1]][:hf.shape[0]]"),
    # shard bounds computed as k * (Vp // S): the last rows lose their owner
    "shard_floor_first": ("return np.array([(k * Vp) // S for k in range(S + 1)], dtype=np.int64)",
                          "return np.array([k * (Vp // S) for k in range(S + 1)], dtype=np.int64)"),
    # padded rows treated as valid ids
    "valid_up_to_Vp": ("valid = (ids >= 0) & (ids < V_real)\n    owner",
                       "valid = (ids >= 0) & (ids < Vp)\n    owner"),
    # embedding of an invalid id not zeroed
    "embed_no_mask": ("E[valid] = W[ids[valid]]", "E[:] = W[np.clip(ids, 0, W.shape[0] - 1)]"),
    # local softmax per shard: each shard normalised against its own maximum
    "local_max": ("s_k = np.stack([np.exp(b - M[:, None]).sum(axis=1) for b in blocks], axis=1)",
                  "s_k = np.stack([np.exp(b - np.max(b, axis=1, keepdims=True)).sum(axis=1) "
                  "for b in blocks], axis=1)"),
    # run sums taken in reverse token order
    "replay_reverse": ("for t in ts[c0:c0 + chunk]:", "for t in reversed(ts[c0:c0 + chunk]):"),
    # run partials summed right to left
    "replay_right_to_left": ("for c0 in range(0, len(ts), chunk):",
                             "for c0 in reversed(range(0, len(ts), chunk)):"),
    # repeated tokens overwrite instead of accumulating
    "embed_bwd_overwrite": ("dW[v] += dEf[t]", "dW[v] = dEf[t]"),
    # negatives taken in sorted order instead of draw order
    "sampled_sorted_negatives": ("    for d in np.asarray(draws, dtype=np.int64):",
                                 "    for d in np.sort(np.asarray(draws, dtype=np.int64)):"),
    # a repeated draw taken twice as a negative
    "sampled_repeats_kept": ("            negs.append(d)\n            taken.add(d)",
                             "            negs.append(d)"),
    # OT-H's second head scored on the next token instead of two ahead
    "oth_shift_one": ("    y1, y2 = tok[1:], tok[2:]", "    y1, y2 = tok[1:], tok[1:-1]"),
    # OT-H's weight left off the second head's gradient
    "oth_unweighted_grad": ("V_real, Vp, ignore_index, g=weight)", "V_real, Vp, ignore_index)"),
    # greedy argmax: ties to the highest class
    "argmax_ties_high": ("    arg = z.argmax(axis=1).astype(np.int64)",
                         "    arg = (z.shape[1] - 1 - z[:, ::-1].argmax(axis=1)).astype(np.int64)"),
    # greedy argmax over the padded classes too
    "argmax_padded": ("    z = logits(h, W, V_real)\n    arg = z.argmax(axis=1).astype(np.int64)",
                      "    z = logits(h, W, W.shape[0])\n    arg = z.argmax(axis=1).astype(np.int64)"),
    # sharded argmax: a later shard wins ties
    "argmax_shard_tie_late": ("        take = m_k > best", "        take = m_k >= best"),
    # n-gram read with the newest token as the highest digit
    "ngram_digit_order": ("        value = sum(v * V ** j for j, v in enumerate(reversed(gram)))",
                          "        value = sum(v * V ** j for j, v in enumerate(gram))"),
    # n-grams running across the start of a sequence
    "ngram_crosses_sequences": ("        pos = t % seq_len if seq_len > 0 else t\n        if pos < n - 1:",
                                "        pos = t\n        if pos < n - 1:"),
    # an n-gram with an invalid id still looked up
    "ngram_keeps_invalid": ("        if any(v < 0 or v >= V for v in gram):\n            continue",
                            "        if False:\n            continue"),
    # bf16 rounding by truncation
    "ngram_truncates": ("    return ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16))",
                        "    return ((u) >> np.uint64(16))"),
    # target positions off by one in the candidate list
    "sampled_pos_shift": ("    pos[valid] = np.searchsorted(uniq, y[valid])",
                          "    pos[valid] = np.searchsorted(uniq, y[valid], side='right')"),
    # max_owner: the gap taken the wrong way round
    "max_owner_gap_sign": ("    return owner, top2[:, 1] - top2[:, 0]", "    return owner, top2[:, 0] - top2[:, 1]"),
    # max_owner: the gap to the third largest logit instead of the second
    "max_owner_gap_third": ("np.sort(z, axis=1)[:, -2:]", "np.sort(z, axis=1)[:, -3:-1]"),
    # max_owner: ties go to the highest column
    "max_owner_ties_high": ("    arg = z.argmax(axis=1)\n    top2",
                            "    arg = z.shape[1] - 1 - z[:, ::-1].argmax(axis=1)\n    top2"),
    # max_owner over the padded classes too
    "max_owner_padded": ("    z = logits(h, W, V_real)\n    arg = z.argmax(axis=1)\n",
                         "    z = logits(h, W, W.shape[0])\n    arg = z.argmax(axis=1)\n"),
    # an ignore value inside the real classes accepted
    "ignore_index_unchecked": ("    if 0 <= ignore_index < V_real:\n        raise", "    if False:\n        raise"),
    # target logit taken from the wrong shard offset
    "target_local_off": ("z_tgt[t] = blocks[owner[t]][t, local[t]]",
                         "z_tgt[t] = blocks[owner[t]][t, max(local[t] - 1, 0)]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    mod = _mutant(old, new)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # AssertionError, or a shape error the mistake causes
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"
