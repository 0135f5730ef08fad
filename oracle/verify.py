"""Scaffold-speculative verification, float64 oracle (test infrastructure only).

Sources (page title, section):

* Fast-dDrive method summary (e.mffb.com.cn), §3.2 "模式二：Scaffold Speculative
  Decoding": scaffold positions of the block are accepted as they are; the MDM
  head drafts every editable position in one forward; one AR forward gives
  p_AR(. | x_<i) at every position and the draft is compared left to right with
  its argmax; a match is accepted and the comparison goes on; at the first
  mismatch the AR prediction is taken, the later drafts are dropped, and one
  bonus token is accepted, so that a round never goes backwards.
* Fast-dDrive (arXiv 2605.23163 translation), abstract and §1: the
  speculative output is identical to pure AR decoding; for test-time scaling
  only the trajectory section is sampled, by sampling the AR verifier.

Readings where the pages are silent or ambiguous:

* AR row e is the AR prediction for the e-th editable slot of the block
  (scaffold slots have no row); row E (one past the last editable slot) is
  the prediction for the position after the block;
* the AR token that replaces the first mismatching draft is itself the bonus
  token; when every draft matches, the bonus is row E's token, which belongs
  to the position after the block;
* editable slots already committed in an earlier round are skipped like
  scaffold; masked slots after the mismatch return to masked (token -1);
* sampled verification draws t = argmax_v (l_v / T + g_v), g = -log(-log u), with
  u supplied per (sequence, row, v) — Gumbel-max, an exact sample of softmax(l/T).
"""
from __future__ import annotations

import math

import numpy as np

MASKED, COMMITTED, SCAFFOLD = 0, 1, 2


def gumbel_scores(row, u, temperature: float) -> np.ndarray:
    """l / T + g with g = -log(-log u), float64."""
    return (np.asarray(row, np.float64) / float(temperature)
            - np.log(-np.log(np.asarray(u, np.float64))))


def _top2_gap(x: np.ndarray) -> float:
    i = int(np.argmax(x))
    best = x[i]
    rest = np.delete(x, i)
    return float(best - rest.max()) if rest.size else math.inf


def spec_verify(tokens, state, ar_logits, noise=None, temperature: float = 1.0) -> dict:
    """Verify one drafted block for each of n_seq sequences.

    tokens/state: [n_seq, L] (masked slots hold the MDM draft); ar_logits:
    [n_seq, E + 1, V]; noise (optional): uniforms of the same shape.
    Returns new tokens/state, accepted_len [n_seq] (slots committed this round,
    bonus included), bonus [n_seq], bonus_pos [n_seq] (slot, or L when after the
    block), and ``margins``: the smallest top-two gap of the sampled scores over
    the rows whose argmax decided the result (inf for greedy rows).
    """
    tokens = np.array(tokens, dtype=np.int64)
    state = np.array(state, dtype=np.int64)
    n_seq, L = tokens.shape
    accepted = np.zeros(n_seq, np.int64)
    bonus = np.zeros(n_seq, np.int64)
    bonus_pos = np.zeros(n_seq, np.int64)
    gap = math.inf
    for r in range(n_seq):
        edit = [p for p in range(L) if state[r, p] != SCAFFOLD]
        E = len(edit)
        assert ar_logits.shape[1] == E + 1

        def ar_token(e: int) -> int:
            nonlocal gap
            if noise is None:
                return int(np.argmax(np.asarray(ar_logits[r, e], np.float64)))
            s = gumbel_scores(ar_logits[r, e], noise[r, e], temperature)
            gap = min(gap, _top2_gap(s))
            return int(np.argmax(s))

        n_acc = 0
        k = E
        for e, p in enumerate(edit):
            if state[r, p] != MASKED:
                continue
            t = ar_token(e)
            if t == tokens[r, p]:
                state[r, p] = COMMITTED
                n_acc += 1
                continue
            k = e
            tokens[r, p] = t
            state[r, p] = COMMITTED
            bonus[r], bonus_pos[r] = t, p
            break
        if k == E:
            bonus[r], bonus_pos[r] = ar_token(E), L
        else:
            for p in edit[k + 1:]:
                if state[r, p] == MASKED:
                    tokens[r, p] = -1
        accepted[r] = n_acc + 1
    return dict(tokens=tokens, state=state, accepted_len=accepted, bonus=bonus,
                bonus_pos=bonus_pos, margins=dict(gumbel=gap))
