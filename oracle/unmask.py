"""Unmask / commit step of masked-diffusion decoding, float64 oracle (test infrastructure only).

Sources (page title, section):

* Fast-dDrive method summary (e.mffb.com.cn), §3.1: the reverse process predicts
  the original token of each masked position.
* Fast-dVLA: Accelerating Discrete Diffusion VLA to Real-Time Performance,
  "关键设计 2. 扩散强制": tokens already unmasked stay fixed.
* same page, "关键设计 4. 流水线并行解码": a block's completion ratio is its
  unmasked count over its size; when the predecessor passes the add threshold
  the block is half-active and commits only predictions above the confidence
  threshold; past the activation threshold it is fully active and, besides the
  confidence filter, commits at least a fraction 1/n of its remaining tokens by
  confidence rank.
* Fast-dDrive method summary, §3.2 "模式二", step 1: scaffold positions are
  auto-accepted and never denoised.

Readings where the pages are silent or loose:

* prediction = argmax over the vocabulary, lowest index on ties; confidence =
  the largest softmax probability = 1 / sum_v exp(l_v - max);
* a candidate is a masked position with a logits row; ``rem`` = candidates of the
  block at step start; completion ratio = non-masked positions (scaffold
  included) / block size, at step start;
* thresholds compare with >= ("passes"): tau on the confidence; the add /
  activation thresholds as exact rationals (done * den >= num * size);
* block 0 of the window follows a complete predecessor (it lies in the cache),
  so it is fully active while it has masked positions; a block with no masked
  position is done;
* fully active: commit {conf >= tau_full} united with the n_min most confident
  candidates, n_min = min(rem, max(k_fixed, ceil(rem * min_frac))), confidence
  ties ranked to the lower position; half active: {conf >= tau_half}.
"""
from __future__ import annotations

from fractions import Fraction
import math

import numpy as np

MASKED, COMMITTED, SCAFFOLD = 0, 1, 2
INACTIVE, HALF, FULL, DONE = 0, 1, 2, 3


def row_stats(row) -> tuple[int, float, float]:
    """(pred, conf, lse) of one logits row in float64."""
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    pred = int(np.flatnonzero(x == m)[0])
    s = np.exp(x - m).sum()
    return pred, float(1.0 / s), float(m + math.log(s))


def block_status(state, block_start, add_thr: Fraction, act_thr: Fraction) -> list[int]:
    """Per-block activation status from the state at step start."""
    bs = [int(x) for x in block_start]
    state = np.asarray(state)
    out = []
    for b in range(len(bs) - 1):
        blk = state[bs[b]:bs[b + 1]]
        if not (blk == MASKED).any():
            out.append(DONE)
            continue
        if b == 0:
            out.append(FULL)
            continue
        prev = state[bs[b - 1]:bs[b]]
        ratio = Fraction(int((prev != MASKED).sum()), len(prev))
        out.append(FULL if ratio >= act_thr else HALF if ratio >= add_thr else INACTIVE)
    return out


def unmask_step(logits, logit_row, block_start, state, tokens, *, tau_full: float,
                tau_half: float, min_frac: Fraction, k_fixed: int, add_thr: Fraction,
                act_thr: Fraction, write_draft: bool = False) -> dict:
    """One unmask/commit step over the active window.

    logits: [R, V]; logit_row[p]: row of position p or -1; state/tokens: [n_pos].
    Returns the new state/tokens and commit [n_pos], n_committed / status
    [n_blocks], pred / conf / lse [n_pos] (-1 / 0 / 0 for non-candidates), and
    ``margins``: the smallest distances of this step's decisions from their
    thresholds (|conf - tau| over the candidates of half/full blocks, and the
    relative confidence gap at each full block's top-n_min cut).

    With ``write_draft`` every candidate left masked also receives its argmax as
    token: the MDM draft of a scaffold-speculative round (Fast-dDrive method
    summary §3.2 "模式二", step 2: one MDM forward drafts all editable positions).
    """
    state = np.array(state, dtype=np.int64)
    tokens = np.array(tokens, dtype=np.int64)
    logit_row = np.asarray(logit_row, dtype=np.int64)
    bs = [int(x) for x in block_start]
    n_pos = len(state)
    pred = np.full(n_pos, -1, dtype=np.int64)
    conf = np.zeros(n_pos)
    lse = np.zeros(n_pos)
    cand = (state == MASKED) & (logit_row >= 0)
    for p in np.flatnonzero(cand):
        pred[p], conf[p], lse[p] = row_stats(logits[logit_row[p]])
    status = block_status(state, bs, add_thr, act_thr)
    commit = np.zeros(n_pos, dtype=np.int64)
    n_committed = []
    tau_margin = math.inf
    rank_margin = math.inf
    for b in range(len(bs) - 1):
        ps = [p for p in range(bs[b], bs[b + 1]) if cand[p]]
        chosen = set()
        if status[b] == HALF:
            chosen = {p for p in ps if conf[p] >= tau_half}
            tau_margin = min([tau_margin] + [abs(conf[p] - tau_half) for p in ps])
        elif status[b] == FULL and ps:
            rem = len(ps)
            n_min = min(rem, max(int(k_fixed), math.ceil(rem * min_frac)))
            ranked = sorted(ps, key=lambda p: (-conf[p], p))
            chosen = {p for p in ps if conf[p] >= tau_full} | set(ranked[:n_min])
            tau_margin = min([tau_margin] + [abs(conf[p] - tau_full) for p in ps])
            if 0 < n_min < rem:
                a, c = conf[ranked[n_min - 1]], conf[ranked[n_min]]
                rank_margin = min(rank_margin, (a - c) / a)
        for p in chosen:
            commit[p] = 1
            tokens[p] = pred[p]
            state[p] = COMMITTED
        n_committed.append(len(chosen))
        if write_draft:
            for p in ps:
                if p not in chosen:
                    tokens[p] = pred[p]
    return dict(state=state, tokens=tokens, commit=commit, n_committed=np.array(n_committed),
                status=np.array(status), pred=pred, conf=conf, lse=lse,
                margins=dict(tau=tau_margin, rank=rank_margin))
