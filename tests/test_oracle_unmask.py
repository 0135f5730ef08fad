"""Pins of the unmask/commit oracle (closed forms, special cases, invariants, the
pages' section table)."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from oracle.unmask import DONE, FULL, HALF, INACTIVE

HERE = os.path.dirname(os.path.abspath(__file__))
M, C_, S = 0, 1, 2


def test_uniform_row_confidence_is_one_over_v():
    for V in (1024, 151936):
        row = np.full(V, 0.25, dtype=np.float32)
        pred, conf, lse = oracle.row_stats(row)
        assert pred == 0 and conf == 1.0 / V and abs(lse - (0.25 + math.log(V))) < 1e-12


def test_single_peak_closed_form():
    """Row (a, 0, ..., 0): conf = e^a / (e^a + V - 1), lse = ln(e^a + V - 1)."""
    V, a = 1000, 3.5
    row = np.zeros(V)
    row[17] = a
    pred, conf, lse = oracle.row_stats(row)
    assert pred == 17
    assert abs(conf - math.exp(a) / (math.exp(a) + V - 1)) < 1e-15
    assert abs(lse - math.log(math.exp(a) + V - 1)) < 1e-12


def test_planted_row_confidence_matches_construction():
    """The generator solves the planted logit from the other entries; the
    oracle's confidence reproduces the probability it reports (to 1e-12)."""
    x, tok, achieved = synth.planted_logits(11, 0, 8, V=5000, bf16=False)
    for r in range(8):
        pred, conf, _ = oracle.row_stats(x[r])
        assert pred == tok[r]
        assert abs(conf - achieved[r]) < 1e-12


def test_argmax_ties_go_to_lowest_index():
    row = np.zeros(64)
    row[[40, 9, 33]] = 2.0
    assert oracle.row_stats(row)[0] == 9


def _step(logits, state, bs, **kw):
    n = len(state)
    params = dict(tau_full=0.9, tau_half=0.9, min_frac=Fraction(1, 4), k_fixed=1,
                  add_thr=Fraction(1, 2), act_thr=Fraction(17, 20))
    params.update(kw)
    return oracle.unmask_step(logits, np.arange(n), bs, state, np.full(n, -1), **params)


def test_status_from_predecessor_ratio_seven_token_blocks():
    """7-token blocks, add 0.5 / act 0.85: predecessor with 3/7 done -> inactive,
    4/7 and 5/7 -> half, 6/7 -> full; block 0 full; a block with nothing masked is done."""
    bs = [0, 7, 14, 21, 28, 35]
    state = np.zeros(35, int)
    state[0:7] = C_            # block 0 complete -> done, block 1 full (7/7)
    state[7:10] = C_           # block 1: 3/7 -> block 2 inactive
    state[14:18] = C_          # block 2: 4/7 -> block 3 half
    state[21:27] = C_          # block 3: 6/7 -> block 4 full
    st = oracle.unmask.block_status(state, bs, Fraction(1, 2), Fraction(17, 20))
    assert st == [DONE, FULL, INACTIVE, HALF, FULL]
    state[14:19] = C_          # block 2: 5/7 -> half
    assert oracle.unmask.block_status(state, bs, Fraction(1, 2), Fraction(17, 20))[3] == HALF


@pytest.mark.parametrize("rem,frac,k,want", [(5, Fraction(1, 4), 1, 2), (4, Fraction(1, 4), 1, 1),
                                             (1, Fraction(1, 4), 1, 1), (1, Fraction(1, 4), 2, 1),
                                             (9, Fraction(1, 4), 4, 4), (32, Fraction(1, 1), 0, 32)])
def test_min_commit_count(rem, frac, k, want):
    """n_min = min(rem, max(k_fixed, ceil(rem * f))), on a full block with tau unreachable."""
    logits = synth.normal_logits(12, rem, rem, V=256, sigma=2.0, bf16=False)
    r = _step(logits, np.zeros(rem, int), [0, rem], tau_full=2.0, min_frac=frac, k_fixed=k)
    assert r["n_committed"][0] == want


def test_full_block_commits_threshold_set_union_top_by_confidence():
    """Full block: {conf >= tau} united with the n_min most confident; ties in
    confidence go to the lower position; scaffold stays untouched."""
    V = 64
    logits = np.zeros((6, V))
    # confidences from a single peak: conf = e^a / (e^a + V - 1)
    peaks = [7.0, 1.0, 6.0, 1.0, 0.5, 6.0]   # positions 2 and 5 tie
    for p, a in enumerate(peaks):
        logits[p, p + 3] = a
    conf = [math.exp(a) / (math.exp(a) + V - 1) for a in peaks]
    state = np.array([M, M, M, M, S, M])
    tau = (conf[0] + conf[2]) / 2                 # only position 0 passes tau
    r = _step(logits, state, [0, 6], tau_full=tau, min_frac=Fraction(2, 5), k_fixed=1)
    # rem = 5 candidates -> n_min = ceil(2) = 2: top two are p0 then p2 (ties p2/p5 -> p2)
    assert list(r["commit"]) == [1, 0, 1, 0, 0, 0]
    assert r["tokens"][0] == 3 and r["tokens"][2] == 5 and r["state"][4] == S
    assert r["tokens"][4] == -1


def test_half_block_commits_only_threshold_set():
    V = 64
    logits = np.zeros((4, V))
    logits[0, 1], logits[1, 2], logits[2, 3] = 8.0, 9.0, 1.0
    state = np.array([C_, C_, C_, C_, M, M, M])  # block 0: 4 of 4 done? no: sizes below
    bs = [0, 4, 7]
    state = np.array([C_, C_, M, M, M, M, M])      # block 0: 2/4 done -> block 1 half
    lr = np.array([-1, -1, -1, -1, 0, 1, 2])
    conf = [math.exp(a) / (math.exp(a) + V - 1) for a in (8.0, 9.0, 1.0)]
    tau = (conf[0] + conf[1]) / 2                 # only the 9.0 row passes
    r = oracle.unmask_step(logits, lr, bs, state, np.full(7, -1), tau_full=2.0, tau_half=tau,
                           min_frac=Fraction(1, 4), k_fixed=1, add_thr=Fraction(1, 2),
                           act_thr=Fraction(17, 20))
    assert list(r["status"]) == [FULL, HALF]
    assert list(r["commit"]) == [0, 0, 0, 0, 0, 1, 0]


def test_invariants_random_windows():
    """Scaffold never changes; commits are a subset of the masked candidates and
    take their argmax; committed tokens never change; full blocks commit at least
    min(rem, n_min); inactive and done blocks commit nothing."""
    g = synth.rng(13)
    for trial in range(20):
        sizes = g.integers(1, 9, size=int(g.integers(1, 4)))
        bs = [0] + list(np.cumsum(sizes))
        n = bs[-1]
        state = g.choice([M, C_, S], size=n, p=[0.6, 0.2, 0.2])
        tokens = np.where(state == M, -1, g.integers(0, 100, size=n))
        logits = synth.normal_logits(14, trial, n, V=300, sigma=2.0, bf16=False)
        r = oracle.unmask_step(logits, np.arange(n), bs, state, tokens, tau_full=0.02, tau_half=0.02,
                               min_frac=Fraction(1, 4), k_fixed=1, add_thr=Fraction(1, 2),
                               act_thr=Fraction(17, 20))
        assert np.all(r["state"][state == S] == S) and np.all(r["tokens"][state != M] == tokens[state != M])
        com = r["commit"].astype(bool)
        assert np.all(state[com] == M)
        for p in np.flatnonzero(com):
            assert r["tokens"][p] == int(np.argmax(logits[p]))
        for b in range(len(bs) - 1):
            blk = slice(bs[b], bs[b + 1])
            rem = int((state[blk] == M).sum())
            if r["status"][b] == FULL:
                assert r["n_committed"][b] >= min(rem, max(1, math.ceil(rem / 4)))
            if r["status"][b] in (INACTIVE, DONE):
                assert r["n_committed"][b] == 0


def test_unreachable_tau_and_full_fraction_commits_greedy_draft():
    """tau > 1 with f = 1 commits every masked position with its argmax: the greedy draft."""
    n = 20
    logits = synth.normal_logits(15, 0, n, V=500, sigma=3.0, bf16=False)
    state = np.zeros(n, int)
    state[[3, 7]] = S
    r = _step(logits, state, [0, n], tau_full=1.5, min_frac=Fraction(1, 1))
    ed = state != S
    assert np.all(r["commit"][ed] == 1) and np.all(r["commit"][~ed] == 0)
    assert np.array_equal(r["tokens"][ed], np.argmax(logits, axis=1)[ed])


def test_block_size_one_commits_left_to_right():
    """B = 1 with k = 1 and tau unreachable: each step commits exactly the
    leftmost masked position (later blocks are inactive until their
    predecessor is done) - autoregressive order."""
    n = 6
    logits = synth.normal_logits(16, 0, n, V=200, sigma=3.0, bf16=False)
    state = np.zeros(n, int)
    tokens = np.full(n, -1)
    bs = list(range(n + 1))
    for step in range(n):
        r = oracle.unmask_step(logits, np.arange(n), bs, state, tokens, tau_full=2.0, tau_half=2.0,
                               min_frac=Fraction(0, 1), k_fixed=1, add_thr=Fraction(1, 2),
                               act_thr=Fraction(17, 20))
        assert list(np.flatnonzero(r["commit"])) == [step]
        state, tokens = r["state"], r["tokens"]


def test_section_table_block_counts_and_scaffold_share():
    """n_s = ceil(|E_s| / d) reproduces the page's block counts 1 / 6 / 1 / 3 at
    d = 32, and the generated layout has those blocks, those editable counts per
    section and about 30% scaffold."""
    gold = json.load(open(os.path.join(HERE, "golden", "ddrive_sections.json")))
    d = gold["d"]
    secs = gold["sections"]
    for s in secs:
        assert -(-s["editable"] // d) == s["blocks"]
    lay = synth.section_layout(1, tuple((s["editable"], s["scaffold"]) for s in secs), d)
    for k, s in enumerate(secs):
        assert int((lay.block_section == k).sum()) == s["blocks"]
        assert int(((lay.section == k) & (lay.scaffold == 0)).sum()) == s["editable"]
    for b in range(lay.n_blocks):
        blk = slice(lay.block_start[b], lay.block_start[b + 1])
        ed = int((lay.scaffold[blk] == 0).sum())
        last = b == lay.n_blocks - 1 or lay.block_section[b + 1] != lay.block_section[b]
        assert ed == d or last
    share = lay.scaffold.mean()
    assert abs(share - gold["scaffold_fraction_about"]) < 0.02


def test_write_draft_fills_every_masked_candidate_with_its_argmax():
    """Draft mode: committed positions as usual; every other masked position with
    a row gets its argmax as token and stays masked; scaffold untouched."""
    n = 12
    logits = synth.normal_logits(17, 0, n, V=300, sigma=3.0, bf16=False)
    state = np.zeros(n, int)
    state[[2, 9]] = S
    lr = np.arange(n)
    lr[5] = -1
    r = oracle.unmask_step(logits, lr, [0, 6, n], state, np.full(n, -1), tau_full=2.0, tau_half=2.0,
                           min_frac=Fraction(1, 4), k_fixed=0, add_thr=Fraction(1, 2),
                           act_thr=Fraction(17, 20), write_draft=True)
    for p in range(n):
        if state[p] == S or lr[p] < 0:
            assert r["tokens"][p] == -1 and r["state"][p] == state[p]
        else:
            assert r["tokens"][p] == int(np.argmax(logits[p]))
            assert r["state"][p] == (C_ if r["commit"][p] else M)
    assert r["commit"].sum() >= 1 and (r["state"] == M).sum() >= 1
