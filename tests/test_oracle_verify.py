"""Pins of the verify oracle: with a toy deterministic AR model, iterated
draft + verify reproduces plain AR decoding exactly (the pages' claim that the
speculative output is identical to pure AR), greedily and with shared
Gumbel noise, for arbitrary drafts."""
import hashlib
import math

import numpy as np
import pytest

import oracle
import synth

M, C_, S = 0, 1, 2
V = 37


def _h(ctx, salt):
    key = repr((int(salt), tuple(int(t) for t in ctx)))
    return int.from_bytes(hashlib.sha256(key.encode()).digest()[:8], "little")


def next_greedy(ctx, salt=0):
    return _h(ctx, salt) % V


def ar_logits_row(ctx, salt=0):
    """Toy model logits for the token after ``ctx``: a seeded normal vector."""
    return synth.rng(_h(ctx, salt) % (2 ** 31)).standard_normal(V)


def sample(ctx, u, T, salt=0):
    return int(np.argmax(ar_logits_row(ctx, salt) / T - np.log(-np.log(u))))


def _greedy_rows(ctx_tokens, edit, L, prompt):
    rows = []
    for p in edit + [L]:
        row = np.zeros(V)
        row[next_greedy(prompt + list(ctx_tokens[:p]))] = 5.0
        rows.append(row)
    return np.array(rows)


def _run_block(prompt, template, drafter, sampled=False, u=None, T=1.0):
    """Decode one block by draft + verify rounds; returns tokens, rounds, last bonus."""
    L = len(template)
    state = np.array([[S if t is not None else M for t in template]])
    tokens = np.array([[t if t is not None else -1 for t in template]])
    edit = [p for p in range(L) if template[p] is None]
    rounds, last = 0, None
    while (state == M).any():
        for p in range(L):
            if state[0, p] == M:
                tokens[0, p] = drafter(rounds, p)
        ctx = tokens[0]
        if sampled:
            rows = np.array([ar_logits_row(prompt + list(ctx[:p])) for p in edit + [L]])
            noise = np.array([u[p] for p in edit + [L]])
            r = oracle.spec_verify(tokens, state, rows[None], noise[None], T)
        else:
            r = oracle.spec_verify(tokens, state, _greedy_rows(ctx, edit, L, prompt)[None])
        assert r["accepted_len"][0] >= 1            # never goes backwards
        tokens, state = r["tokens"], r["state"]
        last = r
        rounds += 1
    return tokens[0], rounds, last


def _reference(prompt, template, sampled=False, u=None, T=1.0):
    out = []
    for p, t in enumerate(template + [None]):
        ctx = prompt + out
        if t is not None:
            out.append(t)
        elif sampled:
            out.append(sample(ctx, u[p], T))
        else:
            out.append(next_greedy(ctx))
    return out


TEMPLATES = [
    [None] * 9,
    [5, None, None, 6, None, None, None, 7, None, 8],
    [None, 1, 1, None, None, 2, None, None],
]


@pytest.mark.parametrize("ti", range(len(TEMPLATES)))
@pytest.mark.parametrize("mode", ["random", "correct", "wrong"])
def test_greedy_draft_verify_equals_ar(ti, mode):
    template = TEMPLATES[ti]
    prompt = [3, 1, 4]
    ref = _reference(prompt, template)
    g = synth.rng(20, ti)

    def drafter(rnd, p):
        if mode == "correct":
            return ref[p]
        if mode == "wrong":
            return (ref[p] + 1) % V
        return int(g.integers(0, V))

    toks, rounds, last = _run_block(prompt, template, drafter)
    assert list(toks) == ref[:len(template)]
    E = sum(t is None for t in template)
    if mode == "correct":
        # one round: E drafts + the bonus for the position after the block
        assert rounds == 1 and last["accepted_len"][0] == E + 1
        assert last["bonus_pos"][0] == len(template) and last["bonus"][0] == ref[len(template)]
    if mode == "wrong":
        assert rounds == E                      # each round commits only the AR token


@pytest.mark.parametrize("ti", range(len(TEMPLATES)))
def test_sampled_draft_verify_equals_ar_sampling(ti):
    """Same Gumbel noise per position: draft + verify gives the AR sample."""
    template = TEMPLATES[ti]
    prompt = [2, 7]
    L = len(template)
    u = synth.uniform_noise(21, ti, (L + 1, V)).astype(np.float64)
    T = 0.7
    ref = _reference(prompt, template, True, u, T)
    g = synth.rng(22, ti)
    toks, _, _ = _run_block(prompt, template, lambda r, p: int(g.integers(0, V)), True, u, T)
    assert list(toks) == ref[:L]


def test_first_mismatch_gives_one_token_and_resets_tail():
    L = 6
    tokens = np.array([[10, 11, 12, 13, 14, 15]])
    state = np.array([[M, M, S, M, M, M]])
    rows = np.zeros((1, 6, 40))
    for e, t in enumerate([9, 11, 13, 14, 15, 30]):   # row 0 disagrees with the draft
        rows[0, e, t] = 1.0
    r = oracle.spec_verify(tokens, state, rows)
    assert r["accepted_len"][0] == 1 and r["bonus"][0] == 9 and r["bonus_pos"][0] == 0
    assert list(r["tokens"][0]) == [9, -1, 12, -1, -1, -1]
    assert list(r["state"][0]) == [C_, M, S, M, M, M]


def test_committed_slots_are_skipped():
    tokens = np.array([[4, 5, 6, 7]])
    state = np.array([[C_, M, M, M]])
    rows = np.zeros((1, 5, 10))
    for e, t in enumerate([1, 5, 6, 2, 3]):        # row 0 belongs to a committed slot
        rows[0, e, t] = 1.0
    r = oracle.spec_verify(tokens, state, rows)
    assert r["accepted_len"][0] == 3 and r["bonus_pos"][0] == 3 and r["bonus"][0] == 2
    assert list(r["tokens"][0]) == [4, 5, 6, 2]


def test_gumbel_score_closed_forms():
    row = np.array([1.0, -2.0, 0.5])
    # u = e^-1 -> -log(-log u) = 0
    np.testing.assert_allclose(oracle.gumbel_scores(row, np.full(3, math.exp(-1)), 2.0), row / 2, atol=1e-15)
    z = np.array([0.3, -1.2, 2.5])
    u = np.exp(-np.exp(-z))
    np.testing.assert_allclose(oracle.gumbel_scores(np.zeros(3), u, 1.0), z, atol=1e-12)


def test_gumbel_max_samples_the_softmax():
    """Gumbel-max with fresh uniforms draws token v with probability softmax(l/T)_v."""
    row = np.array([0.0, 1.0, -0.5, 2.0])
    T = 1.5
    u = synth.uniform_noise(23, 0, (60000, 4)).astype(np.float64)
    picks = np.argmax(row / T - np.log(-np.log(u)), axis=1)
    freq = np.bincount(picks, minlength=4) / len(picks)
    p = np.exp(row / T) / np.exp(row / T).sum()
    np.testing.assert_allclose(freq, p, atol=0.01)
    # the oracle's scores give the same picks
    picks2 = [int(np.argmax(oracle.gumbel_scores(row, u[i], T))) for i in range(2000)]
    assert picks2 == list(picks[:2000])
