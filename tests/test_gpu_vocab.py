"""GPU parity of bd_unmask_step and bd_spec_verify against the float64 oracle,
through the C ABI.  Decisions (argmax, commits, statuses, accepted lengths,
tokens, states) are compared bit for bit; confidence and LSE to fp32 accuracy.
Every input is conditioned so that each decision has a margin (confidence vs
tau >= 1e-4, the confidence gap at a top-n cut >= 1e-5 relative, the Gumbel
score gap of a sampled row >= 1e-3) that fp32 and float64 cannot disagree on;
the tests assert it through the oracle's reported margins."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
import oracle
import synth
from helpers import CONF_RTOL, DEV, bf16, f32, host, i32, status_word, u8

pytestmark = pytest.mark.gpu
V = synth.VOCAB


def _logits_dev(x, bf):
    return bf16(x) if bf else f32(x)


def _gpu_unmask(logits, logit_row, bs, state, tokens, bf, **kw):
    st = u8(state)
    tk = i32(tokens)
    ds = status_word()
    r = bd.bd_unmask_step(_logits_dev(logits, bf), i32(logit_row), i32(bs), st, tk,
                          tau_full=kw["tau_full"], tau_half=kw["tau_half"],
                          min_frac=(kw["min_frac"].numerator, kw["min_frac"].denominator), k_fixed=kw["k_fixed"],
                          add_thr=(kw["add_thr"].numerator, kw["add_thr"].denominator),
                          act_thr=(kw["act_thr"].numerator, kw["act_thr"].denominator), dev_status=ds)
    assert bd.bd_check(ds) == 0
    return {k: host(v) for k, v in r.items()} | dict(state=host(st), tokens=host(tk))


def _compare_unmask(g, o):
    for k in ("commit", "n_committed", "status", "pred", "state", "tokens"):
        assert np.array_equal(g[k].astype(np.int64), np.asarray(o[k], np.int64)), k
    cand = o["pred"] >= 0
    np.testing.assert_allclose(g["conf"][cand], o["conf"][cand], rtol=CONF_RTOL, atol=0)
    np.testing.assert_allclose(g["lse"][cand], o["lse"][cand], rtol=1e-6, atol=1e-6)


def _step_both(logits, logit_row, bs, state, tokens, bf, **kw):
    o = oracle.unmask_step(logits, logit_row, bs, state, tokens, **kw)
    if o["margins"]["tau"] < 1e-4 or o["margins"]["rank"] < 1e-5:
        return None, o
    g = _gpu_unmask(logits, logit_row, bs, state, tokens, bf, **kw)
    _compare_unmask(g, o)
    return g, o


TINY_KW = dict(tau_full=0.9, tau_half=0.9, min_frac=Fraction(1, 4), k_fixed=0, add_thr=Fraction(0, 1),
               act_thr=Fraction(0, 1))


def test_unmask_tiny_config_every_step():
    """[16, 1024] fp32 ~ N(0, 2), two blocks of 8 with 3 scaffold each, both
    blocks fully active; steps until everything is committed."""
    lay = synth.uniform_layout(16, 8, 3, seed=0)
    state = np.where(lay.scaffold == 1, synth.SCAFFOLD, synth.MASKED)
    tokens = np.where(lay.scaffold == 1, 7, -1)
    step = 0
    while (state == synth.MASKED).any():
        for attempt in range(20):
            logits = synth.normal_logits(0, 1000 * step + attempt, 16, 1024, sigma=2.0, bf16=False)
            g, o = _step_both(logits, np.arange(16), lay.block_start, state, tokens, False, **TINY_KW)
            if g is not None:
                break
        assert g is not None
        state, tokens = o["state"], o["tokens"]
        step += 1
    assert step <= 6


def _conditioned_planted(seed, R, Vv, kw, state, logit_row, bs, bf=True):
    for attempt in range(50):
        x, tok, _ = synth.planted_logits(seed, attempt, R, Vv, bf16=bf)
        o = oracle.unmask_step(x, logit_row, bs, state, np.full(len(state), -1), **kw)
        if o["margins"]["tau"] >= 1e-4 and o["margins"]["rank"] >= 1e-5:
            return x
    raise AssertionError("no conditioned draw")


def test_unmask_fast_ddrive_active_block():
    """The first explanation block of the Fast-dDrive layout: 32 editable rows of
    [32, 151936] bf16 logits with a planted peak each, tau = 0.9, fraction 1/4."""
    lay = synth.section_layout(1)
    b = 1
    lo, hi = lay.block_start[b], lay.block_start[b + 1]
    scaf = lay.scaffold[lo:hi]
    n = hi - lo
    state = np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED)
    logit_row = np.full(n, -1)
    logit_row[scaf == 0] = np.arange(int((scaf == 0).sum()))
    R = int((scaf == 0).sum())
    kw = dict(TINY_KW)
    x = _conditioned_planted(1, R, V, kw, state, logit_row, [0, n])
    g, o = _step_both(x, logit_row, [0, n], state, np.full(n, -1), True, **kw)
    assert g is not None and o["n_committed"][0] >= 8


@pytest.mark.parametrize("B", [1, 4, 8, 16, 32])
def test_unmask_wam_block_sweep(B):
    """WAM-Diff2 sweep: one block of B positions, fresh N(0, 3) bf16 rows each
    step, top k = max(1, B/8) by confidence, tau unreachable, at most 8 steps."""
    kw = dict(tau_full=2.0, tau_half=2.0, min_frac=Fraction(0, 1), k_fixed=max(1, B // 8),
              add_thr=Fraction(1, 2), act_thr=Fraction(17, 20))
    state = np.zeros(B, np.int64)
    tokens = np.full(B, -1)
    steps = 0
    while (state == 0).any() and steps < 8:
        for attempt in range(20):
            x = synth.normal_logits(2, 100 * B + 10 * steps + attempt, B, V, sigma=3.0)
            g, o = _step_both(x, np.arange(B), [0, B], state, tokens, True, **kw)
            if g is not None:
                break
        assert g is not None
        assert o["n_committed"][0] == min(kw["k_fixed"], int((state == 0).sum()))
        state, tokens = o["state"], o["tokens"]
        steps += 1
    assert steps == min(8, -(-B // kw["k_fixed"]))


def test_unmask_fast_dvla_pipelined_decode():
    """Fast-dVLA: 10 blocks of 7, up to 3 active (masked ratios 0.2 / 0.6 / 1.0
    at the start), half activation at 1/2 (tau 0.9 only), full at 0.85 (tau 0.9
    plus ceil(rem / 4)); blocks retire once complete; runs until all 70 are
    committed, GPU and oracle each advancing their own state."""
    kw = dict(tau_full=0.9, tau_half=0.9, min_frac=Fraction(1, 4), k_fixed=0, add_thr=Fraction(1, 2),
              act_thr=Fraction(17, 20))
    n_blocks, Bs = 10, 7
    state = np.zeros(n_blocks * Bs, np.int64)
    tokens = np.full(n_blocks * Bs, -1)
    g0 = synth.rng(3, 7)
    state[g0.choice(7, 5, replace=False)] = synth.COMMITTED        # block 0: 2 of 7 masked
    state[7 + g0.choice(7, 3, replace=False)] = synth.COMMITTED    # block 1: 4 of 7 masked
    tokens[state == synth.COMMITTED] = 5
    first, step = 0, 0
    statuses_seen = set()
    while first < n_blocks:
        last = min(n_blocks, first + 3)
        lo, hi = first * Bs, last * Bs
        win_state, win_tok = state[lo:hi], tokens[lo:hi]
        masked = np.flatnonzero(win_state == synth.MASKED)
        logit_row = np.full(hi - lo, -1)
        logit_row[masked] = np.arange(len(masked))
        bs = np.arange(0, hi - lo + 1, Bs)
        for attempt in range(50):
            x, _, _ = synth.planted_logits(3, 1000 * step + attempt, max(1, len(masked)), V)
            g, o = _step_both(x, logit_row, bs, win_state, win_tok, True, **kw)
            if g is not None:
                break
        assert g is not None
        statuses_seen |= set(int(s) for s in o["status"])
        state[lo:hi], tokens[lo:hi] = o["state"], o["tokens"]
        while first < n_blocks and not (state[first * Bs:(first + 1) * Bs] == synth.MASKED).any():
            first += 1
        step += 1
        assert step < 200
    assert bd.FULL in statuses_seen and bd.HALF in statuses_seen


def test_unmask_edge_cases():
    """A done block, a scaffold-only block, exact ties (lowest index wins), a
    vocabulary width that is not a multiple of 8, and a position without a row."""
    Vv, ld = 1003, 1008
    x = np.zeros((4, ld), np.float32)
    x[:, :Vv] = synth.normal_logits(5, 0, 4, Vv, sigma=1.0, bf16=False)
    x[0, [17, 901, 1002]] = 9.0     # tie between three entries
    x[1, 1002] = 12.0               # maximum in the ragged tail
    bs = [0, 2, 4, 7]
    state = np.array([1, 1, 2, 2, 0, 0, 0])
    tokens = np.array([3, 4, 5, 6, -1, -1, -1])
    logit_row = np.array([-1, -1, -1, -1, 0, 1, -1])
    kw = dict(tau_full=0.5, tau_half=0.5, min_frac=Fraction(1, 1), k_fixed=0, add_thr=Fraction(1, 2),
              act_thr=Fraction(17, 20))
    o = oracle.unmask_step(x[:, :Vv], logit_row, bs, state, tokens, **kw)
    st, tk = u8(state), i32(tokens)
    logits = f32(x)[:, :Vv]
    r = bd.bd_unmask_step(logits, i32(logit_row), i32(bs), st, tk, tau_full=0.5, tau_half=0.5, min_frac=(1, 1),
                          k_fixed=0)
    g = {k: host(v) for k, v in r.items()} | dict(state=host(st), tokens=host(tk))
    _compare_unmask(g, o)
    assert g["pred"][4] == 17 and g["pred"][5] == 1002
    assert list(g["status"]) == [bd.DONE, bd.DONE, bd.FULL]


# ================================================================================ verify

def _plant_ar(seed, stream, draft_edit, k, Vv, bf):
    """AR rows agreeing with the draft on the first k editable slots, disagreeing at k."""
    E = len(draft_edit)
    g = synth.rng(seed, 600, stream)
    want = g.integers(0, Vv, size=E + 1)
    want[:k] = draft_edit[:k]
    if k < E:
        want[k] = (draft_edit[k] + 1 + g.integers(0, Vv - 1)) % Vv
    x, tok, _ = synth.planted_logits(seed, stream, E + 1, Vv, sigma=2.0 if not bf else 3.0, tokens=want, bf16=bf)
    assert np.array_equal(tok, want)
    return x


def _gpu_verify(tokens, state, ar, bf, noise=None, T=1.0):
    tk, st = i32(tokens), u8(state)
    ds = status_word()
    acc, bon, bpos = bd.bd_spec_verify(tk, st, _logits_dev(ar, bf), None if noise is None else f32(noise), T,
                                       dev_status=ds)
    assert bd.bd_check(ds) == 0
    return dict(tokens=host(tk), state=host(st), accepted_len=host(acc), bonus=host(bon), bonus_pos=host(bpos))


def _compare_verify(g, o):
    for k in ("tokens", "state", "accepted_len", "bonus", "bonus_pos"):
        assert np.array_equal(g[k].astype(np.int64), np.asarray(o[k], np.int64)), k


def test_verify_tiny_config():
    """16-token draft, AR logits [17, 1024] fp32 with a planted match length k ~ U{0..10}."""
    g = synth.rng(0, 9)
    for trial in range(6):
        draft = g.integers(0, 1024, size=16)
        k = int(g.integers(0, 11))
        ar = _plant_ar(0, trial, draft, k, 1024, False)
        state = np.zeros((1, 16), np.int64)
        o = oracle.spec_verify(draft[None], state, ar[None])
        gg = _gpu_verify(draft[None], state, ar[None], False)
        _compare_verify(gg, o)
        assert o["accepted_len"][0] == k + 1


def test_verify_fast_ddrive_block_with_scaffold():
    """The 33-slot explanation block (32 editable + 1 scaffold), AR [33, 151936]
    bf16; match lengths 0, mid, all (bonus after the block)."""
    lay = synth.section_layout(1)
    lo, hi = lay.block_start[1], lay.block_start[2]
    scaf = lay.scaffold[lo:hi]
    L = hi - lo
    E = int((scaf == 0).sum())
    g = synth.rng(1, 9)
    for k in (0, 13, E):
        draft = g.integers(0, V, size=L)
        state = np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED)
        ar = _plant_ar(1, k, draft[scaf == 0], k, V, True)
        o = oracle.spec_verify(draft[None], state[None], ar[None])
        gg = _gpu_verify(draft[None], state[None], ar[None], True)
        _compare_verify(gg, o)
        assert o["accepted_len"][0] == k + 1
        assert (o["bonus_pos"][0] == L) == (k == E)


def test_verify_skips_committed_slots():
    L, Vv = 10, 512
    draft = np.arange(L) * 3
    state = np.array([1, 1, 2, 0, 0, 2, 0, 0, 0, 0])
    ed = state != 2
    rows_tok = np.concatenate([draft[ed][:2] + 1, draft[ed][2:5], [99, 7, 8, 5]])  # committed rows disagree: ignored
    ar, _, _ = synth.planted_logits(6, 0, len(rows_tok), Vv, tokens=rows_tok, bf16=False)
    o = oracle.spec_verify(draft[None], state[None], ar[None])
    gg = _gpu_verify(draft[None], state[None], ar[None], False)
    _compare_verify(gg, o)
    assert o["accepted_len"][0] == 4


def _conditioned_noise(seed, ar, T, min_gap=1e-3):
    u = synth.uniform_noise(seed, 0, ar.shape)
    flat_u = u.reshape(-1, ar.shape[-1])
    flat_x = ar.reshape(-1, ar.shape[-1])
    for attempt in range(1, 20):
        bad = []
        for r in range(flat_x.shape[0]):
            s = oracle.gumbel_scores(flat_x[r], flat_u[r], T)
            top2 = np.partition(s, -2)[-2:]
            if top2[1] - top2[0] < min_gap:
                bad.append(r)
        if not bad:
            return u
        synth.redraw_noise_rows(seed, 0, flat_u, bad, attempt)
    raise AssertionError("noise could not be conditioned")


@pytest.mark.parametrize("N", [1, 8])
def test_verify_sampled_rollouts(N):
    """Trajectory block of the fork (L = 39: 32 editable + 7 scaffold), N
    rollouts each with their own draft, AR rows and uniforms; Gumbel-max at T = 1."""
    L, E = 39, 32
    g = synth.rng(4, N)
    scaf = np.zeros(L, np.int64)
    scaf[g.choice(L, L - E, replace=False)] = 1
    state = np.tile(np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED), (N, 1))
    drafts = g.integers(0, V, size=(N, L))
    ar = np.stack([_plant_ar(4, 50 * N + r, drafts[r][scaf == 0], int(g.integers(0, E + 1)), V, True)
                   for r in range(N)])
    u = _conditioned_noise(4 + N, ar, 1.0)
    o = oracle.spec_verify(drafts, state, ar, u, 1.0)
    assert o["margins"]["gumbel"] >= 1e-3
    gg = _gpu_verify(drafts, state, ar, True, u, 1.0)
    _compare_verify(gg, o)


def test_unmask_draft_mode_matches_oracle():
    """Draft mode of the speculative round: tau = 0.9 commits, every other
    editable position receives its argmax and stays masked."""
    lay = synth.section_layout(1)
    lo, hi = lay.block_start[2], lay.block_start[3]
    scaf = lay.scaffold[lo:hi]
    n = hi - lo
    state = np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED)
    logit_row = np.full(n, -1)
    logit_row[scaf == 0] = np.arange(int((scaf == 0).sum()))
    kw = dict(tau_full=0.9, tau_half=0.9, min_frac=Fraction(0, 1), k_fixed=0, add_thr=Fraction(1, 2),
              act_thr=Fraction(17, 20))
    x = _conditioned_planted(7, int((scaf == 0).sum()), V, kw, state, logit_row, [0, n])
    o = oracle.unmask_step(x, logit_row, [0, n], state, np.full(n, -1), write_draft=True, **kw)
    st, tk = u8(state), i32(np.full(n, -1))
    r = bd.bd_unmask_step(bf16(x), i32(logit_row), i32([0, n]), st, tk, tau_full=0.9, tau_half=0.9, min_frac=(0, 1),
                          k_fixed=0, write_draft=True)
    g = {k: host(v) for k, v in r.items()} | dict(state=host(st), tokens=host(tk))
    _compare_unmask(g, o)
    assert (g["state"] == synth.MASKED).any() and (g["tokens"][scaf == 0] >= 0).all()


def test_unmask_maximum_window():
    """The largest window the library takes (2,048 positions): 64 blocks of 32
    with 3 scaffold slots each, the first 20 blocks partly committed, Fast-dVLA
    activation thresholds, bf16 logits [masked rows, 4,096] with planted peaks."""
    n_pos, Bsz, Vv = 2048, 32, 4096
    lay = synth.uniform_layout(n_pos, Bsz, scaffold_per_block=3, seed=50)
    g0 = synth.rng(50, 1)
    state = np.where(lay.scaffold == 1, synth.SCAFFOLD, synth.MASKED).astype(np.int64)
    for b in range(20):
        ed = np.flatnonzero(state[b * Bsz:(b + 1) * Bsz] == synth.MASKED) + b * Bsz
        state[g0.choice(ed, size=int(g0.integers(len(ed) // 2, len(ed) + 1)), replace=False)] = synth.COMMITTED
    tokens = np.where(state == synth.MASKED, -1, 7)
    masked = np.flatnonzero(state == synth.MASKED)
    logit_row = np.full(n_pos, -1)
    logit_row[masked] = np.arange(len(masked))
    kw = dict(tau_full=0.9, tau_half=0.9, min_frac=Fraction(1, 4), k_fixed=0, add_thr=Fraction(1, 2),
              act_thr=Fraction(17, 20))
    for attempt in range(20):
        x, _, _ = synth.planted_logits(50, 100 + attempt, len(masked), Vv)
        g, o = _step_both(x, logit_row, lay.block_start, state, tokens, True, **kw)
        if g is not None:
            break
    assert g is not None
    assert {bd.FULL, bd.HALF, bd.INACTIVE} <= set(int(s) for s in o["status"])


def test_verify_maximum_block():
    """The longest verified block (1,024 slots, 1/8 scaffold) for two sequences,
    one matching its draft to the end (bonus after the block), one diverging
    at slot 700; V = 2,048 fp32."""
    L, Vv, n_seq = 1024, 2048, 2
    g = synth.rng(51, 0)
    scaf = np.zeros(L, np.int64)
    scaf[g.choice(L, L // 8, replace=False)] = 1
    E = int((scaf == 0).sum())
    state = np.tile(np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED), (n_seq, 1))
    drafts = g.integers(0, Vv, size=(n_seq, L))
    ar = np.stack([_plant_ar(51, s, drafts[s][scaf == 0], k, Vv, False) for s, k in enumerate((E, 700))])
    o = oracle.spec_verify(drafts, state, ar)
    gg = _gpu_verify(drafts, state, ar, False)
    _compare_verify(gg, o)
    assert list(o["accepted_len"]) == [E + 1, 701] and o["bonus_pos"][0] == L
