"""Pins of the attention oracle against facts the pages and mathematics fix.

Each test would fail for a plausible slip in the oracle: a dropped or extra
visible key, a flipped block comparison, a wrong GQA grouping, a missing
softmax scale, a RoPE sign or pairing error, a wrong LSE base.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _block_end(block_start, i):
    for b in range(len(block_start) - 1):
        if block_start[b] <= i < block_start[b + 1]:
            return block_start[b + 1]
    raise AssertionError


def _case(seed, C, bs, Hq=4, Hkv=2, D=16):
    return synth.attn_case(seed, 0, C=C, block_start=bs, Hq=Hq, Hkv=Hkv, D=D)


@pytest.mark.parametrize("C,bs", [(5, [0, 3, 7, 8]), (0, [0, 4, 6]), (9, [0, 1, 2, 3]), (3, [0, 6])])
def test_zero_query_closed_form(C, bs):
    """Q = 0: every visible key has weight 1/#visible, so o_i is the mean of the
    visible values and lse_i = ln #visible.  #visible(i) = C + end of i's block
    (a block sees the prefix, earlier blocks and itself, never later ones)."""
    c = _case(1, C, bs)
    q = np.zeros_like(c.q)
    o, lse = oracle.block_causal_attention(q, c.k, c.v, C, bs)
    Hq, Hkv = q.shape[1], c.k.shape[0]
    for i in range(bs[-1]):
        nvis = C + _block_end(bs, i)
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            np.testing.assert_allclose(o[i, h], c.v[kv, :nvis].astype(np.float64).mean(0), rtol=0, atol=1e-12)
            assert abs(lse[h, i] - math.log(nvis)) < 1e-12


def test_gqa_grouping_contiguous():
    """Query head h reads KV head h // G: with Q = 0 and a constant value per KV
    head, o[:, h] equals that constant (h % Hkv would read the wrong head)."""
    Hq, Hkv, D, C, bs = 8, 2, 8, 4, [0, 2, 5]
    c = _case(2, C, bs, Hq, Hkv, D)
    v = np.zeros_like(c.v)
    v[0] = 3.0
    v[1] = -7.0
    o, _ = oracle.block_causal_attention(np.zeros_like(c.q), c.k, v, C, bs)
    for h in range(Hq):
        assert np.all(o[:, h] == (3.0 if h < 4 else -7.0))


def _textbook_causal(q, k, v, C):
    """Ordinary causal attention written out with scalar loops."""
    n_q, Hq, D = q.shape
    G = Hq // k.shape[0]
    o = np.zeros((n_q, Hq, D))
    lse = np.zeros((Hq, n_q))
    for i in range(n_q):
        for h in range(Hq):
            kv = h // G
            keys = range(C + i + 1)
            sc = [sum(float(q[i, h, d]) * float(k[kv, j, d]) for d in range(D)) / math.sqrt(D) for j in keys]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            z = sum(w)
            for d in range(D):
                o[i, h, d] = sum(w[j] * float(v[kv, j, d]) for j in keys) / z
            lse[h, i] = mx + math.log(z)
    return o, lse


def test_block_size_one_is_causal():
    """Block size 1 is ordinary autoregressive (causal) attention."""
    C, n_q = 6, 5
    bs = list(range(n_q + 1))
    c = _case(3, C, bs, 4, 2, 8)
    o, lse = oracle.block_causal_attention(c.q, c.k, c.v, C, bs)
    o2, lse2 = _textbook_causal(c.q, c.k, c.v, C)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_single_block_is_bidirectional():
    """One block spanning the whole output: every query sees every key."""
    C, n_q, D = 7, 6, 8
    c = _case(4, C, [0, n_q], 2, 1, D)
    o, lse = oracle.block_causal_attention(c.q, c.k, c.v, C, [0, n_q])
    q = c.q.astype(np.float64)
    k = c.k[0, :C + n_q].astype(np.float64)
    v = c.v[0, :C + n_q].astype(np.float64)
    for h in range(2):
        s = q[:, h] @ k.T / math.sqrt(D)
        w = np.exp(s - s.max(1, keepdims=True))
        np.testing.assert_allclose(o[:, h], (w @ v) / w.sum(1, keepdims=True), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[h], np.log(np.exp(s).sum(1)), rtol=0, atol=1e-12)


def test_later_blocks_do_not_leak():
    """Perturbing a later block's queries, keys and values by 1e4 leaves every
    earlier block's o and lse bitwise unchanged (no logic leak)."""
    C, bs = 10, [0, 3, 6, 9, 12]
    c = _case(5, C, bs)
    o, lse = oracle.block_causal_attention(c.q, c.k, c.v, C, bs)
    for b in range(1, 4):
        q, k, v = c.q.copy(), c.k.copy(), c.v.copy()
        lo = bs[b]
        q[lo:] += 1e4
        k[:, C + lo:] -= 1e4
        v[:, C + lo:] += 1e4
        o2, lse2 = oracle.block_causal_attention(q, k, v, C, bs)
        assert np.array_equal(o[:lo], o2[:lo]) and np.array_equal(lse[:, :lo], lse2[:, :lo])
        assert not np.array_equal(o[lo:], o2[lo:])


def test_brute_force_tiny():
    """Enumerated visible-key lists (no mask matrix) on tiny shapes."""
    g = synth.rng(6)
    for trial in range(6):
        C = int(g.integers(0, 5))
        sizes = g.integers(1, 4, size=int(g.integers(1, 4)))
        bs = [0] + list(np.cumsum(sizes))
        c = _case(100 + trial, C, bs, 2, 1, 4)
        o, lse = oracle.block_causal_attention(c.q, c.k, c.v, C, bs)
        for i in range(bs[-1]):
            b = max(j for j in range(len(bs) - 1) if bs[j] <= i)
            vis = list(range(C)) + [C + a for a in range(bs[-1]) if a < bs[b + 1]]
            for h in range(2):
                sc = np.array([c.q[i, h].astype(float) @ c.k[0, j].astype(float) / 2.0 for j in vis])
                w = np.exp(sc - sc.max())
                ref = (w[:, None] * c.v[0, vis].astype(float)).sum(0) / w.sum()
                np.testing.assert_allclose(o[i, h], ref, rtol=0, atol=1e-12)
                assert abs(lse[h, i] - (sc.max() + math.log(w.sum()))) < 1e-12


def test_softmax_scale_and_lse_hand_case():
    """D = 4, one query, two prefix keys, no active key visible but itself.

    q = (2, 0, 0, 0); keys (1, 0, 0, 0), (0, 0, 0, 0), own key (0, 0, 0, 0):
    scores 2*1/sqrt(4) = 1, 0, 0  ->  weights e, 1, 1 over (e + 2)."""
    q = np.array([[[2.0, 0, 0, 0]]])
    k = np.zeros((1, 3, 4))
    k[0, 0, 0] = 1.0
    v = np.zeros((1, 3, 4))
    v[0, 0] = [1, 0, 0, 0]
    v[0, 1] = [0, 1, 0, 0]
    v[0, 2] = [0, 0, 1, 0]
    o, lse = oracle.block_causal_attention(q, k, v, 2, [0, 1])
    e = math.e
    np.testing.assert_allclose(o[0, 0], [e / (e + 2), 1 / (e + 2), 1 / (e + 2), 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - math.log(e + 2)) < 1e-15


# ------------------------------------------------------------------------ RoPE

def test_round_bf16_hand_values():
    vals = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 1.0 + 2 ** -9, -3.0 - 2 ** -7 - 2 ** -9, 0.0, 2 ** -130]
    want = [1.0, 1.0 + 2 ** -7, 1.0, -3.0 - 2 ** -6, 0.0, 2 ** -130]
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1.0); 1+3*2^-9 is above the tie
    assert list(oracle.round_bf16(np.array(vals))) == want


def test_round_bf16_matches_torch_on_float32():
    """On float32 inputs the oracle's rounding agrees with torch's bfloat16 cast."""
    import torch
    x = synth.rng(7).standard_normal(20000).astype(np.float32) * 37.0
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_rope_two_dim_closed_form():
    """D = 2 is one pair at frequency theta^0 = 1: a rotation by angle p."""
    x = np.array([[0.3, -1.7]] * 4)
    pos = np.array([0, 1, 5, -3])
    r = oracle.rope_rotate(x, pos, 10000.0)
    for j, p in enumerate(pos):
        c, s = math.cos(p), math.sin(p)
        np.testing.assert_allclose(r[j], [0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s], atol=1e-15)


def test_rope_four_dim_pairs_and_frequencies():
    """D = 4, theta = 100: pairs (0, 2) at frequency 1 and (1, 3) at 100^(-1/2) = 0.1."""
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    p = 7
    r = oracle.rope_rotate(x, [p], 100.0)[0]
    a, b = p * 1.0, p * 0.1
    want = [1 * math.cos(a) - 3 * math.sin(a), 2 * math.cos(b) - 4 * math.sin(b),
            3 * math.cos(a) + 1 * math.sin(a), 4 * math.cos(b) + 2 * math.sin(b)]
    np.testing.assert_allclose(r, want, atol=1e-14)


def test_rope_relative_position():
    """rope(q, p + c) . rope(k, s + c) = rope(q, p) . rope(k, s)."""
    g = synth.rng(8)
    q = g.standard_normal((1, 64))
    k = g.standard_normal((1, 64))
    for p, s, c in [(3, 11, 100), (4000, 17, -256), (0, 4305, 256)]:
        a = oracle.rope_rotate(q, [p + c], 1e4) @ oracle.rope_rotate(k, [s + c], 1e4).T
        b = oracle.rope_rotate(q, [p], 1e4) @ oracle.rope_rotate(k, [s], 1e4).T
        assert abs(a - b) < 1e-9 * max(1.0, abs(b))


def test_attention_rope_equals_prerotated_keys():
    """In-operator RoPE of the prefix keys at k_pos - delta equals rotating them
    beforehand (complex-number form, written here independently), rounding to
    bf16, and running the no-RoPE path; the active keys are left alone."""
    C, bs, D = 9, [0, 2, 5], 8
    c = _case(9, C, bs, 4, 2, D)
    k_pos = np.arange(C) * 3 + 40
    delta = 17
    o, lse = oracle.block_causal_attention(c.q, c.k, c.v, C, bs, k_pos=k_pos, delta=delta,
                                           theta=500.0, rope=True)
    half = D // 2
    freq = 500.0 ** (-2.0 * np.arange(half) / D)
    k = c.k.astype(np.float64).copy()
    z = (k[:, :C, :half] + 1j * k[:, :C, half:]) * np.exp(1j * (k_pos - delta)[:, None] * freq[None, :])
    k[:, :C, :half], k[:, :C, half:] = z.real, z.imag
    u = np.ascontiguousarray(k[:, :C]).view(np.uint64)  # round to bf16 on the bits:
    u = (u + np.uint64((1 << 44) - 1) + ((u >> np.uint64(45)) & np.uint64(1))) & ~np.uint64((1 << 45) - 1)
    k[:, :C] = u.view(np.float64)                       # keep 7 of the 52 stored bits, ties to even
    o2, lse2 = oracle.block_causal_attention(c.q, k, c.v, C, bs)
    np.testing.assert_allclose(o, o2, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)


# ------------------------------------------------------------------------ fork

def _fork(N, seed=10, C=7, n_q=4, priv_len=3, bs=(0, 2, 4)):
    return synth.fork_case(seed, 0, N=N, C=C, n_q=n_q, priv_len=priv_len, block_start=bs,
                           Hq=4, Hkv=2, D=8)


def test_fork_zero_query_closed_form():
    """Q = 0: rollout r's query i averages the prefix values, its own private
    rows and its active rows up to the end of i's block."""
    f = _fork(3)
    o, lse = oracle.fork_attention(np.zeros_like(f.q), f.prefix_k, f.prefix_v, f.priv_k, f.priv_v,
                                   f.priv_len, f.block_start)
    for r in range(3):
        for i in range(4):
            end = f.priv_len + _block_end(list(f.block_start), i)
            for h in range(4):
                kv = h // 2
                vals = np.concatenate([f.prefix_v[kv], f.priv_v[r, kv, :end]]).astype(np.float64)
                np.testing.assert_allclose(o[r, i, h], vals.mean(0), atol=1e-12)
                assert abs(lse[r, h, i] - math.log(f.C + end)) < 1e-12


def test_fork_rollouts_are_independent():
    """Changing rollout 1's private rows changes rollout 1 only; identical
    private inputs give identical rollouts."""
    f = _fork(3)
    pk, pv = f.priv_k.copy(), f.priv_v.copy()
    pk[2], pv[2] = pk[0], pv[0]
    q = f.q.copy()
    q[2] = q[0]
    o, lse = oracle.fork_attention(q, f.prefix_k, f.prefix_v, pk, pv, f.priv_len, f.block_start)
    assert np.array_equal(o[0], o[2]) and np.array_equal(lse[0], lse[2])
    pk2 = pk.copy()
    pk2[1] += 5.0
    o2, _ = oracle.fork_attention(q, f.prefix_k, f.prefix_v, pk2, pv, f.priv_len, f.block_start)
    assert np.array_equal(o[[0, 2]], o2[[0, 2]]) and not np.array_equal(o[1], o2[1])


def test_bf16_midpoint_distance_helper():
    """The helper the GPU RoPE test uses to show that its inputs reach elements
    near a bf16 rounding midpoint: hand values (bf16 spacing is 2^-7 on [1, 2):
    1 + 2^-8 is a midpoint, 1 and 1 + 2^-7 are bf16 values half a spacing from
    one; spacing 2^-6 at 3), and rounding by the oracle flips exactly across a
    midpoint."""
    import helpers
    d = helpers.bf16_midpoint_distance(np.array([1.0, 1.0 + 2 ** -8, 1.0 + 2 ** -7, 0.0, -3.0]))
    assert d[0] == 2 ** -8 and d[1] == 0.0 and d[2] == 2 ** -8
    assert np.isinf(d[3]) and d[4] == 2 ** -7
    mid = 1.0 + 2 ** -8 + 2 ** -7          # midpoint between 1 + 2^-7 and 1 + 2^-6
    assert oracle.round_bf16(mid - 1e-12) == 1.0 + 2 ** -7 and oracle.round_bf16(mid + 1e-12) == 1.0 + 2 ** -6
