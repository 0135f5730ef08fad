"""Pins of the streaming-cache oracle (FlashDrive tutorial, "流式推理"): ring
insertion by brute-force bookkeeping, the position-causal mask reducing to
block size 1 causal attention, cross-view causality by enumeration, invariance
to the physical order of the cache, and RoPE in the operator equal to keys
rotated beforehand."""
import numpy as np
import pytest

import oracle
import synth



def _rng(*s):
    return np.random.default_rng(list(s))


def test_insert_keeps_the_last_frames_of_every_view():
    """Insert frames+2 frames, each into the ring slot of its age; after every
    insertion each view's slots hold exactly its last `frames` frames (tracked
    independently as Python lists), positions included; other rows untouched."""
    views, frames, per, Hkv, D = 3, 4, 5, 2, 8
    C = views * frames * per
    g = _rng(1)
    k = g.standard_normal((Hkv, C + 3, D))
    v = g.standard_normal((Hkv, C + 3, D))
    kp = np.full(C, -1, np.int64)
    history = {w: [] for w in range(views)}
    for step in range(frames + 2):
        nk = g.standard_normal((views * per, Hkv, D))
        nv = g.standard_normal((views * per, Hkv, D))
        npos = 1000 * step + np.arange(views * per)
        slot = step % frames
        tail_k, tail_v = k[:, C:].copy(), v[:, C:].copy()
        k, v, kp = oracle.stream_insert(k, v, kp, nk, nv, npos, views, frames, per, slot)
        assert np.array_equal(k[:, C:], tail_k) and np.array_equal(v[:, C:], tail_v)
        for w in range(views):
            history[w].append((slot, nk[w * per:(w + 1) * per], nv[w * per:(w + 1) * per],
                               npos[w * per:(w + 1) * per]))
            history[w] = history[w][-frames:]
            for s_, fk, fv, fp in history[w]:
                rows = slice((w * frames + s_) * per, (w * frames + s_ + 1) * per)
                assert np.array_equal(k[:, rows], fk.transpose(1, 0, 2))
                assert np.array_equal(v[:, rows], fv.transpose(1, 0, 2))
                assert np.array_equal(kp[rows], fp)


def test_insert_does_not_modify_its_inputs():
    k = np.zeros((1, 4, 2)); v = np.zeros((1, 4, 2)); kp = np.zeros(4, np.int64)
    oracle.stream_insert(k, v, kp, np.ones((2, 1, 2)), np.ones((2, 1, 2)), np.array([7, 8]), 2, 2, 1, 1)
    assert not k.any() and not v.any() and not kp.any()


def test_identity_positions_reduce_to_causal_attention():
    """Cache = C0 prefix keys then the new frame's n keys, positions = key index,
    queries at C0 + i: the streaming mask is block-size-1 causal attention over
    prefix + active rows (the block-causal oracle with one block per position)."""
    C0, n, Hq, Hkv, D = 37, 9, 4, 2, 16
    a = synth.attn_case(20, 0, C=C0, block_start=list(range(n + 1)), Hq=Hq, Hkv=Hkv, D=D)
    mask = oracle.streaming_mask(np.arange(C0 + n), 0, C0 + np.arange(n))
    assert np.array_equal(mask, oracle.visibility_mask(C0, list(range(n + 1))))
    o, lse = oracle.stream_attention(a.q, a.k, a.v, C0 + n, None, 0, C0 + np.arange(n))
    o_ref, lse_ref = oracle.block_causal_attention(a.q, a.k, a.v, C0, list(range(n + 1)))
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12)


def _view_major_positions(views, frames, per, t0):
    """Positions of a view-major window whose frames are times t0 .. t0+frames-1."""
    w, f, t = np.meshgrid(np.arange(views), np.arange(frames), np.arange(per), indexing="ij")
    return ((w * frames + f) * per + t).reshape(-1) + t0 * per


def test_cross_view_causality_by_enumeration():
    """View-major positions: a new-frame query of view w sees every key of views
    < w, every history key of view w and the new frame of view w up to itself,
    and nothing of views > w -- checked key by key."""
    views, frames, per = 4, 3, 5
    pos = _view_major_positions(views, frames, per, 0)          # frame frames-1 is the new one
    qpos = np.array([(w * frames + frames - 1) * per + t for w in range(views) for t in range(per)])
    m = oracle.streaming_mask(pos, 0, qpos)
    for qi in range(views * per):
        wq, tq = divmod(qi, per)
        for j in range(views * frames * per):
            wk, rest = divmod(j, frames * per)
            fk, tk = divmod(rest, per)
            want = wk < wq or (wk == wq and (fk < frames - 1 or tk <= tq))
            assert m[qi, j] == want, (qi, j)


def test_order_of_the_cache_does_not_matter():
    """Shuffling the cache rows together with their positions leaves the output
    unchanged (each key carries its position), and a shift of every position
    and of delta by the same amount changes nothing."""
    views, frames, per, Hq, Hkv, D = 2, 3, 4, 4, 2, 16
    C = views * frames * per
    g = _rng(5)
    k = synth.to_bf16(g.standard_normal((Hkv, C, D)).astype(np.float32))
    v = synth.to_bf16(g.standard_normal((Hkv, C, D)).astype(np.float32))
    q = synth.to_bf16(g.standard_normal((views * per, Hq, D)).astype(np.float32))
    pos = _view_major_positions(views, frames, per, 2)
    qpos = np.array([(w * frames + frames - 1) * per + t for w in range(views) for t in range(per)])
    o, lse = oracle.stream_attention(q, k, v, C, pos, 2 * per, qpos, rope=True)
    perm = g.permutation(C)
    o2, lse2 = oracle.stream_attention(q, k[:, perm], v[:, perm], C, pos[perm], 2 * per, qpos, rope=True)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12)
    o3, _ = oracle.stream_attention(q, k, v, C, pos + 100, 2 * per + 100, qpos, rope=True)
    np.testing.assert_allclose(o3, o, rtol=1e-12, atol=1e-12)


def test_rope_in_the_operator_equals_prerotated_keys():
    C, n, Hq, Hkv, D = 40, 6, 4, 2, 16
    g = _rng(7)
    k = synth.to_bf16(g.standard_normal((Hkv, C, D)).astype(np.float32))
    v = synth.to_bf16(g.standard_normal((Hkv, C, D)).astype(np.float32))
    q = synth.to_bf16(g.standard_normal((n, Hq, D)).astype(np.float32))
    pos = g.permutation(C) + 50
    qpos = np.array([10, 25, 45, 60, 80, 95])
    o, lse = oracle.stream_attention(q, k, v, C, pos, 30, qpos, rope=True)
    kr = oracle.round_bf16(oracle.rope_rotate(k, pos - 30, 1e4))
    o2, lse2 = oracle.stream_attention(q, kr, v, C, pos, 30, qpos, rope=False)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12)


def test_query_that_sees_nothing():
    """A query positioned before every key: o = 0, lse = -inf; the other rows are
    unaffected."""
    C, Hq, Hkv, D = 8, 2, 1, 4
    g = _rng(9)
    k, v = g.standard_normal((Hkv, C, D)), g.standard_normal((Hkv, C, D))
    q = g.standard_normal((2, Hq, D))
    o, lse = oracle.stream_attention(q, k, v, C, np.arange(C) + 10, 0, np.array([3, 12]))
    assert not o[0].any() and np.all(np.isneginf(lse[:, 0]))
    s = (q[1, 0] @ k[0, :3].T) * D ** -0.5
    p = np.exp(s - s.max())
    np.testing.assert_allclose(o[1, 0], p @ v[0, :3] / p.sum(), rtol=1e-12)
