"""GPU parity of the streaming cache (FlashDrive tutorial, "流式推理") through
the C ABI: bd_stream_insert bit-exact against the oracle over a run of ring
insertions, and the streaming mask (bd_block_causal_attn with q_pos) against
the float64 oracle -- view-major windows with RoPE at k_pos - delta, ragged
frame sizes, the full 4 x 4 x 256 window with a new 1,024-token frame, the
identity-position case equal to block size 1 causal attention, and queries that
see nothing."""
import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
import oracle
import synth
from helpers import DEV, assert_attn_close, bf16, host, i32, status_word

pytestmark = pytest.mark.gpu


def _window(seed, views, frames, per, Hkv, D, stride_pad=3):
    g = synth.rng(seed, 800)
    C = views * frames * per
    k = synth.to_bf16(g.standard_normal((Hkv, C + stride_pad, D)).astype(np.float32))
    v = synth.to_bf16(g.standard_normal((Hkv, C + stride_pad, D)).astype(np.float32))
    return k, v


def _frame(seed, step, views, per, Hkv, D):
    g = synth.rng(seed, 801, step)
    nk = synth.to_bf16(g.standard_normal((views * per, Hkv, D)).astype(np.float32))
    nv = synth.to_bf16(g.standard_normal((views * per, Hkv, D)).astype(np.float32))
    return nk, nv


def _view_major(views, frames, per, frame_time):
    """Positions of the tokens of view w, frame time f: (w * frames + f) * per + t."""
    w = np.arange(views)[:, None]
    t = np.arange(per)[None, :]
    return ((w * frames + frame_time) * per + t).reshape(-1).astype(np.int32)


@pytest.mark.parametrize("views,frames,per,D", [(4, 4, 64, 128), (3, 2, 37, 64), (4, 4, 256, 128)])
def test_stream_insert_matches_oracle(views, frames, per, D):
    Hkv = 2
    k, v = _window(1, views, frames, per, Hkv, D)
    kp = np.arange(views * frames * per, dtype=np.int32)
    gk, gv, gp = bf16(k), bf16(v), i32(kp)
    for step in range(frames + 2):
        nk, nv = _frame(1, step, views, per, Hkv, D)
        npos = _view_major(views, frames, per, frames + step) + 7
        slot = step % frames
        k, v, kp = oracle.stream_insert(k, v, kp, nk, nv, npos, views, frames, per, slot)
        bd.bd_stream_insert(gk, gv, gp, bf16(nk), bf16(nv), i32(npos), views, frames, per, slot)
        torch.cuda.synchronize()
        assert np.array_equal(host(gk), k) and np.array_equal(host(gv), v)
        assert np.array_equal(host(gp).astype(np.int64), kp.astype(np.int64))


def _stream_case(seed, views, frames, per, Hq, Hkv, D, slides):
    """A window after `slides` insertions: every view's slots hold frame times
    slides .. slides + frames - 1 (ring order), the newest in slot (slides - 1)
    % frames; returns cache, positions, delta and the new frame's queries and
    query positions (all re-based by delta)."""
    k, v = _window(seed, views, frames, per, Hkv, D)
    kp = np.zeros(views * frames * per, np.int32)
    for f in range(frames + slides):
        slot = f % frames
        nk, nv = _frame(seed, f, views, per, Hkv, D)
        k, v, kp = oracle.stream_insert(k, v, kp, nk, nv, _view_major(views, frames, per, f), views, frames, per,
                                        slot)
    delta = slides * per                     # positions slid by `slides` frames
    newest = (frames + slides - 1)
    qpos = (_view_major(views, frames, per, newest) - delta).astype(np.int32)
    g = synth.rng(seed, 802)
    q = synth.to_bf16(g.standard_normal((views * per, Hq, D)).astype(np.float32))
    return k, v, kp, delta, q, qpos


@pytest.mark.parametrize("views,frames,per,D,rope", [(4, 4, 64, 128, True), (3, 3, 50, 128, True),
                                                     (2, 4, 40, 64, False), (4, 4, 256, 128, True)])
def test_streaming_mask_matches_oracle(views, frames, per, D, rope):
    Hq, Hkv = 16, 2
    k, v, kp, delta, q, qpos = _stream_case(3, views, frames, per, Hq, Hkv, D, slides=2)
    C = views * frames * per
    ds = status_word()
    o, lse = bd.bd_block_causal_attn(bf16(q), bf16(k), bf16(v), C, q_pos=i32(qpos),
                                     rope=dict(k_pos=i32(kp), delta=delta, theta=1e4) if rope else
                                     dict(k_pos=i32(kp), delta=delta, theta=1e4, enabled=False),
                                     dev_status=ds)
    assert bd.bd_check(ds) == 0
    o_ref, lse_ref = oracle.stream_attention(q, k, v, C, kp, delta, qpos, rope=rope)
    assert_attn_close(o, lse, o_ref, lse_ref, f"stream {views}x{frames}x{per}")


def test_identity_positions_equal_causal_attention():
    """Positions = key index and queries at C0 + i over a cache holding the new
    rows' own keys: the streaming call equals the plain block size 1 call."""
    C0, n, Hq, Hkv, D = 700, 33, 16, 2, 128
    a = synth.attn_case(21, 0, C=C0, block_start=list(range(n + 1)), Hq=Hq, Hkv=Hkv, D=D)
    q, k, v = bf16(a.q), bf16(a.k), bf16(a.v)
    o1, l1 = bd.bd_block_causal_attn(q, k, v, C0 + n, q_pos=i32(C0 + np.arange(n)))
    o2, l2 = bd.bd_block_causal_attn(q, k, v, C0, block_size=1)
    o_ref, lse_ref = oracle.block_causal_attention(a.q, a.k, a.v, C0, list(range(n + 1)))
    assert_attn_close(o1, l1, o_ref, lse_ref, "streaming")
    assert_attn_close(o2, l2, o_ref, lse_ref, "causal")


def test_queries_that_see_nothing():
    """A query placed before every cached key: o = 0 and lse = -inf; the row
    next to it is unaffected."""
    C, Hq, Hkv, D = 300, 8, 2, 128
    g = synth.rng(22, 0)
    k = synth.to_bf16(g.standard_normal((Hkv, C, D)).astype(np.float32))
    v = synth.to_bf16(g.standard_normal((Hkv, C, D)).astype(np.float32))
    q = synth.to_bf16(g.standard_normal((2, Hq, D)).astype(np.float32))
    kp = (np.arange(C) + 100).astype(np.int32)
    qpos = np.array([50, 250], np.int32)
    ds = status_word()
    o, lse = bd.bd_block_causal_attn(bf16(q), bf16(k), bf16(v), C, q_pos=i32(qpos),
                                     rope=dict(k_pos=i32(kp), delta=0, theta=1e4, enabled=False), dev_status=ds)
    assert bd.bd_check(ds) == 0
    oh, lh = host(o), host(lse)
    assert not oh[0].any() and np.all(np.isneginf(lh[:, 0]))
    o_ref, lse_ref = oracle.stream_attention(q, k, v, C, kp, 0, qpos)
    np.testing.assert_allclose(oh[1], o_ref[1], atol=1e-2, rtol=1e-2)
    np.testing.assert_allclose(lh[:, 1], lse_ref[:, 1], rtol=1e-5)
