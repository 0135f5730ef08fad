"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (same shapes, default KV splits, same inputs): the Fast-dDrive-shaped
speculative round of the bench, the streaming fork with RoPE at N = 1 / 8 / 32,
the WAM-Diff2 and Fast-dVLA attention shapes, and the sampled verifier over 32
rollouts.  The oracle computes every output here (float64, seconds)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
from block_causal_masked_gb300.decode import SpeculativeRound
import oracle
import synth
from helpers import CONF_RTOL, DEV, assert_attn_close, bf16, f32, host, i32, status_word, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ddrive():
    """The Fast-dDrive-shaped round the benchmark times, on the library's
    SpeculativeRound driver."""
    inp = synth.fast_ddrive_round(synth.FAST_DDRIVE.seed)
    t = lambda x, dt: torch.from_numpy(np.array(x, order="C", copy=True)).to(DEV).to(dt)  # noqa: E731
    bf = torch.bfloat16
    rd = SpeculativeRound([t(q, bf) for q, _, _, _ in inp["layers"]], [t(q, bf) for _, q, _, _ in inp["layers"]],
                          [t(k, bf) for _, _, k, _ in inp["layers"]], [t(v, bf) for _, _, _, v in inp["layers"]],
                          inp["C"], t(inp["logits"], bf), t(inp["ar_logits"][None], bf),
                          t(inp["logit_row"], torch.int32), t(inp["state"], torch.uint8),
                          t(inp["tokens"], torch.int32), synth.DDRIVE_TAU)
    return inp, rd


@pytest.mark.parametrize("layer", [0, 17, 35])
def test_bench_round_attention_layers(ddrive, layer):
    """Both attention passes of the bench round (MDM block and causal AR pass)."""
    inp, rd = ddrive
    C, n_q = inp["C"], inp["n_q"]
    q, q_ar, k, v = inp["layers"][layer]
    o, lse = bd.bd_block_causal_attn(rd.q[layer], rd.k[layer], rd.v[layer], C, block_start=rd.block)
    o_ref, lse_ref = oracle.block_causal_attention(q, k, v, C, [0, n_q])
    assert_attn_close(o, lse, o_ref, lse_ref, f"MDM layer {layer}")
    o, lse = bd.bd_block_causal_attn(rd.q_ar[layer], rd.k[layer], rd.v[layer], C, block_size=1)
    o_ref, lse_ref = oracle.block_causal_attention(q_ar, k, v, C, list(range(n_q + 1)))
    assert_attn_close(o, lse, o_ref, lse_ref, f"AR layer {layer}")


def test_bench_round_unmask_and_verify(ddrive):
    """The round's unmask (tau 0.9 + draft) and verify equal the oracle's, and so
    does the committed count the bench reports."""
    inp, rd = ddrive
    n_q = inp["n_q"]
    kw = dict(tau_full=synth.DDRIVE_TAU, tau_half=synth.DDRIVE_TAU, min_frac=Fraction(0, 1), k_fixed=0,
              add_thr=Fraction(1, 2),
              act_thr=Fraction(17, 20), write_draft=True)
    ref = oracle.unmask_step(inp["logits"], inp["logit_row"], [0, n_q], inp["state"], inp["tokens"], **kw)
    assert ref["margins"]["tau"] >= 1e-4
    rd.reset()
    rd.unmask()
    g = {k: host(v) for k, v in rd.um.items()}
    for key in ("commit", "n_committed", "pred"):
        assert np.array_equal(g[key].astype(np.int64), np.asarray(ref[key], np.int64)), key
    assert np.array_equal(host(rd.state).astype(np.int64), ref["state"])
    assert np.array_equal(host(rd.tokens).astype(np.int64), ref["tokens"])
    cand = ref["pred"] >= 0
    np.testing.assert_allclose(g["conf"][cand], ref["conf"][cand], rtol=CONF_RTOL)
    vref = oracle.spec_verify(ref["tokens"][None], ref["state"][None], inp["ar_logits"][None])
    rd.verify()
    assert int(rd.acc[0]) == int(vref["accepted_len"][0]) and int(rd.bonus[0]) == int(vref["bonus"][0])
    assert int(rd.bonus_pos[0]) == int(vref["bonus_pos"][0])
    assert np.array_equal(host(rd.tokens).astype(np.int64), vref["tokens"][0])
    assert np.array_equal(host(rd.state).astype(np.int64), vref["state"][0])
    total, _, _ = oracle.speculative_round(inp["layers"], inp["C"], inp["n_q"], inp["logits"], inp["logit_row"],
                                           inp["state"], inp["tokens"], inp["ar_logits"], synth.DDRIVE_TAU)
    assert rd.committed() == total
    # the round captured as one CUDA graph and replayed commits the same
    rd.capture()
    rd.replay()
    torch.cuda.synchronize()
    assert rd.committed() == total
    assert np.array_equal(host(rd.tokens).astype(np.int64), vref["tokens"][0])


@pytest.mark.parametrize("N", [1, 8, 32])
def test_fork_streaming_full_size(N):
    """Fork over the 4,306-key pre-RoPE streaming prefix (view-major window of
    4 x 4 x 256 + 210 section keys, delta 256): the second trajectory block
    (39 positions, 41 private rows before it) of N rollouts."""
    C = 4096 + 210
    k_pos = synth.streaming_prefix_positions()
    f = synth.fork_case(4, N, N=N, C=C, n_q=39, priv_len=41, block_start=[0, 39], Hq=16, Hkv=2, D=128,
                        k_pos=k_pos, delta=256, theta=1e4)
    ds = status_word()
    o, lse = bd.bd_fork_rollouts(bf16(f.q), bf16(f.prefix_k), bf16(f.prefix_v), bf16(f.priv_k), bf16(f.priv_v),
                                 f.priv_len, C, block_start=i32(f.block_start),
                                 rope=dict(k_pos=i32(k_pos), delta=256, theta=1e4), dev_status=ds)
    assert bd.bd_check(ds) == 0
    o_ref, lse_ref = oracle.fork_attention(f.q, f.prefix_k, f.prefix_v, f.priv_k, f.priv_v, f.priv_len,
                                           f.block_start, k_pos=k_pos, delta=256, theta=1e4, rope=True)
    assert_attn_close(o, lse, o_ref, lse_ref, f"fork N={N}")


@pytest.mark.parametrize("B", [1, 4, 32])
def test_wam_sweep_attention_full_size(B):
    """16/8 heads, prefix 2,048 + the 128 output positions decoded before the block."""
    C = 2048 + 128
    case = synth.attn_case(2, B, C=C, block_start=[0, B], Hq=16, Hkv=8, D=128)
    o, lse = bd.bd_block_causal_attn(bf16(case.q), bf16(case.k), bf16(case.v), C, block_start=i32([0, B]))
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, C, [0, B])
    assert_attn_close(o, lse, o_ref, lse_ref, f"B={B}")


def test_fast_dvla_window_full_size():
    """16/2 heads, 600 prefix keys (512 image + 88 instruction) + 14 decoded
    action tokens, a window of three 7-token blocks."""
    C = 600 + 14
    bs = [0, 7, 14, 21]
    case = synth.attn_case(3, 0, C=C, block_start=bs, Hq=16, Hkv=2, D=128, text_from=512)
    o, lse = bd.bd_block_causal_attn(bf16(case.q), bf16(case.k), bf16(case.v), C, block_start=i32(bs))
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref)


def test_sampled_verify_32_rollouts_full_vocab():
    """The trajectory block of 32 rollouts (39 slots, 32 editable), AR rows
    [32, 33, 151936] bf16, Gumbel noise fp32, temperature 1."""
    N, L, E, V = 32, 39, 32, synth.VOCAB
    g = synth.rng(4, 999)
    scaf = np.zeros(L, np.int64)
    scaf[g.choice(L, L - E, replace=False)] = 1
    state = np.tile(np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED), (N, 1))
    drafts = g.integers(0, V, size=(N, L))
    ar = np.empty((N, E + 1, V), np.float32)
    for r in range(N):
        want = g.integers(0, V, size=E + 1)
        k = int(g.integers(0, E + 1))
        want[:k] = drafts[r][scaf == 0][:k]
        ar[r], _, _ = synth.planted_logits(4, 7000 + r, E + 1, V, tokens=want)
    u = synth.uniform_noise(4, 77, ar.shape)
    flat_u, flat_x = u.reshape(-1, V), ar.reshape(-1, V)
    for attempt in range(1, 20):
        s = flat_x.astype(np.float64) - np.log(-np.log(flat_u.astype(np.float64)))
        top2 = np.partition(s, -2, axis=1)[:, -2:]
        bad = np.flatnonzero(top2[:, 1] - top2[:, 0] < 1e-3)
        if bad.size == 0:
            break
        synth.redraw_noise_rows(4, 77, flat_u, bad, attempt)
    ref = oracle.spec_verify(drafts, state, ar, u, 1.0)
    assert ref["margins"]["gumbel"] >= 1e-3
    tk, st = i32(drafts), u8(state)
    acc, bon, bpos = bd.bd_spec_verify(tk, st, bf16(ar), f32(u), 1.0)
    assert np.array_equal(host(acc).astype(np.int64), ref["accepted_len"])
    assert np.array_equal(host(bon).astype(np.int64), ref["bonus"])
    assert np.array_equal(host(bpos).astype(np.int64), ref["bonus_pos"])
    assert np.array_equal(host(tk).astype(np.int64), ref["tokens"])
    assert np.array_equal(host(st).astype(np.int64), ref["state"])
