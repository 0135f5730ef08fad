"""The device-resident decode loop: the whole 256-token WAM-Diff2 decode at
block size B captured as one CUDA graph (per block: min(8, B/k) denoise steps of
L x bd_block_causal_attn + bd_unmask_step, top k = max(1, B/8) per step; state
and tokens never leave the device).  One replay must commit exactly what the
float64 oracle commits step by step on the same logits, and the attention
launches inside the graph must give the oracle's output."""
from fractions import Fraction

import numpy as np
import pytest

import torch

import oracle
import synth
from block_causal_masked_gb300.decode import BlockDecode
from helpers import DEV, assert_attn_close, host

pytestmark = pytest.mark.gpu
V = synth.VOCAB


def _oracle_decode(B: int):
    """Logits of every step (redrawn until the top-k cut has a margin fp32 cannot
    cross) and the oracle's final state and tokens."""
    n_blocks, steps, k = synth.WAM_TOKENS // B, synth.wam_steps(B), synth.wam_k(B)
    kw = dict(tau_full=2.0, tau_half=2.0, min_frac=Fraction(0, 1), k_fixed=k, add_thr=Fraction(1, 2),
              act_thr=Fraction(17, 20))
    logits = np.empty((n_blocks, steps, B, V), np.float32)
    state = np.zeros(synth.WAM_TOKENS, np.int64)
    tokens = np.full(synth.WAM_TOKENS, -1, np.int64)
    for b in range(n_blocks):
        sl = slice(b * B, (b + 1) * B)
        for s in range(steps):
            for attempt in range(20):
                x = synth.normal_logits(2, 100000 * B + 100 * b + 10 * s + attempt, B, V, sigma=3.0)
                o = oracle.unmask_step(x, np.arange(B), [0, B], state[sl], tokens[sl], **kw)
                if o["margins"]["rank"] >= 1e-5:
                    break
            assert o["margins"]["rank"] >= 1e-5
            logits[b, s] = x
            state[sl], tokens[sl] = o["state"], o["tokens"]
        assert (state[sl] == synth.COMMITTED).all()
    return logits, state, tokens


@pytest.mark.parametrize("B", [1, 8, 32])
def test_wam_decode_graph_matches_oracle(B):
    logits, state_ref, tokens_ref = _oracle_decode(B)
    W = synth.WAM_SWEEP
    g = torch.Generator(device=DEV)
    g.manual_seed(1000 * W.seed + B)
    kv_len = W.prefix + synth.WAM_TOKENS
    q = [torch.randn((B, W.Hq, W.D), generator=g, device=DEV).to(torch.bfloat16) for _ in range(2)]
    kk = [torch.randn((W.Hkv, kv_len, W.D), generator=g, device=DEV).to(torch.bfloat16) for _ in range(2)]
    vv = [torch.randn((W.Hkv, kv_len, W.D), generator=g, device=DEV).to(torch.bfloat16) for _ in range(2)]
    lg = torch.from_numpy(logits).to(DEV).to(torch.bfloat16)
    dec = BlockDecode(q, kk, vv, lg, W.prefix, synth.wam_k(B))
    dec.capture()
    dec.replay()
    assert int(host(dec.dev_status)[0]) == 0
    assert np.array_equal(host(dec.state).astype(np.int64), state_ref)
    assert np.array_equal(host(dec.tokens).astype(np.int64), tokens_ref)
    # the last launch of the graph: layer 1 of the last block's last step
    C = W.prefix + (dec.n_blocks - 1) * B
    q, k, v = (host(t).astype(np.float32) for t in (dec.q[1], dec.kk[1], dec.vv[1]))
    o_ref, lse_ref = oracle.block_causal_attention(q, k, v, C, [0, B])
    assert_attn_close(dec.o, dec.lse, o_ref, lse_ref, f"B={B}")
    # a second replay starts from the reset state and ends in the same place
    dec.replay()
    assert np.array_equal(host(dec.tokens).astype(np.int64), tokens_ref)
