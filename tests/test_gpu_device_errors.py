"""Device-side error paths on the GPU, without a fault or a hang.

* A bounded wait that runs out: every call takes a limit for its pipeline
  waits (wait_limit_ns); at 1 ns the first wait that does not succeed at once
  gives up, the kernel records BD_DEV_TIMEOUT, lets the copies and MMAs it has
  issued land and exits.  bd_check then reports BD_ERR_TIMEOUT, and the next
  ordinary call on the same stream (and, for the vocabulary calls, the same
  workspace) is correct.
* Inputs only the device sees as inconsistent: a block partition that is not
  increasing (unmask) and AR rows that do not match the block's editable slots
  (verify) give BD_ERR_DEVICE_INPUT.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
import oracle
import synth
from helpers import DEV, assert_attn_close, bf16, f32, host, i32, status_word, u8

pytestmark = pytest.mark.gpu

BD_OK, BD_ERR_TIMEOUT, BD_ERR_DEVICE_INPUT = 0, 5, 6
TINY = dict(tau_full=0.9, tau_half=0.9, min_frac=(1, 4), k_fixed=0, add_thr=(0, 1), act_thr=(0, 1))
TINY_F = dict(tau_full=0.9, tau_half=0.9, min_frac=Fraction(1, 4), k_fixed=0, add_thr=Fraction(0, 1),
              act_thr=Fraction(0, 1))


@pytest.mark.parametrize("splits", [1, 4])
def test_attention_wait_timeout_then_normal_call(splits):
    C, bs = 700, [0, 12, 20]
    case = synth.attn_case(60, splits, C=C, block_start=bs, Hq=16, Hkv=2, D=128)
    q, k, v, blk = bf16(case.q), bf16(case.k), bf16(case.v), i32(bs)
    ds = status_word()
    bd.bd_block_causal_attn(q, k, v, C, block_start=blk, num_splits=splits, dev_status=ds, wait_limit_ns=1)
    assert bd.bd_check(ds) == BD_ERR_TIMEOUT
    ds2 = status_word()
    o, lse = bd.bd_block_causal_attn(q, k, v, C, block_start=blk, num_splits=splits, dev_status=ds2)
    assert bd.bd_check(ds2) == BD_OK
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, "after a timed-out call")


def test_fork_with_rope_wait_timeout_then_normal_call():
    k_pos = (np.arange(600) + 256).astype(np.int32)
    f = synth.fork_case(61, 0, N=3, C=600, n_q=12, priv_len=20, block_start=[0, 12], Hq=16, Hkv=2, D=128,
                        k_pos=k_pos, delta=256, theta=1e4)
    args = (bf16(f.q), bf16(f.prefix_k), bf16(f.prefix_v), bf16(f.priv_k), bf16(f.priv_v), f.priv_len, f.C)
    rope = dict(k_pos=i32(k_pos), delta=256, theta=1e4)
    ds = status_word()
    bd.bd_fork_rollouts(*args, block_start=i32(f.block_start), rope=rope, dev_status=ds, wait_limit_ns=1)
    assert bd.bd_check(ds) == BD_ERR_TIMEOUT
    ds2 = status_word()
    o, lse = bd.bd_fork_rollouts(*args, block_start=i32(f.block_start), rope=rope, dev_status=ds2)
    assert bd.bd_check(ds2) == BD_OK
    o_ref, lse_ref = oracle.fork_attention(f.q, f.prefix_k, f.prefix_v, f.priv_k, f.priv_v, f.priv_len,
                                           f.block_start, k_pos=k_pos, delta=256, theta=1e4, rope=True)
    assert_attn_close(o, lse, o_ref, lse_ref, "fork after a timed-out call")


def _tiny_unmask_inputs():
    lay = synth.uniform_layout(16, 8, 3, seed=0)
    state = np.where(lay.scaffold == 1, synth.SCAFFOLD, synth.MASKED)
    tokens = np.where(lay.scaffold == 1, 7, -1)
    logits = synth.normal_logits(0, 0, 16, 1024, sigma=2.0, bf16=False)
    return lay, state, tokens, logits


def test_unmask_wait_timeout_then_normal_call():
    lay, state, tokens, logits = _tiny_unmask_inputs()
    big = synth.normal_logits(62, 0, 32, synth.VOCAB)             # long rows: many pieces per CTA
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)       # one workspace for both calls
    ds = status_word()
    bs32 = i32([0, 32])
    bd.bd_unmask_step(bf16(big), i32(np.arange(32)), bs32, u8(np.zeros(32)), i32(np.full(32, -1)), **TINY,
                      workspace=ws, dev_status=ds, wait_limit_ns=1)
    assert bd.bd_check(ds) == BD_ERR_TIMEOUT
    ref = oracle.unmask_step(logits, np.arange(16), lay.block_start, state, tokens, **TINY_F)
    st, tk = u8(state), i32(tokens)
    ds2 = status_word()
    r = bd.bd_unmask_step(f32(logits), i32(np.arange(16)), i32(lay.block_start), st, tk, **TINY, workspace=ws,
                          dev_status=ds2)
    assert bd.bd_check(ds2) == BD_OK
    assert np.array_equal(host(st), ref["state"]) and np.array_equal(host(tk), ref["tokens"])
    assert np.array_equal(host(r["commit"]), ref["commit"])


def test_verify_wait_timeout_then_normal_call():
    draft = synth.rng(63, 1).integers(0, synth.VOCAB, size=32)
    want = draft.copy()
    want[9] = (want[9] + 1) % synth.VOCAB
    ar, _, _ = synth.planted_logits(63, 3, 33, synth.VOCAB, tokens=np.concatenate([want, [3]]))
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    ds = status_word()
    bd.bd_spec_verify(i32(draft[None]), torch.zeros((1, 32), dtype=torch.uint8, device=DEV), bf16(ar[None]),
                      workspace=ws, dev_status=ds, wait_limit_ns=1)
    assert bd.bd_check(ds) == BD_ERR_TIMEOUT
    ref = oracle.spec_verify(draft[None], np.zeros((1, 32)), ar[None])
    tk = i32(draft[None])
    ds2 = status_word()
    acc, bon, _ = bd.bd_spec_verify(tk, torch.zeros((1, 32), dtype=torch.uint8, device=DEV), bf16(ar[None]),
                                    workspace=ws, dev_status=ds2)
    assert bd.bd_check(ds2) == BD_OK
    assert int(acc[0]) == int(ref["accepted_len"][0]) == 10 and int(bon[0]) == int(ref["bonus"][0])
    assert np.array_equal(host(tk), ref["tokens"])


def test_unmask_inconsistent_partition_is_reported():
    """block_start [0, 10, 6, 16] is not increasing: the deciding CTA refuses to
    apply the commit rule, reports BD_ERR_DEVICE_INPUT and leaves state and
    tokens as they were; the workspace stays usable."""
    lay, state, tokens, logits = _tiny_unmask_inputs()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    st, tk = u8(state), i32(tokens)
    ds = status_word()
    bd.bd_unmask_step(f32(logits), i32(np.arange(16)), i32([0, 10, 6, 16]), st, tk, **TINY, workspace=ws,
                      dev_status=ds)
    assert bd.bd_check(ds) == BD_ERR_DEVICE_INPUT
    assert np.array_equal(host(st), state) and np.array_equal(host(tk), tokens)
    ref = oracle.unmask_step(logits, np.arange(16), lay.block_start, state, tokens, **TINY_F)
    ds2 = status_word()
    bd.bd_unmask_step(f32(logits), i32(np.arange(16)), i32(lay.block_start), st, tk, **TINY, workspace=ws,
                      dev_status=ds2)
    assert bd.bd_check(ds2) == BD_OK
    assert np.array_equal(host(st), ref["state"]) and np.array_equal(host(tk), ref["tokens"])


def test_verify_row_count_mismatch_is_reported():
    """The block has 12 editable slots, so the AR pass must supply 13 rows;
    12 rows give BD_ERR_DEVICE_INPUT."""
    L = 16
    scaf = np.zeros(L, np.int64)
    scaf[[1, 5, 9, 13]] = 1
    state = np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED).astype(np.uint8)
    draft = synth.rng(64, 1).integers(0, 1024, size=L)
    ar = synth.normal_logits(64, 2, 12, 1024, sigma=2.0, bf16=False)
    ds = status_word()
    bd.bd_spec_verify(i32(draft[None]), u8(state[None]), f32(ar[None]), dev_status=ds)
    assert bd.bd_check(ds) == BD_ERR_DEVICE_INPUT
