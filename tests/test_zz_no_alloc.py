"""The allocation-free unmask entry point, for callers that cannot allocate
device memory (a runtime whose memory plan is fixed at start-up, a plug-in host
that hands over only inputs and outputs): bd_unmask_step_noalloc, called through
the C ABI, must give what bd_unmask_step gives with a caller workspace -- on two
calls in a row, of different shapes, that share the library's scratch array.

Kept in a file that pytest collects last, so that a run stopping at its first
failure has run every other test before this one."""
import ctypes as ct

import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
import synth
from helpers import CONF_RTOL, bf16, f32, host, i32, status_word, u8

pytestmark = pytest.mark.gpu


def _args(logits, logit_row, bs, state, tokens, outs, tau):
    a = bd.bd_unmask_args()
    R, V = logits.shape
    a.logits = logits.data_ptr()
    a.logits_dtype = bd.BD_BF16 if logits.dtype == torch.bfloat16 else bd.BD_F32
    a.logits_ld = logits.stride(0)
    a.R, a.V = R, V
    a.logit_row, a.n_pos = logit_row.data_ptr(), state.numel()
    a.block_start, a.n_blocks = bs.data_ptr(), bs.numel() - 1
    a.state, a.tokens = state.data_ptr(), tokens.data_ptr()
    a.tau_full = a.tau_half = tau
    a.min_num, a.min_den, a.k_fixed = 1, 4, 0
    a.add_num, a.add_den, a.act_num, a.act_den = 1, 2, 17, 20
    a.commit, a.n_committed, a.status = outs["commit"].data_ptr(), outs["n_committed"].data_ptr(), \
        outs["status"].data_ptr()
    a.pred, a.conf, a.lse = outs["pred"].data_ptr(), outs["conf"].data_ptr(), outs["lse"].data_ptr()
    a.write_draft = 1
    return a


def _outs(n_pos, n_blocks):
    dev = "cuda:0"
    return dict(commit=torch.empty(n_pos, dtype=torch.uint8, device=dev),
                n_committed=torch.empty(n_blocks, dtype=torch.int32, device=dev),
                status=torch.empty(n_blocks, dtype=torch.int32, device=dev),
                pred=torch.empty(n_pos, dtype=torch.int32, device=dev),
                conf=torch.empty(n_pos, dtype=torch.float32, device=dev),
                lse=torch.empty(n_pos, dtype=torch.float32, device=dev))


def _cases():
    # 1: the Fast-dDrive active block, bf16 [32, 151936] with planted peaks
    lay = synth.section_layout(1)
    lo, hi = lay.block_start[2], lay.block_start[3]
    scaf = lay.scaffold[lo:hi]
    n = hi - lo
    E = int((scaf == 0).sum())
    x, _, _ = synth.planted_logits(31, 0, E, synth.VOCAB)
    lr = np.full(n, -1)
    lr[scaf == 0] = np.arange(E)
    yield bf16(x), lr, [0, n], np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED), 0.9
    # 2: the tiny workload, fp32 [16, 1024], two blocks of 8 with 3 scaffold each
    lay = synth.uniform_layout(16, 8, 3, seed=0)
    x = synth.normal_logits(0, 5, 16, 1024, sigma=2.0, bf16=False)
    yield f32(x), np.arange(16), list(lay.block_start), np.where(lay.scaffold == 1, synth.SCAFFOLD, synth.MASKED), 0.9


def test_noalloc_unmask_equals_workspace_unmask_on_two_calls():
    L = bd.lib()
    L.bd_unmask_step_noalloc.argtypes = [ct.POINTER(bd.bd_unmask_args), ct.c_void_p]
    L.bd_unmask_step_noalloc.restype = ct.c_int
    stream = ct.c_void_p(torch.cuda.current_stream().cuda_stream)
    for logits, lr, bs, state0, tau in _cases():
        n_pos, n_blocks = len(state0), len(bs) - 1
        res = []
        for noalloc in (False, True):
            st, tk = u8(state0), i32(np.full(n_pos, -1))
            lr_d, bs_d = i32(lr), i32(bs)   # kept alive: the struct holds raw pointers only
            outs = _outs(n_pos, n_blocks)
            a = _args(logits, lr_d, bs_d, st, tk, outs, tau)
            ds = status_word()
            a.dev_status = ds.data_ptr()
            if noalloc:
                assert L.bd_unmask_step_noalloc(a, stream) == 0
            else:
                ws = torch.zeros(L.bd_unmask_workspace_size(a), dtype=torch.uint8, device="cuda:0")
                a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
                assert L.bd_unmask_step(a, stream) == 0
            assert bd.bd_check(ds) == 0
            res.append({k: host(v) for k, v in outs.items()} | dict(state=host(st), tokens=host(tk)))
        ref, got = res
        for k in ("commit", "n_committed", "status", "pred", "state", "tokens"):
            assert np.array_equal(ref[k], got[k]), k
        cand = ref["pred"] >= 0
        np.testing.assert_allclose(got["conf"][cand], ref["conf"][cand], rtol=CONF_RTOL, atol=0)
        np.testing.assert_allclose(got["lse"][cand], ref["lse"][cand], rtol=1e-6, atol=1e-6)


def test_noalloc_refuses_problems_beyond_its_scratch():
    L = bd.lib()
    a = bd.bd_unmask_args()
    # the partials of 65,535 logits rows (the most one call takes) need more than the scratch
    a.R, a.V, a.n_pos, a.n_blocks, a.logits_ld = 65535, 151936, 2048, 1, 151936
    a.min_den, a.add_den, a.act_den = 4, 2, 20
    assert L.bd_unmask_workspace_size(a) > (1 << 20)
    L.bd_unmask_step_noalloc.argtypes = [ct.POINTER(bd.bd_unmask_args), ct.c_void_p]
    assert L.bd_unmask_step_noalloc(a, None) == 3   # BD_ERR_WORKSPACE
