"""Device-resident decode drivers: sequences of the library's C-ABI calls on the
current stream, captured as CUDA graphs.  Nothing here computes: every step of
the decode runs in libbd's kernels, and these classes only hold the device
buffers, order the calls and replay them.

SpeculativeRound
    One scaffold-speculative round on one active block (Fast-dDrive method
    summary, §3.2 "模式二", steps 1-3): L x bd_block_causal_attn over the block
    (the MDM pass, the block bidirectional), bd_unmask_step (commits at the
    confidence threshold, draft of the still-masked editable positions),
    L x bd_block_causal_attn again with block size 1 (the AR pass, causal),
    and bd_spec_verify (left-to-right match of the draft, bonus token).
BlockDecode
    A whole block-wise decode (WAM-Diff2 write-up, §三 系统级加速: fixed
    denoising steps per block, the launches captured as CUDA graphs): every
    block of B positions gets `steps` denoise steps, each L x
    bd_block_causal_attn (prefix = the prompt plus the blocks decoded so far)
    and one bd_unmask_step committing the top k by confidence.  Block state and
    tokens stay on the device, and the decode replays as ONE CUDA graph with no
    host round trip between steps.

The attention calls declare the cached prefix ready (``prefix_ready``): the KV
cache of a decode step is written before the step, never inside it.
"""
from __future__ import annotations

import torch

from . import (MASKED, bd_block_causal_attn, bd_spec_verify, bd_unmask_step)

__all__ = ["SpeculativeRound", "BlockDecode"]


def _capture(fn, stream) -> torch.cuda.CUDAGraph:
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


class SpeculativeRound:
    """One scaffold-speculative round on the active block.

    q, q_ar   lists of L bf16 [n_q, Hq, D]: each layer's queries of the MDM and
              of the AR pass
    k, v      lists of L bf16 [Hkv, >= C + n_q, D]: each layer's cache (rows
              [0, C)) and the block's own keys / values (rows [C, C + n_q))
    C         cached keys before the block
    logits    [E, V] bf16 or fp32: the MDM logits of the block's editable rows
    ar_logits [E + 1, V]: the AR logits (row e predicts the e-th editable slot,
              row E the position after the block)
    logit_row int32 [n_q]: logits row of each position, -1 for scaffold
    state0, tokens0   uint8 / int32 [n_q]: the block at the start of the round
    tau       confidence threshold of the MDM commits
    """

    def __init__(self, q, q_ar, k, v, C: int, logits, ar_logits, logit_row, state0, tokens0, tau: float):
        self.q, self.q_ar, self.k, self.v = list(q), list(q_ar), list(k), list(v)
        self.layers = len(self.q)
        self.C = int(C)
        n_q, Hq, D = self.q[0].shape
        dev = self.q[0].device
        self.n_q = n_q
        self.tau = float(tau)
        self.o = torch.empty((n_q, Hq, D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((Hq, n_q), dtype=torch.float32, device=dev)
        self.block = torch.tensor([0, n_q], dtype=torch.int32, device=dev)
        self.logits = logits
        self.ar_logits = ar_logits if ar_logits.dim() == 3 else ar_logits[None]
        self.logit_row = logit_row
        self.state0, self.tokens0 = state0, tokens0
        self.state, self.tokens = state0.clone(), tokens0.clone()
        self.um = dict(commit=torch.empty(n_q, dtype=torch.uint8, device=dev),
                       n_committed=torch.empty(1, dtype=torch.int32, device=dev),
                       status=torch.empty(1, dtype=torch.int32, device=dev),
                       pred=torch.empty(n_q, dtype=torch.int32, device=dev),
                       conf=torch.empty(n_q, dtype=torch.float32, device=dev),
                       lse=torch.empty(n_q, dtype=torch.float32, device=dev))
        self.acc = torch.empty(1, dtype=torch.int32, device=dev)
        self.bonus = torch.empty(1, dtype=torch.int32, device=dev)
        self.bonus_pos = torch.empty(1, dtype=torch.int32, device=dev)
        self.whole = None
        self.graphs = []

    # the four parts of a round, each a sequence of C-ABI calls on the current stream
    def mdm(self):
        for l in range(self.layers):
            bd_block_causal_attn(self.q[l], self.k[l], self.v[l], self.C, block_start=self.block, o=self.o,
                                 lse=self.lse, prefix_ready=True)

    def unmask(self):
        bd_unmask_step(self.logits, self.logit_row, self.block, self.state, self.tokens, tau_full=self.tau,
                       tau_half=self.tau, min_frac=(0, 1), k_fixed=0, write_draft=True, **self.um)

    def ar(self):
        for l in range(self.layers):
            bd_block_causal_attn(self.q_ar[l], self.k[l], self.v[l], self.C, block_size=1, o=self.o,
                                 lse=self.lse, prefix_ready=True)

    def verify(self):
        bd_spec_verify(self.tokens.view(1, -1), self.state.view(1, -1), self.ar_logits, accepted_len=self.acc,
                       bonus=self.bonus, bonus_pos=self.bonus_pos)

    def run(self):
        self.mdm()
        self.unmask()
        self.ar()
        self.verify()

    def reset(self):
        """The block back to its state at the start of the round."""
        self.state.copy_(self.state0)
        self.tokens.copy_(self.tokens0)

    def committed(self) -> int:
        """Editable positions committed by the last round (unmask commits +
        accepted length); reads the device."""
        return int(self.um["n_committed"][0]) + int(self.acc[0])

    def capture(self):
        """Captures the round as one CUDA graph (``whole``: consecutive
        launches overlap through programmatic dependent launch across the part
        boundaries too) and as four graphs, one per part (``graphs``).  The
        round runs once first, outside the capture, to size the workspaces and
        set the kernels' attributes."""
        self.reset()
        self.run()
        torch.cuda.synchronize()
        s = torch.cuda.Stream(self.q[0].device)
        self.graphs = []
        for part in (self.mdm, self.unmask, self.ar, self.verify):
            self.reset()
            torch.cuda.synchronize()
            self.graphs.append(_capture(part, s))
        self.reset()
        torch.cuda.synchronize()
        self.whole = _capture(self.run, s)
        torch.cuda.synchronize()

    def replay(self):
        self.reset()
        self.whole.replay()


class BlockDecode:
    """A whole block-wise decode as one CUDA graph.

    q         list of L bf16 [B, Hq, D]: each layer's queries of the active block
    k, v      lists of L bf16 [Hkv, >= prefix + n_blocks * B, D]: the prompt's
              cache (rows [0, prefix)) followed by the output positions' keys /
              values, block b at rows [prefix + b B, prefix + (b + 1) B)
    logits    bf16 [n_blocks, steps, B, V]: the logits of every denoise step
    prefix    cached prompt keys
    k_fixed   commits per step (the top k by confidence; tau disabled)
    dev_status  optional int32 [1] device status word shared by every call
    """

    def __init__(self, q, k, v, logits, prefix: int, k_fixed: int, dev_status=None, num_splits: int = 0):
        self.q, self.kk, self.vv = list(q), list(k), list(v)
        self.layers = len(self.q)
        self.B, Hq, D = self.q[0].shape
        self.n_blocks, self.steps = int(logits.shape[0]), int(logits.shape[1])
        assert logits.shape[2] == self.B
        self.tokens_total = self.n_blocks * self.B
        self.logits = logits
        self.prefix, self.k = int(prefix), int(k_fixed)
        self.num_splits = num_splits
        dev = self.q[0].device
        self.o = torch.empty((self.B, Hq, D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((Hq, self.B), dtype=torch.float32, device=dev)
        self.block = torch.tensor([0, self.B], dtype=torch.int32, device=dev)
        self.logit_row = torch.arange(self.B, dtype=torch.int32, device=dev)
        self.state = torch.zeros(self.tokens_total, dtype=torch.uint8, device=dev)
        self.tokens = torch.full((self.tokens_total,), -1, dtype=torch.int32, device=dev)
        self.um = dict(commit=torch.empty(self.B, dtype=torch.uint8, device=dev),
                       n_committed=torch.empty(1, dtype=torch.int32, device=dev),
                       status=torch.empty(1, dtype=torch.int32, device=dev),
                       pred=torch.empty(self.B, dtype=torch.int32, device=dev),
                       conf=torch.empty(self.B, dtype=torch.float32, device=dev),
                       lse=torch.empty(self.B, dtype=torch.float32, device=dev))
        self.dev_status = dev_status if dev_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches = self.n_blocks * self.steps * (self.layers + 1)
        self.graph = None

    def step(self, b: int, s: int):
        """Denoise step s of block b: the attention layers, then the commits."""
        B = self.B
        C = self.prefix + b * B
        for l in range(self.layers):
            bd_block_causal_attn(self.q[l], self.kk[l], self.vv[l], C, block_start=self.block, o=self.o,
                                 lse=self.lse, num_splits=self.num_splits, dev_status=self.dev_status,
                                 prefix_ready=True)
        bd_unmask_step(self.logits[b, s], self.logit_row, self.block, self.state[b * B:(b + 1) * B],
                       self.tokens[b * B:(b + 1) * B], tau_full=2.0, tau_half=2.0, min_frac=(0, 1),
                       k_fixed=self.k, add_thr=(1, 2), act_thr=(17, 20), dev_status=self.dev_status, **self.um)

    def reset(self):
        self.state.fill_(MASKED)
        self.tokens.fill_(-1)

    def capture(self):
        """Captures every step of every block as one graph (one step runs
        first, outside the capture, to size the workspaces)."""
        self.step(0, 0)
        torch.cuda.synchronize()
        self.reset()
        s = torch.cuda.Stream(self.q[0].device)

        def all_steps():
            for b in range(self.n_blocks):
                for st in range(self.steps):
                    self.step(b, st)
        self.graph = _capture(all_steps, s)
        torch.cuda.synchronize()

    def replay(self):
        self.reset()
        self.graph.replay()
