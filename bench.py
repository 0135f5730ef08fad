#!/usr/bin/env python3
"""Committed tokens/s of one block-causal masked-diffusion decode round on GB300.

Workload (Fast-dDrive-shaped, seed 1): 16 query / 2 KV heads, head dim 128, bf16,
36 layers; cached prefix = 3,000 tokens (2,700 image-like + 300 text-like) plus
the blocks already decoded (the 92-position critical-objects block and the first
32-position explanation block) = 3,124 keys; active block = the second
explanation block of the 404-position scaffolded output (33 positions: 32
editable + 1 scaffold); vocabulary 151,936.

One step = one scaffold-speculative round on the active block, all through the
library's C ABI (the attention calls declare the cached prefix ready, so each
launch starts fetching it while the previous kernel finishes: the KV cache is
written before a round, never inside it):
  36 x bd_block_causal_attn   (MDM forward, the block bidirectional)
  1  x bd_unmask_step         (argmax / confidence of the 32 editable rows, tau =
                               0.9 commits, draft of the rest)
  36 x bd_block_causal_attn   (AR forward: block size 1, causal)
  1  x bd_spec_verify         (left-to-right match of the draft + bonus token)
committed tokens = unmask commits + verify's accepted length.  The step is
captured as one CUDA graph and timed with CUDA events around its replay; the
per-kernel times of the roofline come from the same round replayed as four
graphs with events between them.  L2 is flushed (256 MiB write) before every
timed step, outside the timed region.

--impl reference runs the float64 CPU oracle on the same inputs instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "committed tokens/s per denoise step; attn & unmask % of HBM/tensor roofline"
UNIT = "tokens/s"
W = synth.FAST_DDRIVE
TAU = synth.DDRIVE_TAU
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------------------ GPU arm

def make_inputs(seed: int) -> dict:
    """Seeded host inputs of one Fast-dDrive-shaped round (synth.fast_ddrive_round)."""
    return synth.fast_ddrive_round(seed)


def gpu_round(inp, device):
    """The library's SpeculativeRound on the workload's inputs, uploaded to the
    device, with a 256 MiB buffer for flushing L2 between timed steps."""
    import torch
    from block_causal_masked_gb300.decode import SpeculativeRound
    t = lambda x, dt: torch.from_numpy(np.array(x, order="C", copy=True)).to(device).to(dt)  # noqa: E731
    bf = torch.bfloat16
    rd = SpeculativeRound([t(q, bf) for q, _, _, _ in inp["layers"]], [t(q, bf) for _, q, _, _ in inp["layers"]],
                          [t(k, bf) for _, _, k, _ in inp["layers"]], [t(v, bf) for _, _, _, v in inp["layers"]],
                          inp["C"], t(inp["logits"], bf), t(inp["ar_logits"][None], bf),
                          t(inp["logit_row"], torch.int32), t(inp["state"], torch.uint8),
                          t(inp["tokens"], torch.int32), TAU)
    rd.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    return rd


def timed_step(rd) -> float:
    """Replays the round (one graph) after an L2 flush; returns its ms."""
    import torch
    rd.reset()
    rd.flush.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    rd.whole.replay()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1)


def timed_parts(rd):
    """Replays the round as its four part graphs with events between them,
    after an L2 flush; returns (step ms, attention ms, unmask ms)."""
    import torch
    rd.reset()
    rd.flush.zero_()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    torch.cuda.synchronize()
    ev[0].record()
    for i, g in enumerate(rd.graphs):
        g.replay()
        ev[i + 1].record()
    ev[4].synchronize()
    tt = [ev[0].elapsed_time(ev[i + 1]) for i in range(4)]
    return tt[3], tt[0] + (tt[2] - tt[1]), tt[1] - tt[0]


def planned_splits(C: int, n_q: int, Hq: int, Hkv: int, D: int) -> int:
    """KV split count the library plans for a plain attention call, read back
    from its workspace size (Hkv x row tiles x S x S owner slices of r(S) rows
    of D bf16 values; none for one split)."""
    import block_causal_masked_gb300 as bd
    a = bd.bd_attn_args()
    a.q = a.k = a.v = a.o = 1 << 20
    a.C, a.n_q, a.Hq, a.Hkv, a.D, a.kv_stride, a.block_size = C, n_q, Hq, Hkv, D, C + n_q, n_q
    ws = bd.lib().bd_attn_workspace_size(a)
    m_tiles = -(-n_q * (Hq // Hkv) // 128)
    for S in range(2, 17):
        r = ((128 + S - 1) // S + 1) & ~1
        if ws == Hkv * m_tiles * S * S * r * 2 * D:
            return S
    return 1


# ------------------------------------------------------------------------------ device-resident decode

WAM = synth.WAM_SWEEP
WAM_TOKENS = synth.WAM_TOKENS


def wam_decode(B: int, layers: int, device, logits=None, seed: int = WAM.seed, num_splits: int = 0):
    """The library's BlockDecode on the WAM-Diff2 sweep at block size B: 16/8
    heads, head dim 128, prompt prefix 2,048, 256 output tokens, top
    synth.wam_k(B) per step, synth.wam_steps(B) steps per block.  Queries and
    the cache are drawn on the device from a seeded generator; logits: float32
    host array [n_blocks, steps, B, V] of bf16 values, or None for seeded
    N(0, 3) rows drawn on the device."""
    import torch
    from block_causal_masked_gb300.decode import BlockDecode
    n_blocks, steps = WAM_TOKENS // B, synth.wam_steps(B)
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + B)
    bf = torch.bfloat16
    kv_len = WAM.prefix + WAM_TOKENS
    q = [torch.randn((B, WAM.Hq, WAM.D), generator=g, device=device).to(bf) for _ in range(layers)]
    kk = [torch.randn((WAM.Hkv, kv_len, WAM.D), generator=g, device=device).to(bf) for _ in range(layers)]
    vv = [torch.randn((WAM.Hkv, kv_len, WAM.D), generator=g, device=device).to(bf) for _ in range(layers)]
    if logits is None:
        lg = (torch.randn((n_blocks, steps, B, synth.VOCAB), generator=g, device=device) * 3.0).to(bf)
    else:
        lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(device).to(bf)
    return BlockDecode(q, kk, vv, lg, WAM.prefix, synth.wam_k(B), num_splits=num_splits)


def run_wam_sweep(args, device):
    """One line per block size: committed tokens/s of the whole decode (one
    CUDA graph), with the per-launch roofline of its attention (at the
    decode's midpoint, prefix 2,048 + 128) and unmask kernels."""
    import torch
    import block_causal_masked_gb300 as bd
    torch.cuda.set_device(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    peaks = measured_peaks()
    lines = []
    for B in (1, 4, 8, 16, 32):
        dec = wam_decode(B, WAM.layers, device)
        t0 = time.time()
        dec.capture()
        cap_s = time.time() - t0
        for _ in range(args.warmup):
            dec.replay()
        torch.cuda.synchronize()
        t = _replay_ms(dec.graph, args.steps, flush, before=dec.reset)
        dec.replay()
        torch.cuda.synchronize()
        committed = int((dec.state == synth.COMMITTED).sum())
        status = int(dec.dev_status[0])
        # per-launch kernel times: one step's 36 attention layers at the
        # decode's midpoint, and 16 independent unmask calls on fresh blocks
        C = WAM.prefix + (dec.n_blocks // 2) * B

        def attn_layers():
            for l in range(WAM.layers):
                bd.bd_block_causal_attn(dec.q[l], dec.kk[l], dec.vv[l], C, block_start=dec.block, o=dec.o,
                                        lse=dec.lse, prefix_ready=True)
        attn_us = _replay_ms(_graph(attn_layers), args.steps, flush) * 1e3 / WAM.layers
        copies = 16
        win = _Window(np.zeros(B), np.full(B, -1), copies, device)
        lgs = [dec.logits[0, 0].clone() for _ in range(copies)]
        outs = [_unmask_outs(B, 1, device) for _ in range(copies)]

        def unmask(i):
            bd.bd_unmask_step(lgs[i], dec.logit_row, dec.block, win.state[i], win.tokens[i], tau_full=2.0,
                              tau_half=2.0, min_frac=(0, 1), k_fixed=dec.k, add_thr=(1, 2), act_thr=(17, 20),
                              **outs[i])
        um_us = _per_launch_us([lambda i=i: unmask(i) for i in range(copies)], win.reset, flush, args.steps)
        nbytes = 2 * WAM.Hkv * (C + B) * WAM.D * 2 + 2 * B * WAM.Hq * WAM.D * 2 + B * WAM.Hq * 4
        kernels = {"attn_kernel": _attn_roof(attn_us, nbytes, 4 * WAM.D * WAM.Hq * B * (C + B), peaks, True),
                   "unmask_kernel": _vocab_roof(um_us, B * synth.VOCAB * 2, peaks)}
        lines.append({"metric": "committed tokens/s (whole decode, one CUDA graph)", "value": committed / t * 1e3,
                      "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_decode": t, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": f"wam_diff2_sweep B={B}: {WAM_TOKENS} tokens, blocks of {B}, top "
                                             f"{dec.k} per step, {dec.steps} steps per block, 16/8 heads, "
                                             f"head dim 128, {WAM.layers} layers, prefix {WAM.prefix}",
                                 "gpu_launches_per_decode": dec.launches, "graph_capture_s": round(cap_s, 2),
                                 "l2": "flushed before every timed decode"},
                      "committed": committed, "dev_status": status, "roofline": kernels})
        del dec, lgs, outs, win
        torch.cuda.empty_cache()
    return lines


# ------------------------------------------------------------------------------ the other workloads

def _graph(fn):
    """fn's launches captured as one CUDA graph (fn runs once first, outside the
    capture, to size workspaces and set kernel attributes)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        fn()
    torch.cuda.synchronize()
    return g


def _replay_ms(g, reps: int, flush, before=None):
    """Median CUDA-event time of `reps` replays, L2 flushed (and `before` run)
    outside the timed region before each."""
    import torch
    ms = []
    for _ in range(reps):
        if before is not None:
            before()
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms)


def _copies(bytes_per_call: int) -> int:
    """Independent input copies for timing a vocabulary kernel back to back:
    enough that the copies together exceed L2, at most 16, at most ~2 GB."""
    return int(max(1, min(16, (2 << 30) // max(1, bytes_per_call))))


def _attn_visible(C: int, block_start, causal: bool = False) -> int:
    """Visible keys summed over the active positions (block-causal, or causal)."""
    n_q = int(block_start[-1])
    if causal:
        return sum(C + i + 1 for i in range(n_q))
    tot = 0
    for b in range(len(block_start) - 1):
        lo, hi = int(block_start[b]), int(block_start[b + 1])
        tot += (hi - lo) * (C + hi)
    return tot


def _attn_roof(us: float, nbytes: float, flops: float, peaks, sustained: bool):
    """Roofline entry of one attention launch: HBM or tensor bound, whichever
    bound is slower at the measured peaks."""
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    tf = (peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops") if peaks else None) or \
        (1700.0 if sustained else 1900.0)
    t_hbm = nbytes / (hbm * 1e9)
    t_tc = flops / (tf * 1e12)
    if t_tc > t_hbm:
        ach = flops / (us * 1e-6) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tf, "unit": "TFLOP/s", "frac": ach / tf,
                "alg_flops_per_launch": flops, "alg_bytes_per_launch": nbytes, "avg_launch_us": us}
    ach = nbytes / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "alg_flops_per_launch": flops, "alg_bytes_per_launch": nbytes, "avg_launch_us": us}


def _vocab_roof(us: float, nbytes: float, peaks):
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    ach = nbytes / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "alg_bytes_per_launch": nbytes, "avg_launch_us": us}


def _extra_line(workload: str, tokens_per_step: float, step_ms: float, args, kernels: dict, extra: dict):
    line = {"metric": METRIC, "value": tokens_per_step / step_ms * 1e3, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload, "l2": "flushed (256 MiB write) before every timed step",
                       "timing": "median of CUDA-event timed graph replays"},
            "committed_per_step": tokens_per_step, "roofline": kernels}
    line.update(extra)
    return line


class _Window:
    """State and tokens of one decode window on the device, `copies` times
    (independent copies for timing a vocabulary kernel back to back), reset to
    their initial values outside timed regions."""

    def __init__(self, state0: np.ndarray, tokens0: np.ndarray, copies: int, dev):
        import torch
        self.s0 = torch.from_numpy(np.ascontiguousarray(state0, dtype=np.uint8)).to(dev)
        self.t0 = torch.from_numpy(np.ascontiguousarray(tokens0, dtype=np.int32)).to(dev)
        self.state = [self.s0.clone() for _ in range(copies)]
        self.tokens = [self.t0.clone() for _ in range(copies)]

    def reset(self):
        for s, t in zip(self.state, self.tokens):
            s.copy_(self.s0)
            t.copy_(self.t0)


def _unmask_outs(n_pos: int, n_blocks: int, dev):
    import torch
    return dict(commit=torch.empty(n_pos, dtype=torch.uint8, device=dev),
                n_committed=torch.empty(n_blocks, dtype=torch.int32, device=dev),
                status=torch.empty(n_blocks, dtype=torch.int32, device=dev),
                pred=torch.empty(n_pos, dtype=torch.int32, device=dev),
                conf=torch.empty(n_pos, dtype=torch.float32, device=dev),
                lse=torch.empty(n_pos, dtype=torch.float32, device=dev))


def _per_launch_us(calls, reset, flush, reps: int) -> float:
    """Per-launch time of `calls` (independent launches, own inputs and outputs
    each) captured back to back in one graph."""
    def run():
        for c in calls:
            c()
    g = _graph(run)
    return _replay_ms(g, reps, flush, before=reset) * 1e3 / len(calls)


def run_tiny(args, dev):
    """Tiny workload, one round: block-causal attention (1 layer, 4/2 heads,
    head dim 64, prefix 256, two blocks of 8 with 3 scaffold each), unmask of the
    16 positions (fp32 logits [16, 1024] ~ N(0, 2), tau 0.9, at least 1/4 of the
    remaining per block, draft of the rest), causal AR attention, verify of the
    draft against AR rows [11, 1024] that agree with it on a seeded prefix."""
    import torch
    import block_causal_masked_gb300 as bd
    T = synth.TINY
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    lay = synth.uniform_layout(16, 8, scaffold_per_block=3, seed=T.seed)
    bs = [0, 8, 16]
    a = synth.attn_case(T.seed, 0, C=T.prefix, block_start=bs, Hq=T.Hq, Hkv=T.Hkv, D=T.D)
    q_ar = synth.attn_case(T.seed, 1000, C=0, block_start=bs, Hq=T.Hq, Hkv=1, D=T.D).q
    logits = synth.normal_logits(T.seed, 1, 16, T.V, sigma=2.0, bf16=False)
    edit = np.flatnonzero(lay.scaffold == 0)
    E = len(edit)
    g = synth.rng(T.seed, 77)
    k = int(g.integers(0, E + 1))
    want = g.integers(0, T.V, size=E + 1)
    want[:k] = np.argmax(logits[edit], axis=1)[:k]          # the draft's tokens on a seeded prefix
    if k < E:
        want[k] = (np.argmax(logits[edit[k]]) + 1) % T.V
    ar, _, _ = synth.planted_logits(T.seed, 2, E + 1, T.V, sigma=2.0, tokens=want, bf16=False)
    state0 = np.where(lay.scaffold == 1, synth.SCAFFOLD, synth.MASKED)
    tokens0 = np.where(lay.scaffold == 1, 11, -1)
    t = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(dt)  # noqa: E731
    bf = torch.bfloat16
    q, k_, v, qa = t(a.q, bf), t(a.k, bf), t(a.v, bf), t(q_ar, bf)
    lg, arl = t(logits, torch.float32), t(ar[None], torch.float32)
    blk = torch.tensor(bs, dtype=torch.int32, device=dev)
    row = torch.arange(16, dtype=torch.int32, device=dev)
    copies = 16
    win = _Window(state0, tokens0, copies, dev)
    outs = [_unmask_outs(16, 2, dev) for _ in range(copies)]
    acc = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(copies)]
    o = torch.empty((16, T.Hq, T.D), dtype=bf, device=dev)
    lse = torch.empty((T.Hq, 16), dtype=torch.float32, device=dev)
    kw = dict(tau_full=0.9, tau_half=0.9, min_frac=(1, 4), k_fixed=0, add_thr=(0, 1), act_thr=(0, 1),
              write_draft=True)

    def attn_mdm():
        bd.bd_block_causal_attn(q, k_, v, T.prefix, block_start=blk, o=o, lse=lse, prefix_ready=True)

    def attn_ar():
        bd.bd_block_causal_attn(qa, k_, v, T.prefix, block_size=1, o=o, lse=lse, prefix_ready=True)

    def unmask(i=0):
        bd.bd_unmask_step(lg, row, blk, win.state[i], win.tokens[i], **kw, **outs[i])

    def verify(i=0):
        bd.bd_spec_verify(win.tokens[i].view(1, -1), win.state[i].view(1, -1), arl, accepted_len=acc[i])

    round_g = _graph(lambda: (attn_mdm(), unmask(), attn_ar(), verify()))
    for _ in range(args.warmup):
        win.reset()
        round_g.replay()
    step_ms = _replay_ms(round_g, args.steps, flush, before=win.reset)
    committed = int(outs[0]["n_committed"].sum()) + int(acc[0][0])
    attn_us = _replay_ms(_graph(lambda: (attn_mdm(), attn_ar())), args.steps, flush) * 1e3 / 2
    um_us = _per_launch_us([lambda i=i: unmask(i) for i in range(copies)], win.reset, flush, args.steps)
    vf_us = _per_launch_us([lambda i=i: verify(i) for i in range(copies)], win.reset, flush, args.steps)
    peaks = measured_peaks()
    vis = (_attn_visible(T.prefix, bs) + _attn_visible(T.prefix, bs, causal=True)) / 2
    nbytes = 2 * T.Hkv * (T.prefix + 16) * T.D * 2 + 2 * 16 * T.Hq * T.D * 2 + 16 * T.Hq * 4
    n_masked = int((state0 == synth.MASKED).sum())
    kernels = {"attn_kernel": _attn_roof(attn_us, nbytes, 4 * T.D * T.Hq * vis, peaks, False),
               "unmask_kernel": _vocab_roof(um_us, n_masked * T.V * 4, peaks),
               "verify_kernel": _vocab_roof(vf_us, (E + 1) * T.V * 4, peaks)}
    return _extra_line("tiny: 1 layer, 4/2 heads, head dim 64, prefix 256, 2 blocks of 8 (3 scaffold each), "
                "fp32 logits [16, 1024]; one round (attention, unmask tau 0.9 + 1/4 + draft, causal AR "
                "attention, verify)", committed, step_ms, args, kernels, {"gpu_launches_per_step": 4})


def run_fast_dvla(args, dev):
    """Fast-dVLA pipelined decode, one denoise step of the 3-block window:
    36 x attention (16/2 heads, head dim 128, prefix 512 image + 88 instruction
    + the 14 action tokens of the two finished blocks, window of three 7-token
    blocks) and one unmask over the window's masked positions (masked ratios
    2/7, 4/7, 7/7; half activation at 1/2 with tau 0.9, full at 0.85 with tau
    0.9 and at least 1/4 of the remaining)."""
    import torch
    import block_causal_masked_gb300 as bd
    F = synth.FAST_DVLA
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    C, bs, n_q = F.prefix + 14, [0, 7, 14, 21], 21
    g0 = synth.rng(F.seed, 7)
    state0 = np.zeros(n_q, np.int64)
    state0[g0.choice(7, 5, replace=False)] = synth.COMMITTED
    state0[7 + g0.choice(7, 3, replace=False)] = synth.COMMITTED
    tokens0 = np.where(state0 == synth.COMMITTED, 5, -1)
    masked = np.flatnonzero(state0 == synth.MASKED)
    logit_row = np.full(n_q, -1, np.int32)
    logit_row[masked] = np.arange(len(masked))
    logits, _, _ = synth.planted_logits(F.seed, 1, len(masked), F.V)
    bf = torch.bfloat16
    t = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(dt)  # noqa: E731
    layers = []
    for l in range(F.layers):
        a = synth.attn_case(F.seed, l, C=C, block_start=bs, Hq=F.Hq, Hkv=F.Hkv, D=F.D, text_from=512)
        layers.append((t(a.q, bf), t(a.k, bf), t(a.v, bf)))
    copies = _copies(len(masked) * F.V * 2)
    lg = [t(logits, bf) for _ in range(copies)]
    row = t(logit_row, torch.int32)
    blk = torch.tensor(bs, dtype=torch.int32, device=dev)
    win = _Window(state0, tokens0, copies, dev)
    outs = [_unmask_outs(n_q, 3, dev) for _ in range(copies)]
    o = torch.empty((n_q, F.Hq, F.D), dtype=bf, device=dev)
    lse = torch.empty((F.Hq, n_q), dtype=torch.float32, device=dev)
    kw = dict(tau_full=0.9, tau_half=0.9, min_frac=(1, 4), k_fixed=0, add_thr=(1, 2), act_thr=(17, 20))

    def attn():
        for q, k, v in layers:
            bd.bd_block_causal_attn(q, k, v, C, block_start=blk, o=o, lse=lse, prefix_ready=True)

    def unmask(i=0):
        bd.bd_unmask_step(lg[i], row, blk, win.state[i], win.tokens[i], **kw, **outs[i])

    step_g = _graph(lambda: (attn(), unmask()))
    for _ in range(args.warmup):
        win.reset()
        step_g.replay()
    step_ms = _replay_ms(step_g, args.steps, flush, before=win.reset)
    committed = int(outs[0]["n_committed"].sum())
    attn_us = _replay_ms(_graph(attn), args.steps, flush) * 1e3 / F.layers
    um_us = _per_launch_us([lambda i=i: unmask(i) for i in range(copies)], win.reset, flush, args.steps)
    peaks = measured_peaks()
    nbytes = 2 * F.Hkv * (C + n_q) * F.D * 2 + 2 * n_q * F.Hq * F.D * 2 + n_q * F.Hq * 4
    kernels = {"attn_kernel": _attn_roof(attn_us, nbytes, 4 * F.D * F.Hq * _attn_visible(C, bs), peaks, True),
               "unmask_kernel": _vocab_roof(um_us, len(masked) * F.V * 2, peaks)}
    return _extra_line(f"fast_dvla: 16/2 heads, head dim 128, 36 layers, prefix {C} keys, window of 3 blocks x 7 "
                f"({len(masked)} masked), vocab 151936; one denoise step (36 attention layers + unmask)",
                committed, step_ms, args, kernels,
                {"gpu_launches_per_step": F.layers + 1, "block_status": outs[0]["status"].tolist()})


def run_fork(args, dev):
    """Shared-prefix fork + streaming cache, one scaffold-speculative round of
    the second trajectory block for N = 1, 8, 32 rollouts: 36 x bd_rope_keys
    (each layer's 4,306 pre-RoPE prefix keys in view-major order rotated at
    k_pos - 256, once for both passes), 36 x bd_fork_rollouts (MDM pass, the
    39-position block bidirectional; 41 private rows of the first trajectory
    block before it), 36 x bd_fork_rollouts (AR pass, causal), then the sampled
    verifier over the N rollouts (AR rows [N, 33,
    151936] bf16 with Gumbel noise fp32).  Inputs are drawn on the device from
    a seeded generator; every rollout's AR rows agree with its draft on a
    seeded number of slots."""
    import torch
    import block_causal_masked_gb300 as bd
    S = synth.FORK_STREAM
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    C, n_q, priv_len, L, E = S.prefix, 39, 41, 39, 32
    k_pos = torch.from_numpy(synth.streaming_prefix_positions()).to(dev)
    rope = dict(k_pos=k_pos, delta=256, theta=1e4)
    bf = torch.bfloat16
    lines = []
    for N in ((args.rollouts,) if getattr(args, "rollouts", None) else (1, 8, 32)):
        gen = torch.Generator(device=dev)
        gen.manual_seed(S.seed * 1000 + N)
        rn = lambda *shape: torch.randn(shape, generator=gen, device=dev).to(bf)  # noqa: E731
        layers = [(rn(N, n_q, S.Hq, S.D), rn(N, n_q, S.Hq, S.D), rn(S.Hkv, C, S.D), rn(S.Hkv, C, S.D),
                   rn(N, S.Hkv, priv_len + n_q, S.D), rn(N, S.Hkv, priv_len + n_q, S.D)) for _ in range(S.layers)]
        blk = torch.tensor([0, n_q], dtype=torch.int32, device=dev)
        o = torch.empty((N, n_q, S.Hq, S.D), dtype=bf, device=dev)
        lse = torch.empty((N, S.Hq, n_q), dtype=torch.float32, device=dev)
        # verify inputs: scaffold slots, drafts, AR rows planted to agree on k_r slots, uniforms
        g = synth.rng(S.seed, 999, N)
        scaf = np.zeros(L, np.int64)
        scaf[g.choice(L, L - E, replace=False)] = 1
        state0 = np.tile(np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED), (N, 1))
        drafts = g.integers(0, S.V, size=(N, L))
        kr = g.integers(0, E + 1, size=N)
        ar = (torch.randn((N, E + 1, S.V), generator=gen, device=dev) * 3.0)
        ed = np.flatnonzero(scaf == 0)
        for r in range(N):
            for e in range(int(kr[r])):
                ar[r, e, int(drafts[r, ed[e]])] = 60.0
            if kr[r] < E:
                ar[r, int(kr[r]), (int(drafts[r, ed[kr[r]]]) + 1) % S.V] = 60.0
        ar = ar.to(bf)
        u = torch.rand((N, E + 1, S.V), generator=gen, device=dev).clamp_(2.0 ** -24, 1.0 - 2.0 ** -24)
        copies = _copies(N * (E + 1) * S.V * 6)
        ars = [ar] + [ar.clone() for _ in range(copies - 1)]
        us = [u] + [u.clone() for _ in range(copies - 1)]
        win = _Window(state0, drafts, copies, dev)
        accs = [torch.empty(N, dtype=torch.int32, device=dev) for _ in range(copies)]
        acc = accs[0]

        # RoPE: each layer's pre-RoPE prefix is rotated once per round (bd_rope_keys)
        # and both passes read the rotated copy
        rot = [torch.empty((S.Hkv, C, S.D), dtype=bf, device=dev) for _ in range(S.layers)]

        def rope_keys():
            for (_, _, pk, _, _, _), r in zip(layers, rot):
                bd.bd_rope_keys(pk, C, rope, out=r)

        def mdm():
            for (q, _, _, pv, rk, rv), r in zip(layers, rot):
                bd.bd_fork_rollouts(q, r, pv, rk, rv, priv_len, C, block_start=blk, o=o, lse=lse)

        def ar_pass():
            for (_, q, _, pv, rk, rv), r in zip(layers, rot):
                bd.bd_fork_rollouts(q, r, pv, rk, rv, priv_len, C, block_size=1, o=o, lse=lse)

        def verify(i=0):
            bd.bd_spec_verify(win.tokens[i], win.state[i], ars[i], us[i], 1.0, accepted_len=accs[i])

        round_g = _graph(lambda: (rope_keys(), mdm(), ar_pass(), verify()))
        reps = max(3, args.steps // (1 + N // 4))
        for _ in range(args.warmup):
            win.reset()
            round_g.replay()
        step_ms = _replay_ms(round_g, reps, flush, before=win.reset)
        committed = int(acc.sum())
        attn_us = _replay_ms(_graph(lambda: (mdm(), ar_pass())), reps, flush) * 1e3 / (2 * S.layers)
        rope_us = _replay_ms(_graph(rope_keys), reps, flush) * 1e3 / S.layers
        vf_us = _per_launch_us([lambda i=i: verify(i) for i in range(copies)], win.reset, flush, reps)
        peaks = measured_peaks()
        vis = N * (_attn_visible(C + priv_len, [0, n_q]) + _attn_visible(C + priv_len, [0, n_q], causal=True)) / 2
        nbytes = (2 * S.Hkv * C * S.D * 2 + N * 2 * S.Hkv * (priv_len + n_q) * S.D * 2
                  + 2 * N * n_q * S.Hq * S.D * 2 + N * n_q * S.Hq * 4)
        kernels = {"attn_kernel": _attn_roof(attn_us, nbytes, 4 * S.D * S.Hq * vis, peaks, True),
                   "rope_prefix_kernel": _vocab_roof(rope_us, 2 * S.Hkv * C * S.D * 2 + C * 4, peaks),
                   "verify_kernel": _vocab_roof(vf_us, N * (E + 1) * S.V * (2 + 4), peaks)}
        lines.append(_extra_line(f"fork_streaming N={N}: 16/2 heads, head dim 128, 36 layers, 4306 pre-RoPE prefix keys "
                    f"(RoPE at k_pos - 256: one bd_rope_keys per layer, read by both passes), trajectory block of "
                    f"39 positions after 41 private rows per rollout; one round (RoPE, MDM fork, causal AR fork, "
                    f"sampled verify of {N} rollouts)",
                    committed, step_ms, args, kernels,
                    {"gpu_launches_per_step": "36 x RoPE + 2 x 36 x attention (+1 when a call splits the rows "
                                              "into two launches) + 1", "rollouts": N}))
        del layers, ar, u, ars, us, rot
        torch.cuda.empty_cache()
    return lines


def run_kv_fp8(args, dev):
    """The FP8 (E4M3) KV-cache variant beside the bf16 attention, per launch, on
    the WAM-Diff2 decode shape (16/8 heads, head dim 128, prefix 2,048 + 128
    decoded, blocks of 32 and of 1) and the Fast-dDrive decode shape (16/2
    heads, 3,124 cached keys, 33 positions): 36 distinct layers back to back in
    a graph, L2 flushed before each replay.  The E4M3 cache holds half the
    bytes; the roofline counts the bytes each variant must read."""
    import torch
    import block_causal_masked_gb300 as bd
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks = measured_peaks()
    shapes = [("wam_diff2 B=32", 16, 8, 2048 + 128, 32), ("wam_diff2 B=1", 16, 8, 2048 + 128, 1),
              ("fast_ddrive", 16, 2, 3124, 33)]
    out = {}
    for name, Hq, Hkv, C, n_q in shapes:
        D, L = 128, 36
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        S = C + n_q
        q = [torch.randn((n_q, Hq, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
        kb = [torch.randn((Hkv, S, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
        vb = [torch.randn((Hkv, S, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
        # E4M3 copies: bytes drawn uniformly over the finite codes, exponent -4 per block
        # (timing only: any bytes run the same instructions)
        k8 = [torch.randint(0, 0x7e, (Hkv, S, D), generator=g, device=dev, dtype=torch.uint8) for _ in range(L)]
        v8 = [torch.randint(0, 0x7e, (Hkv, S, D), generator=g, device=dev, dtype=torch.uint8) for _ in range(L)]
        ex = torch.full((Hkv, -(-S // 128)), -4, dtype=torch.int8, device=dev)
        o = torch.empty((n_q, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((Hq, n_q), dtype=torch.float32, device=dev)
        blk = torch.tensor([0, n_q], dtype=torch.int32, device=dev)

        def bf():
            for l in range(L):
                bd.bd_block_causal_attn(q[l], kb[l], vb[l], C, block_start=blk, o=o, lse=lse, prefix_ready=True)

        def f8():
            for l in range(L):
                bd.bd_block_causal_attn(q[l], k8[l], v8[l], C, block_start=blk, o=o, lse=lse, k_exp=ex, v_exp=ex)
        us_bf = _replay_ms(_graph(bf), args.steps, flush) * 1e3 / L
        us_f8 = _replay_ms(_graph(f8), args.steps, flush) * 1e3 / L
        qo = 2 * n_q * Hq * D * 2 + n_q * Hq * 4
        flops = 4 * D * Hq * n_q * S
        out[name] = {"bf16": _attn_roof(us_bf, qo + 2 * Hkv * S * D * 2, flops, peaks, True),
                     "e4m3": _attn_roof(us_f8, qo + 2 * Hkv * S * D + 2 * Hkv * (-(-S // 128)), flops, peaks, True)}
        del q, kb, vb, k8, v8
        torch.cuda.empty_cache()
    return {"metric": "attention us per launch, bf16 vs FP8 (E4M3) KV cache", "unit": "us", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "dtype": "bf16 / e4m3", "data": "synthetic",
            "config": {"workload": "kv_fp8: 36 layers back to back per shape, L2 flushed before each replay"},
            "roofline": out}


def run_stream(args, dev):
    """FlashDrive streaming step: a new camera frame (4 views x 256 tokens) enters
    the view-major pre-RoPE window of 4 frames per view (4,096 keys, 16/2 heads,
    head dim 128), 36 layers of bd_stream_insert (the frame's K/V into every
    view's ring slot) + bd_block_causal_attn with the streaming mask (the
    frame's 1,024 queries over the window, RoPE at k_pos - delta).  Value: new
    frame tokens per second."""
    import torch
    import block_causal_masked_gb300 as bd
    S = synth.FORK_STREAM
    views, frames, per, Hq, Hkv, D, L = 4, 4, 256, S.Hq, S.Hkv, S.D, S.layers
    C = views * frames * per
    n = views * per
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(S.seed * 1000 + 7)
    bf = torch.bfloat16
    rn = lambda *shape: torch.randn(shape, generator=gen, device=dev).to(bf)  # noqa: E731
    kc = [rn(Hkv, C, D) for _ in range(L)]
    vc = [rn(Hkv, C, D) for _ in range(L)]
    nk = [rn(n, Hkv, D) for _ in range(L)]
    nv = [rn(n, Hkv, D) for _ in range(L)]
    q = [rn(n, Hq, D) for _ in range(L)]
    # window of frame times 1..4 after one slide (delta = one frame); the new
    # frame (time 4) goes into slot 0, where frame 0 was
    w = np.arange(views)[:, None, None]
    f = np.arange(frames)[None, :, None]
    t = np.arange(per)[None, None, :]
    slot_time = np.array([4, 1, 2, 3])[None, :, None]                     # frame time held by each slot
    pos0 = ((w * frames + slot_time) * per + t).reshape(-1).astype(np.int32)
    kpos = torch.from_numpy(pos0).to(dev)
    delta = per
    new_pos = torch.from_numpy(((np.arange(views)[:, None] * frames + 4) * per
                                + np.arange(per)[None, :]).reshape(-1).astype(np.int32)).to(dev)
    qpos = (new_pos - delta).contiguous()
    o = torch.empty((n, Hq, D), dtype=bf, device=dev)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=dev)
    rope = dict(k_pos=kpos, delta=delta, theta=1e4)

    def step():
        for l in range(L):
            bd.bd_stream_insert(kc[l], vc[l], kpos, nk[l], nv[l], new_pos, views, frames, per, 0)
            bd.bd_block_causal_attn(q[l], kc[l], vc[l], C, q_pos=qpos, rope=rope, o=o, lse=lse)

    def attn_only():
        for l in range(L):
            bd.bd_block_causal_attn(q[l], kc[l], vc[l], C, q_pos=qpos, rope=rope, o=o, lse=lse)

    def insert_only():
        for l in range(L):
            bd.bd_stream_insert(kc[l], vc[l], kpos, nk[l], nv[l], new_pos, views, frames, per, 0)

    g = _graph(step)
    for _ in range(args.warmup):
        g.replay()
    step_ms = _replay_ms(g, args.steps, flush)
    attn_us = _replay_ms(_graph(attn_only), args.steps, flush) * 1e3 / L
    ins_us = _replay_ms(_graph(insert_only), args.steps, flush) * 1e3 / L
    peaks = measured_peaks()
    # visible keys per query: every earlier view, its own view's history, its frame up to itself
    pos_np = pos0.astype(np.int64) - delta
    qp = (new_pos.cpu().numpy().astype(np.int64) - delta)
    vis = int((pos_np[None, :] <= qp[:, None]).sum())
    flops = 4 * D * Hq * vis
    nbytes = 2 * Hkv * C * D * 2 + 2 * n * Hq * D * 2 + n * Hq * 4 + C * 4
    kernels = {"attn_kernel": _attn_roof(attn_us, nbytes, flops, peaks, True),
               "stream_insert_kernel": _vocab_roof(ins_us, 2 * 2 * n * Hkv * D * 2 + 2 * n * 4, peaks),
               "rope_prefix_kernel": "inside attn_kernel's time (one launch per attention call)"}
    line = {"metric": "new-frame tokens/s (streaming step: insert + streaming-mask attention, 36 layers)",
            "value": n / step_ms * 1e3, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"stream: 4 views x 4 frames x 256 tokens view-major pre-RoPE window, new "
                                   f"frame of {n} tokens, 16/2 heads, head dim 128, 36 layers, RoPE at k_pos - "
                                   f"{delta}", "l2": "flushed (256 MiB write) before every timed step",
                       "visible_keys_per_query": vis / n},
            "roofline": kernels}
    return line


def algorithmic(inp):
    """Bytes (and FLOPs) the round must move: visible K/V, Q, O, LSE per layer;
    logits rows of masked editable positions; AR rows."""
    C, n_q = inp["C"], inp["n_q"]
    qo = 2 * n_q * W.Hq * W.D * 2 + n_q * W.Hq * 4
    kv_mdm = 2 * W.Hkv * (C + n_q) * W.D * 2
    kv_ar = 2 * W.Hkv * (C + n_q) * W.D * 2          # the last key of the block is visible to its last query
    vis_mdm = n_q * (C + n_q)
    vis_ar = sum(C + i + 1 for i in range(n_q))
    flops_mdm = 4 * W.D * W.Hq * vis_mdm
    flops_ar = 4 * W.D * W.Hq * vis_ar
    unmask_bytes = inp["E"] * W.V * 2
    verify_bytes = (inp["E"] + 1) * W.V * 2
    return dict(attn_bytes=(qo + kv_mdm, qo + kv_ar), attn_flops=(flops_mdm, flops_ar), unmask_bytes=unmask_bytes,
                verify_bytes=verify_bytes)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.proc = None
        self.path = None
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}",
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            # timing starts only once the sampler has written its first row
            t0 = time.time()
            while time.time() - t0 < 5.0 and self.proc.poll() is None:
                with open(self.path) as f:
                    if f.readline().strip():
                        break
                time.sleep(0.02)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l.split(",") for l in open(self.path).read().splitlines() if l.strip()]
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 3 + i and r[3 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def attn_traffic():
    """DRAM bytes per attention launch from the committed ncu capture, if the
    attention kernel's source is still the one that capture measured (else None)."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "attn_kernel_traffic.json")))
        h = hashlib.sha256()
        for f in rec["files"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        return rec["dram_bytes_per_launch"] if h.hexdigest()[:16] == rec["source_sha256_16"] else None
    except (OSError, ValueError, KeyError):
        return None


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def _oracle_sample(inp, budget_s: float):
    """Full oracle rounds until `budget_s` is spent: (rounds, tokens, seconds)."""
    import oracle
    t0 = time.perf_counter()
    steps, tokens = 0, 0
    while True:
        tokens += oracle_round(oracle, inp)
        steps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return steps, tokens, time.perf_counter() - t0


ONE_THREAD_ENV = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                                   "BLIS_NUM_THREADS", "NUMEXPR_NUM_THREADS")}


def cpu_baseline(inp, budget_s: float = 12.0, one_core_budget_s: float = 10.0):
    """The float64 oracle on the host: on every core (numpy's BLAS threads, this
    process), and on one core (a child process pinned to one CPU with one BLAS
    thread), full rounds of the workload until each budget is spent."""
    steps, tokens, dt = _oracle_sample(inp, budget_s)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    out = {"value": tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{steps} full round(s) of the workload (72 attention layers, unmask, verify) in float64 "
                     f"numpy, {dt:.1f} s"}
    env = dict(os.environ, **ONE_THREAD_ENV)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample-s", str(one_core_budget_s)]
    if hasattr(os, "sched_getaffinity"):
        cpu = sorted(os.sched_getaffinity(0))[0]
        cmd = [sys.executable, "-c", f"import os, runpy, sys; os.sched_setaffinity(0, {{{cpu}}}); "
               f"sys.argv = {cmd[1:]!r}; runpy.run_path(sys.argv[0], run_name='__main__')"]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=10 * one_core_budget_s + 120)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        out["one_core"] = {"value": one["tokens"] / one["seconds"], "unit": UNIT, "cores": 1,
                           "sample": f"{one['rounds']} full round(s), {one['seconds']:.1f} s, one CPU, one BLAS "
                                     "thread"}
    except (subprocess.SubprocessError, OSError, ValueError, IndexError, KeyError) as e:
        out["one_core"] = {"value": None, "error": str(e)[:200]}
    return out


def oracle_round(oracle, inp) -> int:
    """Committed tokens of one round by the float64 oracle."""
    return oracle.speculative_round(inp["layers"], inp["C"], inp["n_q"], inp["logits"], inp["logit_row"],
                                    inp["state"], inp["tokens"], inp["ar_logits"], TAU)[0]


def e2e_measure(rd, inp, steps: int):
    """The same round end to end through the library's public calls, captured
    as CUDA graphs the way a serving loop would run them: every step copies
    its inputs (queries of both passes, both logits tensors, state and tokens)
    from pinned host memory and reads its result (committed counts and tokens)
    back to the host, all inside the timed region.  Two device input sets let
    step i+1's copies (on their own stream) overlap step i's kernels."""
    import torch
    hq = [torch.from_numpy(np.array(q, copy=True)).to(torch.bfloat16).pin_memory() for q, _, _, _ in inp["layers"]]
    hqa = [torch.from_numpy(np.array(q, copy=True)).to(torch.bfloat16).pin_memory() for _, q, _, _ in inp["layers"]]
    hl = torch.from_numpy(np.array(inp["logits"], copy=True)).to(torch.bfloat16).pin_memory()
    ha = torch.from_numpy(np.array(inp["ar_logits"][None], copy=True)).to(torch.bfloat16).pin_memory()
    hs = torch.from_numpy(inp["state"].copy()).pin_memory()
    ht = torch.from_numpy(inp["tokens"].copy()).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in hq + hqa + [hl, ha, hs, ht])
    sets = [rd, gpu_round(inp, rd.q[0].device)]
    sets[1].capture()
    outs = [torch.empty(2, dtype=torch.int32).pin_memory() for _ in sets]
    out_tok = [torch.empty_like(ht).pin_memory() for _ in sets]
    d2h = outs[0].numel() * 4 + out_tok[0].numel() * 4
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream(rd.q[0].device)
    copied = [torch.cuda.Event() for _ in sets]
    done = [torch.cuda.Event() for _ in sets]

    def load(i):  # step i's inputs into set i % 2, on the copy stream
        x = sets[i % 2]
        with torch.cuda.stream(copy):
            copy.wait_event(done[i % 2])          # the set's previous round is finished
            for l in range(W.layers):
                x.q[l].copy_(hq[l], non_blocking=True)
                x.q_ar[l].copy_(hqa[l], non_blocking=True)
            x.logits.copy_(hl, non_blocking=True)
            x.ar_logits.copy_(ha, non_blocking=True)
            x.state.copy_(hs, non_blocking=True)
            x.tokens.copy_(ht, non_blocking=True)
            copied[i % 2].record(copy)

    rd.flush.zero_()
    for e in done:
        e.record(compute)
    torch.cuda.synchronize()
    toks = 0
    t0 = time.perf_counter()
    load(0)
    for i in range(steps):
        x = sets[i % 2]
        compute.wait_event(copied[i % 2])
        x.whole.replay()
        outs[i % 2][0:1].copy_(x.um["n_committed"], non_blocking=True)
        outs[i % 2][1:2].copy_(x.acc, non_blocking=True)
        out_tok[i % 2].copy_(x.tokens, non_blocking=True)
        done[i % 2].record(compute)
        if i + 1 < steps:
            load(i + 1)
        if i > 0:                                 # step i - 1's result, read while step i runs
            done[(i - 1) % 2].synchronize()
            toks += int(outs[(i - 1) % 2][0]) + int(outs[(i - 1) % 2][1])
    done[(steps - 1) % 2].synchronize()
    toks += int(outs[(steps - 1) % 2][0]) + int(outs[(steps - 1) % 2][1])
    total = time.perf_counter() - t0
    return {"value": toks / total, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def aggregate(seconds: float, tokens: float, world: int, device="cpu"):
    """Whole-job totals over the ranks: the slowest rank's timed seconds and the
    sum of the committed tokens (each rank decodes its own independent request)."""
    if world == 1:
        return seconds, tokens
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    c = torch.tensor([tokens], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(c)
    return float(t[0]), float(c[0])


def vocab_times(rd, inp, device, reps: int):
    """Per-launch us of the round's unmask and verify calls, each timed as 16
    independent calls (own logits copy, state and tokens) in one graph."""
    import torch
    import block_causal_masked_gb300 as bd
    copies = 16
    n_q = inp["n_q"]
    win = _Window(inp["state"], inp["tokens"], copies, device)
    lgs = [rd.logits] + [rd.logits.clone() for _ in range(copies - 1)]
    ars = [rd.ar_logits] + [rd.ar_logits.clone() for _ in range(copies - 1)]
    outs = [_unmask_outs(n_q, 1, device) for _ in range(copies)]
    accs = [torch.empty(1, dtype=torch.int32, device=device) for _ in range(copies)]

    def unmask(i):
        bd.bd_unmask_step(lgs[i], rd.logit_row, rd.block, win.state[i], win.tokens[i], tau_full=TAU, tau_half=TAU,
                          min_frac=(0, 1), k_fixed=0, write_draft=True, **outs[i])

    def verify(i):
        bd.bd_spec_verify(win.tokens[i].view(1, -1), win.state[i].view(1, -1), ars[i], accepted_len=accs[i])

    um = _per_launch_us([lambda i=i: unmask(i) for i in range(copies)], win.reset, rd.flush, reps)
    vf = _per_launch_us([lambda i=i: verify(i) for i in range(copies)], win.reset, rd.flush, reps)
    return um, vf


def latency_floor(device, flush, reps: int) -> dict:
    """Per-launch time of launches that do almost nothing, 72 back to back in
    one graph (as the round's attention launches are): an empty elementwise
    kernel; the attention kernel on one key tile (one CTA, no cluster); and on
    one 128-key tile per CTA of a 16-CTA cluster (1,920 cached keys + 1, 16
    splits), which adds the cluster launch and the split merge.  The gap between
    a kernel's time and these is in-kernel work; the rest is fixed cost."""
    import torch
    import block_causal_masked_gb300 as bd
    n = 72
    x = torch.zeros(1, device=device)
    empty_us = _replay_ms(_graph(lambda: [x.add_(1.0) for _ in range(n)]), reps, flush) * 1e3 / n
    g = torch.Generator(device=device)
    g.manual_seed(99)
    q = torch.randn((1, 1, 128), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((1, 1921, 128), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((1, 1921, 128), generator=g, device=device).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((1, 1), dtype=torch.float32, device=device)

    def one_tile():
        for _ in range(n):
            bd.bd_block_causal_attn(q, k, v, 0, block_size=1, o=o, lse=lse, num_splits=1, prefix_ready=True)

    def cluster16():
        for _ in range(n):
            bd.bd_block_causal_attn(q, k, v, 1920, block_size=1, o=o, lse=lse, num_splits=16, prefix_ready=True)
    one_us = _replay_ms(_graph(one_tile), reps, flush) * 1e3 / n
    clu_us = _replay_ms(_graph(cluster16), reps, flush) * 1e3 / n
    return {"empty_kernel_us": empty_us, "attn_one_tile_us": one_us, "attn_cluster16_one_tile_each_us": clu_us}


def replica_seed(rank: int) -> int:
    """Seed of the request rank `rank` decodes (independent inputs per replica)."""
    return W.seed + 100 * rank


def run_gpu(args, rank, world, local_rank):
    import torch
    device = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    inp = make_inputs(replica_seed(rank))
    rd = gpu_round(inp, device)
    rd.capture()
    clocks = Clocks(local_rank)
    for _ in range(args.warmup):
        timed_step(rd)
        timed_parts(rd)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    steps_ms = []
    committed = 0
    for _ in range(args.steps):
        steps_ms.append(timed_step(rd))
        committed += rd.committed()
    torch.cuda.synchronize()
    # per-kernel times for the roofline: the attention from the round replayed
    # as four graphs (72 launches in its two attention parts); the vocabulary
    # kernels from 16 independent calls back to back (own logits copies)
    attn_ms = []
    reps = max(3, min(50, args.steps // 4))
    for _ in range(reps):
        _, a, _ = timed_parts(rd)
        attn_ms.append(a)
    unmask_us, verify_us = vocab_times(rd, inp, device, reps)
    floor = latency_floor(device, rd.flush, reps)
    torch.cuda.synchronize()
    total_s = sum(steps_ms) / 1e3
    total_s, committed_all = aggregate(total_s, committed, world, device)
    e2e = e2e_measure(rd, inp, max(3, min(100, args.steps // 2)))
    if rank != 0:
        clocks.stop()
        return None
    alg = algorithmic(inp)
    peaks = measured_peaks()
    attn_launch_s = (sum(attn_ms) / len(attn_ms)) / 1e3 / (2 * W.layers)
    attn_bytes = (alg["attn_bytes"][0] + alg["attn_bytes"][1]) / 2
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = attn_bytes / attn_launch_s / 1e9
    unmask_s = unmask_us / 1e6
    splits = planned_splits(inp["C"], inp["n_q"], W.Hq, W.Hkv, W.D)
    launches_per_step = 2 * W.layers + 2
    line = {
        "metric": METRIC, "value": committed_all / total_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"fast_ddrive: 16/2 heads, head dim 128, 36 layers, prefix {inp['C']} keys, "
                               f"active block {inp['n_q']} positions ({inp['E']} editable), vocab 151936; one "
                               "scaffold-speculative round (MDM attention, unmask tau 0.9 + draft, causal AR "
                               "attention, verify) per step",
                   "decodes_per_gpu": 1, "parallelism": f"replicas x{world}",
                   "l2": "flushed (256 MiB write) before every timed step, outside the timed region",
                   "timing": "CUDA events around one CUDA-graph replay of the round; per-kernel times from "
                             "the round replayed as four graphs with events between them",
                   "committed_per_step": committed_all / world / args.steps,
                   "planted_accept_len": inp["planted_accept"], "attn_splits": splits},
        "roofline": {"bound": "hbm", "kernel": "attn_kernel (bd_block_causal_attn)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": "measured" if peaks else "fallback", "traffic": attn_traffic(),
                     "alg_bytes_per_launch": attn_bytes, "avg_launch_us": attn_launch_s * 1e6,
                     "latency_floor": floor,
                     "unmask": {"alg_bytes": alg["unmask_bytes"], "us": unmask_s * 1e6,
                                "achieved_gbs": alg["unmask_bytes"] / unmask_s / 1e9,
                                "frac": alg["unmask_bytes"] / unmask_s / 1e9 / hbm},
                     "verify": {"alg_bytes": alg["verify_bytes"], "us": verify_us,
                                "achieved_gbs": alg["verify_bytes"] / verify_us / 1e3,
                                "frac": alg["verify_bytes"] / verify_us / 1e3 / hbm}},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "_clocks": clocks,   # stopped by main() once every measured workload has run
    }
    if world == 1:
        line["cpu_baseline"] = cpu_baseline(inp)
    return line


def run_reference(args):
    inp = make_inputs(W.seed)
    import oracle
    for _ in range(args.warmup):
        oracle_round(oracle, inp)
    t0 = time.perf_counter()
    toks = sum(oracle_round(oracle, inp) for _ in range(args.steps))
    dt = time.perf_counter() - t0
    v = toks / dt
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "fast_ddrive (as the GPU arm), float64 oracle on the host cores"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{args.steps} full rounds"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--contract-only", action="store_true",
                    help="print the Fast-dDrive-shaped line without the other workloads' results")
    ap.add_argument("--oracle-sample-s", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--workload", choices=["fast_ddrive", "wam_sweep", "tiny", "fast_dvla", "fork", "stream",
                                           "kv_fp8"],
                    default="fast_ddrive",
                    help="fast_ddrive: the contract's line; the others print extra lines: wam_sweep (the whole "
                         "WAM-Diff2 decode per block size as one CUDA graph), tiny, fast_dvla (one denoise step of "
                         "the 3-block window), fork (one round for N = 1, 8, 32 rollouts), stream (one new camera frame "
                         "into the streaming window: insert + streaming-mask attention), kv_fp8 (bf16 and E4M3 KV "
                         "cache attention per launch)")
    ap.add_argument("--rollouts", type=int, default=None, choices=[1, 8, 32],
                    help="fork workload: only this rollout count (default: 1, 8 and 32)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.oracle_sample_s is not None:       # the one-core oracle timing (a child of cpu_baseline)
        rounds, tokens, secs = _oracle_sample(make_inputs(W.seed), args.oracle_sample_s)
        print(json.dumps({"rounds": rounds, "tokens": tokens, "seconds": secs}), flush=True)
        return 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    extra = {"wam_sweep": run_wam_sweep, "tiny": run_tiny, "fast_dvla": run_fast_dvla, "fork": run_fork,
             "stream": run_stream, "kv_fp8": run_kv_fp8}
    if args.workload in extra:
        import torch
        torch.cuda.set_device(local_rank)
        out = extra[args.workload](args, f"cuda:{local_rank}")
        for ln in (out if isinstance(out, list) else [out]):
            print(json.dumps(ln), flush=True)
        return 0
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = run_gpu(args, rank, world, local_rank)
    if line is not None:
        if world == 1 and not args.contract_only:
            # the other four workloads (and the WAM-Diff2 sweep's five block sizes),
            # each with its per-kernel rooflines, measured after the contract's line
            sub = argparse.Namespace(steps=max(5, min(args.steps, 20)), warmup=3)
            dev = f"cuda:{local_rank}"
            line["configs"] = {"tiny": run_tiny(sub, dev), "fast_dvla": run_fast_dvla(sub, dev),
                               "wam_diff2_sweep": run_wam_sweep(sub, dev), "fork_streaming": run_fork(sub, dev),
                               "stream": run_stream(sub, dev), "kv_fp8": run_kv_fp8(sub, dev)}
        # SM clocks and throttle reasons sampled from the contract's warm-up
        # through the last workload's timed region
        line["clocks"] = line.pop("_clocks").stop()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
