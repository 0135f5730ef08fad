#!/usr/bin/env python3
"""Committed tokens/s of one block-causal masked-diffusion decode round on GB300.

Workload (Fast-dDrive-shaped, seed 1): 16 query / 2 KV heads, head dim 128, bf16,
36 layers; cached prefix = 3,000 tokens (2,700 image-like + 300 text-like) plus
the blocks already decoded (the 92-position critical-objects block and the first
32-position explanation block) = 3,124 keys; active block = the second
explanation block of the 404-position scaffolded output (33 positions: 32
editable + 1 scaffold); vocabulary 151,936.

One step = one scaffold-speculative round on the active block, all through the
library's C ABI:
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
TAU = 0.9
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------------------ inputs

def make_inputs(seed: int):
    """Seeded host inputs of one round (float32 arrays holding bf16 values)."""
    lay = synth.section_layout(W.seed)
    active = 2                                        # second explanation block
    C = W.prefix + int(lay.block_start[active])       # prompt prefix + the blocks decoded before it
    lo, hi = int(lay.block_start[active]), int(lay.block_start[active + 1])
    n_q = hi - lo
    scaf = lay.scaffold[lo:hi].astype(np.int64)
    E = int((scaf == 0).sum())
    layers = []
    for l in range(W.layers):
        a = synth.attn_case(seed, l, C=C, block_start=[0, n_q], Hq=W.Hq, Hkv=W.Hkv, D=W.D, text_from=2700)
        q_ar = synth.attn_case(seed, 1000 + l, C=0, block_start=[0, n_q], Hq=W.Hq, Hkv=1, D=W.D).q
        layers.append((a.q, q_ar, a.k, a.v))
    logits, tok, conf = synth.planted_logits(seed, 1, E, W.V)
    # the draft is the planted token of every editable row; rows at or above tau
    # commit in the unmask step; the AR rows agree with the draft on the first k
    # still-masked slots and disagree at the next one
    g = synth.rng(seed, 77)
    masked_rows = [e for e in range(E) if conf[e] < TAU]
    k = int(g.integers(0, len(masked_rows) + 1))
    want = g.integers(0, W.V, size=E + 1)
    for e in range(E):
        if conf[e] >= TAU or e in masked_rows[:k]:
            want[e] = tok[e]
    if k < len(masked_rows):
        e = masked_rows[k]
        want[e] = (tok[e] + 1) % W.V
    ar_logits, _, _ = synth.planted_logits(seed, 2, E + 1, W.V, tokens=want)
    state = np.where(scaf == 1, synth.SCAFFOLD, synth.MASKED).astype(np.uint8)
    tokens = np.where(scaf == 1, 11, -1).astype(np.int32)
    logit_row = np.full(n_q, -1, np.int32)
    logit_row[scaf == 0] = np.arange(E)
    return dict(C=C, n_q=n_q, E=E, layers=layers, logits=logits, ar_logits=ar_logits, state=state,
                tokens=tokens, logit_row=logit_row, planted_accept=k)


# ------------------------------------------------------------------------------ GPU arm

class GpuRound:
    def __init__(self, inp, device):
        import torch
        import block_causal_masked_gb300 as bd
        self.torch, self.bd, self.dev = torch, bd, device
        self.inp = inp
        t = lambda x, dt: torch.from_numpy(np.array(x, order="C", copy=True)).to(device).to(dt)  # noqa: E731
        bf = torch.bfloat16
        self.q = [t(q, bf) for q, _, _, _ in inp["layers"]]
        self.q_ar = [t(q, bf) for _, q, _, _ in inp["layers"]]
        self.k = [t(k, bf) for _, _, k, _ in inp["layers"]]
        self.v = [t(v, bf) for _, _, _, v in inp["layers"]]
        n_q = inp["n_q"]
        self.o = torch.empty((n_q, W.Hq, W.D), dtype=bf, device=device)
        self.lse = torch.empty((W.Hq, n_q), dtype=torch.float32, device=device)
        self.block = torch.tensor([0, n_q], dtype=torch.int32, device=device)
        self.logits = t(inp["logits"], bf)
        self.ar_logits = t(inp["ar_logits"][None], bf)
        self.logit_row = t(inp["logit_row"], torch.int32)
        self.state0 = t(inp["state"], torch.uint8)
        self.tokens0 = t(inp["tokens"], torch.int32)
        self.state = self.state0.clone()
        self.tokens = self.tokens0.clone()
        self.um = dict(commit=torch.empty(n_q, dtype=torch.uint8, device=device),
                       n_committed=torch.empty(1, dtype=torch.int32, device=device),
                       status=torch.empty(1, dtype=torch.int32, device=device),
                       pred=torch.empty(n_q, dtype=torch.int32, device=device),
                       conf=torch.empty(n_q, dtype=torch.float32, device=device),
                       lse=torch.empty(n_q, dtype=torch.float32, device=device))
        self.acc = torch.empty(1, dtype=torch.int32, device=device)
        self.bonus = torch.empty(1, dtype=torch.int32, device=device)
        self.bonus_pos = torch.empty(1, dtype=torch.int32, device=device)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.launches = 0

    # the four parts of a round, each a sequence of C-ABI calls on the current stream
    def mdm(self):
        for l in range(W.layers):
            self.bd.bd_block_causal_attn(self.q[l], self.k[l], self.v[l], self.inp["C"], block_start=self.block,
                                         o=self.o, lse=self.lse)

    def unmask(self):
        self.bd.bd_unmask_step(self.logits, self.logit_row, self.block, self.state, self.tokens, tau_full=TAU,
                               tau_half=TAU, min_frac=(0, 1), k_fixed=0, write_draft=True, **self.um)

    def ar(self):
        for l in range(W.layers):
            self.bd.bd_block_causal_attn(self.q_ar[l], self.k[l], self.v[l], self.inp["C"], block_size=1,
                                         o=self.o, lse=self.lse)

    def verify(self):
        self.bd.bd_spec_verify(self.tokens.view(1, -1), self.state.view(1, -1), self.ar_logits,
                               accepted_len=self.acc, bonus=self.bonus, bonus_pos=self.bonus_pos)

    def reset(self):
        self.state.copy_(self.state0)
        self.tokens.copy_(self.tokens0)

    def committed(self) -> int:
        return int(self.um["n_committed"][0]) + int(self.acc[0])

    def capture(self):
        torch = self.torch
        self.reset()
        self.mdm(); self.unmask(); self.ar(); self.verify()          # allocate workspaces, set kernel attributes
        torch.cuda.synchronize()
        s = torch.cuda.Stream(self.dev)
        self.graphs = []
        for part in (self.mdm, self.unmask, self.ar, self.verify):
            g = torch.cuda.CUDAGraph()
            self.reset()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                part()
            self.graphs.append(g)
        # the whole round as one graph: consecutive launches overlap through
        # programmatic dependent launch across the part boundaries too
        self.whole = torch.cuda.CUDAGraph()
        self.reset()
        torch.cuda.synchronize()
        with torch.cuda.graph(self.whole, stream=s):
            self.mdm(); self.unmask(); self.ar(); self.verify()
        torch.cuda.synchronize()

    def timed_step(self):
        """Replays the round (one graph); returns its ms."""
        torch = self.torch
        self.reset()
        self.flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        self.whole.replay()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1)

    def timed_parts(self):
        """Replays the round as its four part graphs with events between them;
        returns (step ms, attention ms, unmask ms)."""
        torch = self.torch
        self.reset()
        self.flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        torch.cuda.synchronize()
        ev[0].record()
        for i, g in enumerate(self.graphs):
            g.replay()
            ev[i + 1].record()
        ev[4].synchronize()
        t = [ev[0].elapsed_time(ev[i + 1]) for i in range(4)]
        step = t[3]
        attn = t[0] + (t[2] - t[1])
        unmask = t[1] - t[0]
        return step, attn, unmask

    def attn_splits(self) -> int:
        """KV splits (cluster width) the library plans for this shape."""
        m_tiles = -(-self.inp["n_q"] * (W.Hq // W.Hkv) // 128)
        tiles = -(-self.inp["C"] // 128) + -(-self.inp["n_q"] // 128)
        return max(1, min(152 // (m_tiles * W.Hkv), tiles, 16))


# ------------------------------------------------------------------------------ device-resident decode

WAM = synth.WAM_SWEEP
WAM_TOKENS = 256


def wam_steps(B: int) -> int:
    """Steps per block of the WAM-Diff2 sweep: top k = max(1, B / 8) commits per
    step, at most 8 steps, a block ends once complete."""
    return min(8, -(-B // max(1, B // 8)))


class WamDecode:
    """The whole 256-token WAM-Diff2 decode at block size B as ONE CUDA graph:
    for every block, wam_steps(B) denoise steps of `layers` x
    bd_block_causal_attn (16/8 heads, head dim 128, prefix 2,048 + the blocks
    already decoded) and one bd_unmask_step (top k by confidence).  Block state
    and tokens stay on the device; nothing returns to the host between steps.
    logits: float32 host array [n_blocks, steps, B, V] of bf16 values, or None
    for seeded N(0, 3) rows drawn on the device."""

    def __init__(self, B: int, layers: int, device, logits=None, seed: int = WAM.seed, num_splits: int = 0):
        import torch
        import block_causal_masked_gb300 as bd
        self.torch, self.bd, self.dev = torch, bd, device
        self.B, self.layers, self.num_splits = B, layers, num_splits
        self.n_blocks = WAM_TOKENS // B
        self.steps = wam_steps(B)
        self.k = max(1, B // 8)
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + B)
        bf = torch.bfloat16
        kv_len = WAM.prefix + WAM_TOKENS
        self.q = [torch.randn((B, WAM.Hq, WAM.D), generator=g, device=device).to(bf) for _ in range(layers)]
        self.kk = [torch.randn((WAM.Hkv, kv_len, WAM.D), generator=g, device=device).to(bf) for _ in range(layers)]
        self.vv = [torch.randn((WAM.Hkv, kv_len, WAM.D), generator=g, device=device).to(bf) for _ in range(layers)]
        self.o = torch.empty((B, WAM.Hq, WAM.D), dtype=bf, device=device)
        self.lse = torch.empty((WAM.Hq, B), dtype=torch.float32, device=device)
        if logits is None:
            self.logits = (torch.randn((self.n_blocks, self.steps, B, synth.VOCAB), generator=g, device=device)
                           * 3.0).to(bf)
        else:
            self.logits = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(device).to(bf)
        self.block = torch.tensor([0, B], dtype=torch.int32, device=device)
        self.logit_row = torch.arange(B, dtype=torch.int32, device=device)
        self.state = torch.zeros(WAM_TOKENS, dtype=torch.uint8, device=device)
        self.tokens = torch.full((WAM_TOKENS,), -1, dtype=torch.int32, device=device)
        self.um = dict(commit=torch.empty(B, dtype=torch.uint8, device=device),
                       n_committed=torch.empty(1, dtype=torch.int32, device=device),
                       status=torch.empty(1, dtype=torch.int32, device=device),
                       pred=torch.empty(B, dtype=torch.int32, device=device),
                       conf=torch.empty(B, dtype=torch.float32, device=device),
                       lse=torch.empty(B, dtype=torch.float32, device=device))
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)
        self.launches = self.n_blocks * self.steps * (layers + 1)

    def _block_step(self, b: int, s: int):
        bd, B = self.bd, self.B
        C = WAM.prefix + b * B
        for l in range(self.layers):
            bd.bd_block_causal_attn(self.q[l], self.kk[l], self.vv[l], C, block_start=self.block, o=self.o,
                                    lse=self.lse, num_splits=self.num_splits, dev_status=self.dev_status)
        bd.bd_unmask_step(self.logits[b, s], self.logit_row, self.block, self.state[b * B:(b + 1) * B],
                          self.tokens[b * B:(b + 1) * B], tau_full=2.0, tau_half=2.0, min_frac=(0, 1),
                          k_fixed=self.k, add_thr=(1, 2), act_thr=(17, 20), dev_status=self.dev_status, **self.um)

    def reset(self):
        self.state.zero_()
        self.tokens.fill_(-1)

    def capture(self):
        torch = self.torch
        self._block_step(0, 0)                    # workspaces and kernel attributes, outside the capture
        torch.cuda.synchronize()
        self.reset()
        stream = torch.cuda.Stream(self.dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            for b in range(self.n_blocks):
                for s in range(self.steps):
                    self._block_step(b, s)
        torch.cuda.synchronize()

    def replay(self):
        self.reset()
        self.graph.replay()


def run_wam_sweep(args, device):
    """One JSON line per block size: committed tokens/s of the whole decode."""
    import torch
    torch.cuda.set_device(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    for B in (1, 4, 8, 16, 32):
        dec = WamDecode(B, WAM.layers, device)
        t0 = time.time()
        dec.capture()
        cap_s = time.time() - t0
        for _ in range(args.warmup):
            dec.replay()
        torch.cuda.synchronize()
        ms = []
        for _ in range(args.steps):
            flush.zero_()
            dec.reset()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            dec.graph.replay()
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        committed = int((dec.state == synth.COMMITTED).sum())
        status = int(dec.dev_status[0])
        t = statistics.median(ms)
        print(json.dumps({"metric": "committed tokens/s (whole decode, one CUDA graph)", "value": committed / t * 1e3,
                          "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_decode": t, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": f"wam_diff2_sweep B={B}: {WAM_TOKENS} tokens, blocks of {B}, top "
                                                 f"{dec.k} per step, {dec.steps} steps per block, 16/8 heads, "
                                                 f"head dim 128, {WAM.layers} layers, prefix {WAM.prefix}",
                                     "gpu_launches_per_decode": dec.launches, "graph_capture_s": round(cap_s, 2),
                                     "l2": "flushed before every timed decode"},
                          "committed": committed, "dev_status": status}), flush=True)
        del dec
        torch.cuda.empty_cache()


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


def cpu_baseline(inp, budget_s: float = 12.0):
    """The float64 oracle on the host cores, full rounds until the budget is spent."""
    import oracle
    t0 = time.perf_counter()
    steps, tokens = 0, 0
    while True:
        tokens += oracle_round(oracle, inp)
        steps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{steps} full round(s) of the workload (72 attention layers, unmask, verify) in float64 "
                      f"numpy, {dt:.1f} s"}


def oracle_round(oracle, inp) -> int:
    from fractions import Fraction
    C, n_q = inp["C"], inp["n_q"]
    for q, _, k, v in inp["layers"]:
        oracle.block_causal_attention(q, k, v, C, [0, n_q])
    r = oracle.unmask_step(inp["logits"], inp["logit_row"], [0, n_q], inp["state"], inp["tokens"], tau_full=TAU,
                           tau_half=TAU, min_frac=Fraction(0, 1), k_fixed=0, add_thr=Fraction(1, 2),
                           act_thr=Fraction(17, 20), write_draft=True)
    for _, q, k, v in inp["layers"]:
        oracle.block_causal_attention(q, k, v, C, list(range(n_q + 1)))
    vr = oracle.spec_verify(r["tokens"][None], r["state"][None], inp["ar_logits"][None])
    return int(r["n_committed"][0]) + int(vr["accepted_len"][0])


def e2e_measure(rd, inp, steps: int):
    """The same round end to end through the library's public calls, captured
    as CUDA graphs the way a serving loop would run them: every step copies
    its inputs (queries of both passes, both logits tensors, state and tokens)
    from pinned host memory and reads its result (committed counts and tokens)
    back to the host, all inside the timed region.  Two device input sets let
    step i+1's copies (on their own stream) overlap step i's kernels."""
    torch = rd.torch
    hq = [torch.from_numpy(np.array(q, copy=True)).to(torch.bfloat16).pin_memory() for q, _, _, _ in inp["layers"]]
    hqa = [torch.from_numpy(np.array(q, copy=True)).to(torch.bfloat16).pin_memory() for _, q, _, _ in inp["layers"]]
    hl = torch.from_numpy(np.array(inp["logits"], copy=True)).to(torch.bfloat16).pin_memory()
    ha = torch.from_numpy(np.array(inp["ar_logits"][None], copy=True)).to(torch.bfloat16).pin_memory()
    hs = torch.from_numpy(inp["state"].copy()).pin_memory()
    ht = torch.from_numpy(inp["tokens"].copy()).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in hq + hqa + [hl, ha, hs, ht])
    sets = [rd, GpuRound(inp, rd.dev)]
    sets[1].capture()
    outs = [torch.empty(2, dtype=torch.int32).pin_memory() for _ in sets]
    out_tok = [torch.empty_like(ht).pin_memory() for _ in sets]
    d2h = outs[0].numel() * 4 + out_tok[0].numel() * 4
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream(rd.dev)
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


def replica_seed(rank: int) -> int:
    """Seed of the request rank `rank` decodes (independent inputs per replica)."""
    return W.seed + 100 * rank


def run_gpu(args, rank, world, local_rank):
    import torch
    device = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    inp = make_inputs(replica_seed(rank))
    rd = GpuRound(inp, device)
    rd.capture()
    clocks = Clocks(local_rank)
    for _ in range(args.warmup):
        rd.timed_step()
        rd.timed_parts()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    steps_ms = []
    committed = 0
    for _ in range(args.steps):
        steps_ms.append(rd.timed_step())
        committed += rd.committed()
    torch.cuda.synchronize()
    # per-kernel times for the roofline: the same round as four graphs
    attn_ms, unmask_ms = [], []
    for _ in range(max(3, min(50, args.steps // 4))):
        _, a, u = rd.timed_parts()
        attn_ms.append(a)
        unmask_ms.append(u)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_s = sum(steps_ms) / 1e3
    total_s, committed_all = aggregate(total_s, committed, world, device)
    e2e = e2e_measure(rd, inp, max(3, min(100, args.steps // 2)))
    if rank != 0:
        return None
    alg = algorithmic(inp)
    peaks = measured_peaks()
    attn_launch_s = (sum(attn_ms) / len(attn_ms)) / 1e3 / (2 * W.layers)
    attn_bytes = (alg["attn_bytes"][0] + alg["attn_bytes"][1]) / 2
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = attn_bytes / attn_launch_s / 1e9
    unmask_s = (sum(unmask_ms) / len(unmask_ms)) / 1e3
    splits = rd.attn_splits()
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
                     "unmask": {"alg_bytes": alg["unmask_bytes"], "us": unmask_s * 1e6,
                                "achieved_gbs": alg["unmask_bytes"] / unmask_s / 1e9,
                                "frac": alg["unmask_bytes"] / unmask_s / 1e9 / hbm}},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
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
    ap.add_argument("--workload", choices=["fast_ddrive", "wam_sweep"], default="fast_ddrive",
                    help="wam_sweep: the whole WAM-Diff2 decode per block size as one CUDA graph (extra lines)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload == "wam_sweep":
        run_wam_sweep(args, int(os.environ.get("LOCAL_RANK", "0")))
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
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
