"""Seeded synthetic inputs for the block-causal masked-diffusion decode step.

This module only *draws* numbers and lays them out in the shapes of the workloads
that the pages describe.  It computes nothing of the decode step itself: no
attention, no commit rule, no verification, no sampling.  Both the CPU oracle
(``oracle/``) and the GPU path consume what it returns; neither imports the other.

Every generator takes an explicit integer seed and uses numpy's PCG64 stream,
which gives the same numbers on x86-64 and aarch64.

bf16 values are returned as float32 arrays whose values are exactly
representable in bf16 (round-to-nearest-even), so that converting them to a
bf16 tensor is exact.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence, Tuple

import numpy as np

VOCAB = 151_936  # Qwen2.5/Qwen3 vocabulary width used by the backbones on the pages

# position states shared by every call of the library
MASKED, COMMITTED, SCAFFOLD = 0, 1, 2


def rng(seed: int, *stream: int) -> np.random.Generator:
    """Independent PCG64 stream for ``(seed, *stream)``."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even); returns float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


# --------------------------------------------------------------------------------------
# output layouts
# --------------------------------------------------------------------------------------

@dataclasses.dataclass
class Layout:
    """Positions of a structured output.

    ``scaffold[p]`` is 1 for a frozen template token, ``section[p]`` its section,
    ``block_start`` the block partition over positions (len n_blocks + 1),
    ``block_section[b]`` the section of block b.
    """

    scaffold: np.ndarray
    section: np.ndarray
    block_start: np.ndarray
    block_section: np.ndarray

    @property
    def n_pos(self) -> int:
        return int(self.scaffold.shape[0])

    @property
    def n_blocks(self) -> int:
        return int(self.block_start.shape[0] - 1)


# Fast-dDrive's JSON schema sections: (editable value tokens, scaffold tokens) for
# critical_objects, explanation, future_meta_behavior, trajectory.
DDRIVE_SECTIONS: Tuple[Tuple[int, int], ...] = ((12, 80), (192, 6), (6, 18), (70, 20))


def section_layout(seed: int, sections: Sequence[Tuple[int, int]] = DDRIVE_SECTIONS,
                   d: int = 32) -> Layout:
    """Place each section's scaffold tokens at seeded slots and cut it into blocks.

    A section with E editable tokens is cut into ceil(E/d) blocks of d editable
    tokens (the last one ragged).  A scaffold token belongs to the block of the
    next editable token of its section; trailing scaffold tokens go to the
    section's last block.  So block k >= 1 of a section starts right after the
    section's (k*d)-th editable token.
    """
    g = rng(seed, 101)
    scaffold: List[int] = []
    section: List[int] = []
    starts: List[int] = []
    bsec: List[int] = []
    for s, (n_edit, n_scaf) in enumerate(sections):
        n = n_edit + n_scaf
        flags = np.zeros(n, dtype=np.uint8)
        flags[g.choice(n, size=n_scaf, replace=False)] = 1
        edit_slots = np.flatnonzero(flags == 0)
        base = len(scaffold)
        n_blk = -(-n_edit // d)
        starts.append(base)
        for k in range(1, n_blk):
            starts.append(base + int(edit_slots[k * d - 1]) + 1)
        bsec.extend([s] * n_blk)
        scaffold.extend(int(f) for f in flags)
        section.extend([s] * n)
    starts.append(len(scaffold))
    return Layout(np.array(scaffold, np.uint8), np.array(section, np.int32),
                  np.array(starts, np.int32), np.array(bsec, np.int32))


def uniform_layout(n_pos: int, block: int, scaffold_per_block: int = 0, seed: int = 0) -> Layout:
    """``n_pos`` positions in blocks of ``block``; ``scaffold_per_block`` seeded scaffold slots each."""
    g = rng(seed, 102)
    scaffold = np.zeros(n_pos, np.uint8)
    bs = list(range(0, n_pos, block)) + [n_pos]
    for b in range(len(bs) - 1):
        n = bs[b + 1] - bs[b]
        k = min(scaffold_per_block, n)
        if k:
            scaffold[bs[b] + g.choice(n, size=k, replace=False)] = 1
    return Layout(scaffold, np.zeros(n_pos, np.int32), np.array(bs, np.int32),
                  np.zeros(len(bs) - 1, np.int32))


# --------------------------------------------------------------------------------------
# attention inputs
# --------------------------------------------------------------------------------------

@dataclasses.dataclass
class AttnCase:
    """One layer's attention inputs (bf16 values held in float32).

    q: [n_q, Hq, D]; k, v: [Hkv, kv_stride, D] with rows [0, C) the cached prefix and
    rows [C, C + n_q) the active positions' keys/values; rows past C + n_q are padding.
    ``block_start`` partitions the n_q active positions (len n_blocks + 1).
    """

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    C: int
    block_start: np.ndarray

    @property
    def n_q(self) -> int:
        return int(self.q.shape[0])


def _normal_bf16(g: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    return to_bf16(g.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def attn_case(seed: int, layer: int, *, C: int, block_start: Sequence[int], Hq: int, Hkv: int,
              D: int, text_from: int | None = None, text_bias_norm: float = 2.0,
              kv_pad: int = 0) -> AttnCase:
    """Q/K/V ~ N(0, 1) in bf16.

    Prefix rows ``[text_from, C)`` (text tokens) additionally carry a per-KV-head
    bias vector of norm ``text_bias_norm`` shared by all of them, which makes the
    softmax over those keys more peaked than over the image-like rows.
    """
    g = rng(seed, 200, layer)
    n_q = int(block_start[-1])
    kv_stride = C + n_q + kv_pad
    q = _normal_bf16(g, (n_q, Hq, D))
    k = g.standard_normal((Hkv, kv_stride, D), dtype=np.float32)
    v = g.standard_normal((Hkv, kv_stride, D), dtype=np.float32)
    if text_from is not None and text_from < C:
        bias = g.standard_normal((Hkv, D)).astype(np.float32)
        bias *= np.float32(text_bias_norm) / np.linalg.norm(bias, axis=1, keepdims=True).astype(np.float32)
        k[:, text_from:C, :] += bias[:, None, :]
    k = to_bf16(k)
    v = to_bf16(v)
    return AttnCase(q, k, v, C, np.asarray(block_start, np.int32))


@dataclasses.dataclass
class ForkCase:
    """Shared-prefix fork inputs.

    prefix_k/v: [Hkv, C, D] (pre-RoPE keys when ``k_pos`` is given);
    q: [N, n_q, Hq, D]; priv_k/v: [N, Hkv, priv_len + n_q, D].
    """

    q: np.ndarray
    prefix_k: np.ndarray
    prefix_v: np.ndarray
    priv_k: np.ndarray
    priv_v: np.ndarray
    priv_len: int
    block_start: np.ndarray
    k_pos: np.ndarray | None
    delta: int
    theta: float

    @property
    def N(self) -> int:
        return int(self.q.shape[0])

    @property
    def C(self) -> int:
        return int(self.prefix_k.shape[1])


def streaming_prefix_positions(views: int = 4, frames: int = 4, per_frame: int = 256,
                               sections: int = 210, delta: int = 256) -> np.ndarray:
    """Absolute positions of the cached prefix keys before the window slid by ``delta``.

    The window is stored view-major (all frames of view 0, then view 1, ...).  After
    the slide every key sits at ``k_pos - delta``, i.e. contiguously from 0; the
    section tokens that follow the window continue the count.
    """
    n = views * frames * per_frame + sections
    return (np.arange(n, dtype=np.int64) + delta).astype(np.int32)


def fork_case(seed: int, layer: int, *, N: int, C: int, n_q: int, priv_len: int,
              block_start: Sequence[int], Hq: int, Hkv: int, D: int,
              k_pos: np.ndarray | None = None, delta: int = 0, theta: float = 10000.0) -> ForkCase:
    g = rng(seed, 300, layer)
    q = _normal_bf16(g, (N, n_q, Hq, D))
    pk = _normal_bf16(g, (Hkv, C, D))
    pv = _normal_bf16(g, (Hkv, C, D))
    rk = _normal_bf16(g, (N, Hkv, priv_len + n_q, D))
    rv = _normal_bf16(g, (N, Hkv, priv_len + n_q, D))
    return ForkCase(q, pk, pv, rk, rv, priv_len, np.asarray(block_start, np.int32), k_pos, delta, theta)


# --------------------------------------------------------------------------------------
# vocab logits
# --------------------------------------------------------------------------------------

def normal_logits(seed: int, stream: int, R: int, V: int = VOCAB, sigma: float = 3.0,
                  bf16: bool = True) -> np.ndarray:
    """Rows ~ N(0, sigma^2) (rounded to bf16 unless ``bf16`` is False)."""
    g = rng(seed, 400, stream)
    x = g.standard_normal((R, V), dtype=np.float32) * np.float32(sigma)
    return to_bf16(x) if bf16 else x


def plant_peak(row: np.ndarray, token: int, target: float, bf16: bool = True) -> float:
    """Set ``row[token]`` so that the row's largest softmax probability is about ``target``.

    Input construction: the value is solved from the sum of the other entries'
    exponentials, written in place, rounded to bf16 when ``bf16``; returns the
    probability the planted entry actually has after rounding (computed here in
    float64 from the row as stored).
    """
    rest = np.delete(row.astype(np.float64), token)
    mx = rest.max()
    z_rest = np.exp(rest - mx).sum()
    a = mx + math.log(target * z_rest / (1.0 - target))
    val = np.float32(a)
    if bf16:
        val = to_bf16(np.array([val]))[0]
    row[token] = val
    return float(1.0 / (1.0 + z_rest * math.exp(mx - float(val))))


def planted_logits(seed: int, stream: int, R: int, V: int = VOCAB, sigma: float = 3.0,
                   lo: float = 0.3, hi: float = 0.99, tokens: Sequence[int] | None = None,
                   bf16: bool = True) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """N(0, sigma^2) rows, each with one planted peaked token of probability ~ U(lo, hi).

    Returns (logits [R, V] float32, planted token per row, achieved peak
    probability per row).  ``tokens`` fixes the planted token of each row
    (``-1`` draws one).
    """
    x = normal_logits(seed, stream, R, V, sigma, bf16)
    g = rng(seed, 401, stream)
    tok = g.integers(0, V, size=R)
    if tokens is not None:
        t = np.asarray(tokens)
        tok = np.where(t >= 0, t, tok)
    target = g.uniform(lo, hi, size=R)
    achieved = np.empty(R)
    for r in range(R):
        achieved[r] = plant_peak(x[r], int(tok[r]), float(target[r]), bf16)
    return x, tok.astype(np.int32), achieved


def uniform_noise(seed: int, stream: int, shape) -> np.ndarray:
    """u ~ U[2^-24, 1 - 2^-24] in float32 (the closed range keeps -log(-log u) finite)."""
    g = rng(seed, 500, stream)
    u = g.random(shape, dtype=np.float32)
    return np.clip(u, np.float32(2.0 ** -24), np.float32(1.0 - 2.0 ** -24)).astype(np.float32)


def redraw_rows(seed: int, stream: int, x: np.ndarray, rows: Sequence[int], attempt: int,
                sigma: float = 3.0, bf16: bool = True) -> None:
    """Replace the given rows of ``x`` with fresh N(0, sigma^2) draws (in place)."""
    for r in rows:
        g = rng(seed, 402, stream, int(r), attempt)
        y = g.standard_normal(x.shape[1], dtype=np.float32) * np.float32(sigma)
        x[r] = to_bf16(y) if bf16 else y


def redraw_noise_rows(seed: int, stream: int, u: np.ndarray, rows: Sequence[int], attempt: int) -> None:
    """Replace the given rows of a [R, V] noise array with fresh uniforms (in place)."""
    for r in rows:
        g = rng(seed, 501, stream, int(r), attempt)
        y = g.random(u.shape[-1], dtype=np.float32)
        u[r] = np.clip(y, np.float32(2.0 ** -24), np.float32(1.0 - 2.0 ** -24))


# --------------------------------------------------------------------------------------
# the five workloads (shapes and recipes; sizes from the pages' models)
# --------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    Hq: int
    Hkv: int
    D: int
    layers: int
    prefix: int
    V: int
    logits_bf16: bool


TINY = Workload("tiny", 0, 4, 2, 64, 1, 256, 1024, False)
FAST_DDRIVE = Workload("fast_ddrive", 1, 16, 2, 128, 36, 3000, VOCAB, True)
WAM_SWEEP = Workload("wam_diff2_sweep", 2, 16, 8, 128, 36, 2048, VOCAB, True)
FAST_DVLA = Workload("fast_dvla", 3, 16, 2, 128, 36, 600, VOCAB, True)
FORK_STREAM = Workload("fork_streaming", 4, 16, 2, 128, 36, 4096 + 210, VOCAB, True)
WORKLOADS = {w.name: w for w in (TINY, FAST_DDRIVE, WAM_SWEEP, FAST_DVLA, FORK_STREAM)}


# --------------------------------------------------------------------------------------
# whole-step inputs of the workloads the benchmark times
# --------------------------------------------------------------------------------------

DDRIVE_TAU = 0.9      # confidence threshold of the Fast-dDrive-shaped round's MDM commits
WAM_TOKENS = 256      # output length of the WAM-Diff2 block sweep


def wam_k(B: int) -> int:
    """Commits per denoise step of the WAM-Diff2 sweep at block size B: B / 8, at least 1."""
    return max(1, B // 8)


def wam_steps(B: int) -> int:
    """Denoise steps per block of the WAM-Diff2 sweep: at most 8, and a block
    ends once complete (top k = wam_k(B) commits per step)."""
    return min(8, -(-B // wam_k(B)))


def fast_ddrive_round(seed: int) -> dict:
    """Host inputs of one scaffold-speculative round of the Fast-dDrive-shaped
    workload (float32 arrays holding bf16 values).

    The active block is the second explanation block of the 404-position
    scaffolded output; its cache is the 3,000-token prompt plus the blocks
    decoded before it.  Per layer: the MDM pass's queries, the AR pass's
    queries, K and V (the prompt's 300 text rows carry a shared bias).  MDM
    logits of the editable rows have one planted token each, its softmax
    probability ~ U(0.3, 0.99); the AR rows agree with the planted tokens on
    every row at or above the threshold and on the first ``planted_accept``
    rows below it, and disagree on the next one.
    """
    W = FAST_DDRIVE
    lay = section_layout(W.seed)
    active = 2
    C = W.prefix + int(lay.block_start[active])
    lo, hi = int(lay.block_start[active]), int(lay.block_start[active + 1])
    n_q = hi - lo
    scaf = lay.scaffold[lo:hi].astype(np.int64)
    E = int((scaf == 0).sum())
    layers = []
    for l in range(W.layers):
        a = attn_case(seed, l, C=C, block_start=[0, n_q], Hq=W.Hq, Hkv=W.Hkv, D=W.D, text_from=2700)
        q_ar = attn_case(seed, 1000 + l, C=0, block_start=[0, n_q], Hq=W.Hq, Hkv=1, D=W.D).q
        layers.append((a.q, q_ar, a.k, a.v))
    logits, tok, conf = planted_logits(seed, 1, E, W.V)
    g = rng(seed, 77)
    masked_rows = [e for e in range(E) if conf[e] < DDRIVE_TAU]
    k = int(g.integers(0, len(masked_rows) + 1))
    want = g.integers(0, W.V, size=E + 1)
    for e in range(E):
        if conf[e] >= DDRIVE_TAU or e in masked_rows[:k]:
            want[e] = tok[e]
    if k < len(masked_rows):
        e = masked_rows[k]
        want[e] = (tok[e] + 1) % W.V
    ar_logits, _, _ = planted_logits(seed, 2, E + 1, W.V, tokens=want)
    state = np.where(scaf == 1, SCAFFOLD, MASKED).astype(np.uint8)
    tokens = np.where(scaf == 1, 11, -1).astype(np.int32)
    logit_row = np.full(n_q, -1, np.int32)
    logit_row[scaf == 0] = np.arange(E)
    return dict(C=C, n_q=n_q, E=E, layers=layers, logits=logits, ar_logits=ar_logits, state=state,
                tokens=tokens, logit_row=logit_row, planted_accept=k, planted_conf=conf)


# --------------------------------------------------------------------------------------
# FP8 (E4M3) KV cache: what a cache writer stores
# --------------------------------------------------------------------------------------

KV_BLOCK = 128        # cache rows per power-of-two scale
E4M3_MAX = 448.0


def _e4m3_grid() -> Tuple[np.ndarray, np.ndarray]:
    """The non-negative finite E4M3 values in increasing order and their bytes
    (exponent field e, mantissa m: e = 0 gives m 2^-9, else (8 + m) 2^(e - 10);
    S.1111.111 is not a value)."""
    vals, codes = [], []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append(m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10))
            codes.append((e << 3) | m)
    return np.array(vals), np.array(codes, dtype=np.uint8)


def quantize_kv_e4m3(x: np.ndarray, block: int = KV_BLOCK) -> Tuple[np.ndarray, np.ndarray]:
    """Store x [H, S, D] as E4M3 bytes with one power-of-two scale per (head,
    block of `block` rows): exp = the smallest e with max|x| 2^-e <= 448 in the
    block, then each x 2^-exp rounded to the nearest E4M3 value (ties to the
    even mantissa).  Returns (bytes uint8 [H, S, D], exponents int8 [H, ceil(S / block)])."""
    x = np.asarray(x, dtype=np.float64)
    H, S, D = x.shape
    nb = -(-S // block)
    exps = np.zeros((H, nb), np.int8)
    grid, codes = _e4m3_grid()
    q = np.empty((H, S, D), np.uint8)
    for h in range(H):
        for b in range(nb):
            blk = x[h, b * block:(b + 1) * block]
            amax = float(np.abs(blk).max()) if blk.size else 0.0
            e = int(np.ceil(np.log2(amax / E4M3_MAX))) if amax > 0 else 0
            exps[h, b] = e
            y = np.abs(blk) * 2.0 ** -e
            hi = np.clip(np.searchsorted(grid, y, side="left"), 0, len(grid) - 1)
            lo = np.clip(hi - 1, 0, len(grid) - 1)
            dlo, dhi = y - grid[lo], grid[hi] - y
            pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
            idx = np.where(y >= grid[-1], len(grid) - 1, np.where(pick_hi, hi, lo))
            q[h, b * block:(b + 1) * block] = codes[idx] | np.where(blk < 0, 0x80, 0).astype(np.uint8)
    return q, exps
