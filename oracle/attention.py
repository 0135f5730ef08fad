"""Block-causal attention, float64 oracle (test infrastructure only).

Sources (page title, section):

* Fast-dVLA: Accelerating Discrete Diffusion VLA to Real-Time Performance,
  "关键设计 1. 分块因果注意力": a block sees the prompt prefix, every earlier block
  and itself (bidirectionally), never a later block.
* Fast-dDrive method summary (e.mffb.com.cn), §3.1 "分块因果注意力": output cut
  into blocks, bidirectional inside a block, causal across blocks; the finished
  blocks' K/V are reused as a cache.
* WAM-Diff2 write-up (163.com), §2.1 "Block-Causal 注意力": block size 1 is
  ordinary autoregressive decoding.
* FlashDrive tutorial (agifrontier.github.io), "流式推理": keys are cached
  without position encoding and RoPE is applied inside the operator at the
  re-based position p - Δ.
* Fast-dDrive method summary, §3.3 "共享前缀多轨迹Rollout": N rollouts share one
  prefix KV cache and differ only in their trajectory part.

Readings where the pages are silent:

* query head h uses KV head h // (Hq / Hkv) (contiguous GQA grouping);
* softmax scale D^-1/2, LSE in natural log;
* RoPE is rotate-half over the pairs (d, d + D/2) with frequency theta^(-2d/D);
  the rotated key, an operand of the bf16 QK^T product like any cached key,
  is held in bf16 (round to nearest even) before the product;
* Q and the active positions' keys arrive already rotated; only the cached
  prefix rows are rotated in the operator.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (8 significant bits, ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    m = np.rint(m * 256.0) / 256.0     # keep 8 significant bits; rint rounds half to even
    return np.ldexp(m, e)


def visibility_mask(C: int, block_start) -> np.ndarray:
    """Explicit mask[i, j]: may active position i attend to key j?

    Keys are the C cached prefix rows followed by the n_q active positions.
    Query i in block b(i) sees every prefix key and every active key whose
    block is b(i) or earlier.
    """
    bs = [int(x) for x in block_start]
    n_q = bs[-1]
    block_of = np.empty(n_q, dtype=np.int64)
    for b in range(len(bs) - 1):
        block_of[bs[b]:bs[b + 1]] = b
    mask = np.zeros((n_q, C + n_q), dtype=bool)
    mask[:, :C] = True
    mask[:, C:] = block_of[None, :] <= block_of[:, None]
    return mask


def rope_rotate(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [..., S, D] at integer positions pos [S], in float64."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    freq = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / D)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def block_causal_attention(q, k, v, C: int, block_start, sm_scale: float | None = None,
                           k_pos=None, delta: int = 0, theta: float = 10000.0,
                           rope: bool = False):
    """O and LSE of the active positions' queries over prefix + active keys.

    q: [n_q, Hq, D]; k, v: [Hkv, >= C + n_q, D] (rows [0, C) cached prefix,
    rows [C, C + n_q) active positions).  With ``rope`` the prefix keys are
    pre-RoPE and get rotated at position k_pos[s] - delta (k_pos defaults to s).
    Returns o [n_q, Hq, D] and lse [Hq, n_q], float64.
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, Hq, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    S = C + n_q
    kk = np.array(k[:, :S], dtype=np.float64)
    vv = np.array(v[:, :S], dtype=np.float64)
    if rope and C > 0:
        pos = np.arange(C) if k_pos is None else np.asarray(k_pos[:C], dtype=np.int64)
        kk[:, :C] = round_bf16(rope_rotate(kk[:, :C], pos - int(delta), theta))
    scale = D ** -0.5 if not sm_scale else float(sm_scale)
    mask = visibility_mask(C, block_start)
    o = np.empty((n_q, Hq, D))
    lse = np.empty((Hq, n_q))
    for h in range(Hq):
        kv = h // G
        s = (q[:, h, :] @ kk[kv].T) * scale
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o[:, h, :] = (p @ vv[kv]) / l
        lse[h] = (m + np.log(l))[:, 0]
    return o, lse


def fork_attention(q, prefix_k, prefix_v, priv_k, priv_v, priv_len: int, block_start,
                   sm_scale: float | None = None, k_pos=None, delta: int = 0,
                   theta: float = 10000.0, rope: bool = False):
    """N rollouts forked from one shared prefix.

    Rollout r attends over [prefix ‖ its private rows [0, priv_len) ‖ its active
    block]; the private rows (its earlier trajectory blocks) are visible to all of
    its active queries, the active rows block-causally.  Computed per rollout on
    an explicit concatenation.  q: [N, n_q, Hq, D]; prefix_k/v: [Hkv, C, D];
    priv_k/v: [N, Hkv, priv_len + n_q, D].  Returns o [N, n_q, Hq, D], lse [N, Hq, n_q].
    """
    q = np.asarray(q, dtype=np.float64)
    N, n_q, Hq, D = q.shape
    C = prefix_k.shape[1]
    pk = np.array(prefix_k, dtype=np.float64)
    if rope and C > 0:
        pos = np.arange(C) if k_pos is None else np.asarray(k_pos[:C], dtype=np.int64)
        pk = round_bf16(rope_rotate(pk, pos - int(delta), theta))
    o = np.empty((N, n_q, Hq, D))
    lse = np.empty((N, Hq, n_q))
    for r in range(N):
        k = np.concatenate([pk, np.asarray(priv_k[r, :, :priv_len + n_q], np.float64)], axis=1)
        v = np.concatenate([np.asarray(prefix_v, np.float64),
                            np.asarray(priv_v[r, :, :priv_len + n_q], np.float64)], axis=1)
        o[r], lse[r] = block_causal_attention(q[r], k, v, C + priv_len, block_start, sm_scale)
    return o, lse
