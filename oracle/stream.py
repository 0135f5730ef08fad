"""Streaming new-frame insertion and the streaming attention mask, float64
oracle (test infrastructure only).

Source: FlashDrive tutorial (agifrontier.github.io), section "流式推理":

* only the newest camera frame is encoded; the K/V of the history frames come
  from the cache kept from earlier steps;
* visual tokens are laid out view-major (every frame of camera A, then camera
  B, ...), so the new frame's tokens go into each view's own frame slot, not at
  the end of the cache;
* a causal constraint in the mask makes the new tokens queries over the cached
  history while keeping the causal structure across views;
* keys are stored without position encoding and rotated inside the operator at
  the re-based position p - Δ.

Readings where the page is silent:

* The cache holds a fixed window of ``frames`` frame slots per view.  A step
  overwrites, in every view, the slot the caller names (the slot of that
  view's oldest frame: a ring).  The physical order of keys inside the cache
  does not change attention, because each key carries its own position.
* Positions are integers in the caller's view-major numbering of an
  ever-growing sequence; the operator subtracts Δ (how far the window has slid)
  for RoPE and for the mask alike.
* The streaming mask is causal in those positions: query i sees cached key j
  iff pos(j) - Δ <= q_pos(i).  With view-major positions that is every earlier
  view, the history of the query's own view and its own frame up to itself.
  A query that sees no key gets o = 0 and lse = -inf.
"""
from __future__ import annotations

import numpy as np

from .attention import rope_rotate, round_bf16


def stream_insert(k_cache, v_cache, k_pos, new_k, new_v, new_pos, views: int, frames: int, per_frame: int,
                  slot: int):
    """The cache after writing the new frame into frame slot ``slot`` of every view.

    k_cache, v_cache: [Hkv, >= views * frames * per_frame, D]; k_pos: [views *
    frames * per_frame]; new_k, new_v: [views * per_frame, Hkv, D] (the new
    frame's tokens, view by view); new_pos: [views * per_frame].  Slot s of view
    w holds cache rows [(w * frames + s) * per_frame, ... + per_frame).
    Returns new arrays (k, v, k_pos); the inputs are not modified.
    """
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    kp = np.array(k_pos, copy=True)
    for w in range(views):
        for t in range(per_frame):
            dst = (w * frames + slot) * per_frame + t
            src = w * per_frame + t
            k[:, dst, :] = new_k[src]
            v[:, dst, :] = new_v[src]
            kp[dst] = new_pos[src]
    return k, v, kp


def streaming_mask(k_pos, delta: int, q_pos) -> np.ndarray:
    """mask[i, j]: may the query at q_pos[i] attend to the cached key j?"""
    kp = np.asarray(k_pos, dtype=np.int64) - int(delta)
    return kp[None, :] <= np.asarray(q_pos, dtype=np.int64)[:, None]


def stream_attention(q, k, v, C: int, k_pos, delta: int, q_pos, sm_scale: float | None = None,
                     theta: float = 10000.0, rope: bool = False):
    """O and LSE of queries at positions q_pos over the cached keys [0, C).

    The cache already holds the new frame's own keys (inserted first).  q:
    [n_q, Hq, D]; k, v: [Hkv, >= C, D]; k_pos: [C] (None: key index); with
    ``rope`` the cached keys are pre-RoPE and rotated at k_pos - delta.
    Returns o [n_q, Hq, D] and lse [Hq, n_q], float64.
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, Hq, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    pos = np.arange(C) if k_pos is None else np.asarray(k_pos[:C], dtype=np.int64)
    kk = np.array(k[:, :C], dtype=np.float64)
    vv = np.array(v[:, :C], dtype=np.float64)
    if rope and C > 0:
        kk = round_bf16(rope_rotate(kk, pos - int(delta), theta))
    scale = D ** -0.5 if not sm_scale else float(sm_scale)
    mask = streaming_mask(pos, delta, q_pos)
    o = np.zeros((n_q, Hq, D))
    lse = np.full((Hq, n_q), -np.inf)
    seen = mask.any(axis=1)
    for h in range(Hq):
        kv = h // G
        s = (q[:, h, :] @ kk[kv].T) * scale
        s = np.where(mask, s, -np.inf)
        for i in np.flatnonzero(seen):
            m = s[i].max()
            p = np.exp(s[i] - m)
            l = p.sum()
            o[i, h, :] = (p @ vv[kv]) / l
            lse[h, i] = m + np.log(l)
    return o, lse
