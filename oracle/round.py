"""One scaffold-speculative decode round, float64 oracle (test infrastructure only).

Fast-dDrive method summary (e.mffb.com.cn), §3.2 "模式二：Scaffold Speculative
Decoding", steps 1-3, with the Fast-dDrive-shaped workload's threshold commits
in front: one MDM forward over the active block (block-causal attention, the
block bidirectional), the threshold commits and the draft of every still-masked
editable position from its logits, one AR forward (block size 1: causal), and
the left-to-right verification of the draft with its bonus token.

The composition only calls this package's functions, in the pages' order; each
of them is pinned on its own.
"""
from __future__ import annotations

from fractions import Fraction

from .attention import block_causal_attention
from .unmask import unmask_step
from .verify import spec_verify


def speculative_round(layers, C: int, n_q: int, logits, logit_row, state, tokens, ar_logits, tau: float):
    """Runs the round; returns (committed editable positions, unmask result,
    verify result).  layers: per layer (q_mdm [n_q, Hq, D], q_ar [n_q, Hq, D],
    k, v [Hkv, >= C + n_q, D])."""
    for q, _, k, v in layers:
        block_causal_attention(q, k, v, C, [0, n_q])
    r = unmask_step(logits, logit_row, [0, n_q], state, tokens, tau_full=tau, tau_half=tau,
                    min_frac=Fraction(0, 1), k_fixed=0, add_thr=Fraction(1, 2), act_thr=Fraction(17, 20),
                    write_draft=True)
    for _, q, k, v in layers:
        block_causal_attention(q, k, v, C, list(range(n_q + 1)))
    vr = spec_verify(r["tokens"][None], r["state"][None], ar_logits[None])
    return int(r["n_committed"][0]) + int(vr["accepted_len"][0]), r, vr
