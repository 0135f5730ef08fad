"""Plain, slow, float64 CPU oracle of the block-causal masked-diffusion decode step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The library under ``block_causal_masked_gb300/`` never calls into it and shares no
code with it: the two meet only through the seeded inputs of ``synth/``.

Every function states the method as the pages define it, with no blocking,
fusion or reordering beyond that definition:

* ``attention``  block-causal attention with an explicit mask matrix, GQA,
                 optional RoPE on pre-RoPE cached keys, and the shared-prefix fork.
* ``unmask``     argmax / max-softmax-probability per masked position and the
                 per-block commit rule (scaffold frozen, threshold, minimum
                 fraction, half/full activation from the predecessor's completion).
* ``verify``     scaffold-speculative verification (greedy or Gumbel-max sampled).
* ``stream``     the streaming cache: a new frame written into every view's frame
                 slot, and the streaming (position-causal) attention mask.
* ``round``      one scaffold-speculative round (MDM attention, threshold
                 commits + draft, AR attention, verification), composed of the
                 functions above.
* ``kvquant``    the FP8 (E4M3) KV cache with per-(head, 128-row block)
                 power-of-two scales, dequantised exactly to float64.

Where the pages leave a step open, the docstrings name the reading taken.
Parity of every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (closed forms, special cases, invariants, brute force
and the pages' printed section table); none is unpinned.
"""
from . import attention, kvquant, round, stream, unmask, verify  # noqa: F401
from .attention import (block_causal_attention, fork_attention, rope_rotate,  # noqa: F401
                        round_bf16, visibility_mask)
from .stream import stream_attention, stream_insert, streaming_mask  # noqa: F401
from .unmask import row_stats, unmask_step  # noqa: F401
from .verify import gumbel_scores, spec_verify  # noqa: F401
from .round import speculative_round  # noqa: F401
from .kvquant import dequantize as dequantize_kv, e4m3_value  # noqa: F401

MASKED, COMMITTED, SCAFFOLD = 0, 1, 2
INACTIVE, HALF, FULL, DONE = 0, 1, 2, 3
