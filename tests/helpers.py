"""Shared helpers of the GPU parity tests: moving seeded inputs to the device and
the tolerances the workload fixes.

Attention: |o - o_ref| <= 1e-2 + 1e-2 |o_ref| element-wise, LSE within 1e-5
relative (plus 1e-6 absolute: an LSE near zero -- a row that sees one or two
keys -- is one or two scores, and a score's fp32 error is absolute, about
2^-24 times the sum of |q_d k_d| / sqrt(D) over its D terms, ~5e-7 for N(0, 1)
inputs at D = 128; no relative bound can hold there).  Integer and index
outputs: bit-exact.  Confidences: 2e-6 relative
(fp32 accumulation over the vocabulary against float64); the commit decisions
taken from them are exact because every input is drawn with decision margins
that the tests assert (see the ``margins`` returned by the oracle).
"""
import numpy as np
import torch

import oracle
import synth

DEV = "cuda:0"
O_ATOL, O_RTOL = 1e-2, 1e-2
LSE_RTOL = 1e-5
CONF_RTOL = 2e-6


def bf16(x) -> torch.Tensor:
    return torch.from_numpy(np.array(x, dtype=np.float32, order='C', copy=True)).to(DEV).to(torch.bfloat16)


def f32(x) -> torch.Tensor:
    return torch.from_numpy(np.array(x, dtype=np.float32, order='C', copy=True)).to(DEV)


def i32(x) -> torch.Tensor:
    return torch.from_numpy(np.array(x, dtype=np.int32, order='C', copy=True)).to(DEV)


def u8(x) -> torch.Tensor:
    return torch.from_numpy(np.array(x, dtype=np.uint8, order='C', copy=True)).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def assert_attn_close(o, lse, o_ref, lse_ref, what=""):
    o = host(o).astype(np.float64)
    lse = host(lse).astype(np.float64)
    err = np.abs(o - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outputs off; worst {np.max(err - bound):.3g} over bound"
    lerr = np.abs(lse - lse_ref)
    lb = LSE_RTOL * np.abs(lse_ref) + 1e-6
    assert not (lerr > lb).any(), f"{what}: lse off by up to {np.max(lerr / np.maximum(np.abs(lse_ref), 1e-30)):.3g} relative"


def status_word() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def bf16_midpoint_distance(x) -> np.ndarray:
    """Distance of each float64 value to the nearest midpoint between two bf16
    values (where rounding to bf16 changes its result); +inf for 0."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    m, e = np.frexp(x)                       # x = m * 2**e, 0.5 <= m < 1
    scaled = m * 256.0                       # bf16 values are the integers here
    d = np.abs(scaled - np.floor(scaled) - 0.5) * np.ldexp(1.0, e - 8)
    return np.where(x == 0.0, np.inf, d)
