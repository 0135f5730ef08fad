"""Python binding of libbd, the C-ABI library of the block-causal masked-diffusion
decode step on GB300 (sm_103a).

Argument marshalling only: every function here fills the C struct declared in
``include/bd.h`` from torch tensors (device memory and the current stream) and
calls the library entry point of the same name.  All arithmetic runs in the
library's CUDA kernels; there is no fallback.  If the library cannot be loaded
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as ct
import os
import threading

import torch

from . import _build

__all__ = ["bd_block_causal_attn", "bd_fork_rollouts", "bd_unmask_step", "bd_unmask_step_noalloc",
           "bd_spec_verify", "bd_stream_insert", "bd_rope_keys", "bd_check",
           "bd_status_string", "lib", "BdError", "Workspace", "MASKED", "COMMITTED", "SCAFFOLD",
           "INACTIVE", "HALF", "FULL", "DONE"]

MASKED, COMMITTED, SCAFFOLD = 0, 1, 2
INACTIVE, HALF, FULL, DONE = 0, 1, 2, 3
BD_F32, BD_BF16, BD_E4M3 = 0, 1, 2


class BdError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({bd_status_string(status)})")
        self.status = status


class bd_rope(ct.Structure):
    _fields_ = [("enabled", ct.c_int32), ("k_pos", ct.c_void_p), ("delta", ct.c_int32), ("theta", ct.c_float)]


class bd_attn_args(ct.Structure):
    _fields_ = [("q", ct.c_void_p), ("k", ct.c_void_p), ("v", ct.c_void_p), ("o", ct.c_void_p), ("lse", ct.c_void_p),
                ("block_start", ct.c_void_p), ("n_blocks", ct.c_int32), ("block_size", ct.c_int32),
                ("C", ct.c_int32), ("n_q", ct.c_int32), ("Hq", ct.c_int32), ("Hkv", ct.c_int32), ("D", ct.c_int32),
                ("kv_stride", ct.c_int32), ("sm_scale", ct.c_float), ("rope", bd_rope),
                ("num_splits", ct.c_int32), ("workspace", ct.c_void_p), ("workspace_bytes", ct.c_size_t),
                ("dev_status", ct.c_void_p), ("prefix_ready", ct.c_int32), ("q_pos", ct.c_void_p),
                ("wait_limit_ns", ct.c_uint64), ("kv_dtype", ct.c_int32), ("k_exp", ct.c_void_p),
                ("v_exp", ct.c_void_p)]


class bd_fork_args(ct.Structure):
    _fields_ = [("N", ct.c_int32), ("q", ct.c_void_p), ("prefix_k", ct.c_void_p), ("prefix_v", ct.c_void_p),
                ("prefix_stride", ct.c_int32), ("priv_k", ct.c_void_p), ("priv_v", ct.c_void_p),
                ("priv_stride", ct.c_int32), ("priv_len", ct.c_int32), ("o", ct.c_void_p), ("lse", ct.c_void_p),
                ("block_start", ct.c_void_p), ("n_blocks", ct.c_int32), ("block_size", ct.c_int32),
                ("C", ct.c_int32), ("n_q", ct.c_int32), ("Hq", ct.c_int32), ("Hkv", ct.c_int32), ("D", ct.c_int32),
                ("sm_scale", ct.c_float), ("rope", bd_rope), ("num_splits", ct.c_int32),
                ("workspace", ct.c_void_p), ("workspace_bytes", ct.c_size_t), ("dev_status", ct.c_void_p),
                ("prefix_ready", ct.c_int32), ("wait_limit_ns", ct.c_uint64), ("kv_dtype", ct.c_int32),
                ("prefix_k_exp", ct.c_void_p), ("prefix_v_exp", ct.c_void_p), ("priv_k_exp", ct.c_void_p),
                ("priv_v_exp", ct.c_void_p)]


class bd_stream_insert_args(ct.Structure):
    _fields_ = [("k_cache", ct.c_void_p), ("v_cache", ct.c_void_p), ("k_pos", ct.c_void_p), ("new_k", ct.c_void_p),
                ("new_v", ct.c_void_p), ("new_pos", ct.c_void_p), ("views", ct.c_int32), ("frames", ct.c_int32),
                ("per_frame", ct.c_int32), ("slot", ct.c_int32), ("Hkv", ct.c_int32), ("D", ct.c_int32),
                ("cache_stride", ct.c_int32)]


class bd_rope_keys_args(ct.Structure):
    _fields_ = [("k", ct.c_void_p), ("k_stride", ct.c_int32), ("out", ct.c_void_p), ("Hkv", ct.c_int32),
                ("C", ct.c_int32), ("D", ct.c_int32), ("rope", bd_rope)]


class bd_unmask_args(ct.Structure):
    _fields_ = [("logits", ct.c_void_p), ("logits_dtype", ct.c_int32), ("logits_ld", ct.c_int64),
                ("R", ct.c_int32), ("V", ct.c_int32), ("logit_row", ct.c_void_p), ("n_pos", ct.c_int32),
                ("block_start", ct.c_void_p), ("n_blocks", ct.c_int32), ("state", ct.c_void_p),
                ("tokens", ct.c_void_p), ("tau_full", ct.c_float), ("tau_half", ct.c_float),
                ("min_num", ct.c_int32), ("min_den", ct.c_int32), ("k_fixed", ct.c_int32),
                ("add_num", ct.c_int32), ("add_den", ct.c_int32), ("act_num", ct.c_int32), ("act_den", ct.c_int32),
                ("commit", ct.c_void_p), ("n_committed", ct.c_void_p), ("status", ct.c_void_p),
                ("pred", ct.c_void_p), ("conf", ct.c_void_p), ("lse", ct.c_void_p), ("write_draft", ct.c_int32),
                ("workspace", ct.c_void_p), ("workspace_bytes", ct.c_size_t), ("dev_status", ct.c_void_p),
                ("wait_limit_ns", ct.c_uint64)]


class bd_verify_args(ct.Structure):
    _fields_ = [("n_seq", ct.c_int32), ("L", ct.c_int32), ("tokens", ct.c_void_p), ("state", ct.c_void_p),
                ("ar_logits", ct.c_void_p), ("logits_dtype", ct.c_int32), ("logits_ld", ct.c_int64),
                ("n_rows", ct.c_int32), ("V", ct.c_int32), ("noise", ct.c_void_p), ("temperature", ct.c_float),
                ("accepted_len", ct.c_void_p), ("bonus", ct.c_void_p), ("bonus_pos", ct.c_void_p),
                ("workspace", ct.c_void_p), ("workspace_bytes", ct.c_size_t), ("dev_status", ct.c_void_p),
                ("wait_limit_ns", ct.c_uint64)]


_lib = None
_lock = threading.Lock()


def lib() -> ct.CDLL:
    """The loaded libbd.so (built in-tree on first use when nvcc is present)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ct.CDLL(path)
            for name, argt in (("bd_block_causal_attn", bd_attn_args), ("bd_fork_rollouts", bd_fork_args),
                               ("bd_unmask_step", bd_unmask_args), ("bd_spec_verify", bd_verify_args),
                               ("bd_stream_insert", bd_stream_insert_args), ("bd_rope_keys", bd_rope_keys_args)):
                fn = getattr(L, name)
                fn.argtypes = [ct.POINTER(argt), ct.c_void_p]
                fn.restype = ct.c_int
            for name, argt in (("bd_attn_workspace_size", bd_attn_args), ("bd_fork_workspace_size", bd_fork_args),
                               ("bd_unmask_workspace_size", bd_unmask_args),
                               ("bd_verify_workspace_size", bd_verify_args)):
                fn = getattr(L, name)
                fn.argtypes = [ct.POINTER(argt)]
                fn.restype = ct.c_size_t
            L.bd_status_string.argtypes = [ct.c_int]
            L.bd_status_string.restype = ct.c_char_p
            L.bd_check.argtypes = [ct.c_void_p, ct.c_void_p]
            L.bd_check.restype = ct.c_int
            L.bd_version.restype = ct.c_char_p
            _lib = L
    return _lib


def bd_status_string(status: int) -> str:
    return lib().bd_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ct.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ct.c_void_p(s.cuda_stream)


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise BdError(fn, st)


class Workspace:
    """Zero-filled device scratch grown on demand (one per device and purpose).

    The library leaves its counters at zero after every completed call, so the
    buffer is cleared only when it is (re)allocated."""

    def __init__(self):
        self._buf = {}

    def get(self, nbytes: int, device) -> torch.Tensor | None:
        if nbytes == 0:
            return None
        key = torch.device(device).index
        buf = self._buf.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device)
            self._buf[key] = buf
        return buf


_WS = {"attn": Workspace(), "unmask": Workspace(), "verify": Workspace()}


def _rope(rope) -> bd_rope:
    """dict(k_pos=int32 tensor or None, delta, theta, enabled=True); enabled=False
    passes the positions (for the streaming mask) without rotating the keys."""
    r = bd_rope()
    if rope:
        r.enabled = 1 if rope.get("enabled", True) else 0
        kp = rope.get("k_pos")
        r.k_pos = None if kp is None else kp.data_ptr()
        r.delta = int(rope.get("delta", 0))
        r.theta = float(rope.get("theta", 10000.0))
    return r


def _kv_dtype(k, exps) -> int:
    """BD_E4M3 for a cache of E4M3 bytes (uint8 or float8_e4m3fn tensors, with
    their block exponents), else bf16."""
    fp8 = k.dtype == torch.uint8 or k.dtype == getattr(torch, "float8_e4m3fn", None)
    if fp8 and any(e is None for e in exps):
        raise ValueError("an E4M3 cache needs its block exponents (int8 tensors)")
    for e in exps:
        if e is not None:
            assert e.dtype == torch.int8 and e.is_cuda and e.is_contiguous()
    return BD_E4M3 if fp8 else BD_BF16


def _bs(block_start):
    if block_start is None:
        return None, 0
    assert block_start.dtype == torch.int32 and block_start.is_cuda
    return block_start.data_ptr(), block_start.numel() - 1


def bd_block_causal_attn(q, k, v, C: int, block_start=None, block_size: int = 0, o=None, lse=None,
                         sm_scale: float = 0.0, rope=None, num_splits: int = 0, workspace=None,
                         dev_status=None, stream=None, prefix_ready: bool = False, q_pos=None,
                         wait_limit_ns: int = 0, k_exp=None, v_exp=None):
    """Block-causal attention of the active positions.  q [n_q, Hq, D] bf16;
    k, v [Hkv, kv_stride, D] bf16 (prefix rows [0, C), active rows after), or
    E4M3 bytes (uint8 / float8_e4m3fn) with int8 block exponents k_exp, v_exp
    [Hkv, ceil(kv_stride / 128)].  With q_pos (int32 [n_q]) the streaming mask
    instead: queries over rows [0, C) only, key j visible iff rope k_pos[j] -
    delta <= q_pos[i].  Returns (o [n_q, Hq, D] bf16, lse [Hq, n_q] fp32)."""
    n_q, Hq, D = q.shape
    Hkv, kv_stride, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, n_q), dtype=torch.float32, device=q.device)
    a = bd_attn_args()
    a.q, a.k, a.v, a.o, a.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()
    a.block_start, a.n_blocks = _bs(block_start)
    a.block_size = int(block_size)
    a.C, a.n_q, a.Hq, a.Hkv, a.D, a.kv_stride = int(C), n_q, Hq, Hkv, D, kv_stride
    a.sm_scale = float(sm_scale)
    a.rope = _rope(rope)
    a.num_splits = int(num_splits)
    a.prefix_ready = 1 if prefix_ready else 0
    a.kv_dtype = _kv_dtype(k, (k_exp, v_exp))
    a.k_exp, a.v_exp = _ptr(k_exp), _ptr(v_exp)
    if q_pos is not None:  # part of the plan: set before the workspace is sized
        assert q_pos.dtype == torch.int32 and q_pos.is_cuda and q_pos.numel() == n_q
        a.q_pos = q_pos.data_ptr()
    need = lib().bd_attn_workspace_size(a)
    ws = workspace if workspace is not None else _WS["attn"].get(need, q.device)
    a.workspace = None if ws is None else ws.data_ptr()
    a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    a.dev_status = None if dev_status is None else dev_status.data_ptr()
    a.wait_limit_ns = int(wait_limit_ns)
    _check("bd_block_causal_attn", lib().bd_block_causal_attn(a, _stream(stream)))
    return o, lse


def bd_fork_rollouts(q, prefix_k, prefix_v, priv_k, priv_v, priv_len: int, C: int, block_start=None,
                     block_size: int = 0, o=None, lse=None, sm_scale: float = 0.0, rope=None, num_splits: int = 0,
                     workspace=None, dev_status=None, stream=None, prefix_ready: bool = False,
                     wait_limit_ns: int = 0, prefix_k_exp=None, prefix_v_exp=None, priv_k_exp=None,
                     priv_v_exp=None):
    """N rollouts over one shared prefix.  q [N, n_q, Hq, D]; prefix_k/v [Hkv, prefix_stride, D];
    priv_k/v [N, Hkv, priv_stride, D], bf16 or E4M3 bytes with int8 block exponents
    ([Hkv, ceil(prefix_stride / 128)] and [N, Hkv, ceil(priv_stride / 128)]).
    Returns (o [N, n_q, Hq, D], lse [N, Hq, n_q])."""
    N, n_q, Hq, D = q.shape
    Hkv, prefix_stride, _ = prefix_k.shape
    priv_stride = priv_k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((N, Hq, n_q), dtype=torch.float32, device=q.device)
    a = bd_fork_args()
    a.N, a.q = N, q.data_ptr()
    a.prefix_k, a.prefix_v, a.prefix_stride = prefix_k.data_ptr(), prefix_v.data_ptr(), prefix_stride
    a.priv_k, a.priv_v, a.priv_stride, a.priv_len = priv_k.data_ptr(), priv_v.data_ptr(), priv_stride, int(priv_len)
    a.o, a.lse = o.data_ptr(), lse.data_ptr()
    a.block_start, a.n_blocks = _bs(block_start)
    a.block_size = int(block_size)
    a.C, a.n_q, a.Hq, a.Hkv, a.D = int(C), n_q, Hq, Hkv, D
    a.sm_scale = float(sm_scale)
    a.rope = _rope(rope)
    a.num_splits = int(num_splits)
    a.kv_dtype = _kv_dtype(prefix_k, (prefix_k_exp, prefix_v_exp, priv_k_exp, priv_v_exp))
    a.prefix_k_exp, a.prefix_v_exp = _ptr(prefix_k_exp), _ptr(prefix_v_exp)
    a.priv_k_exp, a.priv_v_exp = _ptr(priv_k_exp), _ptr(priv_v_exp)
    need = lib().bd_fork_workspace_size(a)
    ws = workspace if workspace is not None else _WS["attn"].get(need, q.device)
    a.workspace = None if ws is None else ws.data_ptr()
    a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    a.dev_status = None if dev_status is None else dev_status.data_ptr()
    a.prefix_ready = 1 if prefix_ready else 0
    a.wait_limit_ns = int(wait_limit_ns)
    _check("bd_fork_rollouts", lib().bd_fork_rollouts(a, _stream(stream)))
    return o, lse


def bd_unmask_step(logits, logit_row, block_start, state, tokens, *, tau_full: float, tau_half: float,
                   min_frac=(1, 4), k_fixed: int = 0, add_thr=(1, 2), act_thr=(17, 20), write_draft=False,
                   commit=None,
                   n_committed=None, status=None, pred=None, conf=None, lse=None, workspace=None,
                   dev_status=None, stream=None, wait_limit_ns: int = 0):
    """One unmask/commit step; updates ``state`` and ``tokens`` in place.
    Returns dict(commit, n_committed, status, pred, conf, lse)."""
    R, V = logits.shape
    n_pos = state.numel()
    n_blocks = block_start.numel() - 1
    dev = logits.device
    commit = torch.empty(n_pos, dtype=torch.uint8, device=dev) if commit is None else commit
    n_committed = torch.empty(n_blocks, dtype=torch.int32, device=dev) if n_committed is None else n_committed
    status = torch.empty(n_blocks, dtype=torch.int32, device=dev) if status is None else status
    pred = torch.empty(n_pos, dtype=torch.int32, device=dev) if pred is None else pred
    conf = torch.empty(n_pos, dtype=torch.float32, device=dev) if conf is None else conf
    lse = torch.empty(n_pos, dtype=torch.float32, device=dev) if lse is None else lse
    a = bd_unmask_args()
    a.logits = logits.data_ptr()
    a.logits_dtype = BD_BF16 if logits.dtype == torch.bfloat16 else BD_F32
    a.logits_ld = logits.stride(0) if R > 1 else (V + 7) // 8 * 8
    a.R, a.V = R, V
    a.logit_row, a.n_pos = logit_row.data_ptr(), n_pos
    a.block_start, a.n_blocks = block_start.data_ptr(), n_blocks
    a.state, a.tokens = state.data_ptr(), tokens.data_ptr()
    a.tau_full, a.tau_half = float(tau_full), float(tau_half)
    a.min_num, a.min_den = int(min_frac[0]), int(min_frac[1])
    a.k_fixed = int(k_fixed)
    a.add_num, a.add_den = int(add_thr[0]), int(add_thr[1])
    a.act_num, a.act_den = int(act_thr[0]), int(act_thr[1])
    a.commit, a.n_committed, a.status = commit.data_ptr(), n_committed.data_ptr(), status.data_ptr()
    a.pred, a.conf, a.lse = pred.data_ptr(), conf.data_ptr(), lse.data_ptr()
    a.write_draft = 1 if write_draft else 0
    need = lib().bd_unmask_workspace_size(a)
    ws = workspace if workspace is not None else _WS["unmask"].get(need, dev)
    a.workspace = None if ws is None else ws.data_ptr()
    a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    a.dev_status = None if dev_status is None else dev_status.data_ptr()
    a.wait_limit_ns = int(wait_limit_ns)
    _check("bd_unmask_step", lib().bd_unmask_step(a, _stream(stream)))
    return dict(commit=commit, n_committed=n_committed, status=status, pred=pred, conf=conf, lse=lse)


def bd_spec_verify(tokens, state, ar_logits, noise=None, temperature: float = 1.0, accepted_len=None, bonus=None,
                   bonus_pos=None, workspace=None, dev_status=None, stream=None, wait_limit_ns: int = 0):
    """Scaffold-speculative verify; updates ``tokens``/``state`` [n_seq, L] in place.
    ar_logits [n_seq, n_rows, V]; noise fp32 of the same shape or None.
    Returns (accepted_len, bonus, bonus_pos), int32 [n_seq] each."""
    n_seq, L = tokens.shape
    _, n_rows, V = ar_logits.shape
    dev = tokens.device
    accepted_len = torch.empty(n_seq, dtype=torch.int32, device=dev) if accepted_len is None else accepted_len
    bonus = torch.empty(n_seq, dtype=torch.int32, device=dev) if bonus is None else bonus
    bonus_pos = torch.empty(n_seq, dtype=torch.int32, device=dev) if bonus_pos is None else bonus_pos
    ld = ar_logits.stride(1) if n_rows > 1 else (V + 7) // 8 * 8
    if n_seq > 1 and ar_logits.stride(0) != n_rows * ld:
        raise ValueError("ar_logits: sequences must follow each other at n_rows * row stride")
    if noise is not None and ((n_rows > 1 and noise.stride(1) != ld) or
                              (n_seq > 1 and noise.stride(0) != ar_logits.stride(0))):
        raise ValueError("noise must have the layout of ar_logits")
    a = bd_verify_args()
    a.n_seq, a.L = n_seq, L
    a.tokens, a.state = tokens.data_ptr(), state.data_ptr()
    a.ar_logits = ar_logits.data_ptr()
    a.logits_dtype = BD_BF16 if ar_logits.dtype == torch.bfloat16 else BD_F32
    a.logits_ld = ld
    a.n_rows, a.V = n_rows, V
    a.noise = None if noise is None else noise.data_ptr()
    a.temperature = float(temperature)
    a.accepted_len, a.bonus, a.bonus_pos = accepted_len.data_ptr(), bonus.data_ptr(), bonus_pos.data_ptr()
    need = lib().bd_verify_workspace_size(a)
    ws = workspace if workspace is not None else _WS["verify"].get(need, dev)
    a.workspace = None if ws is None else ws.data_ptr()
    a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    a.dev_status = None if dev_status is None else dev_status.data_ptr()
    a.wait_limit_ns = int(wait_limit_ns)
    _check("bd_spec_verify", lib().bd_spec_verify(a, _stream(stream)))
    return accepted_len, bonus, bonus_pos


def bd_stream_insert(k_cache, v_cache, k_pos, new_k, new_v, new_pos, views: int, frames: int, per_frame: int,
                     slot: int, stream=None) -> None:
    """Writes the new frame (new_k/new_v bf16 [views * per_frame, Hkv, D], view by
    view; new_pos int32 [views * per_frame]) into frame slot ``slot`` of every view
    of the view-major cache (k_cache/v_cache bf16 [Hkv, cache_stride, D]) and its
    positions into k_pos (int32 [views * frames * per_frame])."""
    Hkv, stride, D = k_cache.shape
    a = bd_stream_insert_args()
    a.k_cache, a.v_cache, a.k_pos = k_cache.data_ptr(), v_cache.data_ptr(), k_pos.data_ptr()
    a.new_k, a.new_v, a.new_pos = new_k.data_ptr(), new_v.data_ptr(), new_pos.data_ptr()
    a.views, a.frames, a.per_frame, a.slot = int(views), int(frames), int(per_frame), int(slot)
    a.Hkv, a.D, a.cache_stride = Hkv, D, stride
    _check("bd_stream_insert", lib().bd_stream_insert(a, _stream(stream)))


def bd_rope_keys(k, C: int, rope, out=None, stream=None):
    """The in-operator RoPE rotation written out: keys [0, C) of k (bf16 [Hkv,
    k_stride, D], pre-RoPE) rotated at rope k_pos - delta into out (bf16 [Hkv,
    C, D], created when not given), each element the bf16 rounding of the
    float64 rotation.  Attention calls can then read out with RoPE off."""
    Hkv, k_stride, D = k.shape
    if out is None:
        out = torch.empty((Hkv, C, D), dtype=torch.bfloat16, device=k.device)
    a = bd_rope_keys_args()
    a.k, a.k_stride, a.out = k.data_ptr(), k_stride, out.data_ptr()
    a.Hkv, a.C, a.D = Hkv, int(C), D
    a.rope = _rope(rope)
    _check("bd_rope_keys", lib().bd_rope_keys(a, _stream(stream)))
    return out


def bd_check(dev_status, stream=None) -> int:
    """Synchronises the stream and maps the device status word (0 = ok)."""
    return lib().bd_check(dev_status.data_ptr(), _stream(stream))


def bd_unmask_step_noalloc(logits, logit_row, block_start, state, tokens, *, tau_full: float, tau_half: float,
                           min_frac=(1, 4), k_fixed: int = 0, add_thr=(1, 2), act_thr=(17, 20), write_draft=False,
                           commit=None, n_committed=None, status=None, pred=None, conf=None, lse=None,
                           dev_status=None, stream=None):
    """bd_unmask_step without a workspace: the library's own fixed scratch array
    is used (for callers that cannot allocate device memory).  Output tensors
    not given are created here, as in bd_unmask_step; pass them all to
    allocate nothing on this side either.  Calls that overlap on the GPU race."""
    R, V = logits.shape
    n_pos = state.numel()
    n_blocks = block_start.numel() - 1
    dev = logits.device
    commit = torch.empty(n_pos, dtype=torch.uint8, device=dev) if commit is None else commit
    n_committed = torch.empty(n_blocks, dtype=torch.int32, device=dev) if n_committed is None else n_committed
    status = torch.empty(n_blocks, dtype=torch.int32, device=dev) if status is None else status
    pred = torch.empty(n_pos, dtype=torch.int32, device=dev) if pred is None else pred
    conf = torch.empty(n_pos, dtype=torch.float32, device=dev) if conf is None else conf
    lse = torch.empty(n_pos, dtype=torch.float32, device=dev) if lse is None else lse
    a = bd_unmask_args()
    a.logits = logits.data_ptr()
    a.logits_dtype = BD_BF16 if logits.dtype == torch.bfloat16 else BD_F32
    a.logits_ld = logits.stride(0) if R > 1 else (V + 7) // 8 * 8
    a.R, a.V = R, V
    a.logit_row, a.n_pos = logit_row.data_ptr(), n_pos
    a.block_start, a.n_blocks = block_start.data_ptr(), n_blocks
    a.state, a.tokens = state.data_ptr(), tokens.data_ptr()
    a.tau_full, a.tau_half = float(tau_full), float(tau_half)
    a.min_num, a.min_den = int(min_frac[0]), int(min_frac[1])
    a.k_fixed = int(k_fixed)
    a.add_num, a.add_den = int(add_thr[0]), int(add_thr[1])
    a.act_num, a.act_den = int(act_thr[0]), int(act_thr[1])
    a.commit, a.n_committed, a.status = commit.data_ptr(), n_committed.data_ptr(), status.data_ptr()
    a.pred, a.conf, a.lse = pred.data_ptr(), conf.data_ptr(), lse.data_ptr()
    a.write_draft = 1 if write_draft else 0
    a.dev_status = None if dev_status is None else dev_status.data_ptr()
    fn = lib().bd_unmask_step_noalloc
    fn.argtypes = [ct.POINTER(bd_unmask_args), ct.c_void_p]
    fn.restype = ct.c_int
    _check("bd_unmask_step_noalloc", fn(a, _stream(stream)))
    return dict(commit=commit, n_committed=n_committed, status=status, pred=pred, conf=conf, lse=lse)
