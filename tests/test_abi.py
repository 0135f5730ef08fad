"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/bd.h declares, its ctypes structs match the C layout,
workspace sizing is plain host arithmetic, and invalid arguments are refused
on the host before anything touches CUDA."""
import ctypes as ct
import os
import re
import subprocess

import pytest

import block_causal_masked_gb300 as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bd.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:bd_status|size_t|const char\s*\*)\s*(bd_\w+)\s*\(", src, re.M)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("bd_block_causal_attn", "bd_unmask_step", "bd_spec_verify", "bd_fork_rollouts"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = bd.lib()
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", L._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (bd_\w+)$", out, re.M))
    assert set(_declared()) <= exported


STRUCTS = ["bd_rope", "bd_attn_args", "bd_fork_args", "bd_unmask_args", "bd_verify_args", "bd_stream_insert_args",
           "bd_rope_keys_args"]


def test_ctypes_structs_match_c_layout(tmp_path):
    """sizeof and every field offset, as gcc lays the header out."""
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "bd.h"', "int main(void){"]
    for s in STRUCTS:
        cls = getattr(bd, s)
        lines.append(f'printf("{s} %zu\\n", sizeof({s}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{s}.{f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0;}")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for s in STRUCTS:
        cls = getattr(bd, s)
        assert int(got[s]) == ct.sizeof(cls), s
        for f, _ in cls._fields_:
            assert int(got[f"{s}.{f}"]) == getattr(cls, f).offset, (s, f)


def test_status_strings():
    L = bd.lib()
    for s in range(7):
        assert L.bd_status_string(s) and L.bd_status_string(s) != b"unknown status"
    assert L.bd_status_string(99) == b"unknown status"


FAKE = 1 << 20  # an aligned address that is never dereferenced: every call below fails validation first


def _attn(**kw):
    a = bd.bd_attn_args()
    a.q = a.k = a.v = a.o = FAKE
    a.C, a.n_q, a.Hq, a.Hkv, a.D, a.kv_stride, a.block_size = 100, 8, 4, 2, 128, 200, 8
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), 1), (dict(n_q=0), 1), (dict(C=-1), 1), (dict(kv_stride=50), 1), (dict(block_size=0), 1),
    (dict(D=96), 2), (dict(Hq=5), 2), (dict(q=FAKE + 8), 2), (dict(o=FAKE + 2), 2), (dict(num_splits=17), 1),
    (dict(num_splits=4), 3),  # split partials need a workspace, none given
])
def test_attention_argument_errors_on_host(kw, want):
    a = _attn(**kw)
    assert bd.lib().bd_block_causal_attn(a, None) == want


def test_fork_argument_errors_on_host():
    a = bd.bd_fork_args()
    a.N, a.q, a.prefix_k, a.prefix_v, a.priv_k, a.priv_v, a.o = 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE
    a.C, a.prefix_stride, a.n_q, a.priv_len, a.priv_stride, a.Hq, a.Hkv, a.D, a.block_size = 64, 64, 8, 4, 8, 4, 2, 64, 8
    assert bd.lib().bd_fork_rollouts(a, None) == 1        # priv_stride < priv_len + n_q
    a.priv_stride = 12
    a.N = 0
    assert bd.lib().bd_fork_rollouts(a, None) == 1


def test_workspace_sizes_are_host_arithmetic():
    # split partials: Hkv * row tiles * S * S owner slices of r rows (r = 32 at S = 4) of D bf16
    # values of O; none with one split
    assert bd.lib().bd_attn_workspace_size(_attn(num_splits=4)) == 2 * 1 * 4 * 4 * 32 * 2 * 128
    assert bd.lib().bd_attn_workspace_size(_attn(num_splits=1)) == 0
    u = bd.bd_unmask_args()
    u.R, u.V, u.n_pos, u.n_blocks, u.logits_ld, u.min_den, u.add_den, u.act_den = 32, 151936, 33, 1, 151936, 4, 2, 20
    assert bd.lib().bd_unmask_workspace_size(u) > 0
    u.n_pos = 5000
    assert bd.lib().bd_unmask_workspace_size(u) == 0      # beyond the supported window
    v = bd.bd_verify_args()
    v.n_seq, v.L, v.n_rows, v.V, v.logits_ld = 8, 40, 33, 151936, 151936
    assert bd.lib().bd_verify_workspace_size(v) > 0


def test_vocab_argument_errors_on_host():
    u = bd.bd_unmask_args()
    u.R, u.V, u.n_pos, u.n_blocks, u.logits_ld, u.min_den, u.add_den, u.act_den = 4, 100, 4, 1, 100, 4, 2, 20
    assert bd.lib().bd_unmask_step(u, None) == 1          # ld not a multiple of 8
    u.logits_ld = 104
    assert bd.lib().bd_unmask_step(u, None) == 1          # null pointers
    v = bd.bd_verify_args()
    v.n_seq, v.L, v.n_rows, v.V, v.logits_ld = 1, 4, 9, 100, 104
    assert bd.lib().bd_spec_verify(v, None) == 1          # n_rows > L + 1


def test_stream_insert_argument_errors_on_host():
    a = bd.bd_stream_insert_args()
    a.k_cache = a.v_cache = a.k_pos = a.new_k = a.new_v = a.new_pos = FAKE
    a.views, a.frames, a.per_frame, a.slot, a.Hkv, a.D, a.cache_stride = 4, 4, 256, 0, 2, 128, 4096
    for kw, want in ((dict(slot=4), 1), (dict(slot=-1), 1), (dict(views=0), 1), (dict(cache_stride=4095), 1),
                     (dict(D=96), 2), (dict(new_k=FAKE + 8), 2), (dict(k_pos=None), 1)):
        b = bd.bd_stream_insert_args.from_buffer_copy(a)
        for k, v in kw.items():
            setattr(b, k, v)
        assert bd.lib().bd_stream_insert(b, None) == want, kw


def test_rope_keys_argument_errors_on_host():
    """Bad head dim, misaligned or overlapping buffers, no theta: refused before CUDA."""
    a = bd.bd_rope_keys_args()
    a.k, a.out, a.k_stride, a.Hkv, a.C, a.D = FAKE, FAKE + (1 << 20), 100, 2, 64, 128
    a.rope.theta = 1e4
    for kw, want in ((dict(D=96), 2), (dict(out=FAKE + 8 + (1 << 20)), 2), (dict(out=FAKE + 64), 1),
                     (dict(k_stride=10), 1), (dict(k=None), 1)):
        b = bd.bd_rope_keys_args.from_buffer_copy(a)
        for k, v in kw.items():
            setattr(b, k, v)
        assert bd.lib().bd_rope_keys(b, None) == want, kw
    b = bd.bd_rope_keys_args.from_buffer_copy(a)
    b.rope.theta = 0.0
    assert bd.lib().bd_rope_keys(b, None) == 1


def test_streaming_mask_argument_errors_on_host():
    """With q_pos the active rows are not read (kv_stride >= C suffices), the block
    partition is not needed, and a misaligned q_pos is refused."""
    a = _attn(kv_stride=100, block_size=0, q_pos=FAKE + 2)
    assert bd.lib().bd_block_causal_attn(a, None) == 2
    a = _attn(kv_stride=99, block_size=0, q_pos=FAKE)
    assert bd.lib().bd_block_causal_attn(a, None) == 1


def _planned_splits(**kw):
    """The KV split count the planner picks, read back from the workspace size
    (Hkv * row tiles * S * S owner slices of r(S) rows of D bf16 values; none for
    one split)."""
    a = _attn(num_splits=0, **kw)
    ws = bd.lib().bd_attn_workspace_size(a)
    rows = a.n_q * (a.Hq // a.Hkv)
    m_tiles = (rows + 127) // 128
    if ws == 0:
        return 1
    for s in range(2, 17):
        r = ((128 + s - 1) // s + 1) & ~1
        if ws == a.Hkv * m_tiles * s * s * r * 2 * a.D:
            return s
    raise AssertionError(f"unexpected workspace size {ws}")


@pytest.mark.parametrize("shape,want", [
    # Fast-dDrive decode layer: 26 tiles over 6 clusters -> 16 (the diagonal split among the short ones)
    (dict(C=3124, n_q=33, Hq=16, Hkv=2, kv_stride=3157, block_size=33), 16),
    # Fast-dVLA window: 6 tiles -> 12 (one merge pass of the 256 threads, not two as at 6)
    (dict(C=614, n_q=21, Hq=16, Hkv=2, kv_stride=635, block_size=7), 12),
    # WAM decode, 8 KV heads: 18 tiles over 8 clusters -> 10 (16 would need two waves)
    (dict(C=2176, n_q=1, Hq=16, Hkv=8, kv_stride=2177, block_size=1), 10),
    (dict(C=2176, n_q=32, Hq=16, Hkv=8, kv_stride=2208, block_size=32), 10),
    # a single tile: no split
    (dict(C=100, n_q=8, Hq=4, Hkv=2, kv_stride=200, block_size=8), 1),
])
def test_planner_split_choices(shape, want):
    assert _planned_splits(**shape) == want
