"""GPU parity of bd_block_causal_attn and bd_fork_rollouts against the float64
oracle, through the C ABI, on seeded inputs spanning several K/V tiles, ragged
tails, every block layout the method has (uniform, ragged, block size 1 = causal,
one block = bidirectional), head dims 64/128, GQA ratios 1/2/8, KV splits, and
in-kernel RoPE."""
import zlib

import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
import oracle
import synth
from helpers import DEV, assert_attn_close, bf16, bf16_midpoint_distance, host, i32, status_word

pytestmark = pytest.mark.gpu

CASES = [
    # (name, C, block_start, Hq, Hkv, D, splits)
    ("tiny_cfg", 256, [0, 8, 16], 4, 2, 64, 0),
    ("no_prefix", 0, [0, 5, 9], 8, 8, 128, 0),
    ("ragged_prefix_129", 129, [0, 3, 11, 12], 16, 2, 128, 1),
    ("ragged_prefix_127", 127, [0, 20, 40], 16, 2, 128, 3),
    ("causal_b1", 700, list(range(8)), 16, 8, 128, 0),
    ("one_block", 390, [0, 33], 16, 2, 128, 2),
    ("many_rows", 1000, [0, 33, 66, 92], 16, 2, 128, 0),     # 92 * 8 = 736 packed rows, 6 row tiles
    ("single_key_prefix", 1, [0, 1, 2], 2, 1, 64, 0),
    ("long_prefix", 3092, [0, 33], 16, 2, 128, 0),
]


def _run(case, splits, rope=None, block_start=True):
    bs = torch.tensor(case.block_start, dtype=torch.int32, device=DEV) if block_start else None
    ds = status_word()
    o, lse = bd.bd_block_causal_attn(bf16(case.q), bf16(case.k), bf16(case.v), case.C, block_start=bs,
                                     block_size=0 if block_start else 1, num_splits=splits, rope=rope,
                                     dev_status=ds)
    assert bd.bd_check(ds) == 0
    return o, lse


@pytest.mark.parametrize("name,C,bs,Hq,Hkv,D,splits", CASES, ids=[c[0] for c in CASES])
def test_attention_matches_oracle(name, C, bs, Hq, Hkv, D, splits):
    case = synth.attn_case(10, zlib.crc32(name.encode()) % 1000, C=C, block_start=bs, Hq=Hq, Hkv=Hkv, D=D, kv_pad=5,
                           text_from=max(0, C - 40))
    o, lse = _run(case, splits)
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, name)


def test_uniform_blocks_without_partition_array():
    """block_start = NULL with a block size: the last block ragged (n_q = 13, B = 4)."""
    case = synth.attn_case(11, 0, C=200, block_start=[0, 4, 8, 12, 13], Hq=8, Hkv=2, D=128)
    ds = status_word()
    o, lse = bd.bd_block_causal_attn(bf16(case.q), bf16(case.k), bf16(case.v), case.C, block_size=4, dev_status=ds)
    assert bd.bd_check(ds) == 0
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, case.C, [0, 4, 8, 12, 13])
    assert_attn_close(o, lse, o_ref, lse_ref)


def test_split_count_does_not_change_the_result():
    case = synth.attn_case(12, 0, C=2000, block_start=[0, 16, 33], Hq=16, Hkv=2, D=128)
    """Splits change only rounding: P is rounded to bf16 against each split's own
    running maximum, so O moves by a few bf16 steps while the LSE (summed in
    fp32 before rounding) stays within 1e-6."""
    res = [_run(case, s) for s in (1, 2, 7, 16)]
    for o, lse in res[1:]:
        assert np.allclose(host(lse), host(res[0][1]), rtol=1e-6, atol=1e-6)
        assert np.allclose(host(o), host(res[0][0]), rtol=2e-2, atol=2e-3)


def test_later_blocks_do_not_leak_on_gpu():
    """Perturbing the last block's queries, keys and values leaves the earlier
    blocks' outputs bitwise unchanged on the GPU as well."""
    bs = [0, 7, 14, 21]
    case = synth.attn_case(13, 0, C=600, block_start=bs, Hq=16, Hkv=2, D=128)
    o1, l1 = _run(case, 1)
    case.q[14:] += 50.0
    case.k[:, 600 + 14:] -= 50.0
    case.v[:, 600 + 14:] += 50.0
    o2, l2 = _run(case, 1)
    assert torch.equal(o1[:14], o2[:14]) and torch.equal(l1[:, :14], l2[:, :14])
    assert not torch.equal(o1[14:], o2[14:])


@pytest.mark.parametrize("D", [64, 128])
def test_in_kernel_rope_matches_oracle(D):
    C = 600
    case = synth.attn_case(14, D, C=C, block_start=[0, 12, 20], Hq=16, Hkv=2, D=D)
    k_pos = (np.arange(C) * 3 + 256).astype(np.int32)
    rope = dict(k_pos=i32(k_pos), delta=256, theta=10000.0)
    o, lse = _run(case, 0, rope=rope)
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, C, case.block_start, k_pos=k_pos,
                                                   delta=256, theta=10000.0, rope=True)
    assert_attn_close(o, lse, o_ref, lse_ref, f"rope D={D}")


@pytest.mark.parametrize("D,C,delta,spread", [(128, 4306, 256, 0), (64, 3000, 7, 3), (128, 1024, 12345, 997)])
def test_rotated_prefix_keys_bit_exact(D, C, delta, spread):
    """The operator's rotated copy of the pre-RoPE prefix keys -- the first
    Hkv * C * D bf16 values of the workspace when the call runs unsplit -- is,
    element by element, the bf16 rounding (to nearest even) of the float64
    rotation, on unconditioned N(0, 1) keys: the streaming prefix's view-major
    positions, a strided layout, and positions up to ~1e6.  The inputs reach
    rotated elements within 1e-6 of a bf16 rounding midpoint, where the fp32
    rotation cannot decide the rounding and the float64 one does."""
    if spread == 0:
        k_pos = synth.streaming_prefix_positions()
    else:
        k_pos = (np.arange(C) * spread + delta + 1).astype(np.int32)
    Hkv = 2
    case = synth.attn_case(21 + spread, D, C=C, block_start=[0, 8], Hq=4, Hkv=Hkv, D=D)
    nbytes = Hkv * C * D * 2
    ws = torch.zeros(nbytes + 4096, dtype=torch.uint8, device=DEV)
    ds = status_word()
    bd.bd_block_causal_attn(bf16(case.q), bf16(case.k), bf16(case.v), C, block_start=i32(case.block_start),
                            num_splits=1, workspace=ws, dev_status=ds,
                            rope=dict(k_pos=i32(k_pos), delta=delta, theta=1e4))
    assert bd.bd_check(ds) == 0
    got = host(ws[:nbytes].view(torch.bfloat16)).reshape(Hkv, C, D).astype(np.float64)
    rot = oracle.rope_rotate(case.k[:, :C], k_pos.astype(np.int64) - delta, 1e4)
    ref = oracle.round_bf16(rot)
    bad = got != ref
    assert not bad.any(), f"{bad.sum()} of {bad.size} rotated elements differ"
    assert (bf16_midpoint_distance(rot) < 1e-6).sum() > 0


def test_rope_keys_equal_the_operator_rotation():
    """bd_rope_keys writes the rotation the operator applies: bit-exact to the
    oracle's bf16 rounding of the float64 rotation, and attention over it with
    RoPE off equals attention with RoPE in the operator, bitwise."""
    C = 4096 + 210
    case = synth.attn_case(16, 0, C=C, block_start=[0, 39], Hq=16, Hkv=2, D=128)
    k_pos = synth.streaming_prefix_positions()
    rope = dict(k_pos=i32(k_pos), delta=256, theta=1e4)
    k = bf16(case.k)
    rot = bd.bd_rope_keys(k, C, rope)
    ref = oracle.round_bf16(oracle.rope_rotate(case.k[:, :C], k_pos.astype(np.int64) - 256, 1e4))
    assert np.array_equal(host(rot).astype(np.float64), ref)
    blk = i32(case.block_start)
    o1, l1 = bd.bd_block_causal_attn(bf16(case.q), k, bf16(case.v), C, block_start=blk, rope=rope)
    k2 = k.clone()
    k2[:, :C] = rot
    o2, l2 = bd.bd_block_causal_attn(bf16(case.q), k2, bf16(case.v), C, block_start=blk)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_in_kernel_rope_equals_prerotated_keys():
    """RoPE inside the operator gives bitwise the no-RoPE result on keys rotated
    beforehand (rotated in float64 and rounded to bf16 on the host): the
    operator's rotated keys are those same bf16 values, and the two calls run
    the same plan."""
    C = 4096 + 210
    case = synth.attn_case(15, 0, C=C, block_start=[0, 39], Hq=16, Hkv=2, D=128)
    k_pos = synth.streaming_prefix_positions()
    o, lse = _run(case, 0, rope=dict(k_pos=i32(k_pos), delta=256, theta=1e4))
    k2 = case.k.copy()
    k2[:, :C] = oracle.round_bf16(oracle.rope_rotate(case.k[:, :C], k_pos.astype(np.int64) - 256, 1e4))
    case2 = synth.AttnCase(case.q, k2, case.v, C, case.block_start)
    o2, lse2 = _run(case2, 0)
    assert torch.equal(lse, lse2) and torch.equal(o, o2)


# ---------------------------------------------------------------------------------------- fork

def _fork(seed, N, C, n_q, priv_len, bs, D=128, rope=False):
    k_pos = synth.streaming_prefix_positions(sections=C - 4096) if rope and C > 4096 else None
    if rope and k_pos is None:
        k_pos = (np.arange(C) + 256).astype(np.int32)
    f = synth.fork_case(seed, 0, N=N, C=C, n_q=n_q, priv_len=priv_len, block_start=bs, Hq=16, Hkv=2, D=D,
                        k_pos=k_pos, delta=256 if rope else 0, theta=1e4)
    return f


def _run_fork(f, splits=0, rope=False):
    ds = status_word()
    r = dict(k_pos=i32(f.k_pos), delta=f.delta, theta=f.theta) if rope else None
    o, lse = bd.bd_fork_rollouts(bf16(f.q), bf16(f.prefix_k), bf16(f.prefix_v), bf16(f.priv_k), bf16(f.priv_v),
                                 f.priv_len, f.C, block_start=i32(f.block_start), num_splits=splits, rope=r,
                                 dev_status=ds)
    assert bd.bd_check(ds) == 0
    return o, lse


@pytest.mark.parametrize("N,C,n_q,priv_len,bs,splits", [
    (1, 300, 12, 0, [0, 12], 0),
    (3, 500, 39, 41, [0, 39], 0),
    (8, 1000, 12, 78, [0, 12], 2),
    (5, 129, 20, 130, [0, 10, 20], 1),
])
def test_fork_matches_oracle(N, C, n_q, priv_len, bs, splits):
    f = _fork(20 + N, N, C, n_q, priv_len, bs)
    o, lse = _run_fork(f, splits)
    o_ref, lse_ref = oracle.fork_attention(f.q, f.prefix_k, f.prefix_v, f.priv_k, f.priv_v, priv_len, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, f"fork N={N}")


def test_fork_single_rollout_equals_plain_attention():
    f = _fork(30, 1, 700, 33, 40, [0, 33])
    o, lse = _run_fork(f)
    k = np.concatenate([f.prefix_k, f.priv_k[0]], axis=1)
    v = np.concatenate([f.prefix_v, f.priv_v[0]], axis=1)
    case = synth.AttnCase(f.q[0], k, v, 700 + 40, f.block_start)
    o2, lse2 = _run(case, 0)
    # the two calls may split the keys differently: O a few bf16 steps apart
    assert np.allclose(host(o[0]), host(o2), rtol=2e-2, atol=2e-3)
    assert np.allclose(host(lse[0]), host(lse2), rtol=1e-6, atol=1e-6)


def test_fork_reads_the_prefix_without_writing_it():
    f = _fork(31, 4, 800, 12, 39, [0, 12])
    pk, pv = bf16(f.prefix_k), bf16(f.prefix_v)
    pk0, pv0 = pk.clone(), pv.clone()
    bd.bd_fork_rollouts(bf16(f.q), pk, pv, bf16(f.priv_k), bf16(f.priv_v), f.priv_len, f.C,
                        block_start=i32(f.block_start))
    torch.cuda.synchronize()
    assert torch.equal(pk, pk0) and torch.equal(pv, pv0)


def test_fork_with_rope_matches_oracle():
    f = _fork(32, 4, 4096 + 210, 39, 41, [0, 39], rope=True)
    o, lse = _run_fork(f, rope=True)
    o_ref, lse_ref = oracle.fork_attention(f.q, f.prefix_k, f.prefix_v, f.priv_k, f.priv_v, f.priv_len,
                                           f.block_start, k_pos=f.k_pos, delta=f.delta, theta=f.theta, rope=True)
    assert_attn_close(o, lse, o_ref, lse_ref, "fork rope")


@pytest.mark.parametrize("rope", [False, True])
def test_prefix_ready_matches_default_in_a_graph(rope):
    """prefix_ready = 1 (prefix tiles fetched before the dependency wait) gives
    bitwise the results of the default, for launches chained in one CUDA graph
    where each launch's queries are written by the kernel just before it; with
    RoPE the flag is ignored.  The last launch also matches the oracle."""
    C, bs, n = 1500, [0, 33], 4
    case = synth.attn_case(12, 0, C=C, block_start=bs, Hq=16, Hkv=2, D=128)
    k, v = bf16(case.k), bf16(case.v)
    q0 = bf16(case.q)
    blk = i32(bs)
    kp = torch.arange(C, dtype=torch.int32, device=DEV) + 7
    rp = dict(k_pos=kp, delta=7, theta=1e4) if rope else None

    def chain(flag):
        qs = [torch.empty_like(q0) for _ in range(n)]
        outs = [torch.empty_like(q0) for _ in range(n)]
        lses = [torch.empty((16, 33), dtype=torch.float32, device=DEV) for _ in range(n)]

        def run():
            for i in range(n):
                qs[i].copy_(q0 if i == 0 else outs[i - 1])          # q written by the kernel before
                bd.bd_block_causal_attn(qs[i], k, v, C, block_start=blk, o=outs[i], lse=lses[i], rope=rp,
                                        prefix_ready=flag)
        run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            run()
        for x in outs:
            x.zero_()
        g.replay()
        torch.cuda.synchronize()
        return [host(x) for x in outs], [host(x) for x in lses], host(qs[-1])

    o1, l1, q_last = chain(True)
    o0, l0, _ = chain(False)
    for a, b in zip(o1 + l1, o0 + l0):
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a, b.view(np.uint32)
                              if b.dtype == np.float32 else b)
    kw = dict(k_pos=host(kp), delta=7, theta=1e4, rope=True) if rope else {}
    o_ref, lse_ref = oracle.block_causal_attention(q_last, case.k, case.v, C, bs, **kw)
    assert_attn_close(torch.from_numpy(o1[-1]), torch.from_numpy(l1[-1]), o_ref, lse_ref)


@pytest.mark.parametrize("D", [64, 128])
def test_two_launch_plan_matches_oracle(D):
    """More (row tile, KV head) groups than one wave of SMs: 2,500 positions x 8
    query heads on one KV head = 157 row tiles, run as a bulk launch of 152
    unsplit row tiles and a tail of 5 split wide; block size 100."""
    n_q, C = 2500, 200
    bs = list(range(0, n_q, 100)) + [n_q]
    case = synth.attn_case(40, D, C=C, block_start=bs, Hq=8, Hkv=1, D=D)
    o, lse = _run(case, 0)
    o_ref, lse_ref = oracle.block_causal_attention(case.q, case.k, case.v, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, f"two-launch D={D}")
