"""GPU parity of the FP8 (E4M3) KV-cache attention against the float64 oracle
over the dequantised cache (oracle/kvquant.py), through the C ABI: plain
block-causal attention (head dims 64 / 128, ragged prefixes, block size 1, 92
positions over 6 row tiles, fixed and planned KV splits; the decode shapes
the benchmark times; a call of more row tiles than one wave of SMs, run as two
launches), the shared-prefix fork, closed forms that pin the dequantised values (Q = 0: the mean of exactly
the visible dequantised values), an exponent outside [-15, 7] reported as
BD_ERR_DEVICE_INPUT, and RoPE refused.  Tolerances as for bf16 K/V."""
import zlib

import numpy as np
import pytest
import torch

import block_causal_masked_gb300 as bd
import oracle
import synth
from helpers import DEV, assert_attn_close, bf16, host, i32, status_word, u8

pytestmark = pytest.mark.gpu


def i8(x) -> torch.Tensor:
    return torch.from_numpy(np.array(x, dtype=np.int8, order="C", copy=True)).to(DEV)


def _quantised(case):
    k8, ke = synth.quantize_kv_e4m3(case.k)
    v8, ve = synth.quantize_kv_e4m3(case.v)
    return k8, ke, v8, ve, oracle.dequantize_kv(k8, ke), oracle.dequantize_kv(v8, ve)


def _run8(q, k8, ke, v8, ve, C, bs, splits=0):
    ds = status_word()
    o, lse = bd.bd_block_causal_attn(bf16(q), u8(k8), u8(v8), C, block_start=i32(bs), num_splits=splits,
                                     k_exp=i8(ke), v_exp=i8(ve), dev_status=ds)
    assert bd.bd_check(ds) == 0
    return o, lse


CASES = [
    # (name, C, block_start, Hq, Hkv, D, splits)
    ("tiny_d64", 256, [0, 8, 16], 4, 2, 64, 0),
    ("ragged_129_one_split", 129, [0, 3, 11, 12], 16, 2, 128, 1),
    ("causal_b1_gqa2", 700, list(range(8)), 16, 8, 128, 0),
    ("many_rows", 1000, [0, 33, 66, 92], 16, 2, 128, 0),
    ("long_prefix_4_splits", 3092, [0, 33], 16, 2, 128, 4),
    ("long_prefix_planned", 3092, [0, 33], 16, 2, 128, 0),
]


@pytest.mark.parametrize("name,C,bs,Hq,Hkv,D,splits", CASES, ids=[c[0] for c in CASES])
def test_fp8_attention_matches_oracle(name, C, bs, Hq, Hkv, D, splits):
    case = synth.attn_case(70, zlib.crc32(name.encode()) % 1000, C=C, block_start=bs, Hq=Hq, Hkv=Hkv, D=D,
                           kv_pad=5)
    k8, ke, v8, ve, kd, vd = _quantised(case)
    o, lse = _run8(case.q, k8, ke, v8, ve, C, bs, splits)
    o_ref, lse_ref = oracle.block_causal_attention(case.q, kd, vd, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, name)


BENCH_SHAPES = [
    # the decode shapes bench.py times for the E4M3 cache, one block of n_q positions, planned splits:
    # (name, Hq, Hkv, C, n_q)
    ("wam_diff2_B32", 16, 8, 2048 + 128, 32),
    ("wam_diff2_B1", 16, 8, 2048 + 128, 1),
    ("fast_ddrive", 16, 2, 3124, 33),
]


@pytest.mark.parametrize("name,Hq,Hkv,C,n_q", BENCH_SHAPES, ids=[c[0] for c in BENCH_SHAPES])
def test_fp8_bench_shapes_match_oracle(name, Hq, Hkv, C, n_q):
    bs = [0, n_q]
    case = synth.attn_case(75, zlib.crc32(name.encode()) % 1000, C=C, block_start=bs, Hq=Hq, Hkv=Hkv, D=128)
    k8, ke, v8, ve, kd, vd = _quantised(case)
    o, lse = _run8(case.q, k8, ke, v8, ve, C, bs)
    o_ref, lse_ref = oracle.block_causal_attention(case.q, kd, vd, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, name)


def test_fp8_two_launch_plan_matches_oracle():
    """More (row tile, KV head) groups than one wave of SMs with the E4M3 cache:
    2,500 positions x 8 query heads on one KV head = 157 row tiles, a bulk
    launch of unsplit row tiles and a tail split wide; block size 100."""
    n_q, C = 2500, 200
    bs = list(range(0, n_q, 100)) + [n_q]
    case = synth.attn_case(76, 0, C=C, block_start=bs, Hq=8, Hkv=1, D=128)
    k8, ke, v8, ve, kd, vd = _quantised(case)
    o, lse = _run8(case.q, k8, ke, v8, ve, C, bs)
    o_ref, lse_ref = oracle.block_causal_attention(case.q, kd, vd, C, bs)
    assert_attn_close(o, lse, o_ref, lse_ref, "fp8 two-launch")


def test_fp8_zero_queries_give_the_mean_of_the_dequantised_values():
    """With Q = 0 every visible key has the same weight: o is the mean of exactly
    the visible dequantised V rows (to the bf16 rounding of o: one KV split, so
    no bf16 partials are merged) and lse the log of their count -- a wrong
    exponent, byte order or row would show."""
    C, bs = 300, [0, 5, 12]
    case = synth.attn_case(71, 0, C=C, block_start=bs, Hq=8, Hkv=2, D=128)
    k8, ke, v8, ve, kd, vd = _quantised(case)
    q = np.zeros_like(case.q)
    o, lse = _run8(q, k8, ke, v8, ve, C, bs, splits=1)
    o_ref, lse_ref = oracle.block_causal_attention(q, kd, vd, C, bs)
    np.testing.assert_allclose(host(o), o_ref, rtol=2.0 ** -8, atol=1e-6)
    np.testing.assert_allclose(host(lse), lse_ref, rtol=1e-6)


def test_fp8_fork_matches_oracle():
    N, C, n_q, priv = 3, 600, 12, 20
    f = synth.fork_case(72, 0, N=N, C=C, n_q=n_q, priv_len=priv, block_start=[0, 5, 12], Hq=16, Hkv=2, D=128)
    pk8, pke = synth.quantize_kv_e4m3(f.prefix_k)
    pv8, pve = synth.quantize_kv_e4m3(f.prefix_v)
    rk8 = np.empty(f.priv_k.shape, np.uint8)
    rv8 = np.empty(f.priv_v.shape, np.uint8)
    rke = np.empty((N, 2, 1), np.int8)
    rve = np.empty((N, 2, 1), np.int8)
    for r in range(N):
        rk8[r], rke[r] = synth.quantize_kv_e4m3(f.priv_k[r])
        rv8[r], rve[r] = synth.quantize_kv_e4m3(f.priv_v[r])
    ds = status_word()
    o, lse = bd.bd_fork_rollouts(bf16(f.q), u8(pk8), u8(pv8), u8(rk8), u8(rv8), priv, C,
                                 block_start=i32(f.block_start), prefix_k_exp=i8(pke), prefix_v_exp=i8(pve),
                                 priv_k_exp=i8(rke), priv_v_exp=i8(rve), dev_status=ds)
    assert bd.bd_check(ds) == 0
    rkd = np.stack([oracle.dequantize_kv(rk8[r], rke[r]) for r in range(N)])
    rvd = np.stack([oracle.dequantize_kv(rv8[r], rve[r]) for r in range(N)])
    o_ref, lse_ref = oracle.fork_attention(f.q, oracle.dequantize_kv(pk8, pke), oracle.dequantize_kv(pv8, pve),
                                           rkd, rvd, priv, f.block_start)
    assert_attn_close(o, lse, o_ref, lse_ref, "fp8 fork")


def test_fp8_exponent_out_of_range_is_reported():
    C, bs = 200, [0, 8]
    case = synth.attn_case(73, 0, C=C, block_start=bs, Hq=4, Hkv=2, D=64)
    k8, ke, v8, ve, _, _ = _quantised(case)
    ke = ke.copy()
    ke[1, 0] = 9
    ds = status_word()
    bd.bd_block_causal_attn(bf16(case.q), u8(k8), u8(v8), C, block_start=i32(bs), k_exp=i8(ke), v_exp=i8(ve),
                            dev_status=ds)
    assert bd.bd_check(ds) == 6  # BD_ERR_DEVICE_INPUT


def test_fp8_with_rope_is_refused():
    C, bs = 200, [0, 8]
    case = synth.attn_case(74, 0, C=C, block_start=bs, Hq=4, Hkv=2, D=64)
    k8, ke, v8, ve, _, _ = _quantised(case)
    with pytest.raises(bd.BdError) as e:
        bd.bd_block_causal_attn(bf16(case.q), u8(k8), u8(v8), C, block_start=i32(bs), k_exp=i8(ke),
                                v_exp=i8(ve), rope=dict(k_pos=None, delta=0, theta=1e4))
    assert e.value.status == 2
