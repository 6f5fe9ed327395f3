"""Pins for the oracle's fp64 -> bf16 / fp16 rounding and the exp / SiLU
routine (CPU only).

bf16 rounding is checked against torch's fp32 -> bf16 cast and fp16 against
numpy's fp64 -> fp16 cast (both round to nearest even); exp against the fp64
libm exp to within 2 fp32 ulp.
"""
import math

import numpy as np
import torch

import oracle


def _bf16_ref(x64):
    t = torch.from_numpy(x64.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # force every tie / near-tie pattern of the 16 dropped bits
    low = np.array([0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    bits = np.concatenate([bits, ((bits[:200_000, None] & 0xFFFF0000) | low[None]).ravel()])
    x = bits.view(np.float32)
    x = x[np.isfinite(x)].astype(np.float64)
    assert np.array_equal(oracle.round_bf16(x), _bf16_ref(x))


def test_bf16_overflow_and_specials():
    big = np.array([3.3895313892515355e38, 3.39e38, 1e39, -1e39, 0.0, -0.0, 1e-45])
    got = oracle.round_bf16(big)
    assert got[0] == 0x7F7F                      # largest finite bf16
    assert got[1] == 0x7F7F                      # below the overflow midpoint
    assert got[2] == 0x7F80 and got[3] == 0xFF80
    assert got[4] == 0x0000 and got[5] == 0x8000
    assert got[6] == 0x0000                      # far below the smallest subnormal


def test_bf16_double_rounding_is_avoided():
    # 1 + 2^-8 + 2^-30 is above the bf16 midpoint 1 + 2^-8; rounding through
    # fp32 first would land on the midpoint and round to even (1.0)
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30])
    assert oracle.round_bf16(x)[0] == 0x3F81


def test_fp16_matches_numpy():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(1_000_000) * 10.0 ** rng.integers(-9, 6, size=1_000_000),
        np.array([65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 0.0]),
    ])
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.round_fp16(x), want)


def _ulp32(v):
    v = np.abs(v.astype(np.float32))
    return np.spacing(v).astype(np.float64)


def test_exp_within_two_ulp():
    x = np.concatenate([
        np.linspace(-103.0, 88.7, 2_000_001, dtype=np.float32),
        np.random.default_rng(3).uniform(-20, 20, 1_000_000).astype(np.float32),
        np.array([0.0, 1.0, -1.0, 0.5, 1e-8, -1e-8], np.float32),
    ])
    got = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    normal = ref >= 2.0 ** -126
    err = np.abs(got - ref)[normal] / _ulp32(ref[normal])
    assert err.max() <= 2.0, err.max()
    # subnormal results: absolute error within two subnormal steps
    sub = ~normal
    assert np.all(np.abs(got[sub] - ref[sub]) <= 2 * 2.0 ** -149)


def test_exp_special_values():
    x = np.array([0.0, 88.72, 88.73, 89.5, 200.0, -104.5, -200.0, np.inf, -np.inf], np.float32)
    got = oracle.exp_f32(x)
    assert got[0] == 1.0
    assert np.isfinite(got[1]) and np.isinf(got[2]) and np.isinf(got[3]) and np.isinf(got[4])
    assert got[5] == 0.0 and got[6] == 0.0 and np.isinf(got[7]) and got[8] == 0.0
    assert abs(float(oracle.exp_f32(np.array([1.0], np.float32))[0]) - math.e) < 2.5e-7


def test_silu_against_fp64():
    g = np.concatenate([np.linspace(-30, 30, 600_001, dtype=np.float32),
                        np.array([0.0, 100.0, -100.0, 1e4, -1e4], np.float32)])
    got = oracle.silu_f32(g).astype(np.float64)
    g64 = g.astype(np.float64)
    with np.errstate(over="ignore"):
        ref = g64 / (1.0 + np.exp(-g64))
    ok = np.abs(ref) >= 2.0 ** -126
    err = np.abs(got - ref)[ok] / _ulp32(ref[ok])
    assert err.max() <= 4.0, err.max()
    assert got[-5] == 0.0
    assert got[-4] == 100.0 and got[-2] == 1e4          # g / (1 + ~0) = g exactly
    assert got[-3] == 0.0 and np.signbit(got[-3])       # exp(100) overflows: -100 / inf = -0
