"""GPU parity of static per-tensor activation quant and of the requantization
of a fused weight's per-shard scales to their maximum, against the CPU oracle,
bit-exact.  Inputs are seeded bf16 / fp16 activations and weights quantized by
the oracle one logical shard at a time (each shard with its own absmax/448
scale), as a checkpoint of a fused QKV or gate/up projection stores them."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, require_gpu, to_dev

pytestmark = pytest.mark.gpu

TORCH_DT = {0: torch.bfloat16, 1: torch.float16}


def _static_case(x_bits, dt, scale):
    dev = require_gpu()
    x = to_dev(x_bits, dev).view(TORCH_DT[dt])
    sc = torch.tensor([scale], dtype=torch.float32, device=dev)
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    fm.static_per_tensor_quant_fp8(x, sc, q)
    torch.cuda.synchronize()
    want = oracle.static_quant(x_bits, dt, np.float32(scale))
    got = bits(q)
    bad = np.flatnonzero(got.ravel() != want.ravel())
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


@pytest.mark.parametrize("dt", [0, 1])
@pytest.mark.parametrize("M,K", [(1, 16), (3, 2048), (129, 4096), (8192, 4096)])
def test_static_quant_activations(dt, M, K):
    x = synth.to_bits(synth.quant_input(M, K, TORCH_DT[dt], seed=M + K))
    # the tensor's own absmax / 448 (no saturation) and a smaller scale (saturating tails)
    _, s = oracle.quantize_tensor(x, dt)
    s = float(s)
    _static_case(x, dt, s)
    _static_case(x, dt, s / 8)


@pytest.mark.parametrize("dt", [0, 1])
@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.0e-5, 7.5, 2.0 ** -20, 1.0e30, 2.0 ** -130, 0.0, -0.37])
def test_static_quant_every_16bit_value(dt, scale):
    # every bit pattern of the input type, NaN and infinities included
    _static_case(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16), dt, scale)


def test_static_quant_empty_and_invalid():
    dev = require_gpu()
    sc = torch.ones(1, dtype=torch.float32, device=dev)
    x = torch.zeros(0, dtype=torch.bfloat16, device=dev)
    fm.static_per_tensor_quant_fp8(x, sc, torch.empty(0, dtype=torch.uint8, device=dev))
    x = torch.zeros(24, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fm.Fp8mmError) as e:
        fm.static_per_tensor_quant_fp8(x, sc, torch.empty(24, dtype=torch.uint8, device=dev))
    assert e.value.status == fm.EINVAL


def _fused_weight(widths, K, extra_rows, seed):
    """Codes of a fused weight, each logical shard per-tensor quantized by the oracle."""
    parts, scales = [], []
    for i, w in enumerate(widths):
        W = synth.to_bits(synth.normal((w, K), 0.02 * (1 + i), seed=seed + i))
        q, s = oracle.quantize_tensor(W)
        parts.append(q)
        scales.append(np.float32(s))
    if extra_rows:
        rng = np.random.default_rng(seed)
        parts.append(rng.integers(0, 256, size=(extra_rows, K), dtype=np.uint8))
    return np.concatenate(parts, axis=0), np.array(scales, np.float32)


def _requant_case(codes, scales, widths, in_place):
    dev = require_gpu()
    w = to_dev(codes, dev)
    ss = to_dev(scales, dev)
    out = w if in_place else torch.empty_like(w)
    w_out, smax = fm.requantize_with_max_scale_fp8(w, ss, widths, w_out=out)
    torch.cuda.synchronize()
    want, want_max = oracle.requantize_with_max_scale(codes, scales, widths)
    if np.all(scales == scales[0]):
        # one common scale leaves every code but the NaN codes unchanged
        nan = (codes & 0x7F) == 0x7F
        assert np.array_equal(want[~nan], codes[~nan])
    assert np.float32(smax.item()) == want_max
    got = bits(w_out)
    bad = np.flatnonzero(got.ravel() != want.ravel())
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}"


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("widths,K,extra", [([4096, 1024, 1024], 4096, 0),      # QKV, 8 KV heads of 128
                                            ([14336, 14336], 4096, 0),          # gate / up
                                            ([128, 32, 32], 256, 48),           # rows past the shards
                                            ([16], 16, 0)])
def test_requantize_fused_weights(widths, K, extra, in_place):
    codes, scales = _fused_weight(widths, K, extra, seed=sum(widths) + K)
    _requant_case(codes, scales, widths, in_place)


def test_requantize_every_code_and_scale_ratio():
    # all 256 codes (NaN codes included) under shard scales of assorted ratios to the maximum
    codes = np.tile(np.arange(256, dtype=np.uint8), (12, 1))
    scales = np.array([1.0, 0.5, 0.3, 1e-3, 0.999, 2.0 ** -12], np.float32)
    _requant_case(codes, scales, [2] * 6, in_place=False)
    # equal scales leave every non-NaN code unchanged
    eq = np.full(3, 0.0123, np.float32)
    _requant_case(codes[:6], eq, [2, 2, 2], in_place=False)


def test_requantize_invalid_widths():
    dev = require_gpu()
    w = torch.zeros((8, 32), dtype=torch.uint8, device=dev)
    ss = torch.ones(2, dtype=torch.float32, device=dev)
    with pytest.raises(fm.Fp8mmError) as e:
        fm.requantize_with_max_scale_fp8(w, ss, [6, 6])          # shards past the last row
    assert e.value.status == fm.EINVAL
    with pytest.raises(fm.Fp8mmError):
        fm.requantize_with_max_scale_fp8(w, ss, [])
