"""GPU parity of the int8 group quant and of the row-padded FP8 group quant
with the CPU oracle, bit-exact (codes and scale bits).  Inputs come from the
seeded generators; expected values only from the oracle."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, require_gpu

pytestmark = pytest.mark.gpu

DT = {0: torch.bfloat16, 1: torch.float16}
SENTINEL = 0x5A


def _int8_case(x_cpu, dtype, group, colmajor, fuse):
    dev = require_gpu()
    xb = synth.to_bits(x_cpu)
    M = xb.shape[0]
    K = xb.shape[1] // 2 if fuse else xb.shape[1]
    q = torch.full((M, K), SENTINEL, dtype=torch.int8, device=dev)
    s = torch.zeros(fm.scale_shape(M, K, group, fm.SCALE_FP32, colmajor), dtype=torch.float32, device=dev)
    fm.per_token_group_quant_int8(x_cpu.to(dev), q, s, group, colmajor, fuse)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    q_ref, s_ref = oracle.group_quant_int8(xb, dtype, group, colmajor, fuse)
    q_gpu, s_gpu = bits(q), bits(s)
    bad = np.argwhere(q_gpu != q_ref)
    assert bad.size == 0, f"{len(bad)} code mismatches, first at {bad[:3]}"
    assert np.array_equal(s_gpu.view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 2048), (129, 7168), (4096, 7168)])
@pytest.mark.parametrize("colmajor", [False, True])
def test_int8_plain(dtype, M, K, colmajor):
    _int8_case(synth.quant_input(M, K, DT[dtype], seed=200 + M + K), dtype, 128, colmajor, False)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("fuse", [False, True])
def test_int8_groups_and_fused(group, fuse):
    K = 1024 + 3 * group
    x = synth.quant_input(96, 2 * K if fuse else K, DT[0], seed=group + fuse)
    _int8_case(x, 0, group, True, fuse)
    _int8_case(x, 0, group, False, fuse)


@pytest.mark.parametrize("dtype", [0, 1])
def test_int8_every_16bit_value(dtype):
    # all 65536 bit patterns of the input type, NaN and infinities included,
    # 128 to a group: non-finite groups follow the oracle's clamp
    vals = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    _int8_case(synth.from_bits(vals, DT[dtype]), dtype, 128, False, False)
    _int8_case(synth.from_bits(vals.reshape(1024, 64), DT[dtype]), dtype, 64, True, False)


@pytest.mark.parametrize("K", [1024, 2048 + 16])
def test_int8_whole_row_group(K):
    _int8_case(synth.quant_input(33, K, DT[0], seed=K), 0, K, False, False)


def test_int8_rejects_bad_group():
    dev = require_gpu()
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((4, 128), dtype=torch.int8, device=dev)
    s = torch.zeros((4, 1), dtype=torch.float32, device=dev)
    with pytest.raises(fm.Fp8mmError):
        fm.per_token_group_quant_int8(x, q, s, 96)


def _padded_case(M, M_pad, K, fmt, colmajor, dtype=0, seed=0):
    dev = require_gpu()
    x = synth.quant_input(M, K, DT[dtype], seed=seed)
    q = torch.full((M_pad, K), SENTINEL, dtype=torch.uint8, device=dev)
    shape = fm.scale_shape(M_pad, K, 128, fmt, colmajor)
    s = torch.empty(shape, dtype=fm.scale_dtype(fmt), device=dev)
    s.view(torch.uint8).fill_(SENTINEL)
    fm.per_token_group_quant_fp8_row_padded(x.to(dev), q, s, 128, fmt, colmajor)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    q_ref, s_ref = oracle.group_quant_row_padded(synth.to_bits(x), dtype, 128, M_pad, fmt, colmajor)
    assert np.array_equal(bits(q), q_ref)
    s_gpu = bits(s)
    if colmajor:   # columns past M_pad are padding and are not written
        s_gpu, s_ref = s_gpu[:, :M_pad], s_ref[:, :M_pad]
    assert np.array_equal(s_gpu.view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("fmt,colmajor", [(0, True), (0, False), (1, True), (2, True), (2, False)])
@pytest.mark.parametrize("M,M_pad", [(100, 128), (1, 4), (0, 16), (256, 256), (4000, 4096)])
def test_row_padded(M, M_pad, fmt, colmajor):
    _padded_case(M, M_pad, 2048, fmt, colmajor, seed=M + M_pad)


def test_row_padded_fp16_and_invalid():
    _padded_case(37, 41, 7168, 0, True, dtype=1, seed=5)
    dev = require_gpu()
    x = torch.zeros((8, 128), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((4, 128), dtype=torch.uint8, device=dev)
    s = torch.zeros((1, 4), dtype=torch.float32, device=dev)
    with pytest.raises(fm.Fp8mmError) as e:
        fm.per_token_group_quant_fp8_row_padded(x, q, s, 128)      # M_pad < M
    assert e.value.status == fm.EINVAL
