"""Seeded random shapes and modes for the GEMM and the group quant, against the
oracle (GEMM within the tolerance of gpu_util.check_gemm, quant bit-exact).
The shapes are drawn to land on every tile-table branch, on ragged edges in M,
N and K, and on both the cluster split-K path (M <= 128) and the persistent
kernels."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, check_gemm, gemm_inputs, require_gpu, to_dev

pytestmark = pytest.mark.gpu

AM = {"tensor": (fm.A_TENSOR, oracle.A_TENSOR), "row": (fm.A_ROW, oracle.A_ROW),
      "group": (fm.A_GROUP128, oracle.A_GROUP)}
BM = {"tensor": (fm.B_TENSOR, oracle.B_TENSOR), "col": (fm.B_COL, oracle.B_COL)}


def _gemm_cases(n=24, seed=1234):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        M = int(rng.choice([1, 2, 7, 16, 33, 64, 100, 128, 129, 200, 256, 300, 513, 1100]))
        N = 8 * int(rng.integers(1, 200))
        a_mode = ["tensor", "row", "group"][i % 3]
        b_mode = ["tensor", "col"][(i // 3) % 2]
        K = 128 * int(rng.integers(1, 12)) if a_mode == "group" else 16 * int(rng.integers(1, 90))
        det = bool(rng.integers(0, 4) == 0)
        bias = bool(rng.integers(0, 2))
        out_dtype = int(rng.integers(0, 2))
        cases.append((M, N, K, a_mode, b_mode, det, bias, out_dtype, seed + i))
    return cases


@pytest.mark.parametrize("M,N,K,a_mode,b_mode,det,bias,out_dtype,seed", _gemm_cases())
def test_gemm_fuzz(M, N, K, a_mode, b_mode, det, bias, out_dtype, seed):
    dev = require_gpu()
    A, a_s, B, b_s = gemm_inputs(M, N, K, a_mode, b_mode, seed_a=seed, seed_b=seed + 1)
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=seed + 2)) if bias else None
    out = torch.empty((M, N), dtype=torch.bfloat16 if out_dtype == 0 else torch.float16, device=dev)
    fm.fp8_scaled_mm(to_dev(A, dev), to_dev(B, dev), to_dev(np.ascontiguousarray(a_s, np.float32), dev),
                     to_dev(np.ascontiguousarray(b_s, np.float32), dev), AM[a_mode][0] | BM[b_mode][0], out,
                     bias=to_dev(bias_bits, dev).view(torch.bfloat16) if bias else None, deterministic=det)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    _, exact, sumabs = oracle.gemm(A, B, a_s, b_s, AM[a_mode][1], BM[b_mode][1], bias_bits=bias_bits,
                                   out_dtype=out_dtype, want_exact=True)
    check_gemm(bits(out), exact, sumabs, K, out_dtype, f"fuzz M{M} N{N} K{K} {a_mode}/{b_mode} det={det}")


def _quant_cases(n=24, seed=4321):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        group = int(rng.choice([32, 64, 128]))
        K = group * int(rng.integers(1, 40))
        M = int(rng.choice([1, 3, 15, 16, 17, 100, 257, 1000]))
        fmt = int(rng.integers(0, 3))
        cm = bool(rng.integers(0, 2))
        fuse = bool(rng.integers(0, 2))
        dt = int(rng.integers(0, 2))
        cases.append((M, K, group, fmt, cm, fuse, dt, seed + i))
    return cases


@pytest.mark.parametrize("M,K,group,fmt,cm,fuse,dt,seed", _quant_cases())
def test_quant_fuzz(M, K, group, fmt, cm, fuse, dt, seed):
    dev = require_gpu()
    x = synth.quant_input(M, 2 * K if fuse else K, torch.bfloat16 if dt == 0 else torch.float16, seed=seed)
    q = torch.full((M, K), 0x5A, dtype=torch.uint8, device=dev)
    s = torch.zeros(fm.scale_shape(M, K, group, fmt, cm), dtype=fm.scale_dtype(fmt), device=dev)
    fm.per_token_group_quant_fp8(x.to(dev), q, s, group, fmt, cm, fuse)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    q_ref, s_ref = oracle.group_quant(synth.to_bits(x), dt, group, fmt, cm, fuse)
    assert np.array_equal(bits(q), q_ref)
    s_gpu = bits(s)
    if s_ref.dtype == np.float32:
        assert np.array_equal(s_gpu.view(np.uint32), s_ref.view(np.uint32))
    else:
        assert np.array_equal(s_gpu, s_ref)


def _scaled_mode_cases(n=12, seed=777):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        M = int(rng.choice([1, 17, 128, 129, 300, 1100, 2100]))
        N = 8 * int(rng.integers(1, 300))
        K = 128 * int(rng.integers(1, 20))
        kind = ["ue8m0", "block_f32", "block_ue8m0"][i % 3]
        pad = int(rng.choice([0, 16, 64]))
        cases.append((M, N, K, kind, pad, bool(rng.integers(0, 2)), int(rng.integers(0, 2)), seed + i))
    return cases


@pytest.mark.parametrize("M,N,K,kind,pad,bias,out_dtype,seed", _scaled_mode_cases())
def test_gemm_fuzz_packed_and_block_scales(M, N, K, kind, pad, bias, out_dtype, seed):
    # packed UE8M0 group-128 A scales (as the quant writes them) and 128 x 128 block B
    # scales, with a strided A
    dev = require_gpu()
    X = synth.to_bits(synth.normal((M, K), 1.0, seed=seed))
    W = synth.to_bits(synth.normal((N, K), 0.02, seed=seed + 1))
    if kind == "block_f32":
        A, a_s, _ = oracle.group_quant_canonical(X, 0, 128)
        a_fm, a_or, a_dev = fm.A_GROUP128, oracle.A_GROUP, to_dev(np.ascontiguousarray(a_s, np.float32), dev)
    else:
        A, a_s = oracle.group_quant(X, 0, 128, oracle.SCALE_UE8M0_PACKED, True)
        a_fm, a_or, a_dev = fm.A_GROUP128_UE8M0, oracle.A_GROUP_UE8M0, to_dev(np.ascontiguousarray(a_s), dev)
    if kind.startswith("block"):
        B, b_s = oracle.quantize_blocks(W)
        b_fm, b_or = fm.B_BLOCK128, oracle.B_BLOCK
    else:
        B, b_s = oracle.quantize_rows(W)
        b_fm, b_or = fm.B_COL, oracle.B_COL
    Aw = np.full((M, K + pad), 0x5A, np.uint8)
    Aw[:, :K] = A
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=seed + 2)) if bias else None
    out = torch.empty((M, N), dtype=torch.bfloat16 if out_dtype == 0 else torch.float16, device=dev)
    fm.fp8_scaled_mm(to_dev(Aw, dev), to_dev(B, dev), a_dev, to_dev(np.ascontiguousarray(b_s, np.float32), dev),
                     a_fm | b_fm, out, bias=to_dev(bias_bits, dev).view(torch.bfloat16) if bias else None, K=K)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    _, exact, sumabs = oracle.gemm(Aw, B, a_s, b_s, a_or, b_or, bias_bits=bias_bits, out_dtype=out_dtype, K=K,
                                   want_exact=True)
    check_gemm(bits(out), exact, sumabs, K, out_dtype, f"fuzz M{M} N{N} K{K} {kind} pad{pad}")
