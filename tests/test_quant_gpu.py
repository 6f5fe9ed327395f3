"""GPU parity of per_token_group_quant_fp8 (and its scatter variant) with the
CPU oracle: codes and scales must be bit-exact in every format and layout.

Workload: bf16 / fp16 x ~N(0,1) with 5% of rows x1e-4 and 1% all-zero rows,
tokens M in {1, 64, 512, 8192}, hidden K in {2048, 7168}, group 128, plus
groups 32 / 64, ragged K, group = K, fused SiLU(gate)*up on [M, 2K], and the
topk = 8 of 256 experts scatter."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, require_gpu, to_dev

pytestmark = pytest.mark.gpu

DT = {0: torch.bfloat16, 1: torch.float16}
SENTINEL = 0x5A


def _run_gpu(x_t, group, fmt, colmajor, fuse, K):
    M = x_t.shape[0]
    q = torch.full((M, K), SENTINEL, dtype=torch.uint8, device=x_t.device)
    s = torch.zeros(fm.scale_shape(M, K, group, fmt, colmajor), dtype=fm.scale_dtype(fmt), device=x_t.device)
    fm.per_token_group_quant_fp8(x_t, q, s, group, fmt, colmajor, fuse)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    return bits(q), bits(s)


def _compare(x_cpu, dtype, group, fmt, colmajor, fuse):
    dev = require_gpu()
    xb = synth.to_bits(x_cpu)
    K = xb.shape[1] // 2 if fuse else xb.shape[1]
    q_gpu, s_gpu = _run_gpu(x_cpu.to(dev), group, fmt, colmajor, fuse, K)
    q_ref, s_ref = oracle.group_quant(xb, dtype, group, fmt, colmajor, fuse)
    nq = int(np.count_nonzero(q_gpu != q_ref))
    assert nq == 0, f"{nq} code mismatches, first at {np.argwhere(q_gpu != q_ref)[:3]}"
    if s_ref.dtype == np.float32:
        assert np.array_equal(s_gpu.view(np.uint32), s_ref.view(np.uint32))
    else:
        assert np.array_equal(s_gpu, s_ref)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("M,K", [(1, 2048), (64, 7168), (512, 2048), (512, 7168)])
@pytest.mark.parametrize("fmt,colmajor", [(0, False), (0, True), (1, False), (2, True), (2, False), (1, True)])
def test_config5_plain(dtype, M, K, fmt, colmajor):
    x = synth.quant_input(M, K, DT[dtype], seed=100 + M + K)
    _compare(x, dtype, 128, fmt, colmajor, False)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("fmt,colmajor", [(0, False), (2, True)])
def test_config5_full_size(dtype, fmt, colmajor):
    x = synth.quant_input(8192, 7168, DT[dtype], seed=7)
    _compare(x, dtype, 128, fmt, colmajor, False)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("fmt,colmajor", [(0, False), (2, True), (1, True), (2, False)])
def test_small_groups(dtype, group, fmt, colmajor):
    x = synth.quant_input(96, 1024 + 3 * group if group == 64 else 1024 + group, DT[dtype], seed=21)
    _compare(x, dtype, group, fmt, colmajor, False)


@pytest.mark.parametrize("K", [128, 640, 896, 2176])
def test_ragged_chunks(K):
    # K not a multiple of the 512-element chunk a warp covers
    x = synth.quant_input(37, K, torch.bfloat16, seed=K)
    for fmt, cm in ((0, False), (2, True), (2, False)):
        _compare(x, 0, 128, fmt, cm, False)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("fmt,colmajor", [(0, False), (2, True), (1, False)])
@pytest.mark.parametrize("M,K", [(64, 2048), (300, 7168)])
def test_fused_silu_mul(dtype, fmt, colmajor, M, K):
    x = synth.quant_input(M, 2 * K, DT[dtype], seed=31 + M)
    _compare(x, dtype, 128, fmt, colmajor, True)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("K", [512, 4096, 5376, 7168, 8192, 8208, 12288, 14336, 20480])
@pytest.mark.parametrize("fuse", [False, True])
def test_whole_row_group(dtype, K, fuse):
    # one scale per row: rows held in registers (unfused; 128 threads a row with one to
    # four 16-value segments each up to K = 8192, 256 threads with three or four up to
    # 16384), or two passes
    x = synth.quant_input(33, 2 * K if fuse else K, DT[dtype], seed=41)
    for fmt, cm in ((0, False), (0, True), (2, True)):
        _compare(x, dtype, K, fmt, cm, fuse)


@pytest.mark.parametrize("dtype", [0, 1])
def test_encode_every_16bit_value(dtype):
    # groups whose first element is 448: a = 448, s = 1, multiplier 1, so the
    # codes are the E4M3 encoding of every bf16 / fp16 value with |v| <= 448
    vals = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_bits_to_f64(vals) if dtype == 0 else oracle.fp16_bits_to_f64(vals)
    keep = vals[np.isfinite(v) & (np.abs(v) <= 448)]
    per = 127
    rows = (keep.size + per - 1) // per
    grid = np.zeros((rows, 128), np.uint16)
    big = synth.to_bits(torch.tensor([448.0], dtype=DT[dtype]))[0]
    grid[:, 0] = big
    flat = grid[:, 1:].reshape(-1)
    flat[:keep.size] = keep
    grid[:, 1:] = flat.reshape(rows, per)
    x = synth.from_bits(grid, DT[dtype])
    _compare(x, dtype, 128, 0, False, False)


@pytest.mark.parametrize("dtype", [0, 1])
def test_every_16bit_pattern_with_non_finite(dtype):
    # all 65536 bit patterns, signaling and quiet NaN and infinities included, in
    # their natural order (so whole groups of NaN and inf next to finite groups)
    vals = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for fmt, cm in ((0, False), (2, True)):
        _compare(synth.from_bits(vals.reshape(512, 128), DT[dtype]), dtype, 128, fmt, cm, False)
    _compare(synth.from_bits(vals.reshape(1024, 64), DT[dtype]), dtype, 32, 1, True, False)
    _compare(synth.from_bits(vals.reshape(64, 1024), DT[dtype]), dtype, 1024, 0, False, False)


@pytest.mark.parametrize("M,formats", [(512, ((2, True), (0, True), (0, False))), (8192, ((2, True),))])
def test_scatter_topk8_of_256(M, formats):
    # M = 8192 is the workload the benchmark times (K = 7168, UE8M0 packed column-major)
    dev = require_gpu()
    K = 7168
    x = synth.quant_input(M, K, torch.bfloat16, seed=51)
    dst, R = synth.routing(M, topk=8, num_experts=256)
    for fmt, cm in formats:
        q = torch.full((R, K), SENTINEL, dtype=torch.uint8, device=dev)
        s = torch.zeros(fm.scale_shape(R, K, 128, fmt, cm), dtype=fm.scale_dtype(fmt), device=dev)
        fm.per_token_group_quant_fp8_scatter(x.to(dev), torch.from_numpy(dst).to(dev), q, s, 128, fmt, cm)
        torch.cuda.synchronize()
        assert fm.get_device_status() == 0
        qd, sd = oracle.group_quant_scatter(synth.to_bits(x), 0, 128, dst, R, fmt, cm)
        written = np.zeros(R, bool)
        written[dst.ravel()] = True
        qg = bits(q)
        assert np.array_equal(qg[written], qd[written])
        assert np.all(qg[~written] == SENTINEL)          # padding rows untouched
        sg = bits(s)
        if cm:
            assert np.array_equal(sg[:, :R][:, written].view(np.uint32), sd[:, :R][:, written].view(np.uint32))
        else:
            assert np.array_equal(sg[written].view(np.uint32), sd[written].view(np.uint32))


def test_scatter_skips_negative_and_flags_out_of_range():
    dev = require_gpu()
    M, K = 8, 512
    x = synth.quant_input(M, K, torch.bfloat16, seed=52)
    dst = np.arange(M * 2, dtype=np.int32).reshape(M, 2)
    dst[3, 1] = -1
    q = torch.full((2 * M, K), SENTINEL, dtype=torch.uint8, device=dev)
    s = torch.zeros(fm.scale_shape(2 * M, K, 128, 2, True), dtype=torch.int32, device=dev)
    fm.per_token_group_quant_fp8_scatter(x.to(dev), torch.from_numpy(dst).to(dev), q, s, 128, 2, True)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    assert np.all(bits(q)[7] == SENTINEL)
    dst[5, 0] = 10_000
    fm.per_token_group_quant_fp8_scatter(x.to(dev), torch.from_numpy(dst).to(dev), q, s, 128, 2, True)
    torch.cuda.synchronize()
    assert fm.get_device_status(clear=True) == fm.EINVAL
    assert fm.get_device_status() == 0


def test_empty_batch_launches_nothing():
    dev = require_gpu()
    x = torch.empty((0, 2048), dtype=torch.bfloat16, device=dev)
    q = torch.empty((0, 2048), dtype=torch.uint8, device=dev)
    s = torch.empty((0, 16), dtype=torch.float32, device=dev)
    fm.per_token_group_quant_fp8(x, q, s, 128)


@pytest.mark.parametrize("dtype", [0, 1])
def test_fused_every_16bit_gate(dtype):
    # every finite bf16 / fp16 gate value, with up = 1 and up = -0.75, through the
    # fused SiLU path: the kernel's exp / divide must agree with the oracle's bit for bit
    vals = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_bits_to_f64(vals) if dtype == 0 else oracle.fp16_bits_to_f64(vals)
    gates = vals[np.isfinite(v)]
    K = 128
    rows = (gates.size + K - 1) // K
    g = np.zeros(rows * K, np.uint16)
    g[:gates.size] = gates
    g = g.reshape(rows, K)
    for up_val in (1.0, -0.75):
        up = np.full_like(g, synth.to_bits(torch.tensor([up_val], dtype=DT[dtype]))[0])
        x = synth.from_bits(np.concatenate([g, up], axis=1), DT[dtype])
        _compare(x, dtype, 128, 0, False, True)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("fuse", [False, True])
def test_non_finite_inputs_follow_the_oracle(dtype, fuse):
    # NaN / +-inf sprinkled into some groups: the absmax leaves NaN out and keeps
    # infinities (a reading: the pages are silent on NaN in the absmax); NaN
    # products encode as +448 (the sanitizing clamp)
    M, K = 48, 1024
    x = synth.quant_input(M, 2 * K if fuse else K, DT[dtype], seed=61).float()
    rng = np.random.default_rng(62)
    for val in (float("nan"), float("inf"), float("-inf")):
        r = rng.integers(0, M, 6)
        c = rng.integers(0, x.shape[1], 6)
        x[r, c] = val
    x = x.to(DT[dtype])
    for fmt, cm in ((0, False), (2, True), (1, False)):
        _compare(x, dtype, 128, fmt, cm, fuse)
    _compare(x, dtype, K, 0, False, fuse)


def test_scale_math_matches_ieee_division_for_every_fp32():
    # the kernels form a/448 and 448/a with corrected fused-multiply-add sequences;
    # check them (and the UE8M0 exponent) against IEEE division for every positive
    # finite fp32 amax
    dev = require_gpu()
    counters = torch.zeros(3, dtype=torch.int64, device=dev)
    fm.selftest_scale_math(0, 0x7F800000, counters)
    torch.cuda.synchronize()
    assert counters.tolist() == [0, 0, 0]


def _masked_case(E, T, K, masked, dtype=0, fmt=2, cm=True, seed=81):
    dev = require_gpu()
    x = synth.quant_input(E * T, 2 * K, DT[dtype], seed=seed).reshape(E, T, 2 * K)
    q = torch.full((E, T, K), SENTINEL, dtype=torch.uint8, device=dev)
    s = torch.zeros(fm.masked_scale_shape(E, T, K, 128, fmt, cm), dtype=fm.scale_dtype(fmt), device=dev)
    fm.silu_and_mul_masked_post_quant_fp8(x.to(dev), torch.from_numpy(masked).to(dev), q, s, 128, fmt, cm)
    torch.cuda.synchronize()
    status = fm.get_device_status(clear=True)
    clamped = np.clip(masked, 0, T)
    q_ref, s_ref = oracle.masked_silu_quant(synth.to_bits(x), dtype, clamped, 128, fmt, cm)
    qg = bits(q)
    valid = np.arange(T)[None, :] < clamped[:, None]
    assert np.array_equal(qg[valid], q_ref[valid])
    assert np.all(qg[~valid] == SENTINEL)                  # rows without tokens untouched
    sg = bits(s)
    if s_ref.dtype == np.float32:
        assert np.array_equal(sg.view(np.uint32), s_ref.view(np.uint32))
    else:
        assert np.array_equal(sg, s_ref)
    return status


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("fmt,cm", [(2, True), (0, True), (0, False), (1, True)])
def test_masked_silu_quant_ep_decode(dtype, fmt, cm):
    # 32 local experts of 256 (tokens routed top-8), capacity 256 rows each, K = 2048
    masked = synth.masked_counts(4096, 32)
    assert _masked_case(32, 256, 2048, masked, dtype, fmt, cm) == 0


def test_masked_silu_quant_edges():
    # experts with no tokens, a full expert, a capacity that is not a multiple of 16,
    # and a ragged K
    masked = np.array([0, 100, 1, 37, 0, 99, 16, 17], np.int32)
    assert _masked_case(8, 100, 640, masked, seed=82) == 0
    # counts beyond the capacity are clamped and reported
    masked = np.array([5, 120, 0, 100], np.int32)
    assert _masked_case(4, 100, 512, masked, seed=83) == fm.EINVAL


def test_binding_refuses_strided_views():
    # the entry points read dense extents from a base pointer, so a strided view
    # would be read as if it were dense: the binding refuses it instead
    dev = require_gpu()
    x = torch.zeros((256, 128), dtype=torch.bfloat16, device=dev)
    q, s = fm.alloc_group_quant_outputs(128, 256, 128, fm.SCALE_FP32, False, device=dev)
    with pytest.raises(ValueError, match="contiguous"):
        fm.per_token_group_quant_fp8(x.t(), q, s, 128)
    w = torch.zeros((256, 256), dtype=torch.uint8, device=dev)
    a_s = torch.ones((128, 1), dtype=torch.float32, device=dev)
    w_s = torch.ones((256, 1), dtype=torch.float32, device=dev)
    out = torch.empty((128, 256), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="unit stride"):
        fm.fp8_scaled_mm(q, w.t(), a_s, w_s, fm.A_ROW | fm.B_COL, out)
    out_t = torch.empty((256, 128), dtype=torch.bfloat16, device=dev).t()
    with pytest.raises(ValueError, match="contiguous"):
        fm.fp8_scaled_mm(q, w, a_s, w_s, fm.A_ROW | fm.B_COL, out_t)
    # row-strided operand views (row stride 256 > K = 128) are the supported way to pass a slice
    fm.fp8_scaled_mm(w[:128, :128], w[:, :128], a_s, w_s, fm.A_ROW | fm.B_COL, out)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    assert not out.isnan().any()
