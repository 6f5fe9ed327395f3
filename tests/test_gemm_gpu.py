"""GPU parity of fp8_scaled_mm with the CPU oracle.

Inputs: bf16 activations ~N(0,1) and weights ~N(0,0.02) quantized to E4M3 by
the oracle (per-row / per-channel, per-tensor or group-128 scales), so no
input of the comparison comes from the CUDA path.  Each output element must
be within max(1 ulp, 2^-7 |ref|) of the oracle's exactly accumulated result
(see oracle.parity.check_gemm for the near-cancellation rule).  Large problems
are compared on one row of every 128-row M block (at an in-block offset that
rotates from block to block) against all N, plus the first and last rows, both
sides of tile boundaries and random rows; one prefill shape is compared over
its whole output."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, check_gemm, gemm_inputs, require_gpu, to_dev

pytestmark = pytest.mark.gpu

AMODE = {"tensor": fm.A_TENSOR, "row": fm.A_ROW, "group": fm.A_GROUP128}
BMODE = {"tensor": fm.B_TENSOR, "col": fm.B_COL}
OAMODE = {"tensor": oracle.A_TENSOR, "row": oracle.A_ROW, "group": oracle.A_GROUP}
OBMODE = {"tensor": oracle.B_TENSOR, "col": oracle.B_COL}


def sample_rows(M, n_random=16, seed=0):
    """Rows to compare for a large M: one in every 128-row M block, at offset
    37 b mod 128 in block b, so that every output tile -- whatever wave, raster
    group or tile width computed it -- has a row checked against all N; the first
    and last two rows; both sides of block boundaries spread over M; random rows."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1, M - 2}
    for b in range((M + 127) // 128):
        rows.add(min(M - 1, 128 * b + (37 * b) % 128))
    for b in range(128, M, 128 * max(1, M // 128 // 8)):
        rows.update({b - 1, b})
    rows.update(rng.integers(0, M, size=n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < M), np.int64)


def run_case(M, N, K, a_mode, b_mode, out_dtype=0, bias=False, lda=None, deterministic=False, rows=None,
             seed=0, A=None, a_s=None, B=None, b_s=None):
    dev = require_gpu()
    if A is None:
        A, a_s, B, b_s = gemm_inputs(M, N, K, a_mode, b_mode, seed_a=seed, seed_b=seed + 1, lda=lda)
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=synth.SEED_BIAS)) if bias else None
    out = torch.empty((M, N), dtype=torch.bfloat16 if out_dtype == 0 else torch.float16, device=dev)
    At, Bt = to_dev(A, dev), to_dev(B, dev)
    ast, bst = to_dev(np.ascontiguousarray(a_s, np.float32), dev), to_dev(np.ascontiguousarray(b_s, np.float32), dev)
    biast = to_dev(bias_bits, dev).view(torch.bfloat16) if bias else None
    fm.fp8_scaled_mm(At, Bt, ast, bst, AMODE[a_mode] | BMODE[b_mode], out, bias=biast,
                     deterministic=deterministic, K=K)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    ref_bits, exact, sumabs = oracle.gemm(A, B, a_s, b_s, OAMODE[a_mode], OBMODE[b_mode], bias_bits=bias_bits,
                                          out_dtype=out_dtype, K=K, rows=rows, want_exact=True)
    got = bits(out) if rows is None else bits(out[torch.from_numpy(rows).to(dev)])
    return check_gemm(got, exact, sumabs, K, out_dtype, f"M{M} N{N} K{K} {a_mode}/{b_mode}")


def test_config1_tiny_group128_scales():
    # X [64,512] group-quantized (group 128, fp32 scales), W [256,512] per-channel
    run_case(64, 256, 512, "group", "col")


def test_config1_group_scales_colmajor():
    dev = require_gpu()
    M, N, K = 64, 256, 512
    A, a_s, B, b_s = gemm_inputs(M, N, K, "group", "col", seed_a=3, seed_b=4)
    a_cm = np.zeros((K // 128, oracle.pad4(M)), np.float32)
    a_cm[:, :M] = a_s.T
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fm.fp8_scaled_mm(to_dev(A), to_dev(B), to_dev(a_cm), to_dev(b_s), fm.A_GROUP128_COLMAJOR | fm.B_COL, out)
    torch.cuda.synchronize()
    _, exact, sumabs = oracle.gemm(A, B, a_s, b_s, oracle.A_GROUP, oracle.B_COL, want_exact=True)
    check_gemm(bits(out), exact, sumabs, K)


@pytest.mark.parametrize("N", [4096, 12288, 14336])
@pytest.mark.parametrize("M", [1, 16, 128, 2048, 8192])
def test_config2_per_tensor(M, N):
    rows = None if M <= 128 else sample_rows(M, seed=M)
    run_case(M, N, 4096, "tensor", "tensor", rows=rows, seed=M + N)


@pytest.mark.parametrize("M,K,N", [(8320, 5376, 21504), (8320, 5376, 14336), (23216, 5376, 28672),
                                   (15760, 5376, 28672), (8320, 14336, 5376)])
def test_config3_rowwise_large(M, K, N):
    rows = sample_rows(M, n_random=12, seed=K)
    assert len(rows) >= (M + 127) // 128
    run_case(M, N, K, "row", "col", rows=rows, seed=M)


def test_config3_full_output_8320x14336x5376():
    # the prefill shape with the fewest flops (1.28 TFLOP), every one of its 44.7 M
    # outputs against the oracle
    stats = run_case(8320, 5376, 14336, "row", "col", seed=8320)
    assert stats["n"] == 8320 * 5376


def test_ue8m0_scale_bytes_at_both_ends_of_the_range():
    # the oracle pin's case (bytes 0, 1, 127, 255) through the group-scale kernel: the
    # kernel reads byte 0 as 2^-127 and byte 255 as +inf, as the oracle does
    from test_oracle_gemm import ue8m0_edge_case
    dev = require_gpu()
    A, words, B, b_s = ue8m0_edge_case()
    M, N = A.shape[0], B.shape[0]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fm.fp8_scaled_mm(to_dev(A), to_dev(B), to_dev(words), to_dev(b_s), fm.A_GROUP128_UE8M0 | fm.B_COL, out)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    ref_bits, exact, sumabs = oracle.gemm(A, B, words, b_s, oracle.A_GROUP_UE8M0, oracle.B_COL, want_exact=True)
    got = bits(out)
    check_gemm(got, exact, sumabs, 128, 0, "ue8m0 bytes 0/255", allow_nonfinite=True)
    fin = np.isfinite(exact)
    assert np.array_equal(got[fin], ref_bits[fin])      # these sums are exact: same bits


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (3, 24, 80), (127, 264, 144), (129, 136, 272), (200, 520, 1040),
                                   (257, 1000, 128), (64, 256, 512)])
@pytest.mark.parametrize("a_mode,b_mode", [("row", "col"), ("tensor", "col"), ("row", "tensor")])
def test_edges_and_scale_modes(M, N, K, a_mode, b_mode):
    run_case(M, N, K, a_mode, b_mode, seed=M * 7 + N)


@pytest.mark.parametrize("out_dtype", [0, 1])
@pytest.mark.parametrize("bias", [False, True])
def test_bias_fp16_and_strided_a(out_dtype, bias):
    run_case(300, 4096, 4096, "row", "col", out_dtype=out_dtype, bias=bias, lda=4096 + 64)
    run_case(97, 64, 80, "row", "col", out_dtype=out_dtype, bias=bias, lda=80 + 64)


def test_group_scales_larger():
    run_case(300, 1024, 2048, "group", "col", seed=5)
    run_case(1, 512, 1024, "group", "tensor", seed=6)


def test_empty_and_invalid():
    dev = require_gpu()
    A = torch.zeros((0, 128), dtype=torch.uint8, device=dev)
    B = torch.zeros((64, 128), dtype=torch.uint8, device=dev)
    s = torch.ones(64, dtype=torch.float32, device=dev)
    out = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    fm.fp8_scaled_mm(A, B, s, s, fm.A_ROW | fm.B_COL, out)       # M == 0: nothing launched
    A = torch.zeros((4, 128), dtype=torch.uint8, device=dev)
    out = torch.empty((4, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(fm.Fp8mmError) as e:
        fm.fp8_scaled_mm(A, B, s, s, fm.A_ROW | fm.B_COL, out, K=120)
    assert e.value.status == fm.EINVAL


def test_bounded_wait_reports_timeout_and_context_survives():
    require_gpu()
    assert fm.get_device_status(clear=True) in (0, fm.ETIMEOUT)
    fm.selftest_bounded_wait(50_000_000)           # 50 ms on a barrier nobody arrives on
    assert fm.get_device_status(clear=True) == fm.ETIMEOUT
    assert fm.get_device_status() == 0
    run_case(64, 256, 512, "row", "col")           # the context is still usable


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129])
def test_small_m_boundaries(M):
    # the small-M path (weights as the 128-row MMA operand, K split across a cluster)
    # at every token-block boundary, with a ragged last weight tile
    run_case(M, 1416, 2048, "row", "col", seed=M)


@pytest.mark.parametrize("M,N,K", [(128, 1032, 4096), (97, 4096, 3072), (80, 1416, 2048)],
                         ids=["4-way", "3-way", "2-way"])
def test_small_m_wide_token_block_splits(M, N, K):
    # 128-token blocks split K into up to four ranges; the reduction over them takes
    # eight outputs per pass (two ranges) or four (three or four), ragged rows included
    run_case(M, N, K, "row", "col", seed=M + K, bias=True)


@pytest.mark.parametrize("K", [16, 48, 128, 400, 28672])
def test_small_m_k_extremes(K):
    # K from a single partial K block to the largest K of the workloads
    run_case(8, 256, K, "row", "col", seed=K, bias=True)


def _block_case(M, N, K, seed, ue8m0_a=True, rows=None):
    dev = require_gpu()
    X = synth.to_bits(synth.normal((M, K), 1.0, seed=seed))
    W = synth.to_bits(synth.normal((N, K), 0.02, seed=seed + 1))
    B, b_blk = oracle.quantize_blocks(W)
    if ue8m0_a:
        A, a_words = oracle.group_quant(X, 0, 128, oracle.SCALE_UE8M0_PACKED, True)
        a_dev, a_mode, o_mode, a_ref = to_dev(a_words), fm.A_GROUP128_UE8M0, oracle.A_GROUP_UE8M0, a_words
    else:
        A, a_f, _ = oracle.group_quant_canonical(X, 0, 128)
        a_dev, a_mode, o_mode, a_ref = to_dev(a_f), fm.A_GROUP128, oracle.A_GROUP, a_f
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fm.fp8_scaled_mm(to_dev(A), to_dev(B), a_dev, to_dev(b_blk), a_mode | fm.B_BLOCK128, out)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    _, exact, sumabs = oracle.gemm(A, B, a_ref, b_blk, o_mode, oracle.B_BLOCK, rows=rows, want_exact=True)
    got = bits(out) if rows is None else bits(out[torch.from_numpy(rows).to(dev)])
    return check_gemm(got, exact, sumabs, K, 0, f"block M{M} N{N} K{K}")


@pytest.mark.parametrize("ue8m0_a", [True, False])
def test_block_scaled_gemm(ue8m0_a):
    # A 1 x 128 group scales (the group quant's UE8M0 output read directly, or fp32),
    # B 128 x 128 block scales
    _block_case(512, 7168, 2048, 11, ue8m0_a, rows=sample_rows(512, seed=1))
    _block_case(300, 1000, 1024, 12, ue8m0_a)
    _block_case(1, 136, 256, 13, ue8m0_a)


@pytest.mark.parametrize("M,N,K,a_mode,b_mode,out_dtype,bias", [
    (2048, 4096, 4096, "tensor", "tensor", 0, False),   # the per-tensor configuration's tail-wave shape
    (4096, 4096, 4096, "row", "col", 0, False),
    (1937, 12280, 4096, "row", "col", 1, True),          # ragged M and N, fp16 out, bias
])
def test_tail_wave_shapes(M, N, K, a_mode, b_mode, out_dtype, bias):
    # shapes whose 256-wide tiles leave the last wave badly filled (the tile table then
    # prefers 224- or 192-wide tiles): every output against the oracle, and a second
    # call bit-identical to the first
    dev = require_gpu()
    A, a_s, B, b_s = gemm_inputs(M, N, K, a_mode, b_mode, seed_a=M, seed_b=N)
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=synth.SEED_BIAS)) if bias else None
    odt = torch.bfloat16 if out_dtype == 0 else torch.float16
    args = (to_dev(A), to_dev(B), to_dev(np.ascontiguousarray(a_s, np.float32)),
            to_dev(np.ascontiguousarray(b_s, np.float32)), AMODE[a_mode] | BMODE[b_mode])
    biast = to_dev(bias_bits).view(torch.bfloat16) if bias else None
    outs = []
    for _ in range(2):
        out = torch.empty((M, N), dtype=odt, device=dev)
        fm.fp8_scaled_mm(*args, out, bias=biast)
        outs.append(out)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    _, exact, sumabs = oracle.gemm(A, B, a_s, b_s, OAMODE[a_mode], OBMODE[b_mode], bias_bits=bias_bits,
                                   out_dtype=out_dtype, want_exact=True)
    check_gemm(bits(outs[0]), exact, sumabs, K, out_dtype, f"tail wave M{M} N{N} K{K}")
