"""Guard bands around GEMM outputs.

Every kernel form of fp8_scaled_mm must write exactly its M x N output -- edge
tiles clipped at M and N -- and nothing before or after it.  The output here is a
window of a larger buffer whose margins (16 KB on each side) hold a sentinel;
after the call the margins must be untouched and the window must match the
oracle.  One case per kernel form, each with ragged M and N: the swap-AB split-K
kernel at each token-block width, the 128 x BN kernel at the widths the tile
table picks, the deterministic cluster and fold kernels, and the per-group and
block-scaled kernels (fp16 output and bias included)."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, check_gemm, gemm_inputs, require_gpu, to_dev

pytestmark = pytest.mark.gpu

GUARD = 8192          # sentinel elements on each side of the output
SENTINEL = 0x7A5B     # 16-bit pattern the margins are filled with

AMODE = {"tensor": fm.A_TENSOR, "row": fm.A_ROW, "group": fm.A_GROUP128}
BMODE = {"tensor": fm.B_TENSOR, "col": fm.B_COL}
OAMODE = {"tensor": oracle.A_TENSOR, "row": oracle.A_ROW, "group": oracle.A_GROUP}
OBMODE = {"tensor": oracle.B_TENSOR, "col": oracle.B_COL}


def _guarded_out(M, N, out_dtype, dev):
    buf = torch.full((2 * GUARD + M * N,), SENTINEL, dtype=torch.int16, device=dev)
    out = buf[GUARD:GUARD + M * N].view(M, N).view(torch.bfloat16 if out_dtype == 0 else torch.float16)
    return buf, out


def _check_margins(buf, M, N, what):
    b = buf.cpu().numpy().view(np.uint16)
    before, after = b[:GUARD], b[GUARD + M * N:]
    assert np.all(before == SENTINEL), f"{what}: {int(np.sum(before != SENTINEL))} elements written before the output"
    assert np.all(after == SENTINEL), f"{what}: {int(np.sum(after != SENTINEL))} elements written after the output"


@pytest.mark.parametrize("M,N,K,a_mode,b_mode,out_dtype,bias,det", [
    (5, 264, 256, "row", "col", 0, False, False),        # swap-AB, 16-token block
    (50, 1000, 512, "tensor", "col", 1, True, False),    # swap-AB, 64-token block
    (128, 4104, 256, "row", "tensor", 0, True, False),   # swap-AB, 128-token block
    (300, 520, 512, "row", "col", 0, False, False),      # narrow tiles
    (2048, 4096, 256, "tensor", "tensor", 0, False, False),   # 224-wide tiles
    (1937, 12280, 128, "row", "col", 1, True, False),    # 256-wide tiles, ragged M and N
    (100, 4104, 1024, "row", "col", 0, True, True),      # deterministic, cluster kernel
    (2500, 1000, 512, "row", "col", 1, False, True),     # deterministic, fold kernel
    (300, 1000, 1024, "group", "col", 0, True, False),   # per-group A scales
])
def test_output_written_exactly(M, N, K, a_mode, b_mode, out_dtype, bias, det):
    dev = require_gpu()
    A, a_s, B, b_s = gemm_inputs(M, N, K, a_mode, b_mode, seed_a=M + 1, seed_b=N + 2)
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=synth.SEED_BIAS)) if bias else None
    buf, out = _guarded_out(M, N, out_dtype, dev)
    fm.fp8_scaled_mm(to_dev(A), to_dev(B), to_dev(np.ascontiguousarray(a_s, np.float32)),
                     to_dev(np.ascontiguousarray(b_s, np.float32)), AMODE[a_mode] | BMODE[b_mode], out,
                     bias=to_dev(bias_bits).view(torch.bfloat16) if bias else None, deterministic=det)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    what = f"M{M} N{N} K{K} {a_mode}/{b_mode} det={det}"
    _check_margins(buf, M, N, what)
    _, exact, sumabs = oracle.gemm(A, B, a_s, b_s, OAMODE[a_mode], OBMODE[b_mode], bias_bits=bias_bits,
                                   out_dtype=out_dtype, want_exact=True)
    check_gemm(bits(out), exact, sumabs, K, out_dtype, what)


def test_block_scaled_output_written_exactly():
    dev = require_gpu()
    M, N, K = 300, 1000, 1024
    X = synth.to_bits(synth.normal((M, K), 1.0, seed=21))
    W = synth.to_bits(synth.normal((N, K), 0.02, seed=22))
    B, b_blk = oracle.quantize_blocks(W)
    A, a_words = oracle.group_quant(X, 0, 128, oracle.SCALE_UE8M0_PACKED, True)
    buf, out = _guarded_out(M, N, 0, dev)
    fm.fp8_scaled_mm(to_dev(A), to_dev(B), to_dev(a_words), to_dev(b_blk), fm.A_GROUP128_UE8M0 | fm.B_BLOCK128, out)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    _check_margins(buf, M, N, "block-scaled")
    _, exact, sumabs = oracle.gemm(A, B, a_words, b_blk, oracle.A_GROUP_UE8M0, oracle.B_BLOCK, want_exact=True)
    check_gemm(bits(out), exact, sumabs, K, 0, "block-scaled")
