"""Batch-invariant deterministic mode of fp8_scaled_mm.

Workload: rowwise E4M3, K in {4096, 80 (a tail shorter than one K tile)},
N in {64, 4096}, bf16 and fp16 out, optional bf16 bias ~N(0, 0.1), strided A
(lda = K + 64), M swept 1..4096.  Row i of the result must be bit-identical
whether it is computed in a call of M rows for any M, or in a call that starts
at any prefix / suffix split point; and the M = 4096 result must match the
oracle within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, check_gemm, gemm_inputs, require_gpu, to_dev

pytestmark = pytest.mark.gpu

M_FULL = 4096
# every M up to 300, then a stride that visits every residue of the 128-row tile
M_SWEEP = list(range(1, 301)) + list(range(301, M_FULL + 1, 37)) + [M_FULL - 1, M_FULL]
SPLITS = [1, 2, 37, 64, 100, 101, 127, 128, 129, 1000, 2049, 4000, 4095]


def _setup(K, N, out_dtype, bias):
    dev = require_gpu()
    lda = K + 64
    A, a_s, B, b_s = gemm_inputs(M_FULL, N, K, "row", "col", seed_a=17, seed_b=18, lda=lda)
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=synth.SEED_BIAS)) if bias else None
    t = dict(A=to_dev(A, dev), a_s=to_dev(a_s, dev), B=to_dev(B, dev), b_s=to_dev(b_s, dev),
             bias=to_dev(bias_bits, dev).view(torch.bfloat16) if bias else None,
             odt=torch.bfloat16 if out_dtype == 0 else torch.float16, lda=lda, K=K, N=N)
    return A, a_s, B, b_s, bias_bits, t


def _call(t, start, M):
    out = torch.empty((M, t["N"]), dtype=t["odt"], device=t["A"].device)
    fm.fp8_scaled_mm(t["A"][start:start + M], t["B"], t["a_s"][start:start + M], t["b_s"], fm.A_ROW | fm.B_COL, out,
                     bias=t["bias"], deterministic=True, M=M, K=t["K"], lda=t["lda"])
    return out


@pytest.mark.parametrize("K", [4096, 80])
@pytest.mark.parametrize("N", [64, 4096])
@pytest.mark.parametrize("out_dtype", [0, 1])
@pytest.mark.parametrize("bias", [False, True])
def test_rows_identical_across_M_and_splits(K, N, out_dtype, bias):
    A, a_s, B, b_s, bias_bits, t = _setup(K, N, out_dtype, bias)
    ref = _call(t, 0, M_FULL)
    torch.cuda.synchronize()
    full_sweep = (K == 4096 and N == 4096 and out_dtype == 0 and bias)
    sweep = range(1, M_FULL + 1) if full_sweep else M_SWEEP
    mismatched = []
    for M in sweep:
        if not torch.equal(_call(t, 0, M).view(torch.int16), ref[:M].view(torch.int16)):
            mismatched.append(("prefix", M))
    for s in SPLITS:
        if not torch.equal(_call(t, s, M_FULL - s).view(torch.int16), ref[s:].view(torch.int16)):
            mismatched.append(("suffix", s))
        mid = min(300, M_FULL - s)
        if not torch.equal(_call(t, s, mid).view(torch.int16), ref[s:s + mid].view(torch.int16)):
            mismatched.append(("window", s))
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0
    assert not mismatched, mismatched[:10]
    # and the reference itself is right: every one of its M_FULL x N outputs
    ref_bits, exact, sumabs = oracle.gemm(A, B, a_s, b_s, oracle.A_ROW, oracle.B_COL, bias_bits=bias_bits,
                                          out_dtype=out_dtype, K=K, want_exact=True)
    check_gemm(bits(ref), exact, sumabs, K, out_dtype, f"deterministic K{K} N{N}")


def test_repeat_runs_bit_identical():
    A, a_s, B, b_s, bias_bits, t = _setup(4096, 4096, 0, True)
    r1 = _call(t, 0, 1234)
    r2 = _call(t, 0, 1234)
    torch.cuda.synchronize()
    assert torch.equal(r1.view(torch.int16), r2.view(torch.int16))
