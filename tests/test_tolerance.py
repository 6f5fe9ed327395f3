"""The GEMM parity criterion used by the GPU tests (gpu_util.check_gemm) is
tight enough to catch a wrong kernel and loose enough for a correct one
(CPU only): outputs of an fp32-accumulating GEMM in another summation order
pass, outputs with a plausible kernel mistake fail."""
import numpy as np
import pytest

import oracle
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import check_gemm, gemm_inputs

M, N, K = 64, 96, 512


@pytest.fixture(scope="module")
def case():
    A, a_s, B, b_s = gemm_inputs(M, N, K, "row", "col", seed_a=21, seed_b=22)
    bias = synth.to_bits(synth.normal((N,), 0.1, seed=23))
    out, exact, sumabs = oracle.gemm(A, B, a_s, b_s, oracle.A_ROW, oracle.B_COL, bias_bits=bias, want_exact=True)
    da, db = oracle.e4m3_decode(A), oracle.e4m3_decode(B)
    return dict(A=A, B=B, a_s=a_s, b_s=b_s, bias=bias, out=out, exact=exact, sumabs=sumabs, da=da, db=db)


def _fp32_kernel(c, a_s=None, b_s=None, bias=True, k=K, chunk=128):
    """An fp32-accumulating GEMM with K split into chunks summed in fp32, scaled
    in fp32 and rounded once to bf16: what a correct tensor-core kernel does."""
    a_s = c["a_s"] if a_s is None else a_s
    b_s = c["b_s"] if b_s is None else b_s
    acc = np.zeros((M, N), np.float32)
    for k0 in range(0, k, chunk):
        k1 = min(k0 + chunk, k)
        acc = (acc + (c["da"][:, k0:k1].astype(np.float32) @ c["db"][:, k0:k1].astype(np.float32).T)).astype(
            np.float32)
    v = (acc * np.asarray(a_s, np.float32).reshape(M, 1) * np.asarray(b_s, np.float32).reshape(1, N)).astype(
        np.float32)
    if bias:
        v = (v + oracle.bf16_bits_to_f64(c["bias"]).astype(np.float32)[None, :]).astype(np.float32)
    return oracle.round_bf16(v.astype(np.float64))


def test_accepts_the_oracle_and_an_fp32_kernel(case):
    check_gemm(case["out"], case["exact"], case["sumabs"], K)
    check_gemm(_fp32_kernel(case), case["exact"], case["sumabs"], K)
    check_gemm(_fp32_kernel(case, chunk=32), case["exact"], case["sumabs"], K)


@pytest.mark.parametrize("mistake", ["row scales permuted", "column scales permuted", "bias dropped",
                                     "K tail dropped", "scaled by 1 + 2^-6", "rows shifted", "bias twice"])
def test_rejects_a_wrong_kernel(case, mistake):
    c = case
    if mistake == "row scales permuted":
        got = _fp32_kernel(c, a_s=np.roll(np.asarray(c["a_s"]).reshape(M), 1))
    elif mistake == "column scales permuted":
        got = _fp32_kernel(c, b_s=np.roll(np.asarray(c["b_s"]).reshape(N), 1))
    elif mistake == "bias dropped":
        got = _fp32_kernel(c, bias=False)
    elif mistake == "K tail dropped":
        got = _fp32_kernel(c, k=K - 16)
    elif mistake == "scaled by 1 + 2^-6":
        got = oracle.round_bf16(c["exact"] * (1 + 2.0 ** -6))
    elif mistake == "rows shifted":
        got = np.roll(c["out"], 1, axis=0)
    else:
        got = oracle.round_bf16(c["exact"] + oracle.bf16_bits_to_f64(c["bias"])[None, :])
    with pytest.raises(AssertionError):
        check_gemm(got, c["exact"], c["sumabs"], K)


@pytest.mark.parametrize("chunk", [128, 32])
def test_accepts_an_fp32_kernel_at_the_largest_k(chunk):
    # K = 14336 (the down projection of the prefill shapes): an fp32 accumulation in
    # K chunks still passes, the largest-K case of the accumulation-error allowance
    m, n, k = 16, 64, 14336
    A, a_s, B, b_s = gemm_inputs(m, n, k, "row", "col", seed_a=31, seed_b=32)
    _, exact, sumabs = oracle.gemm(A, B, a_s, b_s, oracle.A_ROW, oracle.B_COL, want_exact=True)
    da, db = oracle.e4m3_decode(A).astype(np.float32), oracle.e4m3_decode(B).astype(np.float32)
    acc = np.zeros((m, n), np.float32)
    for k0 in range(0, k, chunk):
        acc = (acc + da[:, k0:k0 + chunk] @ db[:, k0:k0 + chunk].T).astype(np.float32)
    v = (acc * np.asarray(a_s, np.float32).reshape(m, 1) * np.asarray(b_s, np.float32).reshape(1, n))
    check_gemm(oracle.round_bf16(v.astype(np.float32).astype(np.float64)), exact, sumabs, k)
