"""A GEMM that reads the output of the GEMM before it on the stream.

The small-M GEMMs let the next kernel on the stream launch early (programmatic
dependent launch), and every GEMM launches as such a dependent; the second GEMM
must still read its operand only after the first has finished writing it.

GEMM 1 (M = 16, K = 16, codes 0 and +-1, unit scales) writes small integers
(|v| <= 16) in bf16, whose bytes are all finite E4M3 codes; GEMM 2 takes those
bytes as its A operand (K = 2 N1).  GEMM 1's output buffer is zeroed and its A
operand changed before every round, so a GEMM 2 that read too early would see
zeros or the previous round's values.  Rounds run eagerly on one stream and as
replays of a captured CUDA graph; both GEMMs are compared with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from gpu_util import bits, check_gemm, require_gpu, to_dev

pytestmark = pytest.mark.gpu

M, K1, N1, N2 = 16, 16, 1024, 4096
K2 = 2 * N1
ONE, MINUS_ONE = 0x38, 0xB8   # E4M3 codes of +1 and -1


def _ternary_codes(shape, seed):
    rng = np.random.default_rng(seed)
    return rng.choice(np.array([0, ONE, MINUS_ONE], np.uint8), size=shape, p=[0.5, 0.25, 0.25])


def _check_round(A1, B1, B2, out1, out2, what):
    o1 = bits(out1)
    _, exact1, sumabs1 = oracle.gemm(A1, B1, np.ones(1, np.float32), np.ones(1, np.float32), oracle.A_TENSOR,
                                     oracle.B_TENSOR, want_exact=True)
    assert np.all(np.abs(exact1) <= 16) and np.all(exact1 == np.round(exact1))
    check_gemm(o1, exact1, sumabs1, K1, 0, what + " (first GEMM)")
    A2 = np.ascontiguousarray(o1).view(np.uint8).reshape(M, K2)   # the bytes the second GEMM read
    _, exact2, sumabs2 = oracle.gemm(A2, B2, np.ones(1, np.float32), np.full(1, 0.01, np.float32),
                                     oracle.A_TENSOR, oracle.B_TENSOR, want_exact=True)
    check_gemm(bits(out2), exact2, sumabs2, K2, 0, what + " (second GEMM)")


def test_second_gemm_reads_first_gemms_output():
    dev = require_gpu()
    B1 = _ternary_codes((N1, K1), 101)
    B2 = np.random.default_rng(102).integers(0, 0x7E, size=(N2, K2), dtype=np.uint8)
    b1, b2 = to_dev(B1, dev), to_dev(B2, dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    s2 = torch.full((1,), 0.01, dtype=torch.float32, device=dev)
    a1 = torch.empty((M, K1), dtype=torch.uint8, device=dev)
    out1 = torch.empty((M, N1), dtype=torch.bfloat16, device=dev)
    out2 = torch.empty((M, N2), dtype=torch.bfloat16, device=dev)
    a2 = out1.view(torch.uint8)   # [M, 2 N1]: the first GEMM's output bytes

    def pair(stream):
        out1.zero_()
        fm.fp8_scaled_mm(a1, b1, one, one, fm.A_TENSOR | fm.B_TENSOR, out1, stream=stream)
        fm.fp8_scaled_mm(a2, b2, one, s2, fm.A_TENSOR | fm.B_TENSOR, out2, stream=stream)

    st = torch.cuda.Stream()
    for r in range(4):
        A1 = _ternary_codes((M, K1), 200 + r)
        a1.copy_(torch.from_numpy(A1))
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            pair(st)
        st.synchronize()
        assert fm.get_device_status() == 0
        _check_round(A1, B1, B2, out1, out2, f"eager round {r}")

    graph = torch.cuda.CUDAGraph()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(graph, stream=st):
            pair(torch.cuda.current_stream())
    torch.cuda.synchronize()
    for r in range(4):
        A1 = _ternary_codes((M, K1), 300 + r)
        a1.copy_(torch.from_numpy(A1))
        out2.fill_(0)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert fm.get_device_status() == 0
        _check_round(A1, B1, B2, out1, out2, f"graph round {r}")


@pytest.mark.parametrize("group", [N1, 128], ids=["per_token", "group128"])
def test_quant_reads_previous_gemms_output(group):
    # a decode layer: GEMM 1 writes out1 (bf16 small integers); the quant -- also a
    # programmatic dependent of the work before it -- reads out1 as its input; GEMM 2
    # consumes the codes and scales.  out1 is zeroed and GEMM 1's A changed every round.
    dev = require_gpu()
    B1 = _ternary_codes((N1, K1), 111)
    B2 = np.random.default_rng(112).integers(0, 0x7E, size=(N2, N1), dtype=np.uint8)
    b1, b2 = to_dev(B1, dev), to_dev(B2, dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    s2 = torch.full((N2, 1), 0.01, dtype=torch.float32, device=dev)
    a1 = torch.empty((M, K1), dtype=torch.uint8, device=dev)
    out1 = torch.empty((M, N1), dtype=torch.bfloat16, device=dev)
    q = torch.empty((M, N1), dtype=torch.uint8, device=dev)
    s = torch.empty((M, N1 // group), dtype=torch.float32, device=dev)
    out2 = torch.empty((M, N2), dtype=torch.bfloat16, device=dev)
    a_mode = fm.A_ROW if group == N1 else fm.A_GROUP128

    def layer(stream):
        out1.zero_()
        fm.fp8_scaled_mm(a1, b1, one, one, fm.A_TENSOR | fm.B_TENSOR, out1, stream=stream)
        fm.per_token_group_quant_fp8(out1, q, s, group, stream=stream)
        fm.fp8_scaled_mm(q, b2, s, s2, a_mode | fm.B_COL, out2, stream=stream)

    def check(A1, what):
        o1 = bits(out1)
        _, exact1, _ = oracle.gemm(A1, B1, np.ones(1, np.float32), np.ones(1, np.float32), oracle.A_TENSOR,
                                   oracle.B_TENSOR, want_exact=True)
        assert np.array_equal(oracle.bf16_bits_to_f64(o1), exact1), what + ": first GEMM"
        q_ref, s_ref = oracle.group_quant(o1, 0, group, oracle.SCALE_FP32, False, False)
        assert np.array_equal(bits(q), q_ref), what + ": codes"
        assert np.array_equal(bits(s).view(np.uint32), s_ref.view(np.uint32)), what + ": scales"
        _, exact2, sumabs2 = oracle.gemm(q_ref, B2, s_ref, np.full(N2, 0.01, np.float32),
                                         oracle.A_ROW if group == N1 else oracle.A_GROUP, oracle.B_COL,
                                         want_exact=True)
        check_gemm(bits(out2), exact2, sumabs2, N1, 0, what + ": second GEMM")

    st = torch.cuda.Stream()
    for r in range(3):
        A1 = _ternary_codes((M, K1), 400 + r)
        a1.copy_(torch.from_numpy(A1))
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            layer(st)
        st.synchronize()
        assert fm.get_device_status() == 0
        check(A1, f"eager round {r}")
    graph = torch.cuda.CUDAGraph()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(graph, stream=st):
            layer(torch.cuda.current_stream())
    torch.cuda.synchronize()
    for r in range(3):
        A1 = _ternary_codes((M, K1), 500 + r)
        a1.copy_(torch.from_numpy(A1))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert fm.get_device_status() == 0
        check(A1, f"graph round {r}")
