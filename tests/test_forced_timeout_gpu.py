"""Forced timeouts inside the real kernels: failure detection without a GPU fault.

fp8mm_set_wait_timeout_ns shortens the limit of the GEMM and group-quant
pipelines' bounded waits, so that real waits -- for a stage's TMA loads, for an
accumulator, for a cluster peer -- give up in mid-run.  For every GEMM form, the
group quant (plain and fused) and several limits:
the call returns; the device status word reads FP8MM_ETIMEOUT (or FP8MM_OK if no
wait outlasted the limit); every output element is either still the sentinel the
buffer was filled with or the correct value (a kernel that gives up leaves the
tiles or items it had not finished unwritten); and the next call, with the default limit,
is correct and clean (the context survives).  The drains -- a producer waiting
for its own loads, an MMA thread for its own MMAs -- keep the full limit, so no
copy or MMA is still in flight when a CTA frees its TMEM or exits."""
import numpy as np
import pytest
import torch

import oracle
import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import bits, check_gemm, gemm_inputs, require_gpu, to_dev

pytestmark = pytest.mark.gpu

SENTINEL = 0x7A5B
LIMITS_NS = (100, 1000, 20000)
AMODE = {"tensor": fm.A_TENSOR, "row": fm.A_ROW, "group": fm.A_GROUP128}
BMODE = {"tensor": fm.B_TENSOR, "col": fm.B_COL}
OAMODE = {"tensor": oracle.A_TENSOR, "row": oracle.A_ROW, "group": oracle.A_GROUP}
OBMODE = {"tensor": oracle.B_TENSOR, "col": oracle.B_COL}

CASES = [
    # M, N, K, a_mode, b_mode, out_dtype, bias, deterministic      kernel form
    (5, 264, 2048, "row", "col", 0, False, False),                # swap-AB split-K, 16-token block
    (50, 1000, 1024, "tensor", "col", 1, True, False),            # swap-AB, 64-token block
    (2048, 4096, 2048, "tensor", "tensor", 0, False, False),      # 128 x 224 tiles
    (1937, 12280, 512, "row", "col", 1, True, False),             # 128 x BN tiles, ragged
    (100, 4104, 2048, "row", "col", 0, True, True),               # deterministic, cluster kernel
    (2500, 1000, 1024, "row", "col", 1, False, True),             # deterministic, fold kernel
    (300, 1000, 2048, "group", "col", 0, True, False),            # per-group A scales
]


@pytest.fixture(autouse=True)
def _default_limit_after():
    yield
    fm.set_wait_timeout_ns(0)


def _run(M, N, K, out_dtype, launch):
    dev = require_gpu()
    buf = torch.full((M * N,), SENTINEL, dtype=torch.int16, device=dev)
    out = buf.view(M, N).view(torch.bfloat16 if out_dtype == 0 else torch.float16)
    launch(out)
    torch.cuda.synchronize()
    return out, fm.get_device_status(clear=True)


def _check_written(out, exact, sumabs, K, out_dtype, what):
    got = bits(out).reshape(-1)
    written = got != SENTINEL
    if written.any():
        check_gemm(got[written], exact.reshape(-1)[written], sumabs.reshape(-1)[written], K, out_dtype, what)
    return int(written.sum())


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"M{c[0]}_N{c[1]}_K{c[2]}_{c[3]}{'_det' if c[7] else ''}")
def test_short_wait_limit_gives_up_cleanly(case):
    M, N, K, a_mode, b_mode, out_dtype, bias, det = case
    require_gpu()
    A, a_s, B, b_s = gemm_inputs(M, N, K, a_mode, b_mode, seed_a=M + 7, seed_b=N + 9)
    bias_bits = synth.to_bits(synth.normal((N,), 0.1, seed=synth.SEED_BIAS)) if bias else None
    At, Bt = to_dev(A), to_dev(B)
    ast, bst = to_dev(np.ascontiguousarray(a_s, np.float32)), to_dev(np.ascontiguousarray(b_s, np.float32))
    biast = to_dev(bias_bits).view(torch.bfloat16) if bias else None
    _, exact, sumabs = oracle.gemm(A, B, a_s, b_s, OAMODE[a_mode], OBMODE[b_mode], bias_bits=bias_bits,
                                   out_dtype=out_dtype, want_exact=True)

    def launch(out):
        fm.fp8_scaled_mm(At, Bt, ast, bst, AMODE[a_mode] | BMODE[b_mode], out, bias=biast, deterministic=det)

    assert fm.get_device_status(clear=True) == fm.OK
    outcomes = []
    for limit in LIMITS_NS:
        fm.set_wait_timeout_ns(limit)
        out, status = _run(M, N, K, out_dtype, launch)
        fm.set_wait_timeout_ns(0)
        assert status in (fm.OK, fm.ETIMEOUT), (limit, status)
        n = _check_written(out, exact, sumabs, K, out_dtype, f"limit {limit} ns")
        if status == fm.OK:
            assert n == M * N, f"limit {limit} ns: status OK but {M * N - n} outputs unwritten"
        outcomes.append((limit, status, n))
    # the shortest limit is far below one HBM round trip: some wait must have given up
    assert outcomes[0][1] == fm.ETIMEOUT, outcomes
    # and the context is intact: the default limit gives the full, correct result
    out, status = _run(M, N, K, out_dtype, launch)
    assert status == fm.OK
    check_gemm(bits(out), exact, sumabs, K, out_dtype, "after the forced timeouts")


QSENT = 0x5A


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("fmt,colmajor", [(0, False), (2, True)])
def test_quant_short_wait_limit_gives_up_cleanly(fuse, fmt, colmajor):
    dev = require_gpu()
    M, K = 4096, 7168
    x = synth.quant_input(M, 2 * K if fuse else K, torch.bfloat16, seed=77)
    q_ref, s_ref = oracle.group_quant(synth.to_bits(x), 0, 128, fmt, colmajor, fuse)
    s_ref = s_ref.view(np.uint32)
    xd = x.to(dev)

    def run():
        q = torch.full((M, K), QSENT, dtype=torch.uint8, device=dev)
        s = torch.empty(fm.scale_shape(M, K, 128, fmt, colmajor), dtype=fm.scale_dtype(fmt), device=dev)
        s.view(torch.uint8).fill_(QSENT)
        fm.per_token_group_quant_fp8(xd, q, s, 128, fmt, colmajor, fuse)
        torch.cuda.synchronize()
        return bits(q), bits(s).view(np.uint32), fm.get_device_status(clear=True)

    assert fm.get_device_status(clear=True) == fm.OK
    statuses = []
    for limit in LIMITS_NS:
        fm.set_wait_timeout_ns(limit)
        qg, sg, status = run()
        fm.set_wait_timeout_ns(0)
        assert status in (fm.OK, fm.ETIMEOUT), (limit, status)
        assert np.all((qg == q_ref) | (qg == QSENT)), f"limit {limit} ns: wrong codes written"
        assert np.all((sg == s_ref) | (sg == 0x5A5A5A5A)), f"limit {limit} ns: wrong scales written"
        if status == fm.OK:
            assert np.array_equal(qg, q_ref)
        statuses.append(status)
    assert statuses[0] == fm.ETIMEOUT, statuses
    qg, sg, status = run()
    assert status == fm.OK and np.array_equal(qg, q_ref)
    padded = sg != 0x5A5A5A5A
    assert np.array_equal(sg[padded], s_ref[padded])


def test_wait_limit_argument_checks():
    require_gpu()
    with pytest.raises(fm.Fp8mmError):
        fm.set_wait_timeout_ns(-1)
    with pytest.raises(fm.Fp8mmError):
        fm.set_wait_timeout_ns(3_000_000_000)
    fm.set_wait_timeout_ns(0)
