"""Pins for the oracle's scaled FP8 GEMM (CPU only).

The accumulation is pinned by exact integer arithmetic (every E4M3 value
times 2^9 is an integer, so sum_k A B * 2^18 is an int64 dot product) and by
brute-force rational arithmetic on tiny matrices; scales by power-of-two
values whose products are exact, chosen per row / per column so that a
transposed index fails; the final rounding by the separately pinned
fp64 -> bf16 / fp16 routine.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C          # no NaN codes
    return c


def _int_form(codes):
    v = oracle.e4m3_decode(codes) * 512.0          # integers in [-229376, 229376]
    assert np.all(v == np.round(v))
    return v.astype(np.int64)


def test_accumulation_is_exact_int64():
    rng = np.random.default_rng(0)
    A = _codes(rng, (48, 4096))
    B = _codes(rng, (40, 4096))
    out, exact, _ = oracle.gemm(A, B, np.float32(1), np.float32(1), oracle.A_TENSOR, oracle.B_TENSOR,
                                want_exact=True)
    acc = _int_form(A) @ _int_form(B).T            # exact in int64
    assert np.array_equal(exact, acc.astype(np.float64) / 2.0 ** 18)
    assert np.array_equal(out, oracle.round_bf16(acc / 2.0 ** 18))
    # scalar scales that are powers of two scale the exact sum exactly
    _, e2, _ = oracle.gemm(A, B, np.float32(2.0 ** -3), np.float32(2.0 ** 5), oracle.A_TENSOR, oracle.B_TENSOR,
                           want_exact=True)
    assert np.array_equal(e2, acc.astype(np.float64) / 2.0 ** 16)


def test_extreme_accumulation_k28672():
    # largest-magnitude operands at the largest K of the workloads: still exact
    K = 28672
    A = np.full((2, K), 0x7E, np.uint8)
    B = np.full((3, K), 0x7E, np.uint8)
    B[1, ::2] = 0xFE
    B[2, 1] = 0x01
    _, exact, _ = oracle.gemm(A, B, np.float32(1), np.float32(1), 0, 0, want_exact=True)
    assert exact[0, 0] == 448.0 * 448.0 * K
    assert exact[0, 1] == 0.0
    assert exact[0, 2] == 448.0 * 448.0 * (K - 1) + 448.0 * 2.0 ** -9


def test_tiny_bruteforce_rational():
    rng = np.random.default_rng(1)
    for trial in range(6):
        M, N, K = rng.integers(1, 5), rng.integers(1, 5), int(rng.integers(1, 5)) * 16
        A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
        a_s = (rng.random(M) + 0.1).astype(np.float32)
        b_s = (rng.random(N) + 0.1).astype(np.float32)
        bias = rng.integers(0, 0x7F00, size=N).astype(np.uint16) & 0xBFFF   # finite bf16
        out, exact, _ = oracle.gemm(A, B, a_s, b_s, oracle.A_ROW, oracle.B_COL, bias_bits=bias,
                                    want_exact=True)
        da = oracle.e4m3_decode(A)
        db = oracle.e4m3_decode(B)
        bv = oracle.bf16_bits_to_f64(bias)
        for m in range(M):
            for n in range(N):
                s = sum(Fraction(float(da[m, k])) * Fraction(float(db[n, k])) for k in range(K))
                ref = s * Fraction(float(a_s[m])) * Fraction(float(b_s[n])) + Fraction(float(bv[n]))
                assert abs(Fraction(float(exact[m, n])) - ref) <= abs(ref) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 1000)
                assert out[m, n] == oracle.round_bf16(np.array([float(ref)]))[0]


def test_row_and_column_scales_are_not_transposed():
    rng = np.random.default_rng(2)
    M, N, K = 8, 12, 256
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    a_s = (2.0 ** np.arange(M)).astype(np.float32)
    b_s = (2.0 ** (-2 * np.arange(N))).astype(np.float32)
    _, exact, _ = oracle.gemm(A, B, a_s, b_s, oracle.A_ROW, oracle.B_COL, want_exact=True)
    acc = (_int_form(A) @ _int_form(B).T).astype(np.float64) / 2.0 ** 18
    want = acc * (2.0 ** np.arange(M))[:, None] * (2.0 ** (-2 * np.arange(N)))[None, :]
    assert np.array_equal(exact, want)


def test_group_scales():
    rng = np.random.default_rng(3)
    M, N, K = 6, 10, 512
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    G = K // 128
    # constant across groups: identical to the per-row mode
    a_row = (rng.random(M) + 0.5).astype(np.float32)
    a_grp = np.repeat(a_row[:, None], G, axis=1)
    b = (rng.random(N) + 0.5).astype(np.float32)
    o1, e1, _ = oracle.gemm(A, B, a_row, b, oracle.A_ROW, oracle.B_COL, want_exact=True)
    o2, e2, sabs = oracle.gemm(A, B, a_grp, b, oracle.A_GROUP, oracle.B_COL, want_exact=True)
    assert np.array_equal(o1, o2)
    # the per-group products a_s * acc_g round in fp64: a few ulp of sum |terms|
    assert np.all(np.abs(e1 - e2) <= sabs * 2.0 ** -50)
    # power-of-two group scales: sum_g 2^g * (partial sum over group g), exact
    a_pow = np.tile((2.0 ** np.arange(G)).astype(np.float32), (M, 1))
    _, e3, _ = oracle.gemm(A, B, a_pow, np.float32(1), oracle.A_GROUP, oracle.B_TENSOR, want_exact=True)
    IA, IB = _int_form(A), _int_form(B)
    want = sum((IA[:, g * 128:(g + 1) * 128] @ IB[:, g * 128:(g + 1) * 128].T) * 2 ** g for g in range(G))
    assert np.array_equal(e3, want.astype(np.float64) / 2.0 ** 18)
    # column-major group scales [G, pad4(M)] give the same result
    a_cm = np.zeros((G, oracle.pad4(M)), np.float32)
    a_cm[:, :M] = a_pow.T
    _, e4, _ = oracle.gemm(A, B, a_cm, np.float32(1), oracle.A_GROUP_COLMAJOR, oracle.B_TENSOR, want_exact=True)
    assert np.array_equal(e3, e4)


def test_bias_strided_a_and_rows():
    rng = np.random.default_rng(4)
    M, N, K = 9, 16, 80
    A_wide = _codes(rng, (M, K + 64))
    B = _codes(rng, (N, K))
    bias = (rng.standard_normal(N) * 0.1).astype(np.float32)
    bias_bits = (bias.view(np.uint32) >> 16).astype(np.uint16)
    a_s, b_s = np.float32(0.03), np.float32(0.5)
    o1, e1, _ = oracle.gemm(A_wide, B, a_s, b_s, 0, 0, bias_bits=bias_bits, K=K, want_exact=True)
    o2, e2, _ = oracle.gemm(np.ascontiguousarray(A_wide[:, :K]), B, a_s, b_s, 0, 0, want_exact=True)
    assert np.allclose(e1 - e2, oracle.bf16_bits_to_f64(bias_bits)[None, :], rtol=0, atol=1e-12)
    rows = np.array([8, 0, 3])
    o3 = oracle.gemm(A_wide, B, a_s, b_s, 0, 0, bias_bits=bias_bits, K=K, rows=rows)
    assert np.array_equal(o3, o1[rows])


def test_fp16_output_rounding():
    rng = np.random.default_rng(5)
    A, B = _codes(rng, (4, 128)), _codes(rng, (8, 128))
    o, e, _ = oracle.gemm(A, B, np.float32(1e-3), np.float32(1), 0, 0, out_dtype=1, want_exact=True)
    assert np.array_equal(o, e.astype(np.float16).view(np.uint16))


def test_block_scales_and_packed_ue8m0_a_scales():
    # per-group A scales x 128 x 128 block B scales: with powers of two the result is
    # exact and equals sum_g a[m,g] b[n/128,g] partial_g computed here in int64
    rng = np.random.default_rng(6)
    M, N, K = 5, 300, 384
    G = K // 128
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    ea = rng.integers(120, 134, size=(M, G))                  # UE8M0 exponent bytes
    eb = rng.integers(-3, 4, size=((N + 127) // 128, G))
    a_f = (2.0 ** (ea - 127)).astype(np.float32)
    b_blk = (2.0 ** eb).astype(np.float32)
    _, e1, _ = oracle.gemm(A, B, a_f, b_blk, oracle.A_GROUP, oracle.B_BLOCK, want_exact=True)
    IA, IB = _int_form(A), _int_form(B)
    want = np.zeros((M, N))
    for g in range(G):
        part = (IA[:, g * 128:(g + 1) * 128] @ IB[:, g * 128:(g + 1) * 128].T).astype(np.float64) / 2.0 ** 18
        want += part * (2.0 ** (ea[:, g] - 127))[:, None] * (2.0 ** eb[np.arange(N) // 128, g])[None, :]
    assert np.array_equal(e1, want)
    # the same A scales as packed UE8M0 words, column-major [ceil(G/4), pad4(M)]
    words = np.zeros(((G + 3) // 4, oracle.pad4(M)), np.uint32)
    for g in range(G):
        words[g // 4, :M] |= ea[:, g].astype(np.uint32) << np.uint32(8 * (g % 4))
    _, e2, _ = oracle.gemm(A, B, words.view(np.int32), b_blk, oracle.A_GROUP_UE8M0, oracle.B_BLOCK, want_exact=True)
    assert np.array_equal(e1, e2)
    # block scales constant over N blocks reduce to the column-scale-free group mode
    _, e3, _ = oracle.gemm(A, B, a_f, np.ones(((N + 127) // 128, G), np.float32), oracle.A_GROUP, oracle.B_BLOCK,
                           want_exact=True)
    _, e4, _ = oracle.gemm(A, B, a_f, np.float32(1), oracle.A_GROUP, oracle.B_TENSOR, want_exact=True)
    assert np.array_equal(e3, e4)


def ue8m0_edge_case():
    """Inputs of the UE8M0 byte-range pin (also run on the GPU): K = 128, every A
    and B code 1.0 (0x38) except B row 2, all zero; so each row's single K block
    sums to 128, or to 0 in column 2.  A scale bytes per row: 0, 1, 127, 255;
    column scales 2^100, 2^-120, 1 and 2^100 for the other columns."""
    M, N, K = 4, 8, 128
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    B[2] = 0
    e = [0, 1, 127, 255]
    words = np.zeros((1, oracle.pad4(M)), np.uint32)
    words[0, :M] = e                      # group 0 sits in byte 0 of word 0
    b_s = np.full(N, 2.0 ** 100, np.float32)
    b_s[1] = 2.0 ** -120
    b_s[2] = 1.0
    return A, words.view(np.int32), B, b_s


def test_ue8m0_scale_bytes_at_both_ends_of_the_range():
    # A UE8M0 byte e stands for the fp32 scale 2^(e-127) (the Quant PR's fp32 form of
    # a UE8M0 scale, Modifications 3), taken as an fp32 value like every other scale:
    # byte 0 is the subnormal 2^-127 (not 0), byte 255 overflows to +inf (not the
    # finite fp64 2^128).  Expected bf16 bits worked out by hand:
    #   row 0, 128 * 2^-127 * 2^100 = 2^-20   -> 0x3580;  * 2^-120 = 2^-240, below
    #          the smallest bf16 subnormal (2^-133) -> 0;  column 2: 0
    #   row 1, 128 * 2^-126 * 2^100 = 2^-19   -> 0x3600;  2^-239 -> 0
    #   row 2, 128 * 2^100 = 2^107            -> 0x7500;  2^-113 -> 0x0700
    #   row 3, inf in every column with a non-zero sum (with the fp64 2^128 column 1
    #          would be the finite 2^15); column 2: inf * 0 = NaN
    A, words, B, b_s = ue8m0_edge_case()
    out, exact, _ = oracle.gemm(A, B, words, b_s, oracle.A_GROUP_UE8M0, oracle.B_COL, want_exact=True)
    assert out[0, 0] == 0x3580 and out[0, 1] == 0x0000 and out[0, 2] == 0x0000
    assert out[1, 0] == 0x3600 and out[1, 1] == 0x0000
    assert out[2, 0] == 0x7500 and out[2, 1] == 0x0700 and out[2, 2] == 0x0000
    assert np.all(out[:3, 3:] == out[:3, :1])
    assert exact[3, 0] == np.inf and exact[3, 1] == np.inf and np.isnan(exact[3, 2])
    assert out[3, 0] == 0x7F80 and out[3, 1] == 0x7F80 and (out[3, 2] & 0x7F80) == 0x7F80 and out[3, 2] & 0x7F
