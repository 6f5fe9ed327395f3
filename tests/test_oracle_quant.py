"""Pins for the oracle's per-token group quant (CPU only).

Hand-computed groups and layouts come from text fixtures under
tests/golden/; the rest are properties that hold for any correct
implementation: the dequantized codes reproduce the input within half an
E4M3 step, the largest element maps to +-448 under fp32 scales, UE8M0 scales
are the smallest power of two >= amax/448, and special cases reduce to
simpler ones (group = whole row, SiLU(gate) = gate for large gates).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_mm_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    cases, cur = [], None
    with open(os.path.join(GOLD, "quant_hand_groups.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "case":
                cur = {"name": rest[0]}
                cases.append(cur)
            else:
                cur[key] = rest
    return cases


def _bits(values, dtype):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16 if dtype == 0 else torch.float16)
    return synth.to_bits(t)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_groups(case):
    dtype = {"bf16": 0, "fp16": 1}[case["dtype"][0]]
    group = int(case["group"][0])
    ue8m0 = bool(int(case["ue8m0"][0]))
    vals = [float(v) for v in case["values"]]
    x = np.zeros((1, group), np.uint16)
    x[0, :len(vals)] = _bits(vals, dtype)
    q, s, e = oracle.group_quant_canonical(x, dtype, group, False, ue8m0)
    want = np.zeros(group, np.uint8)
    want[:len(vals)] = [int(c, 16) for c in case["codes"]]
    assert np.array_equal(q[0], want), [hex(c) for c in q[0, :len(vals)]]
    assert s.view(np.uint32)[0, 0] == int(case["scale"][0], 16), hex(s.view(np.uint32)[0, 0])
    if case["byte"][0] != "-":
        assert e[0, 0] == int(case["byte"][0])


def test_ue8m0_packing_fixture():
    rows = {"rowmajor": [], "colmajor": []}
    with open(os.path.join(GOLD, "ue8m0_packing.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                rows[key].append([int(v, 16) for v in vals])
    x = np.zeros((2, 768), np.uint16)
    for g in range(6):
        x[0, g * 128] = _bits([2.0 ** (g - 3)], 0)[0]
    for colmajor, key in ((False, "rowmajor"), (True, "colmajor")):
        _, s = oracle.group_quant(x, 0, 128, oracle.SCALE_UE8M0_PACKED, colmajor)
        want = np.array(rows[key], np.uint32).view(np.int32)
        assert s.dtype == np.int32 and np.array_equal(s, want), (key, [[hex(v) for v in r] for r in s.view(np.uint32)])


def _check_properties(x_bits, dtype, group, fuse, ue8m0):
    q, s, e = oracle.group_quant_canonical(x_bits, dtype, group, fuse, ue8m0)
    M, K = q.shape
    G = K // group
    if dtype == 0:
        xv = oracle.bf16_bits_to_f64(x_bits)
    else:
        xv = oracle.fp16_bits_to_f64(x_bits)
    if fuse:
        gate, up = xv[:, :K], xv[:, K:]
        with np.errstate(over="ignore"):
            v = gate / (1.0 + np.exp(-gate)) * up
    else:
        v = xv
    vg = v.reshape(M, G, group)
    amax = np.abs(vg).max(axis=2)
    a = np.maximum(amax, float(np.float32(1e-10)))
    s64 = s.astype(np.float64)
    # fp32 rounding of a/448; with SiLU in front, the fp32 SiLU also moves amax by a few ulp
    rel = 2.0 ** -20 if fuse else 2.0 ** -23
    if ue8m0:
        # smallest power of two >= a/448
        assert np.all(np.log2(s64) == np.round(np.log2(s64)))
        assert np.all(s64 >= a / 448 * (1 - rel))
        assert np.all(s64 < 2 * a / 448 * (1 + rel))
        assert np.array_equal(s64, 2.0 ** (e.astype(np.float64) - 127))
    else:
        assert np.all(np.abs(s64 - a / 448) <= a / 448 * rel)
    deq = oracle.e4m3_decode(q).reshape(M, G, group)
    scaled = vg / s64[:, :, None]                 # the value the code should represent
    tol = np.maximum(np.abs(scaled) * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20) + np.abs(scaled) * 2.0 ** -20
    if fuse:
        tol = tol + np.abs(scaled) * 2.0 ** -20 * 8   # fp32 SiLU rounding
    err = np.abs(deq - np.clip(scaled, -448, 448))
    assert np.all(err <= tol), float((err - tol).max())
    assert np.all(np.abs(deq) <= 448)
    if not ue8m0 and not fuse:
        # the absmax element of every non-zero group lands on +-448
        idx = np.abs(vg).argmax(axis=2)
        top = np.take_along_axis(deq, idx[:, :, None], axis=2)[:, :, 0]
        nz = amax >= 1e-10
        assert np.all(np.abs(top[nz]) == 448.0)
    return q, s, e


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("ue8m0", [False, True])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_properties_config5_like(dtype, ue8m0, group):
    x = synth.quant_input(128, 2048, torch.bfloat16 if dtype == 0 else torch.float16, seed=11)
    _check_properties(synth.to_bits(x), dtype, group, False, ue8m0)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_properties_fused(dtype, ue8m0):
    x = synth.quant_input(64, 2 * 1024, torch.bfloat16 if dtype == 0 else torch.float16, seed=12)
    _check_properties(synth.to_bits(x), dtype, 128, True, ue8m0)


def test_fp16_small_groups_never_saturate():
    # the PR's failure signature: 4095/4096 codes +-448 for fp16 groups with
    # amax < 6.8e-3 under UE8M0.  Correct output keeps them in range.
    x = (synth.normal((32, 4096), 1.0, seed=5) * 1e-3).to(torch.float16)
    q, s, e = oracle.group_quant_canonical(synth.to_bits(x), 1, 128, False, True)
    assert np.all(e < 127 - 14)           # multipliers above 65504 were in use
    # a +-448 code only where the scaled value rounds there (>= 432), i.e. at
    # most the group's largest elements -- not whole groups
    v = oracle.fp16_bits_to_f64(synth.to_bits(x)).reshape(32, 32, 128)
    scaled = np.abs(v) / s.astype(np.float64)[:, :, None]
    sat = ((q & 0x7F) == 0x7E).reshape(32, 32, 128)
    assert np.all(scaled[sat] >= 432)
    assert sat.sum() < 0.01 * sat.size


def test_whole_row_group_is_per_row():
    x = synth.to_bits(synth.normal((16, 512), 1.0, seed=6))
    q1, s1, _ = oracle.group_quant_canonical(x, 0, 512)
    q2, s2 = oracle.quantize_rows(x, 0)
    assert np.array_equal(q1, q2) and np.array_equal(s1[:, 0], s2)
    # and equals the group quant of each row taken on its own
    for m in (0, 7, 15):
        qm, sm, _ = oracle.group_quant_canonical(x[m:m + 1], 0, 512)
        assert np.array_equal(qm[0], q1[m]) and sm[0, 0] == s1[m, 0]


def test_fused_large_gate_is_identity():
    # SiLU(g) = g / (1 + exp(-g)) and exp(-g) < 2^-25 for g >= 18, so in fp32
    # SiLU(g) == g; with up = 1 the fused quant equals the plain quant of gate.
    rng = np.random.default_rng(4)
    gate = torch.tensor(rng.uniform(18, 300, (8, 256)), dtype=torch.float32)
    gate[:, ::7] *= 1e-2          # mix in ordinary values too (those must differ)
    up = torch.ones_like(gate)
    xf = synth.to_bits(torch.cat([gate, up], 1).to(torch.bfloat16))
    xg = synth.to_bits(gate.to(torch.bfloat16))
    qf, sf, _ = oracle.group_quant_canonical(xf, 0, 128, True)
    qg, sg, _ = oracle.group_quant_canonical(xg, 0, 128, False)
    big = (gate.to(torch.bfloat16).float().numpy() >= 18)
    assert np.array_equal(sf, sg)          # every group's absmax is a large gate
    assert np.array_equal(qf[big], qg[big])
    assert not np.array_equal(qf[~big], qg[~big])
    # gate and up halves are not interchangeable
    xs = synth.to_bits(torch.cat([up, gate], 1).to(torch.bfloat16))
    qs, _, _ = oracle.group_quant_canonical(xs, 0, 128, True)
    assert not np.array_equal(qs, qf)


def test_fused_zero_up_keeps_sign_of_silu():
    gate = torch.tensor([[-3.0, 2.0] + [0.0] * 126], dtype=torch.float32)
    up = torch.zeros_like(gate)
    x = synth.to_bits(torch.cat([gate, up], 1).to(torch.bfloat16))
    q, s, _ = oracle.group_quant_canonical(x, 0, 128, True)
    assert q[0, 0] == 0x80 and q[0, 1] == 0x00       # -0 keeps its sign bit
    assert s.view(np.uint32)[0, 0] == 0x2A7B5123


def test_layouts_agree():
    x = synth.to_bits(synth.quant_input(10, 1024, seed=8))
    for fmt in (0, 1, 2):
        _, rm = oracle.group_quant(x, 0, 128, fmt, False)
        _, cm = oracle.group_quant(x, 0, 128, fmt, True)
        assert cm.shape[1] == 12 and np.all(cm[:, 10:] == 0)
        assert np.array_equal(cm[:, :10].T, rm)


def test_scatter_rows_equal_plain_rows():
    x = synth.to_bits(synth.quant_input(40, 512, seed=9))
    dst, R = synth.routing(40, topk=8, num_experts=16, align=8)
    assert len(np.unique(dst)) == dst.size and dst.min() >= 0 and dst.max() < R
    q, s = oracle.group_quant(x, 0, 128, oracle.SCALE_UE8M0_PACKED, True)
    qd, sd = oracle.group_quant_scatter(x, 0, 128, dst, R)
    for m in range(40):
        for d in dst[m]:
            assert np.array_equal(qd[d], q[m]) and np.array_equal(sd[:, d], s[:, m])
    untouched = np.setdiff1d(np.arange(R), dst.ravel())
    assert np.all(qd[untouched] == 0) and np.all(sd[:, untouched] == 0)


def test_masked_layout_is_the_fused_quant_of_the_valid_rows():
    # x [E=3, T=5, 2K]: expert e holds masked_m[e] tokens; each valid row is the
    # fused quant of that row alone, padding rows and experts with no tokens stay 0
    E, T, K = 3, 5, 256
    x = synth.to_bits(synth.quant_input(E * T, 2 * K, seed=71)).reshape(E, T, 2 * K)
    masked = np.array([5, 0, 2], np.int32)
    for fmt, cm in ((oracle.SCALE_UE8M0_PACKED, True), (oracle.SCALE_FP32, True), (oracle.SCALE_FP32, False)):
        q, s = oracle.masked_silu_quant(x, 0, masked, 128, fmt, cm)
        for e in range(E):
            n = masked[e]
            if n:
                qr, sr = oracle.group_quant(x[e, :n], 0, 128, fmt, cm, fuse_silu_mul=True)
                assert np.array_equal(q[e, :n], qr)
                if cm:
                    assert np.array_equal(s[e][:, :n], sr[:, :n])
                else:
                    assert np.array_equal(s[e * T:e * T + n], sr)
            assert np.all(q[e, n:] == 0)
        if cm:
            assert s.shape == (E, 2 if fmt == oracle.SCALE_FP32 else 1, 8)
            assert np.all(s[1] == 0) and np.all(s[:, :, T:] == 0)


def test_masked_counts_sum_to_routed_tokens():
    c = synth.masked_counts(4096, 256)
    assert c.sum() == 4096 * 8 and c.dtype == np.int32
    assert np.array_equal(synth.masked_counts(4096, 32), c[:32])


def test_block_quant_is_groupwise_per_block():
    # each 128 x 128 block: absmax/448 scale, its largest element at +-448, and the
    # same codes as the group quant of the block taken as one row
    w = synth.to_bits(synth.normal((200, 384), 0.02, seed=91))
    q, s = oracle.quantize_blocks(w)
    assert q.shape == (200, 384) and s.shape == (2, 3)
    v = oracle.bf16_bits_to_f64(w)
    for i in range(2):
        for j in range(3):
            blk = v[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            a = np.abs(blk).max()
            assert abs(s[i, j] - a / 448) <= a / 448 * 2.0 ** -23
            deq = oracle.e4m3_decode(q[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128])
            assert np.abs(deq).max() == 448.0


def test_static_quant_pins():
    x = synth.to_bits(synth.normal((4, 512), 3.0, seed=92))
    v = oracle.bf16_bits_to_f64(x)
    # scale 1: the codes are the encoding of the values themselves
    assert np.array_equal(oracle.static_quant(x, 0, 1.0), oracle.e4m3_encode(v.astype(np.float32)))
    # a power-of-two scale divides exactly
    assert np.array_equal(oracle.static_quant(x, 0, 0.25), oracle.e4m3_encode((v * 4).astype(np.float32)))
    # beyond the range the codes saturate to +-448
    q = oracle.static_quant(x, 0, 1e-3)
    assert np.all(np.abs(oracle.e4m3_decode(q)) <= 448) and np.any((q & 0x7F) == 0x7E)
    # an IEEE divide, not a multiply by the reciprocal: 87.5 / 7 = 12.5 exactly, the
    # midpoint of 12 (0x54) and 13 (0x55), which goes to the even code 0x54;
    # fl32(1/7) = (1/7)(1 + 4.47e-8) would give 87.5 * fl32(1/7) = 12.50000056,
    # rounded to 12.5 + 2^-20 and so to 13
    xb = np.array([0x42AF, 0xC2AF], np.uint16)                  # bf16 87.5, -87.5
    assert list(oracle.static_quant(xb, 0, 7.0)) == [0x54, 0xD4]
    xh = np.array([0x5578, 0xD578], np.uint16)                  # fp16 87.5, -87.5
    assert list(oracle.static_quant(xh, 1, 7.0)) == [0x54, 0xD4]


def test_requantize_with_max_scale_pins():
    rng = np.random.default_rng(93)
    w = rng.integers(0, 256, size=(100, 64), dtype=np.uint8)
    w[(w & 0x7F) == 0x7F] = 0x30
    widths = [32, 48, 16]                   # rows 96..99 lie past the shards and are copied
    # equal shard scales: nothing changes
    out, smax = oracle.requantize_with_max_scale(w, [0.5, 0.5, 0.5], widths)
    assert np.array_equal(out, w) and smax == np.float32(0.5)
    # a shard whose scale is s_max / 4: its values are divided by 4 exactly, then re-encoded
    out, smax = oracle.requantize_with_max_scale(w, [1.0, 0.25, 1.0], widths)
    assert smax == 1.0
    assert np.array_equal(out[:32], w[:32]) and np.array_equal(out[80:], w[80:])
    mid = oracle.e4m3_decode(w[32:80]) / 4
    assert np.array_equal(out[32:80], oracle.e4m3_encode(mid.astype(np.float32)))
    # the dequantized weight is fp32: code 0x11 is d = 9*2^-8 and the shard scale
    # s = 0x4089C71C = 2257351*2^-19, so d*s = 20316159*2^-27, a 25-bit odd
    # significand whose rounding to fp32 is a tie, resolved to the even 20316160*2^-27
    # = 155*2^-10.  Divided by s_max = 5 that is 31*2^-10 exactly, the midpoint of
    # 15*2^-9 (0x0F) and 16*2^-9 (0x10): the even code 0x10.  (Without the fp32
    # rounding of d*s the quotient lies just below the midpoint: 0x0F.)
    s_i = np.array([0x4089C71C], np.uint32).view(np.float32)[0]
    out, smax = oracle.requantize_with_max_scale(np.array([[0x11], [0x11]], np.uint8), [s_i, 5.0], [1, 1])
    assert smax == np.float32(5.0) and out[0, 0] == 0x10


def test_int8_encode_pins():
    # ties go to the even neighbour; the clamp takes NaN to +127 and saturates
    x = np.array([0.5, 1.5, 2.5, -0.5, -2.5, 126.5, 127.49, 300.0, -300.0, np.nan, np.inf, -np.inf, -127.5],
                 np.float32)
    want = np.array([0, 2, 2, 0, -2, 126, 127, 127, -128, 127, 127, -128, -128], np.int8)
    assert np.array_equal(oracle.i8_encode(x), want)
    # finite values in range reduce to numpy's round-half-to-even
    r = (np.random.default_rng(94).standard_normal(20000) * 60).astype(np.float32)
    r[::7] = np.round(r[::7]) + 0.5
    assert np.array_equal(oracle.i8_encode(r), np.clip(np.rint(r), -128, 127).astype(np.int8))


def test_int8_multiplier_is_an_ieee_quotient():
    # a = 143/64: fl32(127/a) = 14900045*2^-18, and a times it is 127 + 1.8e-7, which
    # rounds to 127 (code 127).  v = a/2 = 143/128 gives v*mult = 63.5 + 9e-8 exactly,
    # which rounds to 63.5, a tie that goes to the even 64.  (The reciprocal of the
    # stored scale fl32(a/127) = 0x3C902041 is one ulp smaller and would give
    # 63.499996 -> 63.)
    x = np.zeros((1, 128), np.uint16)
    x[0, :3] = [0x400F, 0x3F8F, 0xBF8F]                     # bf16 143/64, 143/128, -143/128
    q, s = oracle.group_quant_int8(x, 0, 128)
    assert list(q[0, :3]) == [127, 64, -64] and not q[0, 3:].any()
    assert s.view(np.uint32)[0, 0] == 0x3C902041


def test_int8_group_quant_properties():
    x = synth.to_bits(synth.quant_input(64, 1024, seed=95))
    v = oracle.bf16_bits_to_f64(x)
    q, s = oracle.group_quant_int8(x, 0, 128)
    assert q.dtype == np.int8 and s.shape == (64, 8)
    g = v.reshape(64, 8, 128)
    a = np.maximum(np.abs(g).max(axis=2), 1e-10)
    # scale = absmax / 127 to fp32 rounding, and the same absmax as the fp8 quant sees
    assert np.all(np.abs(s - a / 127) <= a / 127 * 2.0 ** -23)
    _, s8, _ = oracle.group_quant_canonical(x, 0, 128)
    assert np.all(np.abs(s * 127.0 - s8 * 448.0) <= a * 2.0 ** -21)
    qg = q.reshape(64, 8, 128).astype(np.int64)
    nz = np.abs(g).max(axis=2) > 0
    # the largest element of every non-zero group maps to +-127, all codes within it
    assert np.all(np.abs(qg).max(axis=2)[nz] == 127) and np.all(np.abs(qg) <= 127)
    # dequantization is within half a step (plus the multiplier's rounding)
    err = np.abs(qg * s[:, :, None] - g)
    assert np.all(err <= s[:, :, None] * (0.5 + 2.0 ** -16))
    # an all-zero group: zero codes, floor scale
    z = np.zeros((1, 128), np.uint16)
    qz, sz = oracle.group_quant_int8(z, 0, 128)
    assert not qz.any() and sz[0, 0] == np.float32(np.float32(1e-10) / np.float32(127))
    # negating the input negates the codes
    qn, sn = oracle.group_quant_int8(x ^ np.uint16(0x8000), 0, 128)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    # column-major scales are the transpose, padded to a multiple of 4 rows
    _, scm = oracle.group_quant_int8(x[:6], 0, 128, colmajor=True)
    assert scm.shape == (8, 8) and np.array_equal(scm[:, :6], s[:6].T) and not scm[:, 6:].any()


def test_int8_fused_silu_mul_against_fp64():
    x = synth.to_bits(synth.normal((8, 512), 2.0, seed=96))
    q, s = oracle.group_quant_int8(x, 0, 128, fuse_silu_mul=True)
    v = oracle.bf16_bits_to_f64(x)
    gate, up = v[:, :256], v[:, 256:]
    ref = gate / (1.0 + np.exp(-gate)) * up
    err = np.abs(q.astype(np.float64).reshape(8, 2, 128) * s[:, :, None] - ref.reshape(8, 2, 128))
    assert np.all(err <= s[:, :, None] * (0.5 + 2.0 ** -12))


def test_row_padded_pins():
    x = synth.to_bits(synth.quant_input(10, 512, seed=97))
    for fmt, cm in [(oracle.SCALE_FP32, True), (oracle.SCALE_FP32, False), (oracle.SCALE_UE8M0_PACKED, True)]:
        q, sc = oracle.group_quant(x, 0, 128, fmt, cm)
        qp, scp = oracle.group_quant_row_padded(x, 0, 128, 16, fmt, cm)
        assert qp.shape == (16, 512) and np.array_equal(qp[:10], q) and not qp[10:].any()
        if cm:
            assert scp.shape[1] == 16 and np.array_equal(scp[:, :10], sc[:, :10]) and not scp[:, 10:].any()
        else:
            assert scp.shape[0] == 16 and np.array_equal(scp[:10], sc) and not scp[10:].any()


@pytest.mark.parametrize("pos", [0, 1, 63, 127])
@pytest.mark.parametrize("nan_bits", [0x7F81, 0xFFC0, 0x7FC1])
def test_absmax_skips_every_nan_wherever_it_sits(pos, nan_bits):
    # signaling (0x7F81) or quiet NaN at any position: the scale is that of the group
    # with the NaN replaced by 0, in both output formats, and the NaN encodes at +max
    x = synth.to_bits(synth.quant_input(1, 128, seed=98))
    y = x.copy()
    y[0, pos] = nan_bits
    x[0, pos] = 0
    _, s_ref, _ = oracle.group_quant_canonical(x, 0, 128)
    q, s, _ = oracle.group_quant_canonical(y, 0, 128)
    assert s[0, 0] == s_ref[0, 0] and q[0, pos] == 0x7E
    qi, si = oracle.group_quant_int8(y, 0, 128)
    _, si_ref = oracle.group_quant_int8(x, 0, 128)
    assert si[0, 0] == si_ref[0, 0] and qi[0, pos] == 127
