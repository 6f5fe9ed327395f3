"""CPU oracle for the FP8 linear-layer hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``fp8_scaled_gemm_mm_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``fp8_oracle.c`` (plain C, IEEE fp32/fp64, no FMA
contraction); this module marshals numpy arrays and lays scales out in the
layouts the cited pull requests name, with plain indexing:

* per-token group quant -- sglang PR #33533 "[JIT] per_token_group_quant: fix
  the fp16 UE8M0 multiplier overflow, 1.23x on the fused EP-MoE path, unify
  the scale allocation" (Modifications 1-3; the scale-format table in
  section 3: fp32, fp32 power of two 2^(e-127), UE8M0 bytes packed four to an
  int32; row-major or column-major "TMA-aligned" layouts).
* the topk scatter variant -- same PR, second commit note: one token quantized
  once and replicated to its destination rows, the scale written into the
  MN-major grouped-GEMM buffer.  The oracle is, as the PR's own test is, the
  non-scatter result with its rows mapped.
* scaled FP8 GEMM -- sglang PR #34318 "[Kernel] Route large SM90
  row/column-scaled FP8 GEMMs to Torch" (Summary: E4M3FN inputs, fp32
  row/column scales, bf16 out) and the prhub summary of sglang PR #33148
  (per-tensor scalar scales; the bias argument of ``apply``).

Every function here is pinned by ``tests/test_oracle_*.py`` against values
and properties that do not come from this code.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

EPS = np.float32(1e-10)          # the group-absmax floor
FP8_MAX = 448.0                  # largest finite E4M3FN value

# scale formats (shared vocabulary with the C ABI's `ue8m0` argument)
SCALE_FP32 = 0
SCALE_FP32_POW2 = 1
SCALE_UE8M0_PACKED = 2

# GEMM scale modes, A side (low nibble) and B side (high nibble)
A_TENSOR, A_ROW, A_GROUP, A_GROUP_COLMAJOR, A_GROUP_UE8M0 = 0, 1, 2, 3, 4
B_TENSOR, B_COL, B_BLOCK = 0, 1, 2


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        L.oracle_decode_e4m3.argtypes = [P, P, I64]
        L.oracle_encode_e4m3.argtypes = [P, P, I64]
        L.oracle_round_bf16.argtypes = [P, P, I64]
        L.oracle_round_fp16.argtypes = [P, P, I64]
        L.oracle_exp_f32.argtypes = [P, P, I64]
        L.oracle_silu_f32.argtypes = [P, P, I64]
        L.oracle_group_quant.argtypes = [P, I, I64, I64, I64, I, I, P, P, P]
        L.oracle_encode_i8.argtypes = [P, P, I64]
        L.oracle_group_quant_int8.argtypes = [P, I, I64, I64, I64, I, P, P]
        L.oracle_group_quant.restype = I
        L.oracle_gemm.argtypes = [P, I64, P, I64, I64, I64, I64, P, I, I64, P, I, P, I, P, I64,
                                  P, P, P, I]
        L.oracle_gemm.restype = I
        L.oracle_num_threads.restype = I
        _LIB = L
    return _LIB


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads() -> int:
    return lib().oracle_num_threads()


# ---------------------------------------------------------------- E4M3 ---

def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().oracle_decode_e4m3(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    v = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_encode_e4m3(_ptr(v), _ptr(out), v.size)
    return out


# ------------------------------------------------------ 16-bit rounding ---

def round_bf16(x) -> np.ndarray:
    """fp64 -> bf16 bit patterns, round to nearest even."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_round_bf16(_ptr(v), _ptr(out), v.size)
    return out


def round_fp16(x) -> np.ndarray:
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_round_fp16(_ptr(v), _ptr(out), v.size)
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def fp16_bits_to_f64(bits) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ----------------------------------------------------------- exp / SiLU ---

def exp_f32(x) -> np.ndarray:
    v = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(v.shape, np.float32)
    lib().oracle_exp_f32(_ptr(v), _ptr(out), v.size)
    return out


def silu_f32(x) -> np.ndarray:
    v = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(v.shape, np.float32)
    lib().oracle_silu_f32(_ptr(v), _ptr(out), v.size)
    return out


# --------------------------------------------------------- group quant ---

def group_quant_canonical(x_bits, x_dtype: int, group: int, fuse_silu_mul: bool = False,
                          ue8m0: bool = False):
    """Per-token group quant, canonical outputs.

    x_bits: uint16 [M, K] (or [M, 2K] when fused) holding bf16 (x_dtype 0)
    or fp16 (x_dtype 1) bit patterns.  Returns (q uint8 [M, K], s float32
    [M, G], e uint8 [M, G]) where s is the scale value and e the UE8M0 byte.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M = x.shape[0]
    K = x.shape[1] // 2 if fuse_silu_mul else x.shape[1]
    if K % group:
        raise ValueError("group must divide K")
    G = K // group
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, G), np.float32)
    e = np.empty((M, G), np.uint8)
    rc = lib().oracle_group_quant(_ptr(x), x_dtype, M, K, group, int(fuse_silu_mul), int(ue8m0),
                                  _ptr(q), _ptr(s), _ptr(e))
    if rc != 0:
        raise RuntimeError(f"oracle_group_quant failed ({rc})")
    return q, s, e


def i8_encode(x) -> np.ndarray:
    """fp32 -> int8: NaN -> +127, clamp to [-128, 127], round half to even."""
    v = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(v.shape, np.int8)
    lib().oracle_encode_i8(_ptr(v), _ptr(out), v.size)
    return out


def group_quant_int8(x_bits, x_dtype: int, group: int, colmajor: bool = False, fuse_silu_mul: bool = False):
    """int8 per-token group quant (fp32 scales max(amax, 1e-10)/127).
    Returns (q int8 [M, K], scales laid out row-major [M, G] or column-major
    [G, pad4(M)])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M = x.shape[0]
    K = x.shape[1] // 2 if fuse_silu_mul else x.shape[1]
    if K % group:
        raise ValueError("group must divide K")
    q = np.empty((M, K), np.int8)
    s = np.empty((M, K // group), np.float32)
    rc = lib().oracle_group_quant_int8(_ptr(x), x_dtype, M, K, group, int(fuse_silu_mul), _ptr(q), _ptr(s))
    if rc != 0:
        raise RuntimeError(f"oracle_group_quant_int8 failed ({rc})")
    return q, layout_scales(s, None, SCALE_FP32, colmajor)


def group_quant_row_padded(x_bits, x_dtype: int, group: int, m_pad: int, fmt: int = SCALE_FP32,
                           colmajor: bool = True):
    """Row-padded group quant: outputs sized for m_pad >= M rows; rows M..m_pad-1
    get zero codes and zero scales (the row padding plus tail zeroing of the
    entry-point dedup notes of sglang PR #33533)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x.shape
    if m_pad < M:
        raise ValueError("m_pad < M")
    q, s, e = group_quant_canonical(x, x_dtype, group, False, fmt != SCALE_FP32)
    qp = np.zeros((m_pad, K), np.uint8)
    qp[:M] = q
    sp = np.zeros((m_pad, s.shape[1]), np.float32)
    sp[:M] = s
    ep = np.zeros((m_pad, s.shape[1]), np.uint8)
    ep[:M] = e
    return qp, layout_scales(sp, ep, fmt, colmajor)


def pad4(n: int) -> int:
    return (n + 3) // 4 * 4


def layout_scales(s, e, fmt: int, colmajor: bool, rows_total: int = None, row_map=None):
    """Lay per-(row, group) scales out as the kernel stores them.

    fmt 0/1: float32; row-major [R, G] or column-major [G, pad4(R)].
    fmt 2:   UE8M0 bytes, four groups per int32 (group 4j+b in byte b);
             row-major [R, ceil(G/4)] or column-major [ceil(G/4), pad4(R)].
    Unwritten entries (padding, unused bytes of the last word) are 0.
    row_map (optional) gives, for each source row, the destination rows
    (-1 = none) -- the scatter variant; rows_total is then the number of
    destination rows.
    """
    M, G = s.shape
    R = M if rows_total is None else rows_total
    if row_map is None:
        pairs = [(m, m) for m in range(M)]
    else:
        pairs = [(m, int(d)) for m in range(M) for d in row_map[m] if d >= 0]
    if fmt in (SCALE_FP32, SCALE_FP32_POW2):
        if colmajor:
            out = np.zeros((G, pad4(R)), np.float32)
            for m, d in pairs:
                out[:, d] = s[m]
        else:
            out = np.zeros((R, G), np.float32)
            for m, d in pairs:
                out[d] = s[m]
        return out
    W = (G + 3) // 4
    words = np.zeros((M, W), np.uint32)
    for g in range(G):
        words[:, g // 4] |= e[:, g].astype(np.uint32) << np.uint32(8 * (g % 4))
    words = words.view(np.int32)
    if colmajor:
        out = np.zeros((W, pad4(R)), np.int32)
        for m, d in pairs:
            out[:, d] = words[m]
    else:
        out = np.zeros((R, W), np.int32)
        for m, d in pairs:
            out[d] = words[m]
    return out


def group_quant(x_bits, x_dtype: int, group: int, fmt: int = SCALE_FP32, colmajor: bool = False,
                fuse_silu_mul: bool = False):
    """per_token_group_quant_fp8: returns (q [M, K] uint8, laid-out scales)."""
    q, s, e = group_quant_canonical(x_bits, x_dtype, group, fuse_silu_mul, fmt != SCALE_FP32)
    return q, layout_scales(s, e, fmt, colmajor)


def group_quant_scatter(x_bits, x_dtype: int, group: int, dst_row, num_dst_rows: int,
                        fmt: int = SCALE_UE8M0_PACKED, colmajor: bool = True):
    """Topk scatter variant: the non-scatter result of row m written to every
    destination row dst_row[m, t] >= 0.  Untouched destination rows are 0."""
    q, s, e = group_quant_canonical(x_bits, x_dtype, group, False, fmt != SCALE_FP32)
    dst = np.asarray(dst_row)
    qd = np.zeros((num_dst_rows, q.shape[1]), np.uint8)
    for m in range(q.shape[0]):
        for d in dst[m]:
            if d >= 0:
                qd[d] = q[m]
    return qd, layout_scales(s, e, fmt, colmajor, rows_total=num_dst_rows, row_map=dst)


def masked_silu_quant(x_bits, x_dtype: int, masked_m, group: int, fmt: int = SCALE_UE8M0_PACKED,
                      colmajor: bool = True):
    """Masked fused SiLU*up group quant on the expert-major layout x [E, T, 2K]
    (the EP-MoE decode path of sglang PR #33533, Speed Tests): rows t <
    masked_m[e] of expert e get the fused group quant of that row; others stay 0.

    Returns (q uint8 [E, T, K], scales): row-major scales as group_quant with
    E*T rows; column-major per expert, [E, G or ceil(G/4), pad4(T)].
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    E, T, K2 = x.shape
    K = K2 // 2
    G = K // group
    q = np.zeros((E, T, K), np.uint8)
    s_all = np.zeros((E, T, G), np.float32)
    e_all = np.zeros((E, T, G), np.uint8)
    written = np.zeros((E, T), bool)
    for e in range(E):
        n = int(masked_m[e])
        if n <= 0:
            continue
        qe, se, ee = group_quant_canonical(x[e, :n], x_dtype, group, True, fmt != SCALE_FP32)
        q[e, :n] = qe
        s_all[e, :n] = se
        e_all[e, :n] = ee
        written[e, :n] = True
    if not colmajor:
        flat_s = s_all.reshape(E * T, G)
        flat_e = e_all.reshape(E * T, G)
        lay = layout_scales(flat_s, flat_e, fmt, False)
        lay[~written.reshape(-1)] = 0
        return q, lay
    outs = []
    for e in range(E):
        lay = layout_scales(s_all[e], e_all[e], fmt, True)     # [cols, pad4(T)]
        lay[:, :T][:, ~written[e]] = 0
        lay[:, T:] = 0
        outs.append(lay)
    return q, np.stack(outs)


def quantize_rows(x_bits, x_dtype: int = 0):
    """Per-row (per-output-channel) E4M3 quantization with fp32 scale
    absmax/448: the group quant with one group per row."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q, s, _ = group_quant_canonical(x, x_dtype, x.shape[1])
    return q, s[:, 0].copy()


def quantize_blocks(w_bits, block: int = 128, x_dtype: int = 0):
    """128 x 128 block quantization of a weight [N, K]: each block gets the
    group-quant formula with the whole block as one group (scale absmax/448).
    Returns (codes [N, K], scales float32 [ceil(N/block), K/block])."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w.shape
    nb, kb = (N + block - 1) // block, K // block
    q = np.empty((N, K), np.uint8)
    s = np.empty((nb, kb), np.float32)
    for i in range(nb):
        rows = w[i * block:(i + 1) * block]
        for j in range(kb):
            blk = np.ascontiguousarray(rows[:, j * block:(j + 1) * block])
            qb, sb, _ = group_quant_canonical(blk.reshape(1, -1), x_dtype, blk.size)
            q[i * block:(i + 1) * block, j * block:(j + 1) * block] = qb.reshape(blk.shape)
            s[i, j] = sb[0, 0]
    return q, s


def static_quant(x_bits, x_dtype: int, scale):
    """Static per-tensor activation quant with a given fp32 scale (the prhub
    summary of sglang PR #33148, Key source snippets: the checkpoint's activation
    scale input_scale.max() is used as it is): q = E4M3(fl32(x / scale))."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    v = (bf16_bits_to_f64(x) if x_dtype == 0 else fp16_bits_to_f64(x)).astype(np.float32)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        r = v / np.float32(scale)                     # IEEE fp32 division
    return e4m3_encode(r)


def requantize_with_max_scale(w_codes, shard_scales, logical_widths):
    """Fused weight with per-logical-shard scales -> one per-tensor scale (same
    snippets: process_weights_after_loading): s_max = max_i s_i and every row of
    shard i becomes E4M3(fl32(fl32(decode(q) * s_i) / s_max)).
    Returns (codes, s_max)."""
    w = np.ascontiguousarray(w_codes, dtype=np.uint8)
    s = np.asarray(shard_scales, dtype=np.float32)
    s_max = np.float32(s.max())
    out = np.empty_like(w)
    start = 0
    for i, width in enumerate(logical_widths):
        deq = (e4m3_decode(w[start:start + width]).astype(np.float32) * s[i]).astype(np.float32)
        out[start:start + width] = e4m3_encode((deq / s_max).astype(np.float32))
        start += width
    out[start:] = w[start:]
    return out, s_max


def quantize_tensor(x_bits, x_dtype: int = 0):
    """Per-tensor E4M3 quantization with one fp32 scale absmax/448: the same
    formula with the whole tensor as one group."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    flat = x.reshape(1, -1)
    q, s, _ = group_quant_canonical(flat, x_dtype, flat.shape[1])
    return q.reshape(x.shape), np.float32(s[0, 0])


# ---------------------------------------------------------------- GEMM ---

def gemm(A, B, a_scale, b_scale, a_mode: int, b_mode: int, bias_bits=None, out_dtype: int = 0,
         K: int = None, rows=None, want_exact: bool = False, threads: int = 0):
    """Scaled FP8 GEMM: out[m, n] = round(a_s * b_s * sum_k A[m,k] B[n,k] (+ bias[n])).

    A: uint8 [M, lda] (first K columns used), B: uint8 [N, ldb].
    a_scale: float32 scalar / [M] / [M, K/128] (a_mode 2) / [K/128, ld] (a_mode 3) /
    int32 packed UE8M0 words [ceil(K/512), ld] (a_mode 4).
    b_scale: float32 scalar / [N] / [ceil(N/128), K/128] (b_mode 2, with a per-group a_mode).
    Returns out bits (uint16 [rows, N]) and, if want_exact, the fp64 value
    before rounding and sum |a_s b_s A B| (for accumulation-error bounds).
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    M, lda = A.shape
    N, ldb = B.shape
    K = lda if K is None else K
    if a_mode == A_GROUP_UE8M0:    # packed UE8M0 words, passed through bit for bit
        a_s = np.ascontiguousarray(np.asarray(a_scale, dtype=np.int32)).view(np.float32)
    else:
        a_s = np.ascontiguousarray(np.atleast_1d(a_scale), dtype=np.float32)
    b_s = np.ascontiguousarray(np.atleast_1d(b_scale), dtype=np.float32)
    a_ld = a_s.shape[1] if a_s.ndim == 2 else 0
    bias = None if bias_bits is None else np.ascontiguousarray(bias_bits, dtype=np.uint16)
    if rows is None:
        rr = None
        n_rows = M
    else:
        rr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rr.size
    out = np.empty((n_rows, N), np.uint16)
    exact = np.empty((n_rows, N), np.float64) if want_exact else None
    sumabs = np.empty((n_rows, N), np.float64) if want_exact else None
    rc = lib().oracle_gemm(_ptr(A), lda, _ptr(B), ldb, M, N, K, _ptr(a_s), a_mode, a_ld, _ptr(b_s),
                           b_mode, _ptr(bias), out_dtype, _ptr(rr), n_rows, _ptr(out), _ptr(exact),
                           _ptr(sumabs), threads)
    if rc <= 0:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    if want_exact:
        return out, exact, sumabs
    return out
