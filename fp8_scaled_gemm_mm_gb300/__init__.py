"""Python binding of libfp8mm, the GB300 (sm_103a) FP8 linear-layer hot path.

Thin marshalling over the C ABI declared in ``include/fp8mm.h``: every function
here passes device pointers, sizes and the current CUDA stream to the library
and raises ``Fp8mmError`` on a non-zero status.  All arithmetic happens in the
library's CUDA kernels; there is no other implementation to fall back to, and
importing this module fails loudly if the library has not been built.

Operations (see the header for full semantics):
  per_token_group_quant_fp8             bf16/fp16 -> E4M3FN codes + scales (group 32/64/128 or
                                        the whole row; fp32, pow-2 or packed UE8M0 scales; fused
                                        SiLU(gate) * up)
  per_token_group_quant_fp8_scatter     the same, written to topk destination rows
  silu_and_mul_masked_post_quant_fp8    fused quant of the expert-major [E, T, 2K] layout
  per_token_group_quant_int8            int8 codes with fp32 scales
  per_token_group_quant_fp8_row_padded  outputs sized for M_pad >= M rows, tail rows zeroed
  static_per_tensor_quant_fp8           E4M3(x / s) with a given scale
  requantize_with_max_scale_fp8         a fused weight's shards brought to their largest scale
  fp8_scaled_mm                         out = round(a_s * b_s * A B^T (+ bias)); per-tensor,
                                        per-row/column, group-128 A and 128 x 128 block B scales;
                                        deterministic (batch-invariant) mode
Diagnostics: get_device_status, selftest_bounded_wait, selftest_scale_math,
set_wait_timeout_ns.

Every call is asynchronous on the given stream (default: torch's current one);
buffers are the caller's, the library allocates nothing per call.

    q, s = fm.alloc_group_quant_outputs(M, K, 128, fm.SCALE_UE8M0_PACKED, True, device="cuda")
    fm.per_token_group_quant_fp8(x, q, s, 128, fm.SCALE_UE8M0_PACKED, True)
    fm.fp8_scaled_mm(q, w_codes, s, w_block_scales, fm.A_GROUP128_UE8M0 | fm.B_BLOCK128, out)
"""
import ctypes
import os

import torch

__all__ = [
    "Fp8mmError", "lib", "per_token_group_quant_fp8", "per_token_group_quant_fp8_scatter",
    "fp8_scaled_mm", "silu_and_mul_masked_post_quant_fp8", "static_per_tensor_quant_fp8",
    "per_token_group_quant_int8", "per_token_group_quant_fp8_row_padded",
    "requantize_with_max_scale_fp8", "masked_scale_shape", "get_device_status", "selftest_bounded_wait",
    "selftest_scale_math", "set_wait_timeout_ns", "scale_shape", "scale_dtype",
    "alloc_group_quant_outputs", "SCALE_FP32", "SCALE_FP32_POW2", "SCALE_UE8M0_PACKED",
    "A_TENSOR", "A_ROW", "A_GROUP128", "A_GROUP128_COLMAJOR", "A_GROUP128_UE8M0", "B_TENSOR", "B_COL",
    "B_BLOCK128",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp8mm.so")

# status codes
OK, EINVAL, EALIGN, EUNSUPPORTED, ECUDA, ETIMEOUT = 0, -1, -2, -3, -4, -5
# scale formats of the group quant
SCALE_FP32, SCALE_FP32_POW2, SCALE_UE8M0_PACKED = 0, 1, 2
# GEMM scale modes
A_TENSOR, A_ROW, A_GROUP128, A_GROUP128_COLMAJOR, A_GROUP128_UE8M0 = 0x0, 0x1, 0x2, 0x3, 0x4
B_TENSOR, B_COL, B_BLOCK128 = 0x00, 0x10, 0x20

_DTYPE_CODE = {torch.bfloat16: 0, torch.float16: 1}


class Fp8mmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib().fp8mm_status_string(status).decode()} ({status})")


_LIB = None


def lib():
    """The loaded libfp8mm (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libfp8mm is not built ({LIB_PATH} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.fp8_scaled_mm.argtypes = [P, P, P, P, I, P, P, I, I64, I64, I64, I64, I64, I, P]
        L.fp8_scaled_mm.restype = I
        L.per_token_group_quant_fp8.argtypes = [P, I, P, P, I64, I64, I, I, I, I, P]
        L.per_token_group_quant_fp8.restype = I
        L.per_token_group_quant_fp8_scatter.argtypes = [P, I, P, I, I64, P, P, I64, I64, I, I, I, P]
        L.per_token_group_quant_fp8_scatter.restype = I
        L.silu_and_mul_masked_post_quant_fp8.argtypes = [P, I, P, I64, I64, I64, P, P, I, I, I, P]
        L.silu_and_mul_masked_post_quant_fp8.restype = I
        L.per_token_group_quant_int8.argtypes = [P, I, P, P, I64, I64, I, I, I, P]
        L.per_token_group_quant_int8.restype = I
        L.per_token_group_quant_fp8_row_padded.argtypes = [P, I, P, P, I64, I64, I64, I, I, I, P]
        L.per_token_group_quant_fp8_row_padded.restype = I
        L.static_per_tensor_quant_fp8.argtypes = [P, I, P, P, I64, P]
        L.static_per_tensor_quant_fp8.restype = I
        L.requantize_with_max_scale_fp8.argtypes = [P, P, P, P, I, I64, I64, P, P]
        L.requantize_with_max_scale_fp8.restype = I
        L.fp8mm_get_device_status.argtypes = [I, I]
        L.fp8mm_get_device_status.restype = I
        L.fp8mm_selftest_bounded_wait.argtypes = [I64, P]
        L.fp8mm_selftest_bounded_wait.restype = I
        L.fp8mm_set_wait_timeout_ns.argtypes = [I64]
        L.fp8mm_set_wait_timeout_ns.restype = I
        L.fp8mm_selftest_scale_math.argtypes = [ctypes.c_uint32, ctypes.c_uint32, P, P]
        L.fp8mm_selftest_scale_math.restype = I
        L.fp8mm_status_string.argtypes = [I]
        L.fp8mm_status_string.restype = ctypes.c_char_p
        L.fp8mm_version.restype = I
        _LIB = L
    return _LIB


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, name="tensor", row_strided=False):
    """Device address of t for the C ABI.  The entry points take a base pointer
    and dense extents (the GEMM operands also a row stride), so a tensor has to
    live on a CUDA device and be contiguous; a 2-D GEMM operand only needs unit
    stride along its last dimension.  A host tensor's address would be read as
    a device address, and a strided view would be read as if it were dense, so
    both are refused here.  Plain ints pass through as raw device addresses."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
    if t.numel() > 0:
        if row_strided and t.dim() == 2:
            if t.stride(1) != 1:
                raise ValueError(f"{name} needs unit stride along its last dimension, got strides {t.stride()}")
        elif not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous, got strides {t.stride()} for shape {tuple(t.shape)}")
    return t.data_ptr()


def _check(status: int, what: str):
    if status != OK:
        raise Fp8mmError(status, what)


# ----------------------------------------------------------- group quant

def scale_shape(rows: int, K: int, group: int, fmt: int, colmajor: bool):
    """Shape of the scale tensor the kernels write (see include/fp8mm.h)."""
    G = K // group
    W = (G + 3) // 4
    pad = (rows + 3) // 4 * 4
    if fmt == SCALE_UE8M0_PACKED:
        return (W, pad) if colmajor else (rows, W)
    return (G, pad) if colmajor else (rows, G)


def scale_dtype(fmt: int):
    return torch.int32 if fmt == SCALE_UE8M0_PACKED else torch.float32


def alloc_group_quant_outputs(rows: int, K: int, group: int, fmt: int = SCALE_FP32, colmajor: bool = False,
                              device="cuda", zero: bool = False):
    """Allocate codes [rows, K] uint8 and the scale tensor for these flags."""
    mk = torch.zeros if zero else torch.empty
    q = mk((rows, K), dtype=torch.uint8, device=device)
    s = mk(scale_shape(rows, K, group, fmt, colmajor), dtype=scale_dtype(fmt), device=device)
    return q, s


def per_token_group_quant_fp8(x, q, s, group: int, ue8m0: int = SCALE_FP32, scale_colmajor: bool = False,
                              fuse_silu_mul: bool = False, stream=None, x_dtype=None, M=None, K=None):
    """Quantize x [M, K] (or [M, 2K] with fuse_silu_mul) into q [M, K] and s."""
    if x_dtype is None:
        x_dtype = _DTYPE_CODE[x.dtype]
    if M is None:
        M = x.shape[0]
    if K is None:
        K = x.shape[1] // 2 if fuse_silu_mul else x.shape[1]
    st = lib().per_token_group_quant_fp8(_ptr(x, "x"), x_dtype, _ptr(q, "q"), _ptr(s, "s"), M, K, group,
                                         int(ue8m0), int(bool(scale_colmajor)), int(bool(fuse_silu_mul)),
                                         _stream(stream))
    _check(st, "per_token_group_quant_fp8")


def per_token_group_quant_int8(x, q, s, group: int, scale_colmajor: bool = False, fuse_silu_mul: bool = False,
                               stream=None):
    """int8 group quant: x [M, K] (or [M, 2K] fused) -> q int8 [M, K], s fp32."""
    M = x.shape[0]
    K = x.shape[1] // 2 if fuse_silu_mul else x.shape[1]
    st = lib().per_token_group_quant_int8(_ptr(x, "x"), _DTYPE_CODE[x.dtype], _ptr(q, "q"), _ptr(s, "s"), M, K,
                                          group, int(bool(scale_colmajor)), int(bool(fuse_silu_mul)),
                                          _stream(stream))
    _check(st, "per_token_group_quant_int8")


def per_token_group_quant_fp8_row_padded(x, q, s, group: int, ue8m0: int = SCALE_FP32, scale_colmajor: bool = True,
                                         stream=None):
    """Group quant of x [M, K] into q [M_pad, K] / s sized for M_pad = q.shape[0]
    rows; rows M .. M_pad-1 are zeroed."""
    M, K = x.shape
    st = lib().per_token_group_quant_fp8_row_padded(_ptr(x, "x"), _DTYPE_CODE[x.dtype], _ptr(q, "q"),
                                                    _ptr(s, "s"), M, q.shape[0], K, group, int(ue8m0),
                                                    int(bool(scale_colmajor)), _stream(stream))
    _check(st, "per_token_group_quant_fp8_row_padded")


def per_token_group_quant_fp8_scatter(x, dst_row, q, s, group: int, ue8m0: int = SCALE_UE8M0_PACKED,
                                      scale_colmajor: bool = True, stream=None, x_dtype=None, M=None, K=None,
                                      topk=None, num_dst_rows=None):
    """Quantize x [M, K] once per token and write it to rows dst_row[m, :] of q / s."""
    if x_dtype is None:
        x_dtype = _DTYPE_CODE[x.dtype]
    if M is None:
        M, K = x.shape
    if topk is None:
        topk = dst_row.shape[1]
    if num_dst_rows is None:
        num_dst_rows = q.shape[0]
    st = lib().per_token_group_quant_fp8_scatter(_ptr(x, "x"), x_dtype, _ptr(dst_row, "dst_row"), topk,
                                                 num_dst_rows, _ptr(q, "q"), _ptr(s, "s"), M, K, group, int(ue8m0),
                                                 int(bool(scale_colmajor)), _stream(stream))
    _check(st, "per_token_group_quant_fp8_scatter")


def masked_scale_shape(E: int, T: int, K: int, group: int, fmt: int, colmajor: bool):
    """Shape of the scale tensor of silu_and_mul_masked_post_quant_fp8."""
    if not colmajor:
        return scale_shape(E * T, K, group, fmt, False)
    G = K // group
    cols = (G + 3) // 4 if fmt == SCALE_UE8M0_PACKED else G
    return (E, cols, (T + 3) // 4 * 4)


def silu_and_mul_masked_post_quant_fp8(x, masked_m, q, s, group: int, ue8m0: int = SCALE_UE8M0_PACKED,
                                       scale_colmajor: bool = True, stream=None):
    """x [E, T, 2K] -> q [E, T, K] and s for the first masked_m[e] rows of each expert."""
    E, T, K2 = x.shape
    st = lib().silu_and_mul_masked_post_quant_fp8(_ptr(x, "x"), _DTYPE_CODE[x.dtype], _ptr(masked_m, "masked_m"),
                                                  E, T, K2 // 2, _ptr(q, "q"), _ptr(s, "s"), group, int(ue8m0),
                                                  int(bool(scale_colmajor)), _stream(stream))
    _check(st, "silu_and_mul_masked_post_quant_fp8")


def static_per_tensor_quant_fp8(x, scale, q, stream=None):
    """q = E4M3(x / scale[0]) elementwise (static activation scale)."""
    st = lib().static_per_tensor_quant_fp8(_ptr(x, "x"), _DTYPE_CODE[x.dtype], _ptr(scale, "scale"), _ptr(q, "q"),
                                           x.numel(), _stream(stream))
    _check(st, "static_per_tensor_quant_fp8")


def requantize_with_max_scale_fp8(w, shard_scales, logical_widths, w_out=None, max_scale_out=None, stream=None):
    """Bring a fused weight's per-shard scales to their maximum; returns (w_out, s_max tensor [1])."""
    N, K = w.shape
    if w_out is None:
        w_out = w
    if max_scale_out is None:
        max_scale_out = torch.empty(1, dtype=torch.float32, device=w.device)
    widths = (ctypes.c_int64 * len(logical_widths))(*[int(v) for v in logical_widths])
    st = lib().requantize_with_max_scale_fp8(_ptr(w, "w"), _ptr(w_out, "w_out"), _ptr(shard_scales, "shard_scales"),
                                             ctypes.cast(widths, ctypes.c_void_p), len(logical_widths), N, K,
                                             _ptr(max_scale_out, "max_scale_out"), _stream(stream))
    _check(st, "requantize_with_max_scale_fp8")
    return w_out, max_scale_out


# ------------------------------------------------------------------ GEMM

def fp8_scaled_mm(A, B, a_scale, b_scale, scale_mode: int, out, bias=None, deterministic: bool = False,
                  stream=None, M=None, N=None, K=None, lda=None, ldb=None):
    """out [M, N] (bf16 / fp16) = round(a_s * b_s * A[:, :K] B[:, :K]^T (+ bias)).

    A: uint8 / float8_e4m3fn [M, lda], B: [N, ldb] (row strides in elements).
    """
    if M is None:
        M = A.shape[0]
    if N is None:
        N = B.shape[0]
    if K is None:
        K = A.shape[1]
    if lda is None:
        lda = A.stride(0) if A.dim() == 2 else K
    if ldb is None:
        ldb = B.stride(0) if B.dim() == 2 else K
    out_dtype = _DTYPE_CODE[out.dtype] if isinstance(out, torch.Tensor) else 0
    st = lib().fp8_scaled_mm(_ptr(A, "A", True), _ptr(B, "B", True), _ptr(a_scale, "a_scale"),
                             _ptr(b_scale, "b_scale"), int(scale_mode), _ptr(bias, "bias"), _ptr(out, "out"),
                             out_dtype, M, N, K, lda, ldb, int(bool(deterministic)), _stream(stream))
    _check(st, "fp8_scaled_mm")


# ------------------------------------------------------------ diagnostics

def get_device_status(device: int = -1, clear: bool = True) -> int:
    return lib().fp8mm_get_device_status(device, int(clear))


def selftest_scale_math(bits_lo: int, bits_hi: int, counters, stream=None):
    """Compare the quant kernels' scale arithmetic with IEEE division over a range
    of fp32 bit patterns; adds mismatch counts to counters (int64 [3], device)."""
    _check(lib().fp8mm_selftest_scale_math(int(bits_lo), int(bits_hi), _ptr(counters, "counters"), _stream(stream)),
           "fp8mm_selftest_scale_math")


def selftest_bounded_wait(timeout_ns: int, stream=None):
    _check(lib().fp8mm_selftest_bounded_wait(int(timeout_ns), _stream(stream)), "fp8mm_selftest_bounded_wait")


def set_wait_timeout_ns(timeout_ns: int):
    """Limit of the GEMM and group-quant kernels' pipeline waits for later launches
    (0: the default)."""
    _check(lib().fp8mm_set_wait_timeout_ns(int(timeout_ns)), "fp8mm_set_wait_timeout_ns")
