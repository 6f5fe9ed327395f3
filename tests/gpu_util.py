"""Shared helpers of the GPU parity tests: device placement and the GEMM
tolerance check.  Inputs come from the seeded generators and, for the GEMM,
are quantized by the CPU oracle; expected values come only from the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_mm_gb300 import synth


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp8_scaled_gemm_mm_gb300 as fm
    fm.lib()   # fail loudly if the library is missing
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.to(dev)


def bits(t: torch.Tensor) -> np.ndarray:
    """GPU tensor -> numpy with the same bytes (uint16 for 16-bit types)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_to_f64(b: np.ndarray, out_dtype: int) -> np.ndarray:
    return oracle.bf16_bits_to_f64(b) if out_dtype == 0 else oracle.fp16_bits_to_f64(b)


def ulp_of(ref: np.ndarray, out_dtype: int) -> np.ndarray:
    mbits, emin = (7, -126) if out_dtype == 0 else (10, -14)
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** (emin - 1))))
    e = np.maximum(e, emin)
    return 2.0 ** (e - mbits)


def check_gemm(got_bits, exact, sumabs, K: int, out_dtype: int = 0, what: str = ""):
    """Elementwise check of the GEMM output against the oracle.

    Criterion: |got - ref| <= max(1 ulp of ref in the output format, 2^-7 |ref|).
    Where an output nearly cancels (|ref| << the magnitude of its terms) the
    fp32 accumulation of any GPU kernel can exceed that literal bound; such
    elements must instead lie within ulp(ref) + 2 K 2^-24 sum|a_s b_s A B|,
    the worst-case error of fp32 summation of K terms, and must be rare.
    Returns a dict of statistics.
    """
    got = out_to_f64(got_bits, out_dtype)
    ref = exact
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    diff = np.abs(got - ref)
    ulp = ulp_of(ref, out_dtype)
    lit = np.maximum(ulp, 2.0 ** -7 * np.abs(ref))
    acc = ulp + 2.0 * K * 2.0 ** -24 * sumabs
    bad_lit = diff > lit
    bad = bad_lit & (diff > acc)
    stats = {
        "n": int(diff.size),
        "literal_violations": int(bad_lit.sum()),
        "hard_violations": int(bad.sum()),
        "max_rel_to_sumabs": float((diff / np.maximum(sumabs, 1e-300)).max()),
    }
    assert stats["hard_violations"] == 0, (what, stats, np.argwhere(bad)[:5])
    assert stats["literal_violations"] <= max(2, 1e-4 * diff.size), (what, stats)
    return stats


def gemm_inputs(M, N, K, a_mode, b_mode, seed_a=synth.SEED_A, seed_b=synth.SEED_B, lda=None):
    """bf16 X ~N(0,1) [M,K], W ~N(0,0.02) [N,K] quantized by the oracle.

    a_mode: 'tensor' | 'row' | 'group' (group 128, fp32 scales)
    b_mode: 'tensor' | 'col'
    Returns (A codes [M, lda], a_scale, B codes [N, K], b_scale).
    """
    X = synth.to_bits(synth.normal((M, K), 1.0, seed=seed_a))
    W = synth.to_bits(synth.normal((N, K), 0.02, seed=seed_b))
    if a_mode == "tensor":
        A, a_s = oracle.quantize_tensor(X)
        a_s = np.array([a_s], np.float32)
    elif a_mode == "row":
        A, a_s = oracle.quantize_rows(X)
    else:
        A, a_s, _ = oracle.group_quant_canonical(X, 0, 128)
    if b_mode == "tensor":
        B, b_s = oracle.quantize_tensor(W)
        b_s = np.array([b_s], np.float32)
    else:
        B, b_s = oracle.quantize_rows(W)
    if lda is not None and lda != K:
        Aw = np.zeros((M, lda), np.uint8)
        Aw[:, :K] = A
        Aw[:, K:] = 0x5A          # junk beyond K must not be read
        A = Aw
    return A, a_s, B, b_s
