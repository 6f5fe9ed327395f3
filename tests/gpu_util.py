"""Shared helpers of the GPU parity tests: device placement, byte views and the
GEMM inputs.  Inputs come from the seeded generators and, for the GEMM, are
quantized by the CPU oracle; expected values come only from the oracle, and the
GEMM tolerance rule is oracle.parity.check_gemm."""
import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_mm_gb300 import synth
from oracle.parity import check_gemm, out_to_f64, ulp_of  # noqa: F401  (the parity criterion)


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
