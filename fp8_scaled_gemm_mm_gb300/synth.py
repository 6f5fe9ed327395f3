"""Seeded synthetic inputs for tests and benchmarks.

This module only draws random numbers and builds index structures; it holds
none of the quantization or GEMM arithmetic, so both the CUDA path and the
CPU oracle can be fed from it.

Distributions follow the workloads of the cited pull requests:
* GEMM activations ~N(0, 1) and weights ~N(0, 0.02) in bf16, bias ~N(0, 0.1)
  (sglang PR #34318 "Route large SM90 row/column-scaled FP8 GEMMs to Torch",
  Kernel results table; sglang PR #44861 Modifications: bias, strided input,
  BF16/FP16, K = 80 tail).
* group-quant inputs ~N(0, 1) with a fraction of rows scaled by 1e-4 and a
  fraction all zero, so that tiny groups (the fp16 UE8M0 overflow regime of
  sglang PR #33533, Modifications section 1) and the absmax floor both occur.
* topk routing: each token picks `topk` distinct experts out of
  `num_experts`; expert regions are laid out back to back, each padded to a
  multiple of `align` rows, tokens inside a region ordered by token index.
"""
import numpy as np
import torch

SEED_A = 0
SEED_B = 1
SEED_BIAS = 2
SEED_ROUTING = 3


def _gen(seed: int, device="cpu"):
    return torch.Generator(device=device).manual_seed(int(seed))


def normal(shape, std: float = 1.0, seed: int = 0, dtype=torch.bfloat16, device="cpu"):
    """N(0, std^2) samples drawn in fp32 and stored as `dtype`."""
    g = _gen(seed, device)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def quant_input(M: int, K: int, dtype=torch.bfloat16, seed: int = SEED_A, small_frac: float = 0.05,
                zero_frac: float = 0.01, device="cpu"):
    """Group-quant activations: N(0, 1), with `small_frac` of the rows scaled
    by 1e-4 and `zero_frac` of the rows all zero (rows chosen by the seed).
    Row selection is done in fp32 before the cast to `dtype`."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    pick = torch.rand((M,), generator=g, device=device)
    small = pick < small_frac
    zero = (pick >= small_frac) & (pick < small_frac + zero_frac)
    x[small] *= 1e-4
    x[zero] = 0.0
    return x.to(dtype)


def routing(M: int, topk: int = 8, num_experts: int = 256, seed: int = SEED_ROUTING,
            align: int = 128):
    """Destination rows for the topk scatter.

    Returns (dst_row int32 [M, topk], num_dst_rows).  Every token goes to
    `topk` distinct experts; destination row = start of the expert's region +
    the token's rank among the expert's tokens.  Regions are padded to a
    multiple of `align`; padding rows are never written.
    """
    g = _gen(seed)
    scores = torch.rand((M, num_experts), generator=g)
    experts = scores.topk(topk, dim=1).indices.numpy().astype(np.int64)     # [M, topk]
    tok = np.repeat(np.arange(M, dtype=np.int64), topk)
    exp = experts.reshape(-1)
    order = np.lexsort((tok, exp))                    # by expert, then token
    counts = np.bincount(exp, minlength=num_experts)
    padded = (counts + align - 1) // align * align
    start = np.concatenate([[0], np.cumsum(padded)[:-1]])
    first = np.concatenate([[0], np.cumsum(counts)[:-1]])
    rank = np.empty(M * topk, np.int64)
    rank[order] = np.arange(M * topk) - first[exp[order]]
    dst = (start[exp] + rank).reshape(M, topk).astype(np.int32)
    return dst, int(padded.sum())


def masked_counts(tokens: int, local_experts: int, topk: int = 8, num_experts: int = 256,
                  seed: int = SEED_ROUTING):
    """Tokens held by each of the first `local_experts` experts after routing
    `tokens` tokens to `topk` of `num_experts` experts (the per-expert counts of
    an expert-parallel dispatch), int32 [local_experts]."""
    g = _gen(seed)
    scores = torch.rand((tokens, num_experts), generator=g)
    experts = scores.topk(topk, dim=1).indices.reshape(-1).numpy()
    return np.bincount(experts, minlength=num_experts)[:local_experts].astype(np.int32)


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 / fp16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray, dtype=torch.bfloat16) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(dtype)
