"""The seeded input generators produce the workloads the design notes state
(CPU only): value distributions, the share of tiny and all-zero rows, the
routing layout of the topk scatter and the expert counts of the masked
layout, all reproducible from their seeds."""
import numpy as np
import torch

from fp8_scaled_gemm_mm_gb300 import synth


def test_generators_are_reproducible():
    a = synth.to_bits(synth.quant_input(64, 256, seed=5))
    assert np.array_equal(a, synth.to_bits(synth.quant_input(64, 256, seed=5)))
    assert not np.array_equal(a, synth.to_bits(synth.quant_input(64, 256, seed=6)))
    assert np.array_equal(synth.routing(50)[0], synth.routing(50)[0])
    assert np.array_equal(synth.masked_counts(1000, 8), synth.masked_counts(1000, 8))


def test_normal_std():
    for std in (1.0, 0.02, 0.1):
        x = synth.normal((512, 512), std, seed=3).float()
        assert abs(x.mean().item()) < 5e-3 * std / 0.1 + 1e-3 * std
        assert abs(x.std().item() / std - 1) < 0.01


def test_quant_input_row_mix():
    M, K = 8192, 256
    x = synth.quant_input(M, K, seed=0).float()
    amax = x.abs().amax(dim=1)
    zero = amax == 0
    tiny = (amax > 0) & (amax < 1e-2)
    # 1 % all-zero rows, 5 % rows scaled by 1e-4 (binomial spread: +- 4 sigma)
    assert abs(zero.sum().item() - 0.01 * M) < 4 * (0.01 * 0.99 * M) ** 0.5
    assert abs(tiny.sum().item() - 0.05 * M) < 4 * (0.05 * 0.95 * M) ** 0.5
    normal_rows = x[~zero & ~tiny]
    assert abs(normal_rows.std().item() - 1) < 0.01
    assert abs(x[tiny].std().item() / 1e-4 - 1) < 0.05
    # the rows are chosen before the cast: fp16 has the same zero and tiny rows
    h = synth.quant_input(M, K, torch.float16, seed=0).float()
    hmax = h.abs().amax(dim=1)
    assert torch.equal(hmax == 0, zero) and torch.equal((hmax > 0) & (hmax < 1e-2), tiny)


def test_routing_layout():
    M, topk, E, align = 300, 8, 64, 16
    dst, R = synth.routing(M, topk=topk, num_experts=E, align=align)
    assert dst.shape == (M, topk) and dst.dtype == np.int32
    assert R % align == 0
    used = np.sort(dst.ravel())
    assert len(np.unique(used)) == M * topk and used[0] >= 0 and used[-1] < R
    # every expert region starts on an `align` boundary and is filled from its start:
    # the used rows form runs that each begin at a multiple of `align`
    breaks = np.flatnonzero(np.diff(used) != 1) + 1
    starts = used[np.concatenate([[0], breaks])]
    assert np.all(starts % align == 0)
    # padding per region is below `align`, so at most E*(align-1) rows are unused
    assert R - M * topk <= E * (align - 1)


def test_routing_orders_tokens_within_an_expert():
    # regions start on multiples of `align`, so each aligned block of rows belongs to
    # one expert; inside it the rows hold that expert's tokens in increasing order
    align = 8
    dst, R = synth.routing(200, topk=2, num_experts=6, align=align)
    token_of_row = np.full(R, -1)
    for m in range(dst.shape[0]):
        token_of_row[dst[m]] = m
    for b in range(0, R, align):
        t = token_of_row[b:b + align]
        t = t[t >= 0]
        assert np.all(np.diff(t) > 0), (b, t)
        # rows are filled from the start of the block: no hole before a used row
        assert np.all(token_of_row[b:b + len(t)] >= 0)


def test_masked_counts():
    c = synth.masked_counts(4096, 256)
    assert c.sum() == 4096 * 8 and np.all(c <= 4096) and c.dtype == np.int32
    assert np.array_equal(synth.masked_counts(4096, 32), c[:32])
    # about tokens * topk / experts each
    assert abs(c.mean() - 128) < 1e-9 and c.min() > 64 and c.max() < 192


def test_bits_round_trip():
    x = synth.normal((33, 17), 1.0, seed=4)
    b = synth.to_bits(x)
    assert b.dtype == np.uint16 and b.shape == (33, 17)
    assert torch.equal(synth.from_bits(b, torch.bfloat16), x)
    h = x.to(torch.float16)
    assert torch.equal(synth.from_bits(synth.to_bits(h), torch.float16), h)
