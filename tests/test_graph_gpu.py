"""Every entry point launches asynchronously on the caller's stream with no host
synchronisation or per-call allocation, so a sequence of them can be captured
in a CUDA graph and replayed (the deterministic-linear PR tests graph replay of
its linears).  Captured replays over fresh inputs must reproduce eager results
bit for bit (every kernel here has a fixed reduction order)."""
import numpy as np
import pytest
import torch

import fp8_scaled_gemm_mm_gb300 as fm
from fp8_scaled_gemm_mm_gb300 import synth
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def _pipeline(bufs):
    """Quant -> GEMM chains for a prefill-like and a decode-like row count, the
    block-scaled GEMM and the masked fused quant, all on the current stream."""
    b = bufs
    fm.per_token_group_quant_fp8(b["x"], b["a"], b["a_s"], b["x"].shape[1])
    fm.fp8_scaled_mm(b["a"], b["w"], b["a_s"], b["w_s"], fm.A_ROW | fm.B_COL, b["out"], bias=b["bias"])
    fm.per_token_group_quant_fp8(b["xd"], b["ad"], b["ad_s"], b["xd"].shape[1])
    fm.fp8_scaled_mm(b["ad"], b["w"], b["ad_s"], b["w_s"], fm.A_ROW | fm.B_COL, b["outd"])
    fm.fp8_scaled_mm(b["ad"], b["w"], b["ad_s"], b["w_s"], fm.A_ROW | fm.B_COL, b["outdet"], deterministic=True)
    fm.per_token_group_quant_fp8(b["x"], b["ag"], b["ag_s"], 128, fm.SCALE_UE8M0_PACKED, True)
    fm.fp8_scaled_mm(b["ag"], b["w"], b["ag_s"], b["w_blk"], fm.A_GROUP128_UE8M0 | fm.B_BLOCK128, b["outg"])
    fm.silu_and_mul_masked_post_quant_fp8(b["xm"], b["mm"], b["qm"], b["sm"], 128)
    fm.fp8_scaled_mm(b["sa"], b["sw"], b["ss"], b["ss"], fm.A_TENSOR | fm.B_TENSOR, b["outsk"])   # a tail-wave shape


def _make(dev):
    M, Md, K, N = 512, 8, 1024, 768
    E, T, KM = 4, 64, 256
    w = torch.empty((N, K), dtype=torch.uint8, device=dev)
    w_s = torch.empty((N, 1), dtype=torch.float32, device=dev)
    fm.per_token_group_quant_fp8(synth.normal((N, K), 0.02, seed=31, device=dev), w, w_s, K)
    b = dict(
        x=torch.empty((M, K), dtype=torch.bfloat16, device=dev),
        xd=torch.empty((Md, K), dtype=torch.bfloat16, device=dev),
        xm=torch.empty((E, T, 2 * KM), dtype=torch.bfloat16, device=dev),
        mm=torch.tensor([64, 3, 0, 17], dtype=torch.int32, device=dev),
        w=w, w_s=w_s,
        w_blk=(torch.rand(((N + 127) // 128, K // 128), generator=torch.Generator(device=dev).manual_seed(3),
                          device=dev) * 1e-3 + 1e-4),
        bias=synth.normal((N,), 0.1, seed=32, device=dev),
        a=torch.empty((M, K), dtype=torch.uint8, device=dev),
        a_s=torch.empty((M, 1), dtype=torch.float32, device=dev),
        ad=torch.empty((Md, K), dtype=torch.uint8, device=dev),
        ad_s=torch.empty((Md, 1), dtype=torch.float32, device=dev),
        ag=torch.empty((M, K), dtype=torch.uint8, device=dev),
        ag_s=torch.empty(fm.scale_shape(M, K, 128, fm.SCALE_UE8M0_PACKED, True), dtype=torch.int32, device=dev),
        out=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
        outd=torch.empty((Md, N), dtype=torch.bfloat16, device=dev),
        outdet=torch.empty((Md, N), dtype=torch.bfloat16, device=dev),
        outg=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
        sa=torch.randint(0, 126, (2048, 4096), generator=torch.Generator(device=dev).manual_seed(5),
                         dtype=torch.uint8, device=dev),
        sw=torch.randint(0, 126, (4096, 4096), generator=torch.Generator(device=dev).manual_seed(6),
                         dtype=torch.uint8, device=dev),
        ss=torch.full((1,), 0.01, dtype=torch.float32, device=dev),
        outsk=torch.empty((2048, 4096), dtype=torch.bfloat16, device=dev),
        qm=torch.zeros((E, T, KM), dtype=torch.uint8, device=dev),
        sm=torch.zeros(fm.masked_scale_shape(E, T, KM, 128, fm.SCALE_UE8M0_PACKED, True), dtype=torch.int32,
                       device=dev),
    )
    return b


def _fill(b, seed, dev):
    b["x"].copy_(synth.quant_input(*b["x"].shape, seed=seed, device=dev))
    b["xd"].copy_(synth.quant_input(*b["xd"].shape, seed=seed + 1, device=dev))
    b["xm"].copy_(synth.quant_input(b["xm"].shape[0] * b["xm"].shape[1], b["xm"].shape[2], seed=seed + 2,
                                    device=dev).reshape(b["xm"].shape))


OUTS = ("a", "a_s", "out", "ad", "outd", "outdet", "ag", "ag_s", "outg", "qm", "sm", "outsk")


def test_graph_replay_matches_eager():
    dev = require_gpu()
    b = _make(dev)
    _fill(b, 100, dev)
    _pipeline(b)                     # first calls: per-device set-up happens here, outside capture
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _pipeline(b)
    torch.cuda.synchronize()
    assert fm.get_device_status() == 0

    for seed in (200, 300, 400):
        _fill(b, seed, dev)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        replayed = {k: b[k].clone() for k in OUTS}
        _pipeline(b)                 # eager on the same inputs
        torch.cuda.synchronize()
        for k in OUTS:
            assert torch.equal(replayed[k].view(torch.uint8), b[k].view(torch.uint8)), (seed, k)
        assert fm.get_device_status() == 0
