#!/usr/bin/env python3
"""Benchmark of the FP8 linear hot path on GB300.

One step = the five large rowwise-scaled prefill GEMMs of the kernel table of
sglang PR #34318 ("Kernel results": M x K x N = 8320x5376x21504,
8320x5376x14336, 23216x5376x28672, 15760x5376x28672, 8320x14336x5376), each
preceded by the per-token quantization of its bf16 activation (group = K, fp32
row scales) that produces the GEMM's A operand:

    X bf16 [M,K] --per_token_group_quant_fp8--> A e4m3 [M,K], a_s [M]
    A, B e4m3 [N,K], a_s, b_s [N] --fp8_scaled_mm--> D bf16 [M,N]

Weights are ~N(0, 0.02) bf16 quantized per output channel once at set-up (by
the same quant kernel), activations ~N(0, 1); inputs stay resident in HBM.
value = sum 2MNK over the step / step time (TFLOP/s), aggregated over ranks.

Also reported: the group-128 quant kernel alone on its largest workload
(M=8192, K=7168 bf16, UE8M0 packed column-major scales, plain and fused
SiLU*up) in GB/s; the roofline of the dominant kernel (the GEMM); the
end-to-end figure through the C ABI with host buffers; the oracle timed on
the host cores on a bounded sample (cpu_baseline); SM clocks sampled during
the timed region.

--impl reference times the CPU oracle (the only reference implementation of
this path) on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 scaled-GEMM TFLOP/s & % of FP8 peak; group-quant GB/s & % of HBM peak"
SHAPES = [(8320, 5376, 21504), (8320, 5376, 14336), (23216, 5376, 28672), (15760, 5376, 28672),
          (8320, 14336, 5376)]  # (M, K, N)
# torch._scaled_mm on H100 80GB for the same five shapes (sglang PR #34318, Kernel results): sum 2MNK / sum time
H100_TORCH_US = [1351.1, 896.4, 5295.9, 3570.9, 843.9]
QUANT_M, QUANT_K = 8192, 7168
FP8_OVER_BF16 = 2.0      # nominal dense FP8 : BF16 tensor rate on GB300 (4.5 : 2.25 PFLOP/s)
NOMINAL_FP8_DENSE_TFLOPS = 4500.0   # GB300 dense FP8 tensor rate, nominal (context for the measured-peak fraction)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
L2_FLUSH_BYTES = 512 << 20


def workload_config(world):
    """The `config` object of the JSON line; the same for both arms."""
    return {"workload": "large rowwise-scaled FP8 prefill GEMMs (5 shapes) + per-token activation quant",
            "shapes_MxKxN": [list(s) for s in SHAPES], "out": "bf16", "scales": "fp32 per-row x per-col",
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then {L2_FLUSH_BYTES >> 20} "
                  "MiB read so no dirty lines remain), outside the step events",
            "parallelism": f"replicas x{world} (no data-path collective)"}


def flops(M, K, N):
    return 2.0 * M * N * K


def h100_reference_tflops():
    return sum(flops(*s) for s in SHAPES) / (sum(H100_TORCH_US) * 1e-6) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def _code_only(text):
    """C/C++ source without comments and blank-line or indentation differences, so
    that editing a comment does not count as changing a kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":                       # string / char literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (ln.strip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def source_hash(*rel):
    """Hash of the code (comments and layout ignored) of the given source files."""
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel, current_hash, key="bytes_per_launch"):
    """Per-launch DRAM bytes (read + write) from a committed ncu capture, if it
    was taken on the current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_hash") != current_hash:
        return None
    return d.get(key)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ multi-rank

class L2Flush:
    """Evicts the L2 between timed launches: writes a buffer four times the L2, then
    reads another as large, so that the L2 holds neither the timed kernel's data nor
    dirty lines whose write-back the next kernel would pay for."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink.copy_(self.r.sum())   # a plain fp32 reduction: reads the buffer, writes a scalar


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of per-rank timings over the process group (every
    rank receives the result); the job is as slow as its slowest rank."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_value(world, step_flops, step_ms):
    """Whole-job throughput in TFLOP/s: every rank runs the same step on its own
    GPU (replicas, weak scaling), so the job does world * step_flops per step in
    the slowest rank's step time."""
    return world * step_flops / (step_ms * 1e-3) / 1e12


# ------------------------------------------------------------- GPU bench

def run_gpu(args, rank, world, local_rank):
    import torch
    import fp8_scaled_gemm_mm_gb300 as fm
    from fp8_scaled_gemm_mm_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    fm.lib()

    # ---- set-up: resident inputs, weights quantized once per output channel
    work = []
    for i, (M, K, N) in enumerate(SHAPES):
        X = synth.normal((M, K), 1.0, seed=synth.SEED_A + 10 * i, device=dev)
        W = synth.normal((N, K), 0.02, seed=synth.SEED_B + 10 * i, device=dev)
        B = torch.empty((N, K), dtype=torch.uint8, device=dev)
        b_s = torch.empty((N, 1), dtype=torch.float32, device=dev)
        fm.per_token_group_quant_fp8(W, B, b_s, K)
        del W
        A = torch.empty((M, K), dtype=torch.uint8, device=dev)
        a_s = torch.empty((M, 1), dtype=torch.float32, device=dev)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        work.append(dict(M=M, K=K, N=N, X=X, A=A, a_s=a_s, B=B, b_s=b_s, D=D))
    flush = L2Flush(torch, dev)
    torch.cuda.synchronize()

    step_flops = sum(flops(w["M"], w["K"], w["N"]) for w in work)
    step_quant_bytes = sum(w["M"] * w["K"] * 3 + w["M"] * 4 for w in work)
    n_events = 2 * len(work) + 1

    def step(ev):
        ev[0].record()
        for i, w in enumerate(work):
            fm.per_token_group_quant_fp8(w["X"], w["A"], w["a_s"], w["K"])
            ev[2 * i + 1].record()
            fm.fp8_scaled_mm(w["A"], w["B"], w["a_s"], w["b_s"], fm.A_ROW | fm.B_COL, w["D"])
            ev[2 * i + 2].record()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        flush()
        step([torch.cuda.Event(enable_timing=True) for _ in range(n_events)])
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush()                       # L2 flush between timed steps (not inside them)
        step(evs[k])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if rank == 0 else None

    step_ms, gemm_ms, quant_ms = [], [], []
    per_shape_gemm = [0.0] * len(work)
    for ev in evs:
        step_ms.append(ev[0].elapsed_time(ev[-1]))
        g = q = 0.0
        for i in range(len(work)):
            q += ev[2 * i].elapsed_time(ev[2 * i + 1])
            gi = ev[2 * i + 1].elapsed_time(ev[2 * i + 2])
            g += gi
            per_shape_gemm[i] += gi
        gemm_ms.append(g)
        quant_ms.append(q)
    tot_step_ms = sum(step_ms)
    tot_gemm_ms = sum(gemm_ms)
    tot_quant_ms = sum(quant_ms)
    if world > 1:
        tot_step_ms, tot_gemm_ms, tot_quant_ms = max_over_ranks([tot_step_ms, tot_gemm_ms, tot_quant_ms], dev)

    # ---- group-128 quant on its largest workload (plain and fused), rank 0 only
    quant_obj = None
    if rank == 0:
        quant_obj = bench_group_quant(torch, fm, synth, dev, flush)

    widened = per_tensor = determ = scatter = sweep = tiny = decode = chain = layers_obj = None
    if rank == 0:
        peaks, _ = load_peaks()
        scatter = bench_scatter(torch, fm, synth, dev, flush)
        sweep = bench_quant_sweep(torch, fm, synth, dev, flush, peaks["hbm_gbs"])
        tiny = bench_tiny_config(torch, fm, synth, dev, flush)
        widened = bench_widened(torch, fm, synth, dev, flush, work[0])
        per_tensor = bench_per_tensor(torch, fm, dev, flush)
        determ = bench_deterministic(torch, fm, dev, flush)
        decode = bench_decode_step(torch, fm, synth, dev, flush, peaks["hbm_gbs"])
        chain = bench_decode_chain(torch, fm, dev, flush, peaks["hbm_gbs"])
        layers_obj = bench_decode_layers(torch, fm, dev, flush, peaks["hbm_gbs"])

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if rank == 0 and not args.no_e2e:
        e2e = bench_e2e(torch, fm, work, flush, args)

    res = dict(step_ms=tot_step_ms / args.steps, gemm_ms=tot_gemm_ms / args.steps,
               quant_ms=tot_quant_ms / args.steps, wall=wall, step_flops=step_flops,
               step_quant_bytes=step_quant_bytes, clocks=clocks, quant=quant_obj, e2e=e2e, widened=widened,
               per_tensor=per_tensor, determ=determ, scatter=scatter, sweep=sweep, tiny=tiny, decode=decode, chain=chain, layers=layers_obj,
               per_shape_gemm_ms=[x / args.steps for x in per_shape_gemm], launches=2 * len(work) * args.steps)
    return res


def bench_group_quant(torch, fm, synth, dev, flush, reps=20):
    M, K = QUANT_M, QUANT_K
    out = {}
    for name, fuse in (("plain", False), ("fused_silu_mul", True)):
        x = synth.quant_input(M, 2 * K if fuse else K, torch.bfloat16, seed=5, device=dev)
        q, s = fm.alloc_group_quant_outputs(M, K, 128, fm.SCALE_UE8M0_PACKED, True, device=dev)
        for _ in range(3):
            fm.per_token_group_quant_fp8(x, q, s, 128, fm.SCALE_UE8M0_PACKED, True, fuse)
        ts = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fm.per_token_group_quant_fp8(x, q, s, 128, fm.SCALE_UE8M0_PACKED, True, fuse)
            b.record()
            ts.append((a, b))
        torch.cuda.synchronize()
        us = trimmed_mean([a.elapsed_time(b) for a, b in ts]) * 1e3
        nbytes = M * K * 2 * (2 if fuse else 1) + M * K + (K // 512) * ((M + 3) // 4 * 4) * 4
        out[name] = {"us": round(us, 2), "bytes": nbytes, "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}
    # masked fused SiLU*up quant on the expert-parallel decode layout: 32 local experts
    # of 256 (4096 tokens routed top-8), capacity 256 rows, K = 2048; bytes of the rows
    # that hold tokens only
    import numpy as np
    E, T, KM = 32, 256, 2048
    counts = synth.masked_counts(4096, E)
    xm = synth.quant_input(E * T, 2 * KM, torch.bfloat16, seed=6, device=dev).reshape(E, T, 2 * KM)
    mm = torch.from_numpy(counts).to(dev)
    qm = torch.empty((E, T, KM), dtype=torch.uint8, device=dev)
    sm = torch.empty(fm.masked_scale_shape(E, T, KM, 128, fm.SCALE_UE8M0_PACKED, True), dtype=torch.int32, device=dev)
    for _ in range(3):
        fm.silu_and_mul_masked_post_quant_fp8(xm, mm, qm, sm, 128)
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fm.silu_and_mul_masked_post_quant_fp8(xm, mm, qm, sm, 128)
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    us = trimmed_mean([a.elapsed_time(b) for a, b in ts]) * 1e3
    rows = int(np.asarray(counts).sum())
    nbytes = rows * KM * 5 + rows * (KM // 512) * 4
    out["masked_silu_mul_ep_decode"] = {"us": round(us, 2), "bytes": nbytes, "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                                        "workload": f"E={E} T={T} K={KM}, {rows} token rows"}
    # the same quant as a graph-captured decode runs it: 16 launches on distinct inputs
    # replayed back to back from one CUDA graph (each a programmatic dependent of the one
    # before), per-launch time
    L = 16
    xs = [synth.quant_input(E * T, 2 * KM, torch.bfloat16, seed=60 + i, device=dev).reshape(E, T, 2 * KM)
          for i in range(L)]
    qs = [torch.empty_like(qm) for _ in range(L)]
    ss = [torch.empty_like(sm) for _ in range(L)]
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())

    def chain(stream):
        for i in range(L):
            fm.silu_and_mul_masked_post_quant_fp8(xs[i], mm, qs[i], ss[i], 128, stream=stream)
    with torch.cuda.stream(st):
        chain(st)
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            chain(torch.cuda.current_stream())
    torch.cuda.synchronize()
    tg = []
    for _ in range(10):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        tg.append(a.elapsed_time(b) * 1e3 / L)
    ug = statistics.median(tg)
    out["masked_silu_mul_ep_decode"]["graph_chain_16"] = {"us_per_launch": round(ug, 2),
                                                          "gbs": round(nbytes / (ug * 1e-6) / 1e9, 1)}
    del graph, xs, qs, ss
    return out


def scatter_workload(torch, fm, synth, dev, M=QUANT_M, K=QUANT_K):
    """Topk scatter of the group-128 quant: M tokens of K bf16, each quantized once and
    written to 8 of 256 expert rows (seeded routing, expert regions padded to 128
    rows), UE8M0 scales packed column-major.  Returns (launch, algorithmic bytes):
    2K read and 8 x (K codes + K/512 scale words) written per token."""
    import numpy as np
    x = synth.quant_input(M, K, torch.bfloat16, seed=53, device=dev)
    dst, R = synth.routing(M, topk=8, num_experts=256)
    dst_t = torch.from_numpy(dst).to(dev)
    q, s = fm.alloc_group_quant_outputs(R, K, 128, fm.SCALE_UE8M0_PACKED, True, device=dev)
    written = int(np.count_nonzero(dst >= 0))
    nbytes = M * K * 2 + written * (K + (K // 512) * 4) + dst.size * 4

    def launch():
        fm.per_token_group_quant_fp8_scatter(x, dst_t, q, s, 128, fm.SCALE_UE8M0_PACKED, True)
    return launch, nbytes, R


def bench_scatter(torch, fm, synth, dev, flush, reps=20):
    launch, nbytes, R = scatter_workload(torch, fm, synth, dev)
    us = _median_us(torch, flush, launch, reps)
    return {"workload": f"M={QUANT_M} K={QUANT_K} bf16, group 128, topk 8 of 256 experts -> {R} rows, UE8M0 "
                        "packed column-major scales", "us": round(us, 2), "bytes": nbytes,
            "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}


def bench_quant_sweep(torch, fm, synth, dev, flush, hbm_peak, reps=10):
    """Every standalone group-quant cell of the quant configuration: tokens M in
    1, 64, 512, 8192; hidden K in 2048, 7168; bf16 and fp16; fp32 row-major and UE8M0
    packed column-major scales; group 128.  Cells whose ideal time at the HBM peak is
    under 5 us are marked launch-bound (an empty launch measures a few us this way)."""
    out = []
    for K in (2048, 7168):
        for M in (1, 64, 512, 8192):
            for dt_name, dt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
                x = synth.quant_input(M, K, dt, seed=200 + M + K, device=dev)
                for fmt_name, fmt, cm in (("fp32_rowmajor", fm.SCALE_FP32, False),
                                          ("ue8m0_colmajor", fm.SCALE_UE8M0_PACKED, True)):
                    q, sc = fm.alloc_group_quant_outputs(M, K, 128, fmt, cm, device=dev)
                    us = _median_us(torch, flush, lambda: fm.per_token_group_quant_fp8(x, q, sc, 128, fmt, cm), reps)
                    nbytes = M * K * 3 + sc.numel() * 4
                    ideal = nbytes / (hbm_peak * 1e9) * 1e6
                    out.append({"M": M, "K": K, "dtype": dt_name, "scales": fmt_name, "us": round(us, 2),
                                "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                                "frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4),
                                "bound": "launch" if ideal < 5.0 else "hbm"})
    return out


def bench_tiny_config(torch, fm, synth, dev, flush, reps=20):
    """The tiny rowwise configuration: X bf16 [64, 512] group-128 quantized (fp32
    scales), then the GEMM against a per-channel-quantized W [256, 512] with the
    per-group A scales.  Launch-bound at this size; reported in us per launch."""
    M, N, K = 64, 256, 512
    X = synth.normal((M, K), 1.0, seed=synth.SEED_A, device=dev)
    W = synth.normal((N, K), 0.02, seed=synth.SEED_B, device=dev)
    B = torch.empty((N, K), dtype=torch.uint8, device=dev)
    b_s = torch.empty((N, 1), dtype=torch.float32, device=dev)
    fm.per_token_group_quant_fp8(W, B, b_s, K)
    A = torch.empty((M, K), dtype=torch.uint8, device=dev)
    a_s = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    q_us = _median_us(torch, flush, lambda: fm.per_token_group_quant_fp8(X, A, a_s, 128), reps)
    g_us = _median_us(torch, flush, lambda: fm.fp8_scaled_mm(A, B, a_s, b_s, fm.A_GROUP128 | fm.B_COL, D), reps)
    return {"workload": "X [64,512] group-128 quant + GEMM with W [256,512], group-128 A x per-column B scales",
            "quant_us": round(q_us, 2), "gemm_us": round(g_us, 2),
            "gemm_tflops": round(flops(M, K, N) / (g_us * 1e-6) / 1e12, 3), "bound": "launch"}


def trimmed_mean(xs):
    """Mean of the middle half of the samples.  Event timestamps on this part come in
    steps of about 2 us, so a median of a few-us kernel sits on one step; the mean of
    many samples whose phase against the steps varies resolves finer."""
    xs = sorted(xs)
    q = len(xs) // 4
    mid = xs[q:len(xs) - q] or xs
    return sum(mid) / len(mid)


def _median_us(torch, flush, fn, reps):
    """Event-timed launch of fn, the L2 evicted before each; trimmed mean in us (at
    least 40 samples for launches shorter than 50 us)."""
    for _ in range(3):
        fn()
    ts = []
    n = reps
    for i in range(max(reps, 40)):
        if i == reps and ts:
            torch.cuda.synchronize()
            if min(a.elapsed_time(b) for a, b in ts) * 1e3 > 50.0:
                break
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    return trimmed_mean([a.elapsed_time(b) for a, b in ts]) * 1e3


def bench_widened(torch, fm, synth, dev, flush, w0, reps=10):
    """The paths beyond the headline step, each alone on one workload:
    block-scaled GEMM (A 1x128 UE8M0 group scales x B 128x128 block scales) on the
    first prefill shape, and the HBM-bound quant variants on M=8192, K=7168."""
    out = {}
    M, K, N = w0["M"], w0["K"], w0["N"]
    words = fm.scale_shape(M, K, 128, fm.SCALE_UE8M0_PACKED, True)
    a_w = torch.empty(words, dtype=torch.int32, device=dev)
    A = torch.empty((M, K), dtype=torch.uint8, device=dev)
    fm.per_token_group_quant_fp8(w0["X"], A, a_w, 128, fm.SCALE_UE8M0_PACKED, True)
    b_blk = torch.rand(((N + 127) // 128, K // 128), generator=torch.Generator(device=dev).manual_seed(7),
                       device=dev) * 1e-3 + 1e-4
    us = _median_us(torch, flush, lambda: fm.fp8_scaled_mm(A, w0["B"], a_w, b_blk, fm.A_GROUP128_UE8M0 | fm.B_BLOCK128,
                                                           w0["D"]), reps)
    out["block_scaled_gemm"] = {"workload": f"{M}x{K}x{N}, A group-128 UE8M0 (packed, column-major) x B 128x128 fp32",
                                "us": round(us, 1), "tflops": round(flops(M, K, N) / (us * 1e-6) / 1e12, 1)}
    del A, a_w
    QM, QK = QUANT_M, QUANT_K
    x = synth.quant_input(QM, QK, torch.bfloat16, seed=8, device=dev)
    q = torch.empty((QM, QK), dtype=torch.uint8, device=dev)
    sc = torch.full((1,), 0.01, dtype=torch.float32, device=dev)
    us = _median_us(torch, flush, lambda: fm.static_per_tensor_quant_fp8(x, sc, q), reps)
    out["static_per_tensor_quant"] = {"workload": f"{QM}x{QK} bf16", "us": round(us, 2), "bytes": QM * QK * 3}
    qi = q.view(torch.int8)
    si = torch.empty(fm.scale_shape(QM, QK, 128, fm.SCALE_FP32, True), dtype=torch.float32, device=dev)
    us = _median_us(torch, flush, lambda: fm.per_token_group_quant_int8(x, qi, si, 128, True), reps)
    out["int8_group_quant"] = {"workload": f"{QM}x{QK} bf16, group 128, fp32 column-major scales",
                               "us": round(us, 2), "bytes": QM * QK * 3 + si.numel() * 4}
    MP = QM
    xs = x[: QM - 192]
    sp = torch.empty(fm.scale_shape(MP, QK, 128, fm.SCALE_FP32, True), dtype=torch.float32, device=dev)
    us = _median_us(torch, flush, lambda: fm.per_token_group_quant_fp8_row_padded(xs, q, sp, 128), reps)
    out["row_padded_group_quant"] = {"workload": f"M={QM - 192} padded to {MP}, K={QK} bf16, group 128, fp32 "
                                                 "column-major scales", "us": round(us, 2),
                                     "bytes": (QM - 192) * QK * 2 + MP * QK + sp.numel() * 4}
    del x, xs, q, sp, si
    NW, KW = 2 * 14336, 4096
    w = torch.randint(0, 126, (NW, KW), generator=torch.Generator(device=dev).manual_seed(9), dtype=torch.uint8,
                      device=dev)
    w_out = torch.empty_like(w)
    ss = torch.tensor([0.011, 0.013], dtype=torch.float32, device=dev)
    us = _median_us(torch, flush, lambda: fm.requantize_with_max_scale_fp8(w, ss, [14336, 14336], w_out=w_out), reps)
    out["requantize_with_max_scale"] = {"workload": f"gate/up weight {NW}x{KW}, 2 shards", "us": round(us, 2),
                                        "bytes": NW * KW * 2}
    for v in out.values():
        if "bytes" in v:
            v["gbs"] = round(v["bytes"] / (v["us"] * 1e-6) / 1e9, 1)
    return out


def bench_per_tensor(torch, fm, dev, flush, reps=10):
    """Per-tensor scaled GEMMs at K = 4096 for every (M, N) of the per-tensor
    configuration (M in 1, 16, 128, 2048, 8192; N in 4096, 12288, 14336), L2 flushed
    before each timed launch.  M <= 128 is HBM-bound (the weight streams once),
    larger M tensor-bound."""
    K = 4096
    g = torch.Generator(device=dev).manual_seed(11)
    out = []
    for N in (4096, 12288, 14336):
        B = torch.randint(0, 126, (N, K), generator=g, dtype=torch.uint8, device=dev)
        for M in (1, 16, 128, 2048, 8192):
            A = torch.randint(0, 126, (M, K), generator=g, dtype=torch.uint8, device=dev)
            a_s = torch.full((1,), 0.02, dtype=torch.float32, device=dev)
            b_s = torch.full((1,), 0.001, dtype=torch.float32, device=dev)
            D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            us = _median_us(torch, flush, lambda: fm.fp8_scaled_mm(A, B, a_s, b_s, fm.A_TENSOR | fm.B_TENSOR, D),
                            reps)
            nbytes = M * K + N * K + 2 * M * N
            out.append({"M": M, "N": N, "K": K, "us": round(us, 2),
                        "tflops": round(flops(M, K, N) / (us * 1e-6) / 1e12, 1),
                        "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "bound": "hbm" if M <= 128 else "tensor"})
            del A, D
        del B
    return out


def bench_decode_step(torch, fm, synth, dev, flush, hbm_peak, reps=10):
    """Decode-shaped linear, K = 4096: the per-token quant of x [M, K] bf16 (one fp32
    scale per row) followed by the rowwise GEMM against a per-channel E4M3 weight
    [N, K], timed as one pair (the GEMM is launched as a programmatic dependent of the
    quant, so its set-up and first weight prefetches overlap the quant's end), next to
    each kernel alone.  Bytes: x read, codes and scales written and read back, the
    weight and the bf16 output."""
    K = 4096
    out = []
    for N in (4096, 14336):
        W = synth.normal((N, K), 0.02, seed=41, device=dev)
        B = torch.empty((N, K), dtype=torch.uint8, device=dev)
        b_s = torch.empty((N, 1), dtype=torch.float32, device=dev)
        fm.per_token_group_quant_fp8(W, B, b_s, K)
        del W
        for M in (1, 16, 64):
            x = synth.normal((M, K), 1.0, seed=42 + M, device=dev)
            A = torch.empty((M, K), dtype=torch.uint8, device=dev)
            a_s = torch.empty((M, 1), dtype=torch.float32, device=dev)
            D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            quant = lambda: fm.per_token_group_quant_fp8(x, A, a_s, K)
            gemm = lambda: fm.fp8_scaled_mm(A, B, a_s, b_s, fm.A_ROW | fm.B_COL, D)

            def pair():
                quant()
                gemm()
            t_pair = _median_us(torch, flush, pair, reps)
            t_q = _median_us(torch, flush, quant, reps)
            t_g = _median_us(torch, flush, gemm, reps)
            nbytes = 2 * M * K + 2 * (M * K + 4 * M) + N * K + 4 * N + 2 * M * N
            out.append({"M": M, "N": N, "K": K, "us_pair": round(t_pair, 2), "us_quant_alone": round(t_q, 2),
                        "us_gemm_alone": round(t_g, 2), "gbs": round(nbytes / (t_pair * 1e-6) / 1e9, 1),
                        "frac": round(nbytes / (t_pair * 1e-6) / 1e9 / hbm_peak, 4)})
            del x, A, a_s, D
        del B, b_s
    return out


def bench_decode_chain(torch, fm, dev, flush, hbm_peak, layers=16, reps=10):
    """A decode step's chain of GEMMs, K = 4096: x [M, K] against `layers` distinct
    per-tensor-scaled E4M3 weights [N, K] (layers x N x K bytes, far beyond L2),
    launched back to back and replayed from one CUDA graph; each GEMM is a
    programmatic dependent of the one before, whose early trigger lets it set up and
    prefetch weight tiles while that one finishes.  Per-GEMM time = replay time /
    layers (L2 evicted before each replay); bytes per GEMM: weight, x and the bf16
    output."""
    K = 4096
    g = torch.Generator(device=dev).manual_seed(17)
    out = []
    for N in (4096, 14336):
        Ws = [torch.randint(0, 126, (N, K), generator=g, dtype=torch.uint8, device=dev) for _ in range(layers)]
        for M in (1, 16):
            x = torch.randint(0, 126, (M, K), generator=g, dtype=torch.uint8, device=dev)
            a_s = torch.full((1,), 0.02, dtype=torch.float32, device=dev)
            b_s = torch.full((1,), 0.001, dtype=torch.float32, device=dev)
            outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(layers)]
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())

            def chain(stream):
                for i in range(layers):
                    fm.fp8_scaled_mm(x, Ws[i], a_s, b_s, fm.A_TENSOR | fm.B_TENSOR, outs[i], stream=stream)
            with torch.cuda.stream(st):
                chain(st)                 # set-up outside the capture
                st.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=st):
                    chain(torch.cuda.current_stream())
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                graph.replay()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            us = statistics.median(ts) / layers
            nbytes = N * K + M * K + 2 * M * N
            out.append({"M": M, "N": N, "K": K, "layers": layers, "us_per_gemm": round(us, 2),
                        "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                        "frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4)})
            del graph, x, outs
        del Ws
        torch.cuda.empty_cache()
    return out


def bench_decode_layers(torch, fm, dev, flush, hbm_peak, layers=16, reps=10):
    """A decode step's chain of linear layers, K = 4096: per layer the per-token quant
    of its activation x_i [M, K] bf16 (one fp32 scale per row) and the rowwise GEMM
    against its own per-channel E4M3 weight [N, K]; `layers` layers back to back,
    replayed from one CUDA graph, every kernel a programmatic dependent of the one
    before.  Per-layer time = replay time / layers (L2 evicted before each replay);
    bytes per layer: x read, codes and scales written and read back, the weight and
    the bf16 output."""
    K = 4096
    g = torch.Generator(device=dev).manual_seed(23)
    out = []
    for N in (4096, 14336):
        Ws = [torch.randint(0, 126, (N, K), generator=g, dtype=torch.uint8, device=dev) for _ in range(layers)]
        bs = torch.full((N, 1), 0.001, dtype=torch.float32, device=dev)
        for M in (1, 16):
            xs = [torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16) for _ in range(layers)]
            As = [torch.empty((M, K), dtype=torch.uint8, device=dev) for _ in range(layers)]
            ass = [torch.empty((M, 1), dtype=torch.float32, device=dev) for _ in range(layers)]
            outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(layers)]
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())

            def chain(stream):
                for i in range(layers):
                    fm.per_token_group_quant_fp8(xs[i], As[i], ass[i], K, stream=stream)
                    fm.fp8_scaled_mm(As[i], Ws[i], ass[i], bs, fm.A_ROW | fm.B_COL, outs[i], stream=stream)
            with torch.cuda.stream(st):
                chain(st)                 # set-up outside the capture
                st.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=st):
                    chain(torch.cuda.current_stream())
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                graph.replay()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            us = statistics.median(ts) / layers
            nbytes = 2 * M * K + 2 * (M * K + 4 * M) + N * K + 4 * N + 2 * M * N
            out.append({"M": M, "N": N, "K": K, "layers": layers, "us_per_layer": round(us, 2),
                        "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                        "frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4)})
            del graph, xs, As, ass, outs
        del Ws
        torch.cuda.empty_cache()
    return out


def bench_deterministic(torch, fm, dev, flush, reps=10):
    """Cost of the deterministic (batch-invariant) mode on the deterministic
    configuration's shapes (K = 4096, N in 64, 4096, lda = K + 64, bf16 out with
    bias): event-timed normal and deterministic launches, L2 flushed before each."""
    g = torch.Generator(device=dev).manual_seed(12)
    out = []
    K = 4096
    for N in (64, 4096):
        B = torch.randint(0, 126, (N, K), generator=g, dtype=torch.uint8, device=dev)
        b_s = torch.rand((N, 1), generator=g, device=dev) * 1e-3
        bias = (torch.rand((N,), generator=g, device=dev) - 0.5).to(torch.bfloat16)
        for M in (1, 16, 128, 1024, 4096):
            A = torch.randint(0, 126, (M, K + 64), generator=g, dtype=torch.uint8, device=dev)
            a_s = torch.rand((M, 1), generator=g, device=dev) + 0.5
            D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            t = {}
            for det in (False, True):
                t[det] = _median_us(torch, flush, lambda: fm.fp8_scaled_mm(A, B, a_s, b_s, fm.A_ROW | fm.B_COL, D,
                                                                           bias=bias, deterministic=det, K=K), reps)
            out.append({"M": M, "N": N, "K": K, "us": round(t[False], 2), "us_deterministic": round(t[True], 2),
                        "ratio": round(t[True] / t[False], 3)})
    return out


def bench_e2e(torch, fm, work, flush, args):
    """Same step through the C ABI from pinned host buffers: H2D of each
    activation, quant + GEMM, D2H of each output, all inside the timed region.
    Copies in, compute and copies out run on three streams ordered by events, so
    the copy of shape i+1's activation and of shape i-1's output overlap the
    GEMM of shape i (every shape has its own buffers)."""
    host_x = [torch.empty(w["X"].shape, dtype=torch.bfloat16, pin_memory=True) for w in work]
    for hx, w in zip(host_x, work):
        hx.copy_(w["X"].cpu())
    host_d = [torch.empty(w["D"].shape, dtype=torch.bfloat16, pin_memory=True) for w in work]
    h2d = sum(h.numel() * 2 for h in host_x)
    d2h = sum(h.numel() * 2 for h in host_d)
    steps = max(3, min(args.steps, 10))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_cmp = torch.cuda.current_stream()

    def one():
        ev_in = [torch.cuda.Event() for _ in work]
        ev_cmp = [torch.cuda.Event() for _ in work]
        with torch.cuda.stream(s_in):
            for i, (hx, w) in enumerate(zip(host_x, work)):
                w["X"].copy_(hx, non_blocking=True)
                ev_in[i].record(s_in)
        for i, w in enumerate(work):
            s_cmp.wait_event(ev_in[i])
            fm.per_token_group_quant_fp8(w["X"], w["A"], w["a_s"], w["K"], stream=s_cmp)
            fm.fp8_scaled_mm(w["A"], w["B"], w["a_s"], w["b_s"], fm.A_ROW | fm.B_COL, w["D"], stream=s_cmp)
            ev_cmp[i].record(s_cmp)
        with torch.cuda.stream(s_out):
            for i, (hd, w) in enumerate(zip(host_d, work)):
                s_out.wait_event(ev_cmp[i])
                hd.copy_(w["D"], non_blocking=True)

    one()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        one()
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    step_flops = sum(flops(w["M"], w["K"], w["N"]) for w in work)
    return {"value": round(step_flops / t / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(t * 1e3, 3), "steps": steps}


# ---------------------------------------------------- single-kernel cases

def _widened_case(torch, fm, synth, dev, case):
    """(launch, bytes) of one widened kernel on the workload bench_widened times."""
    QM, QK = QUANT_M, QUANT_K
    if case == "quant_masked":
        E, T, KM = 32, 256, 2048
        counts = synth.masked_counts(4096, E)
        xm = synth.quant_input(E * T, 2 * KM, torch.bfloat16, seed=6, device=dev).reshape(E, T, 2 * KM)
        mm = torch.from_numpy(counts).to(dev)
        qm = torch.empty((E, T, KM), dtype=torch.uint8, device=dev)
        sm = torch.empty(fm.masked_scale_shape(E, T, KM, 128, fm.SCALE_UE8M0_PACKED, True), dtype=torch.int32,
                         device=dev)
        rows = int(counts.sum())
        return (lambda: fm.silu_and_mul_masked_post_quant_fp8(xm, mm, qm, sm, 128)), rows * KM * 5 + rows * (KM // 512) * 4
    if case == "requant":
        NW, KW = 2 * 14336, 4096
        w = torch.randint(0, 126, (NW, KW), generator=torch.Generator(device=dev).manual_seed(9), dtype=torch.uint8,
                          device=dev)
        w_out = torch.empty_like(w)
        ss = torch.tensor([0.011, 0.013], dtype=torch.float32, device=dev)
        return (lambda: fm.requantize_with_max_scale_fp8(w, ss, [14336, 14336], w_out=w_out)), NW * KW * 2
    x = synth.quant_input(QM, QK, torch.bfloat16, seed=8, device=dev)
    q = torch.empty((QM, QK), dtype=torch.uint8, device=dev)
    if case == "static_quant":
        sc = torch.full((1,), 0.01, dtype=torch.float32, device=dev)
        return (lambda: fm.static_per_tensor_quant_fp8(x, sc, q)), QM * QK * 3
    if case == "quant_int8":
        si = torch.empty(fm.scale_shape(QM, QK, 128, fm.SCALE_FP32, True), dtype=torch.float32, device=dev)
        qi = q.view(torch.int8)
        return (lambda: fm.per_token_group_quant_int8(x, qi, si, 128, True)), QM * QK * 3 + si.numel() * 4
    xs = x[: QM - 192]
    sp = torch.empty(fm.scale_shape(QM, QK, 128, fm.SCALE_FP32, True), dtype=torch.float32, device=dev)
    return ((lambda: fm.per_token_group_quant_fp8_row_padded(xs, q, sp, 128)),
            (QM - 192) * QK * 2 + QM * QK + sp.numel() * 4)


def run_kernel_case(args):
    """Launch one kernel on its workload warmup + steps times (for profilers)
    and print its event-timed median.  gemm: a prefill shape (--shape, default
    8320x5376x21504) or --mnk M,K,N, rowwise scales; gemm_block: the same
    shapes with group-128 UE8M0 A scales and 128x128 B block scales; quant / quant_fused:
    group-128 quant of M=8192, K=7168 bf16 with UE8M0 packed column-major
    scales; quant_masked: the masked fused quant on the EP decode layout (E=32,
    T=256, K=2048); quant_int8 / quant_row_padded / static_quant / requant: the
    widened paths on the workloads the benchmark reports for them."""
    import torch
    import fp8_scaled_gemm_mm_gb300 as fm
    from fp8_scaled_gemm_mm_gb300 import synth
    dev = torch.device("cuda", 0)
    if args.kernel_case in ("gemm", "gemm_block"):
        M, K, N = SHAPES[args.shape] if not args.mnk else tuple(int(v) for v in args.mnk.split(","))
        X = synth.normal((M, K), 1.0, seed=1, device=dev)
        W = synth.normal((N, K), 0.02, seed=2, device=dev)
        A = torch.empty((M, K), dtype=torch.uint8, device=dev)
        B = torch.empty((N, K), dtype=torch.uint8, device=dev)
        a_s = torch.empty((M, 1), dtype=torch.float32, device=dev)
        b_s = torch.empty((N, 1), dtype=torch.float32, device=dev)
        fm.per_token_group_quant_fp8(X, A, a_s, K)
        fm.per_token_group_quant_fp8(W, B, b_s, K)
        del X, W
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        work = flops(M, K, N)

        def launch():
            fm.fp8_scaled_mm(A, B, a_s, b_s, fm.A_ROW | fm.B_COL, D, deterministic=args.deterministic)

        if args.kernel_case == "gemm_block":
            a_s = torch.empty(fm.scale_shape(M, K, 128, fm.SCALE_UE8M0_PACKED, True), dtype=torch.int32, device=dev)
            X = synth.normal((M, K), 1.0, seed=1, device=dev)
            fm.per_token_group_quant_fp8(X, A, a_s, 128, fm.SCALE_UE8M0_PACKED, True)
            del X
            b_s = torch.rand(((N + 127) // 128, K // 128), generator=torch.Generator(device=dev).manual_seed(7),
                             device=dev) * 1e-3 + 1e-4

            def launch():
                fm.fp8_scaled_mm(A, B, a_s, b_s, fm.A_GROUP128_UE8M0 | fm.B_BLOCK128, D)
    elif args.kernel_case in ("quant_masked", "quant_int8", "quant_row_padded", "static_quant", "requant"):
        launch, work = _widened_case(torch, fm, synth, dev, args.kernel_case)
    elif args.kernel_case == "scatter":
        launch, work, _ = scatter_workload(torch, fm, synth, dev)
    else:
        fuse = args.kernel_case == "quant_fused"
        M, K = QUANT_M, QUANT_K
        x = synth.quant_input(M, 2 * K if fuse else K, torch.bfloat16, seed=5, device=dev)
        q, s = fm.alloc_group_quant_outputs(M, K, 128, fm.SCALE_UE8M0_PACKED, True, device=dev)
        work = M * K * 2 * (2 if fuse else 1) + M * K + (K // 512) * ((M + 3) // 4 * 4) * 4

        def launch():
            fm.per_token_group_quant_fp8(x, q, s, 128, fm.SCALE_UE8M0_PACKED, True, fuse)
    for _ in range(args.warmup):
        launch()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in ts) * 1e3
    is_gemm = args.kernel_case.startswith("gemm")
    rate = work / (us * 1e-6) / (1e12 if is_gemm else 1e9)
    print(json.dumps({"kernel_case": args.kernel_case, "us": round(us, 2),
                      ("tflops" if is_gemm else "gbs"): round(rate, 1)}), flush=True)
    return 0


# --------------------------------------------------------- CPU reference

_ORACLE_WEIGHTS = {}


def oracle_sample(rows_per_shape, seed=0):
    """Run the oracle's quant + GEMM on `rows_per_shape` rows of every shape.
    Returns (flops done, seconds, threads)."""
    import oracle
    from fp8_scaled_gemm_mm_gb300 import synth
    done = 0.0
    elapsed = 0.0
    threads = oracle.num_threads()
    for i, (M, K, N) in enumerate(SHAPES):
        X = synth.to_bits(synth.normal((rows_per_shape, K), 1.0, seed=1000 + 10 * seed + i))
        if i not in _ORACLE_WEIGHTS:              # weight preparation: once, not timed
            W = synth.to_bits(synth.normal((N, K), 0.02, seed=2000 + i))
            _ORACLE_WEIGHTS[i] = oracle.quantize_rows(W)
        B, b_s = _ORACLE_WEIGHTS[i]
        t0 = time.perf_counter()
        A, a_s = oracle.quantize_rows(X)
        oracle.gemm(A, B, a_s, b_s, oracle.A_ROW, oracle.B_COL, threads=threads)
        elapsed += time.perf_counter() - t0
        done += flops(rows_per_shape, K, N)
    return done, elapsed, threads


def cpu_baseline(rows_per_shape):
    done, sec, threads = oracle_sample(rows_per_shape)
    return {"value": round(done / sec / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows_per_shape} rows of each of the 5 shapes: per-row quant + fp64 GEMM over all N "
                      f"({done / 1e9:.1f} GFLOP, {sec:.1f} s)"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(rows)
    tot_f = tot_s = 0.0
    threads = 1
    t_wall = time.perf_counter()
    for k in range(args.steps):
        f, s, threads = oracle_sample(rows, seed=k)
        tot_f += f
        tot_s += s
    wall = time.perf_counter() - t_wall
    value = tot_f / tot_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows of each of the 5 shapes per step (per-row quant + fp64 GEMM over "
                                   "all N); the oracle times a bounded sample of the workload"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2),
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=480, help="oracle rows per shape for cpu_baseline")
    ap.add_argument("--ref-rows", type=int, default=16, help="oracle rows per shape per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernel-case", choices=["gemm", "gemm_block", "quant", "quant_fused", "quant_masked",
                                              "quant_int8", "quant_row_padded", "static_quant", "requant",
                                              "scatter"],
                    default=None,
                    help="run a single kernel on its workload (for profilers) instead of the benchmark")
    ap.add_argument("--shape", type=int, default=0, help="prefill shape index for --kernel-case gemm")
    ap.add_argument("--mnk", default=None, help="M,K,N for --kernel-case gemm instead of a prefill shape")
    ap.add_argument("--deterministic", action="store_true", help="--kernel-case gemm in the batch-invariant mode")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.kernel_case:
        return run_kernel_case(args)

    import torch
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    res = run_gpu(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return 0

    peaks, peak_kind = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    hbm_peak = peaks["hbm_gbs"]
    value = job_value(world, res["step_flops"], res["step_ms"])
    gemm_tflops = res["step_flops"] / (res["gemm_ms"] * 1e-3) / 1e12
    quant_gbs = res["step_quant_bytes"] / (res["quant_ms"] * 1e-3) / 1e9
    ghash = source_hash("fp8_scaled_gemm_mm_gb300/csrc/gemm.cu", "fp8_scaled_gemm_mm_gb300/csrc/ptx.cuh")
    qhash = source_hash("fp8_scaled_gemm_mm_gb300/csrc/quant.cu", "fp8_scaled_gemm_mm_gb300/csrc/ptx.cuh")
    traffic = load_traffic("gemm", ghash)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["step_ms"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / world / h100_reference_tflops(), 3),
        "vs_baseline_note": "per-GPU value / torch._scaled_mm on H100 80GB for the same five shapes "
                            f"({h100_reference_tflops():.0f} TFLOP/s, sglang PR #34318 kernel table; other hardware)",
        "dtype": "e4m3 x e4m3 -> fp32 accumulate -> bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, bf16, quantized on device)",
        "config": workload_config(world),
        "gemm": {"tflops": round(gemm_tflops, 2), "ms_per_step": round(res["gemm_ms"], 4),
                 "frac_of_measured_peak": round(gemm_tflops / fp8_peak, 4),
                 "frac_of_nominal_dense_fp8": round(gemm_tflops / NOMINAL_FP8_DENSE_TFLOPS, 4),
                 "per_shape_tflops": [round(flops(*s) / (t * 1e-3) / 1e12, 1)
                                      for s, t in zip(SHAPES, res["per_shape_gemm_ms"])]},
        "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 2), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                     "traffic": traffic,
                     "peak_note": f"{peak_kind} bf16 burst {peaks['bf16_tflops']} TFLOP/s x {FP8_OVER_BF16} "
                                  "(nominal fp8:bf16 dense ratio)",
                     "traffic_note": "dram read+write bytes of one launch of the 8320x5376x21504 shape (ncu)",
                     "kernel": "fp8_gemm_kernel", "source_hash": ghash},
        "activation_quant": {"gbs": round(quant_gbs, 1), "frac_hbm": round(quant_gbs / hbm_peak, 4),
                             "ms_per_step": round(res["quant_ms"], 4)},
        "group_quant": None,
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "e2e": res["e2e"],
        "cpu_baseline": None,
        "wall_s": round(res["wall"], 3),
    }
    if res["quant"]:
        gq = res["quant"]
        line["group_quant"] = {
            "workload": f"M={QUANT_M} K={QUANT_K} bf16, group 128, UE8M0 packed column-major scales",
            "bound": "hbm", "peak_gbs": hbm_peak, "source_hash": qhash,
            **{k: dict(v, frac=round(v["gbs"] / hbm_peak, 4)) for k, v in gq.items()}}
        gc = line["group_quant"]["masked_silu_mul_ep_decode"].get("graph_chain_16")
        if gc:
            gc["frac"] = round(gc["gbs"] / hbm_peak, 4)
        line["group_quant"]["plain"]["traffic"] = load_traffic("group_quant", qhash)
        line["group_quant"]["fused_silu_mul"]["traffic"] = load_traffic("group_quant", qhash,
                                                                        "fused_bytes_per_launch")
    if res["scatter"]:
        sc = dict(res["scatter"])
        sc["frac"] = round(sc["gbs"] / hbm_peak, 4)
        sc["bound"] = "hbm"
        sc["traffic"] = load_traffic("scatter", qhash)
        line["scatter"] = sc
    if res["sweep"]:
        line["group_quant_sweep"] = {"note": "every standalone quant cell (group 128), event-timed, L2 flushed before "
                                             "each launch; frac of the HBM peak", "cells": res["sweep"]}
    if res["tiny"]:
        line["tiny_group_gemm"] = res["tiny"]
    if res["decode"]:
        line["decode_step_k4096"] = {"note": "per-token quant + rowwise GEMM timed as one pair (the GEMM a "
                                             "programmatic dependent of the quant) and each alone; L2 flushed "
                                             "before each; frac of the HBM peak for the pair's bytes",
                                     "shapes": res["decode"]}
    if res.get("chain"):
        line["decode_chain_k4096"] = {"note": "16 decode GEMMs (distinct per-tensor-scaled weights) back to back in one "
                                              "CUDA graph, each a programmatic dependent of the one before; per-GEMM "
                                              "time, L2 evicted before each replay; frac of HBM",
                                      "shapes": res["chain"]}
    if res.get("layers"):
        line["decode_layers_k4096"] = {"note": "16 decode layers (per-token quant + rowwise GEMM, own weights) back to "
                                               "back in one CUDA graph, every kernel a programmatic dependent of the one "
                                               "before; per-layer time, L2 evicted before each replay; frac of HBM",
                                       "shapes": res["layers"]}
    if res["widened"]:
        wd = res["widened"]
        for k, v in wd.items():
            if "gbs" in v:
                v["frac_hbm"] = round(v["gbs"] / hbm_peak, 4)
            if "tflops" in v:
                v["frac_fp8_peak"] = round(v["tflops"] / fp8_peak, 4)
        line["widened"] = wd
    if res["per_tensor"]:
        for v in res["per_tensor"]:
            v["frac"] = round(v["gbs"] / hbm_peak if v["bound"] == "hbm" else v["tflops"] / fp8_peak, 4)
        line["per_tensor_k4096"] = {"note": "per-tensor scales, L2 flushed before each launch, event-timed; "
                                            "frac of HBM (M <= 128) or of the FP8 peak", "shapes": res["per_tensor"]}
    if res["determ"]:
        line["deterministic_cost_k4096"] = {"note": "rowwise scales, bias, lda = K + 64; event-timed normal vs "
                                                    "deterministic launches, L2 flushed before each",
                                            "shapes": res["determ"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_rows)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
