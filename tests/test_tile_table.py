"""The GEMM planner's host logic, on the CPU: the shape-keyed tile table and the
split count of the small-M path (tests/c_abi/tile_table.cu compiles the
library's sources into a host program that answers plan queries; no kernel
runs).

Checked: deterministic mode picks its tile from N alone, so every M (every
prefix or suffix of the rows) runs the same tile and reduction (sglang PR #44861,
Modifications: fixed reduction tiles); group scales always take the group
kernel's tile; the widest tile wins wherever it fills the machine; the split
count keeps each of its stated limits and is the largest that does."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BK = 128
SMS = 152


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is needed to build the planner probe")
    exe = str(tmp_path_factory.mktemp("tile_table") / "tile_table")
    # device code to PTX only (no ptxas): the probe calls host functions alone
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=compute_103a", "-std=c++17",
                           "--expt-relaxed-constexpr", "-w", "-I", os.path.join(ROOT, "include"), "-o", exe,
                           os.path.join(ROOT, "tests", "c_abi", "tile_table.cu")])

    def ask(lines):
        r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
        return [tuple(int(v) for v in ln.split()) for ln in r.stdout.strip().splitlines()]
    return ask


def _configs(plan, shapes, det=0, group=0, sms=SMS):
    return plan([f"config {M} {N} {det} {group} {sms}" for M, N in shapes])


def test_deterministic_tile_depends_on_n_only(plan):
    Ms = [1, 2, 7, 16, 37, 64, 100, 101, 128, 129, 1000, 4096, 23216]
    for N in (64, 128, 256, 1024, 4096, 14336, 28672):
        got = set(_configs(plan, [(M, N) for M in Ms], det=1))
        assert len(got) == 1, (N, got)
        bn, _ = got.pop()
        assert bn in (64, 128, 256)
    # and it does not depend on the machine size either
    assert _configs(plan, [(512, 4096)], det=1, sms=148) == _configs(plan, [(512, 4096)], det=1, sms=SMS)


def test_group_scales_take_the_group_tile(plan):
    got = set(_configs(plan, [(M, N) for M in (1, 64, 8320) for N in (256, 5376, 28672)], group=1))
    assert got == {(256, 4)}


def test_prefill_shapes_take_the_widest_tile(plan):
    # the five prefill shapes fill every wave of 128 x 256 tiles almost exactly
    shapes = [(8320, 21504), (8320, 14336), (23216, 28672), (15760, 28672), (8320, 5376)]
    assert all(bn == 256 for bn, _ in _configs(plan, shapes))


def test_narrow_tiles_only_when_they_save_a_wave(plan):
    # a narrower tile is chosen only if it needs fewer waves than 256-wide tiles, if the
    # 256-wide tiles fit in one partly idle wave (narrower ones then use more SMs), or if
    # in the same number of waves it leaves fewer SMs idle in the last one (M = 2048,
    # N = 4096: 256 tiles of 256 columns are 1.68 waves, 304 tiles of 224 exactly 2)
    for M in (256, 384, 1024, 2048, 8192):
        for N in (512, 1024, 1536, 2048, 4096, 12288, 14336):
            (bn, _), = _configs(plan, [(M, N)])
            if bn != 256:
                mblk = -(-M // 128)
                tiles = lambda w: mblk * -(-N // w)
                waves = lambda w: -(-tiles(w) // SMS)
                fill = lambda w: tiles(w) / (waves(w) * SMS)
                assert waves(bn) <= waves(256), (M, N, bn)
                assert waves(bn) < waves(256) or waves(256) == 1 or fill(bn) > fill(256), (M, N, bn)
    (bn, _), = _configs(plan, [(2048, 4096)])
    assert bn == 224
    (bn, _), = _configs(plan, [(8320, 21504)])      # full waves: the widest tile
    assert bn == 256


def test_split_count_limits_and_maximality(plan):
    cases = [(M, N, kb) for M in (1, 8, 16, 17, 32, 33, 64, 65, 100, 128) for N in (256, 1024, 4096, 14336, 28672)
             for kb in (1, 2, 3, 8, 32, 112)]
    got = plan([f"splits {M} {N} {kb} {SMS}" for M, N, kb in cases])

    def limits_ok(M, N, kb, s):
        tiles = -(-N // 128) * -(-M // 128)
        bt = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
        return (s <= 8 and s * 2 <= kb and tiles * s <= 2 * SMS   # cluster size, 2 K blocks a slice, residency
                # partials written and read below half the weight slice (all of it for 128-token blocks)
                and s <= kb * BK // ((8 if bt == 128 else 16) * bt))
    for (M, N, kb), (s,) in zip(cases, got):
        assert s >= 1
        if s > 1:
            assert limits_ok(M, N, kb, s), (M, N, kb, s)
        assert not limits_ok(M, N, kb, s + 1), (M, N, kb, s)   # the largest count that keeps them


def test_deterministic_split_depends_on_n_and_k_only(plan):
    # the batch-invariant K split: the tile width from N alone (the same as the table's
    # deterministic row), at most eight K ranges (one cluster) of at least two K blocks,
    # and one range when K is a single block (the K = 80 tail case)
    Ns = (8, 64, 256, 1000, 1024, 4096, 12288, 14336, 28672)
    kbs = (1, 2, 3, 5, 32, 42, 112)
    got = plan([f"det {N} {kb}" for N in Ns for kb in kbs])
    cfg = {N: c for N, c in zip(Ns, _configs(plan, [(1, N) for N in Ns], det=1))}
    for (N, kb), (bn, s) in zip([(N, kb) for N in Ns for kb in kbs], got):
        assert bn == cfg[N][0], (N, bn)
        assert 1 <= s <= 8, (N, kb, s)
        assert s == 1 or kb // s >= 2, (N, kb, s)
        if kb == 1:
            assert s == 1
    # the workloads' shapes: K = 4096 (32 blocks): four ranges for N = 4096, eight for N = 64
    assert plan(["det 4096 32"]) == [(256, 4)]
    assert plan(["det 64 32"]) == [(64, 8)]
