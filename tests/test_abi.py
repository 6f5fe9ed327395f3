"""The C-ABI library builds, loads and exports every symbol its header
declares; host-side validation rejects bad arguments before any CUDA call
(CPU only: nothing here launches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            names += re.findall(r"FP8MM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


@pytest.fixture(scope="module")
def L():
    from fp8_scaled_gemm_mm_gb300 import build
    build.build()
    import fp8_scaled_gemm_mm_gb300 as fm
    return fm.lib()


def test_header_declares_the_entry_points():
    names = set(_declared())
    for n in ("fp8_scaled_mm", "per_token_group_quant_fp8", "per_token_group_quant_fp8_scatter",
              "fp8mm_get_device_status", "fp8mm_status_string", "fp8mm_version"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.fp8mm_version() >> 16 == 1
    for code in (0, -1, -2, -3, -4, -5):
        assert L.fp8mm_status_string(code).startswith(b"FP8MM_")


def test_quant_argument_validation(L):
    q = L.per_token_group_quant_fp8
    fake = 1 << 20   # never dereferenced: validation fails first
    # K not a multiple of 16, group not dividing K, bad group, bad dtype, bad format
    assert q(fake, 0, fake, fake, 4, 72, 32, 0, 0, 0, None) == -1
    assert q(fake, 0, fake, fake, 4, 2048 + 64, 128, 0, 0, 0, None) == -1
    assert q(fake, 0, fake, fake, 4, 2048, 96, 0, 0, 0, None) == -1
    assert q(fake, 2, fake, fake, 4, 2048, 128, 0, 0, 0, None) == -1
    assert q(fake, 0, fake, fake, 4, 2048, 128, 3, 0, 0, None) == -1
    assert q(fake, 0, fake, fake, -1, 2048, 128, 0, 0, 0, None) == -1
    # empty batch: nothing to do, nothing launched
    assert q(None, 0, None, None, 0, 2048, 128, 0, 0, 0, None) == 0
    # null pointers with work to do
    assert q(None, 0, fake, fake, 4, 2048, 128, 0, 0, 0, None) == -1
    # misaligned input / codes
    assert q(fake + 2, 0, fake, fake, 4, 2048, 128, 0, 0, 0, None) == -2
    assert q(fake, 0, fake + 8, fake, 4, 2048, 128, 0, 0, 0, None) == -2
    s = L.per_token_group_quant_fp8_scatter
    assert s(fake, 0, None, 8, 64, fake, fake, 4, 2048, 128, 2, 1, None) == -1
    assert s(fake, 0, fake, 0, 64, fake, fake, 4, 2048, 128, 2, 1, None) == -1


def test_gemm_argument_validation(L):
    g = L.fp8_scaled_mm
    f = 1 << 20
    ok_args = dict(A=f, B=f + (1 << 24), a=f + (2 << 24), b=f + (3 << 24), mode=0x11, bias=None, out=f + (4 << 24),
                   od=0, M=64, N=256, K=512, lda=512, ldb=512, det=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return g(a["A"], a["B"], a["a"], a["b"], a["mode"], a["bias"], a["out"], a["od"], a["M"], a["N"], a["K"],
                 a["lda"], a["ldb"], a["det"], None)

    assert call(K=72, lda=80, ldb=80) == -1           # K % 16
    assert call(K=0) == -1                            # empty reduction
    assert call(lda=256) == -1                        # lda < K
    assert call(lda=520) == -2                        # lda % 16
    assert call(N=260) == -2                          # N % 8
    assert call(mode=0x5) == -1                       # bad A mode
    assert call(mode=0x31) == -1                      # bad B mode
    assert call(mode=0x21) == -1                      # block B scales need per-group A scales
    assert call(od=2) == -1                           # bad out dtype
    assert call(mode=0x12, K=80, lda=80, ldb=80) == -1  # group scales need K % 128
    assert call(A=f + 8) == -2                        # misaligned A
    assert call(out=f + 4) == -2                      # misaligned out
    assert call(out=f + 16) == -1                     # out overlaps A
    assert call(M=0) == 0                             # empty: no launch
    assert call(A=None) == -1


def test_masked_and_new_entry_validation(L):
    f = 1 << 20
    m = L.silu_and_mul_masked_post_quant_fp8
    # more experts than a CTA stages, T not positive, bad group: rejected before any launch
    assert m(f, 0, f, 1025, 64, 256, f, f, 128, 2, 1, None) == -1
    assert m(f, 0, f, 4, -1, 256, f, f, 128, 2, 1, None) == -1
    assert m(f, 0, f, 4, 64, 256, f, f, 96, 2, 1, None) == -1
    assert m(None, 0, None, 0, 64, 256, None, None, 128, 2, 1, None) == 0     # no experts: no-op
    i8 = L.per_token_group_quant_int8
    assert i8(f, 0, f, f, 4, 2048, 96, 0, 0, None) == -1                   # bad group
    assert i8(f, 0, f + 8, f, 4, 2048, 128, 0, 0, None) == -2              # misaligned codes
    rp = L.per_token_group_quant_fp8_row_padded
    assert rp(f, 0, f, f, 8, 4, 128, 128, 0, 1, None) == -1                # M_pad < M
    assert rp(f, 0, f, f, 8, 16, 128, 128, 3, 1, None) == -1               # bad format
    sq = L.static_per_tensor_quant_fp8
    assert sq(f, 0, f, f, 24, None) == -1                                   # numel % 16
    assert sq(f, 2, f, f, 32, None) == -1                                   # bad dtype
    rq = L.requantize_with_max_scale_fp8
    w = (ctypes.c_int64 * 2)(6, 6)
    assert rq(f, f, f, ctypes.cast(w, ctypes.c_void_p), 2, 8, 32, f, None) == -1   # shards past N
    assert rq(f, f, f, ctypes.cast(w, ctypes.c_void_p), 0, 8, 32, f, None) == -1   # no shards


def test_wait_limit_setting_validation(L):
    # host-side only: a negative limit or one above the 2 s default is rejected;
    # 0 restores the default
    L.fp8mm_set_wait_timeout_ns.argtypes = [ctypes.c_int64]
    assert L.fp8mm_set_wait_timeout_ns(-1) == -1
    assert L.fp8mm_set_wait_timeout_ns(2_000_000_001) == -1
    assert L.fp8mm_set_wait_timeout_ns(1000) == 0
    assert L.fp8mm_set_wait_timeout_ns(2_000_000_000) == 0
    assert L.fp8mm_set_wait_timeout_ns(0) == 0


def test_plain_c_consumer(L, tmp_path):
    # the header compiles as C11 and a C program links the library and gets the
    # documented statuses back (host-side paths only)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.join(ROOT, "fp8_scaled_gemm_mm_gb300", "_build")
    exe = str(tmp_path / "consumer")
    subprocess.check_call([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c_abi", "consumer.c"), "-L", lib_dir, "-lfp8mm",
                           "-Wl,-rpath," + lib_dir, "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c consumer ok" in r.stdout


def test_binding_refuses_host_tensors(L):
    # a host tensor's address must never reach a kernel: the binding raises
    # before it calls into the library
    import torch
    import fp8_scaled_gemm_mm_gb300 as fm
    x = torch.zeros((4, 128), dtype=torch.bfloat16)
    q = torch.zeros((4, 128), dtype=torch.uint8)
    s = torch.zeros((4, 1), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.per_token_group_quant_fp8(x, q, s, 128)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.static_per_tensor_quant_fp8(x, torch.ones(1), q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fp8_scaled_mm(q, q, s, s, fm.A_ROW | fm.B_COL, x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.requantize_with_max_scale_fp8(q, torch.ones(2), [2, 2], max_scale_out=torch.ones(1))


def test_gemm_validation_fuzz(L):
    # Random argument sets, each breaking at least one documented rule (or empty):
    # every one must come back as EINVAL / EALIGN (or OK for an empty problem) with
    # nothing launched.  Runs only where no GPU is present, so that a validation
    # bug could never send the fake pointers to a kernel.
    import random
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: run without a GPU")
    g = L.fp8_scaled_mm
    rng = random.Random(7)
    base = 1 << 24
    big = 1 << 31
    checked = 0
    while checked < 3000:
        M = rng.choice([-3, 0, 1, 17, 128, 129, 4096, big])
        N = rng.choice([-1, 0, 8, 12, 256, 4096, big])
        K = rng.choice([-16, 0, 8, 16, 72, 80, 128, 512, big])
        lda = max(K, 0) + rng.choice([-16, 0, 0, 8, 16, 64])
        ldb = max(K, 0) + rng.choice([-16, 0, 0, 8, 16])
        a_mode, b_mode = rng.choice([0, 1, 2, 3, 4, 5]), rng.choice([0, 1, 2, 3])
        extra = rng.choice([0, 0, 0, 0x100])
        od = rng.choice([0, 1, 1, 2])
        ptrs = [base + (i << 40) + rng.choice([0, 0, 0, 2, 4, 8]) for i in range(5)]
        if rng.random() < 0.1:
            ptrs[rng.randrange(5)] = None
        A, B, a_s, b_s, out = ptrs
        bias = rng.choice([None, base + (6 << 40), base + (6 << 40) + 1])
        group = a_mode in (2, 3, 4)
        rules_broken = (M < 0 or N < 0 or a_mode > 4 or b_mode > 2 or extra or (b_mode == 2 and not group)
                        or od not in (0, 1) or max(M, N, K) > big - 1 or K <= 0 or K % 16 or lda < K or ldb < K
                        or lda % 16 or ldb % 16 or N % 8 or (group and K % 128))
        empty = M == 0 or N == 0
        if not rules_broken and not empty:
            rules_broken = (None in (A, B, a_s, b_s, out) or any(p % 16 for p in (A, B, out))
                            or a_s % 4 or b_s % 4 or (bias is not None and bias % 2))
        if not rules_broken and not empty:
            continue                      # a valid request would try to launch: not sent
        st = g(A, B, a_s, b_s, a_mode | (b_mode << 4) | extra, bias, out, od, M, N, K, lda, ldb, 0, None)
        if rules_broken:
            assert st in (-1, -2), (st, M, N, K, lda, ldb, a_mode, b_mode, extra, od, ptrs, bias)
        else:
            assert st == 0, (st, M, N, K)
        checked += 1


def test_quant_validation_fuzz(L):
    # As for the GEMM: requests that break a documented rule (or are empty) only,
    # never sent where a GPU is present.
    import random
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: run without a GPU")
    q = L.per_token_group_quant_fp8
    rng = random.Random(11)
    base = 1 << 24
    checked = 0
    while checked < 3000:
        M = rng.choice([-2, 0, 1, 33, 8192, 1 << 31])
        K = rng.choice([-128, 0, 8, 16, 96, 128, 2048, 7168, 2048 + 64])
        group = rng.choice([16, 32, 64, 96, 128, 256, K])
        dt = rng.choice([0, 1, 1, 2])
        fmt = rng.choice([-1, 0, 1, 2, 3])
        cm, fuse = rng.randrange(2), rng.randrange(2)
        ptrs = [base + (i << 40) + rng.choice([0, 0, 0, 2, 4, 8]) for i in range(3)]
        if rng.random() < 0.1:
            ptrs[rng.randrange(3)] = None
        x, qq, s = ptrs
        rules_broken = (M < 0 or K <= 0 or dt not in (0, 1) or fmt not in (0, 1, 2)
                        or group not in (32, 64, 128, K) or group <= 0 or K % 16 or K % group)
        empty = M == 0
        if not rules_broken and not empty:
            rules_broken = (M > (1 << 31) - 1 or None in ptrs or x % 16 or qq % 16 or s % 4)
        if not rules_broken and not empty:
            continue
        st = q(x, dt, qq, s, M, K, group, fmt, cm, fuse, None)
        if rules_broken:
            assert st in (-1, -2), (st, M, K, group, dt, fmt, ptrs)
        else:
            assert st == 0, (st, M, K, group)
        checked += 1
