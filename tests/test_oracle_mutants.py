"""The oracle's pins must catch a plausible mistake anywhere in it.

Each case below plants one mistake in a copy of the oracle (a wrong constant,
sign, index, rounding rule, operand order or layout), and the oracle pin tests
(tests/test_oracle_*.py) then run against that copy in a child process: at
least one pin has to fail.  The unchanged copy runs too, as the control that
has to pass.  Everything happens on the CPU; the CUDA library is not involved.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C_SRC = "fp8_oracle.c"
PY_SRC = "__init__.py"

# (name, file, [(text, replacement, occurrences to replace)])
MUTANTS = [
    # E4M3
    ("e4m3 ties away from zero", C_SRC, [("double k = nearbyint(a / q);", "double k = round(a / q);", 1)]),
    ("e4m3 overflow gives the NaN code", C_SRC,
     [("if (a >= 448.0) return sign | 0x7E;", "if (a >= 464.0) return sign | 0x7F;", 1)]),
    ("e4m3 subnormal spacing 2^-10", C_SRC,
     [("q = ldexp(1.0, -9);                  /* subnormal spacing */", "q = ldexp(1.0, -10);", 1)]),
    ("e4m3 decode with exponent bias 8", C_SRC,
     [("v = ldexp(8.0 + (double)m, e - 10);", "v = ldexp(8.0 + (double)m, e - 11);", 1)]),
    ("e4m3 NaN input gives the NaN code", C_SRC, [("if (isnan(x)) return 0x7E;", "if (isnan(x)) return 0x7F;", 1)]),
    ("e4m3 negative zero loses its sign", C_SRC,
     [("uint8_t sign = signbit(x) ? 0x80 : 0x00;", "uint8_t sign = x < 0.0f ? 0x80 : 0x00;", 1)]),
    # 16-bit rounding
    ("bf16 rounding truncates", C_SRC,
     [("double r = nearbyint(a / q) * q;", "double r = floor(a / q) * q;", 1)]),
    ("fp16 smallest normal exponent -15", C_SRC,
     [("double r = round_binary(fabs(v), 10, -14, 15);", "double r = round_binary(fabs(v), 10, -15, 15);", 1)]),
    # exp / SiLU
    ("exp polynomial drops the x^6 term", C_SRC,
     [("p = fmaf(p, r, 1.0f / 720.0f);", "p = fmaf(p, r, 0.0f);", 1)]),
    ("exp drops the ln2 tail", C_SRC, [("r = fmaf(-n, ln2_lo, r);", "", 1)]),
    ("silu with exp(+g)", C_SRC, [("float e = exp_cw7(-g);", "float e = exp_cw7(g);", 1)]),
    ("fused gate and up swapped", C_SRC,
     [("float gate = load_x(x, x_dtype, m * ldx + k);", "float gate = load_x(x, x_dtype, m * ldx + K + k);", 1),
      ("float up = load_x(x, x_dtype, m * ldx + K + k);", "float up = load_x(x, x_dtype, m * ldx + k);", 1)]),
    # group quant
    ("absmax without the absolute value", C_SRC, [("float a = fabsf(v);", "float a = v;", 1)]),
    ("absmax through fmaxf, NaNs not skipped", C_SRC,
     [("if (isnan(v)) return amax;\n  float a = fabsf(v);\n  return a > amax ? a : amax;",
       "return fmaxf(amax, fabsf(v));", 1)]),
    ("absmax floor 1e-12", C_SRC, [("float a = fmaxf(amax, 1e-10f);", "float a = fmaxf(amax, 1e-12f);", 1)]),
    ("scale divisor 447", C_SRC, [("float sc = a / 448.0f;", "float sc = a / 447.0f;", 1)]),
    ("multiplier as the reciprocal of the scale", C_SRC, [("mult = 448.0f / a;", "mult = 1.0f / sc;", 1)]),
    ("ue8m0 rounds the exponent down", C_SRC,
     [("int ex = be + ((bits & 0x7FFFFF) != 0);", "int ex = be;", 1)]),
    ("ue8m0 multiplier off by a factor two", C_SRC,
     [("mult = pow2f_exact(127 - ex);", "mult = pow2f_exact(128 - ex);", 1)]),
    ("GEMM UE8M0 scale byte decoded in fp64 (byte 255 finite)", C_SRC,
     [("return (double)ldexpf(1.0f, (int)e - 127);", "return ldexp(1.0, (int)e - 127);", 1)]),
    ("GEMM UE8M0 scale byte 0 decoded as zero", C_SRC,
     [("return (double)ldexpf(1.0f, (int)e - 127);", "return e ? (double)ldexpf(1.0f, (int)e - 127) : 0.0;", 1)]),
    # int8
    ("int8 ties away from zero", C_SRC,
     [("if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0)) n = f + 1.0;", "if (r >= 0.5) n = f + 1.0;", 1)]),
    ("int8 NaN gives -128", C_SRC, [("if (isnan(x)) return 127;", "if (isnan(x)) return -128;", 1)]),
    ("int8 scale divisor 128", C_SRC, [("s[m * G + g] = a / 127.0f;", "s[m * G + g] = a / 128.0f;", 1)]),
    ("int8 clamp symmetric at -127", C_SRC, [("if (c < -128.0) c = -128.0;", "if (c < -127.0) c = -127.0;", 1)]),
    # GEMM
    ("gemm group width 64", C_SRC, [("const int64_t group = 128;", "const int64_t group = 64;", 1)]),
    ("gemm row scales ignored", C_SRC,
     [("case 1: return (double)j->a_scale[m];", "case 1: return (double)j->a_scale[0];", 1)]),
    ("gemm column scale read per row", C_SRC,
     [("(j->b_mode == 1 ? (double)j->b_scale[n] : 1.0)", "(j->b_mode == 1 ? (double)j->b_scale[m % j->N] : 1.0)",
       1)]),
    ("gemm group scales ignore the row", C_SRC,
     [("case 2: return (double)j->a_scale[m * j->a_ld + g];", "case 2: return (double)j->a_scale[g];", 1)]),
    ("gemm ue8m0 bytes in reverse order", C_SRC, [(">> (8 * (g % 4))", ">> (8 * (3 - g % 4))", 1)]),
    ("gemm block scales ignore the row block", C_SRC,
     [("return (double)j->b_scale[(n / 128) * j->b_ld + g];", "return (double)j->b_scale[g];", 1)]),
    ("gemm bias dropped", C_SRC, [("if (j->bias) val +=", "if (0) val +=", 1)]),
    ("gemm bias scaled with the product", C_SRC,
     [("if (j->bias) val += (double)bf16_to_float(j->bias[n]);",
       "if (j->bias) val += (double)bf16_to_float(j->bias[n]) * bs;", 1)]),
    ("gemm accumulates in fp32", C_SRC, [("double p = lut[a[k]] * lut[b[k]];\n          acc += p;",
                                          "double p = lut[a[k]] * lut[b[k]];\n          acc = (float)(acc + p);", 1)]),
    ("exp overflow threshold too low", C_SRC, [("if (x > 89.0f) return INFINITY;", "if (x > 80.0f) return INFINITY;", 1)]),
    ("exp 2^n split loses a factor two", C_SRC, [("int n2 = ni - n1;", "int n2 = ni - n1 - (ni < 0);", 1)]),
    ("silu denominator 1 - exp(-g)", C_SRC, [("float d = 1.0f + e;", "float d = 1.0f - e;", 1)]),
    ("ue8m0 byte one below the scale's exponent", C_SRC, [("eb = (uint8_t)ex;", "eb = (uint8_t)(ex - 1);", 1)]),
    ("e4m3 subnormal code off by one", C_SRC,
     [("return (uint8_t)(r / ldexp(1.0, -9)); /* subnormal: m */", "return (uint8_t)(r / ldexp(1.0, -9) - 1);", 1)]),
    ("bf16 overflow one binade late", C_SRC,
     [("if (r >= ldexp(1.0, emax + 1)) return INFINITY;", "if (r >= ldexp(1.0, emax + 2)) return INFINITY;", 1)]),
    ("fp16 decode subnormals one binade low", C_SRC,
     [("else if (e == 0) v = ldexp((double)m, -24);", "else if (e == 0) v = ldexp((double)m, -25);", 1)]),
    ("int8 fused path with gate and up swapped", C_SRC,
     [("v[i] = silu_f32(load_x(x, x_dtype, m * ldx + k)) * load_x(x, x_dtype, m * ldx + K + k);",
       "v[i] = silu_f32(load_x(x, x_dtype, m * ldx + K + k)) * load_x(x, x_dtype, m * ldx + k);", 1)]),
    ("int8 multiplier as the reciprocal of the scale", C_SRC,
     [("float mult = 127.0f / a;", "float mult = 1.0f / (a / 127.0f);", 1)]),
    ("gemm column-major group scales read row-major", C_SRC,
     [("case 3: return (double)j->a_scale[g * j->a_ld + m];", "case 3: return (double)j->a_scale[g];", 1)]),
    ("gemm per-tensor B scale ignored", C_SRC,
     [("double bs = j->b_mode == 0 ? (double)j->b_scale[0]", "double bs = j->b_mode == 0 ? 1.0", 1)]),
    ("row-major ue8m0 words laid out column-major", PY_SRC,
     [("        out = np.zeros((R, W), np.int32)\n        for m, d in pairs:\n            out[d] = words[m]",
       "        out = np.zeros((R, W), np.int32)\n        for m, d in pairs:\n            out[d] = words[m][::-1]", 1)]),
    ("requant zeroes the rows past the shards", PY_SRC, [("out[start:] = w[start:]", "out[start:] = 0", 1)]),
    ("static quant reads fp16 as bf16", PY_SRC,
     [("v = (bf16_bits_to_f64(x) if x_dtype == 0 else fp16_bits_to_f64(x)).astype(np.float32)",
       "v = bf16_bits_to_f64(x).astype(np.float32)", 1)]),
    ("block quant scales transposed", PY_SRC, [("s[i, j] = sb[0, 0]", "s[j % nb, i % kb] = sb[0, 0]", 1)]),
    ("scatter codes written to the first destination only", PY_SRC,
     [("        for d in dst[m]:\n            if d >= 0:\n                qd[d] = q[m]",
       "        for d in dst[m][:1]:\n            if d >= 0:\n                qd[d] = q[m]", 1)]),
    # layouts and the Python-level paths
    ("column-major scales without the pad-4 stride", PY_SRC,
     [("out = np.zeros((G, pad4(R)), np.float32)", "out = np.zeros((G, R), np.float32)", 1)]),
    ("ue8m0 words packed in reverse byte order", PY_SRC,
     [("<< np.uint32(8 * (g % 4))", "<< np.uint32(8 * (3 - g % 4))", 1)]),
    ("scatter writes only the first destination's scales", PY_SRC,
     [("for d in row_map[m] if d >= 0]", "for d in row_map[m][:1] if d >= 0]", 1)]),
    ("static quant multiplies by the reciprocal scale", PY_SRC,
     [("r = v / np.float32(scale)", "r = v * (np.float32(1.0) / np.float32(scale))", 1)]),
    ("requant divides by the shard's own scale", PY_SRC,
     [("(deq / s_max).astype(np.float32)", "(deq / s[i]).astype(np.float32)", 1)]),
    ("requant keeps the decode in fp64", PY_SRC,
     [("deq = (e4m3_decode(w[start:start + width]).astype(np.float32) * s[i]).astype(np.float32)",
       "deq = e4m3_decode(w[start:start + width]) * np.float64(s[i])", 1)]),
    ("masked quant writes every row of an expert", PY_SRC, [("n = int(masked_m[e])", "n = T", 1)]),
    ("row padding repeats the last row", PY_SRC, [("qp = np.zeros((m_pad, K), np.uint8)",
                                                    "qp = np.repeat(q[-1:], m_pad, axis=0) if M else "
                                                    "np.zeros((m_pad, K), np.uint8)", 1)]),
]

PIN_TESTS = ["tests/test_oracle_quant.py", "tests/test_oracle_gemm.py", "tests/test_oracle_rounding.py",
             "tests/test_oracle_e4m3.py"]

CHILD = """
import sys
sys.path.insert(0, {root!r})
import oracle                       # the planted copy, cached before the suite puts the repository first
assert oracle.__file__.startswith({root!r}), oracle.__file__
import pytest
sys.exit(pytest.main({args!r}))
"""


def _plant(dst, file, edits):
    pkg = os.path.join(dst, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    path = os.path.join(pkg, file)
    text = open(path).read()
    for old, new, count in edits:
        assert text.count(old) >= count, f"mutation site not found in oracle/{file}: {old!r}"
        text = text.replace(old, new, count)
    open(path, "w").write(text)


def _run(dst):
    args = [os.path.join(ROOT, t) for t in PIN_TESTS] + ["-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                                                         "--rootdir", ROOT, "-W", "ignore"]
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=dst, args=args)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is needed to build the planted copies")
    jobs = [("control (no mistake)", C_SRC, [])] + MUTANTS
    dirs = []
    for i, (_, file, edits) in enumerate(jobs):
        d = str(tmp_path / f"m{i:02d}")
        os.makedirs(d)
        _plant(d, file, edits)
        dirs.append(d)
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(_run, dirs))
    rc0, log0 = results[0]
    assert rc0 == 0, f"the unchanged copy of the oracle fails its pins:\n{log0}"
    survivors = [name for (name, _, _), (rc, _) in zip(jobs[1:], results[1:]) if rc == 0]
    broken = [(name, rc, log) for (name, _, _), (rc, log) in zip(jobs[1:], results[1:]) if rc not in (0, 1)]
    assert not broken, "planted copies that did not run to a test verdict:\n" + "\n".join(
        f"{n}: rc={rc}\n{log}" for n, rc, log in broken)
    assert not survivors, f"mistakes no pin catches: {survivors}"
