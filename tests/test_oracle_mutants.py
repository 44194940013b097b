"""Planted mistakes in the CPU oracle must fail its pins.

Each case copies the oracle package (and the pin module with what it
imports) to a temporary directory, makes ONE plausible mistake in the copy
(a wrong sign, index, constant, stream or rounding rule, a dropped term, a
transposed operand), builds it, and runs ``tests/test_oracle_pins.py``
against it.  The pins pass on an unmutated copy and must fail on every
mutant: a mistake that no pin notices is a hole in the pins.  Everything
runs on the CPU; the repository's own oracle is never modified.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C = "oracle/hlq_oracle.c"
PY = "oracle/__init__.py"
COPIED = ["oracle/__init__.py", "oracle/hlq_oracle.c", "tests/__init__.py",
          "tests/exact_ref.py", "tests/test_oracle_pins.py",
          "tests/golden/sequency16.txt"]

# (name, file, text in the oracle, replacement); each text occurs once.
MUTANTS = [
    # Hadamard matrix and sequency order
    ("H negated", C, "return (ones % 2 == 0) ? 1 : -1;",
     "return (ones % 2 == 1) ? 1 : -1;"),
    ("H from i|j", C, "int both = i & j, ones = 0;", "int both = i | j, ones = 0;"),
    ("sequency reversed", C, "sigma[changes] = i;", "sigma[15 - changes] = i;"),
    # exact sums: rounding and signs
    ("ties away from zero", C, "if (half && (sticky || (keep & 1u)))", "if (half)"),
    ("sticky bit dropped", C, "if (half && (sticky || (keep & 1u)))",
     "if (half && (keep & 1u))"),
    ("H signs ignored", C, "if (h[j] < 0)\n            neg = !neg;", ""),
    ("normal exponent off by one", C, "*pos = (int)e - 1;", "*pos = (int)e;"),
    # transforms
    ("HQ coefficient order", C, "&H[i * 16], &src[r * cols + 16 * b], 1, 16);",
     "&H[(15 - i) * 16], &src[r * cols + 16 * b], 1, 16);"),
    ("HQ along rows, rows swapped", C,
     "&H[i * 16], &src[16 * b * cols + c], (ptrdiff_t)cols,",
     "&H[(i ^ 1) * 16], &src[16 * b * cols + c], (ptrdiff_t)cols,"),
    ("HLA natural order", C,
     "&H[sigma[k] * 16], &src[16 * b * C + c], (ptrdiff_t)C, 16);",
     "&H[k * 16], &src[16 * b * C + c], (ptrdiff_t)C, 16);"),
    ("HLA coefficient-major layout", C,
     "out[c * Tp + rank * b + k] = exact_signed_sum(",
     "out[c * Tp + b + (T / 16) * k] = exact_signed_sum("),
    ("fp64 HQ sign", C, "s += H[i * 16 + j] * src[r * cols + 16 * b + j];",
     "s -= H[i * 16 + j] * src[r * cols + 16 * b + j];"),
    ("fp64 HQ along rows, one row negated", C,
     "s += H[i * 16 + j] * src[(16 * b + j) * cols + c];",
     "s += H[j * 16 + i] * src[(16 * b + j) * cols + c] * (i == 3 ? -1 : 1);"),
    ("fp64 HLA natural order", C,
     "s += H[sigma[k] * 16 + j] * src[(16 * b + j) * C + c];",
     "s += H[k * 16 + j] * src[(16 * b + j) * C + c];"),
    # Philox4x32-10 and the word of an element
    ("Philox Weyl constant", C, "k1 += 0xBB67AE85u;", "k1 += 0xBB67AE86u;"),
    ("Philox 7 rounds", C, "for (int round = 0; round < 10; ++round) {",
     "for (int round = 0; round < 7; ++round) {"),
    ("Philox multiplier", C, "(uint64_t)0xD2511F53u * c0;", "(uint64_t)0xD2511F55u * c0;"),
    ("Philox key halves swapped", C,
     "uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};",
     "uint32_t key[2] = {(uint32_t)(seed >> 32), (uint32_t)seed};"),
    ("Philox word order", C, "return out[e % 4];", "return out[3 - e % 4];"),
    ("Philox stream in counter word 3", C, "(uint32_t)((e / 4) >> 32), stream, 0};",
     "(uint32_t)((e / 4) >> 32), 0, stream};"),
    # quantizers
    ("SR comparison reversed", C, "r = f + ((u < frac) ? 1.0f : 0.0f);",
     "r = f + ((u > frac) ? 1.0f : 0.0f);"),
    ("SR uniform scaled by 2^-23", C, "(float)(word >> 8) * 0x1p-24f;",
     "(float)(word >> 8) * 0x1p-23f;"),
    ("SR from the low 24 bits", C, "(float)(word >> 8) * 0x1p-24f;",
     "(float)(word & 0xffffffu) * 0x1p-24f;"),
    ("RNE ties away", C, "r = rintf(x);", "r = roundf(x);"),
    ("RNE truncates", C, "r = rintf(x);", "r = truncf(x);"),
    ("upper clamp dropped", C, "if (r > (float)qmax)\n        r = (float)qmax;", ""),
    ("lower clamp dropped", C, "if (r < (float)-qmax)\n        r = (float)-qmax;", ""),
    ("scaling by a reciprocal", C, "float x = y / s;", "float x = y * (1.0f / s);"),
    ("zero scale gives code 1", C, "if (s == 0.0f)\n        return 0;",
     "if (s == 0.0f)\n        return 1;"),
    ("RNE scale over qmax + 1", C, "float s = amax / (float)qmax;\n    *scale = s;",
     "float s = amax / (float)(qmax + 1);\n    *scale = s;"),
    ("HQ scale over qmax + 1", C, "float s = amax / (float)qmax;\n        if (gran == 1)",
     "float s = amax / (float)(qmax + 1);\n        if (gran == 1)"),
    ("row number of a sample ignored", C, "int64_t row = row_ids ? row_ids[r] : r;",
     "int64_t row = r;"),
    ("element index transposed", C, "uint64_t e = (uint64_t)(row * cols + c);",
     "uint64_t e = (uint64_t)(c * nrows + row);"),
    ("per-token maximum without abs", C,
     "if (fabsf(Y[r * cols + c]) > amax)\n                    amax = fabsf(Y[r * cols + c]);",
     "if (Y[r * cols + c] > amax)\n                    amax = Y[r * cols + c];"),
    ("tensor maximum without abs", C,
     "        if (fabsf(v[i]) > amax)\n            amax = fabsf(v[i]);\n    return amax;",
     "        if (v[i] > amax)\n            amax = v[i];\n    return amax;"),
    ("nibbles swapped", C,
     "packed[k] = (uint8_t)(((uint8_t)codes[2 * k] & 0x0fu) |\n"
     "                              (((uint8_t)codes[2 * k + 1] & 0x0fu) << 4));",
     "packed[k] = (uint8_t)(((uint8_t)codes[2 * k + 1] & 0x0fu) |\n"
     "                              (((uint8_t)codes[2 * k] & 0x0fu) << 4));"),
    # GEMM and dequantization
    ("GEMM B transposed", C, "s += (int64_t)A[m * K + k] * (int64_t)B[n * K + k];",
     "s += (int64_t)A[m * K + k] * (int64_t)B[k * N + n];"),
    ("GEMM products in int8", C, "s += (int64_t)A[m * K + k] * (int64_t)B[n * K + k];",
     "s += (int8_t)(A[m * K + k] * B[n * K + k]);"),
    ("g_x without 1/16", C,
     "g_x[t * Cin + i] = (double)acc[t * Cin + i] * sg * (double)s_w / 16.0;",
     "g_x[t * Cin + i] = (double)acc[t * Cin + i] * sg * (double)s_w;"),
    ("g_x token scale ignored", C, "double sg = (double)s_gy[gran_gy == 1 ? t : 0];",
     "double sg = (double)s_gy[0];"),
    ("g_w over 8", C, "(double)s_x / 16.0;", "(double)s_x / 8.0;"),
    ("g_w channel scale ignored", C, "(double)s_x[i] / 16.0;", "(double)s_x[0] / 16.0;"),
    # composition of the paths
    ("w on the g_y stream", PY,
     "qWt, s_w = hq_quantize(Wt, PER_TENSOR, rnd, seed, STREAM_W)",
     "qWt, s_w = hq_quantize(Wt, PER_TENSOR, rnd, seed, STREAM_GY)"),
    ("w per row", PY, "qWt, s_w = hq_quantize(Wt, PER_TENSOR, rnd, seed, STREAM_W)",
     "qWt, s_w = hq_quantize(Wt, PER_TOKEN, rnd, seed, STREAM_W)"),
    ("g_y transformed along tokens", PY, "Y = hq_transform(g_y, axis=0)\n    qY, s_gy",
     "Y = hq_transform(g_y, axis=1)\n    qY, s_gy"),
    ("g_y granularity ignored", PY,
     "qY, s_gy = hq_quantize(Y, gran_gy, rnd, seed, STREAM_GY)",
     "qY, s_gy = hq_quantize(Y, PER_TOKEN, rnd, seed, STREAM_GY)"),
    ("g_y on the w stream", PY,
     "qY, s_gy = hq_quantize(Y, gran_gy, rnd, seed, STREAM_GY)",
     "qY, s_gy = hq_quantize(Y, gran_gy, rnd, seed, STREAM_W)"),
    ("ablation g_y on stream 0", PY,
     "qg, s_g = hq_quantize(Yg, PER_TENSOR, rnd, seed, STREAM_GY_T)",
     "qg, s_g = hq_quantize(Yg, PER_TENSOR, rnd, seed, STREAM_GY)"),
    ("ablation x on stream 2", PY,
     "qx, s_x = hq_quantize(Yx, PER_TENSOR, rnd, seed, STREAM_X_T)",
     "qx, s_x = hq_quantize(Yx, PER_TENSOR, rnd, seed, STREAM_GY_T)"),
    ("ablation x along channels", PY, "Yx = hq_transform(x, axis=1)",
     "Yx = hq_transform(x, axis=0)"),
    ("g_w rank fixed at 8", PY, "Gb = hla_transform(g_y, rank)", "Gb = hla_transform(g_y, 8)"),
    ("stored activation rank fixed at 8", PY, "Xb = hla_transform(x, rank)",
     "Xb = hla_transform(x, 8)"),
    ("per-channel scales ignored", PY, "    if not per_channel:\n        return rne_quantize",
     "    if True:\n        return rne_quantize"),
    ("g_x ablation w as int4", PY, "qW, s_w = int8_quantize(Wb)",
     "qW, s_w = rne_quantize(Wb, 7)"),
    ("g_x ablation scale of w used twice", PY,
     "g_x = dequant_gx(acc, np.array([s_g], np.float32), PER_TENSOR, s_w)",
     "g_x = dequant_gx(acc, np.array([s_w], np.float32), PER_TENSOR, s_w)"),
    ("LQS comparison reversed", PY,
     "choice = PER_TOKEN if m_tensor > threshold * m_token else PER_TENSOR",
     "choice = PER_TOKEN if m_token > threshold * m_tensor else PER_TENSOR"),
    ("LQS threshold ignored", PY,
     "choice = PER_TOKEN if m_tensor > threshold * m_token else PER_TENSOR",
     "choice = PER_TOKEN if m_tensor > m_token else PER_TENSOR"),
    ("LQS error with SR", PY, "q, s = hq_quantize(Y, gran, RNE, 0, STREAM_GY)",
     "q, s = hq_quantize(Y, gran, SR, 0, STREAM_GY)"),
    ("LQS error with the first token's scale", PY,
     "sc = (np.asarray(s, np.float64)[:, None] if gran == PER_TOKEN",
     "sc = (np.float64(s[0]) if gran == PER_TOKEN"),
    ("g_w channel scales collapsed", PY,
     "g_w = dequant_gw(acc, s_g, s_x)\n    return dict(Gb=Gb",
     "g_w = dequant_gw(acc, s_g, np.max(s_x))\n    return dict(Gb=Gb"),
]


def _copy(dst, mutant=None):
    for rel in COPIED:
        os.makedirs(os.path.join(dst, os.path.dirname(rel)), exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), os.path.join(dst, rel))
    with open(os.path.join(dst, "tests", "conftest.py"), "w") as f:
        f.write("")
    if mutant is not None:
        _, rel, old, new = mutant
        path = os.path.join(dst, rel)
        with open(path) as f:
            src = f.read()
        with open(path, "w") as f:
            f.write(src.replace(old, new))


def _run(dst):
    """(build ok, pytest return code, last line of the pin run)."""
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    env["PYTHONDONTWRITEBYTECODE"] = "1"
    b = subprocess.run([sys.executable, "-c", "import oracle; oracle.build()"],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=300)
    if b.returncode != 0:
        return False, None, b.stderr[-300:]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    return True, r.returncode, lines[-1] if lines else r.stderr[-300:]


def test_each_mutant_text_occurs_once():
    for name, rel, old, _ in MUTANTS:
        with open(os.path.join(ROOT, rel)) as f:
            assert f.read().count(old) == 1, name


def test_pins_fail_on_every_planted_mistake(tmp_path):
    control = tmp_path / "control"
    _copy(str(control))
    ok, rc, last = _run(str(control))
    assert ok and rc == 0, f"the unmutated copy must pass the pins: {last}"

    def one(i):
        dst = str(tmp_path / f"m{i}")
        _copy(dst, MUTANTS[i])
        return MUTANTS[i][0], _run(dst)

    workers = max(1, min(8, os.cpu_count() or 1))
    survivors, broken = [], []
    with cf.ThreadPoolExecutor(workers) as ex:
        for name, (ok, rc, last) in ex.map(one, range(len(MUTANTS))):
            if not ok:
                broken.append(f"{name}: does not build: {last}")
            elif rc == 0:
                survivors.append(name)
            elif rc != 1:
                broken.append(f"{name}: pytest status {rc}: {last}")
    assert not broken, broken
    assert not survivors, f"mutants no pin notices: {survivors}"

