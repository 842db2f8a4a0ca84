"""The pins catch plausible mistakes in the oracle.

Each case copies oracle/mxq_oracle.c, plants one mistake (a wrong constant,
sign, index, stride, rounding mode, dropped rule or transposed operand),
builds the copy, and runs the oracle pin tests against it: every planted
mistake must make at least one pin fail.  Mistakes are planted only in the
CPU oracle, never on a GPU.

Not covered on purpose: the MX9 prime bit order and the MX6 code bit layout,
which the pages never print (parity unpinned for both).
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mxq_oracle.c")
PINS = ["tests/test_oracle_mxfp8_pins.py", "tests/test_oracle_mx9_pins.py",
        "tests/test_oracle_mx_variants_pins.py", "tests/test_oracle_dual_twin.py"]

MUTATIONS = [
    ("E4M3 max 480 instead of 448", "amax <= ldexp(448.0, mid - 127)", "amax <= ldexp(480.0, mid - 127)"),
    ("scale bias off by one", "amax <= ldexp(448.0, mid - 127)", "amax <= ldexp(448.0, mid - 126)"),
    ("strict instead of non-strict cutoff", "amax <= ldexp(448.0, mid - 127)", "amax < ldexp(448.0, mid - 127)"),
    ("multiplier sign flipped", "q[i * qstride] = oracle_e4m3_encode(ldexp(v, 127 - s));",
     "q[i * qstride] = oracle_e4m3_encode(ldexp(v, s - 127));"),
    ("32x1 NaN-dropped multiplier sign", "0x7F : oracle_e4m3_encode(ldexp(v, 127 - s))",
     "0x7F : oracle_e4m3_encode(ldexp(v, s - 127))"),
    ("E4M3 exponent bias 8", "code = (E + 7) * 8 + ((int)n - 8);", "code = (E + 8) * 8 + ((int)n - 8);"),
    ("E4M3 truncation", "n = nearbyint(ldexp(a, 3 - E));", "n = floor(ldexp(a, 3 - E));"),
    ("E4M3 sign dropped", "return (uint8_t)(sign | code);", "return (uint8_t)code;"),
    ("rowwise Inf saturates", "s = colwise ? 254 : 255;", "s = 254;"),
    ("colwise Inf poisons", "s = colwise ? 254 : 255;", "s = 255;"),
    ("NaN does not poison colwise", "    if (any_nan)\n        s = 255;\n    else if (any_inf)\n        s = colwise",
     "    if (any_nan && !colwise)\n        s = 255;\n    else if (any_inf)\n        s = colwise"),
    ("blocked layout row stride", "c / 4) * 512 + (r % 32) * 16 +", "c / 4) * 512 + (r % 32) * 4 +"),
    ("blocked layout 32-row group stride", "((r % 128) / 32) * 4 + (c % 4)", "((r % 128) / 32) * 16 + (c % 4)"),
    ("atoms column-major", "((r / 128) * (C / 4) + c / 4) * 512", "((c / 4) * (R / 128) + r / 128) * 512"),
    ("slab offset uses M", "s_col[N * lo / 32 +\n", "s_col[M * lo / 32 +\n"),
    ("swizzle slab offset uses M", "s_col[N * lo / 32 + oracle_blocked_index", "s_col[M * lo / 32 + oracle_blocked_index"),
    ("swizzle reads s_rm transposed", "s_rm[n * (M / 32) + c];", "s_rm[c * N + n];"),
    ("tail not zeroed", "for (b = N * end / 32; b < N * M / 32; ++b) s_col[b] = 0;", "(void)b;"),
    ("q_col not transposed", "q_col + n * M + row, 1);\n                if (in_group)",
     "q_col + row * N + n, N);\n                if (in_group)"),
    ("MX9 offset 7", "    int k = E - 6 - tau;\n    return k < -126 ? -126 : k;", "    int k = E - 7 - tau;\n    return k < -126 ? -126 : k;"),
    ("MX9 prime polarity flipped", "            int tau = tp < E;\n            int k = mx9_k(E, tau);",
     "            int tau = tp >= E;\n            int k = mx9_k(E, tau);"),
    ("MX9 no -126 clamp", "    int k = E - 6 - tau;\n    return k < -126 ? -126 : k;", "    int k = E - 6 - tau;\n    return k;"),
    ("MX9 clamp to 128", "                if (r > 127.0) r = 127.0;", "                if (r > 128.0) r = 128.0;"),
    ("MX9 truncation", "                r = nearbyint(ldexp(v, -k));", "                r = trunc(ldexp(v, -k));"),
    ("MX9 bf16 exponent bits", "return (int)((u >> 7) & 0xFF) - 127;", "return (int)((u >> 8) & 0xFF) - 127;"),
    ("MX6 offset 4", "d = fmt == ORC_FMT_MX9 ? 6 : 3, qmax", "d = fmt == ORC_FMT_MX9 ? 6 : 4, qmax"),
    ("packed record fields swapped", "        mx_block(v, t, fmt, &rec[0], &rec[1], q);", "        mx_block(v, t, fmt, &rec[1], &rec[0], q);"),
    ("axis-0 index transposed", "int64_t idx = axis == 1 ? line * ld + pos : pos * ld + line;",
     "int64_t idx = axis == 1 ? line * ld + pos : line * ld + pos;"),
    ("packed pack no -126 clamp", "        int k = E - d - tau;\n        if (k < -126) k = -126;\n",
     "        int k = E - d - tau;\n"),
    ("packed pack ties away from zero", "            r = nearbyint(ldexp(v[i], -k));",
     "            r = round(ldexp(v[i], -k));"),
    ("packed unpack no -126 clamp", "            k = E - d - tau;\n            if (k < -126) k = -126;\n",
     "            k = E - d - tau;\n"),
]


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


def _run_mutation(source: str, old: str, new: str):
    """Build the oracle with one planted mistake and run the pins against it."""
    mutated = source.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mut.c")
        so = os.path.join(d, "libmut.so")
        open(c, "w").write(mutated)
        subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-fno-fast-math",
                        "-ffp-contract=off", "-w", c, "-o", so, "-lm"], check=True)
        env = dict(os.environ, MXQ_ORACLE_LIB=so)
        return subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p",
                               "no:cacheprovider", "-m", "not gpu"], cwd=ROOT, env=env,
                              capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def results(source):
    """Every mutation's pin run, several at a time (each is its own process)."""
    from concurrent.futures import ThreadPoolExecutor
    for name, old, _ in MUTATIONS:
        assert source.count(old) == 1, f"mutation site not found or not unique: {name}"
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        futs = {name: ex.submit(_run_mutation, source, old, new) for name, old, new in MUTATIONS}
        return {name: f.result() for name, f in futs.items()}


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(results, name, old, new):
    r = results[name]
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin"
    assert "failed" in r.stdout, r.stdout[-2000:]
