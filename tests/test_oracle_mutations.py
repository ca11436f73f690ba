"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a scratch copy of ``oracle/oracle.c`` (a
dropped term, a wrong sign, index or bound, a swapped operand), rebuilds that
copy with gcc and runs the oracle pins (``test_oracle_*.py``) against it: every
mutant must fail at least one pin.  Nothing here touches the GPU or the CUDA
library; the mistakes are planted in the oracle, on the CPU.

Each mutation names the exact source text it replaces and how often that text
occurs, so an edit of the oracle that moves it fails here loudly instead of
leaving a mutant unapplied.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text, occurrences of text in oracle.c, which occurrence to change, replacement)
MUTATIONS = [
    ("e4m3 subnormal exponent", "v = ldexp((double)m / 8.0, -6);", 1, 0,
     "v = ldexp((double)m / 8.0, -7);"),
    ("e4m3 normal bias", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", 1, 0,
     "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("encode ties away from even", "pick = (c % 2 == 0) ? c : c + 1;", 1, 0, "pick = c + 1;"),
    ("encode overflows to NaN instead of saturating", "return s | 126;", 1, 0, "return s | 0x7F;"),
    ("encode drops the sign", "return s | (uint8_t)pick;", 1, 0, "return (uint8_t)pick;"),
    ("scale divisor", "return num / 448.0f;", 1, 0, "return num / 447.0f;"),
    ("scale of an all-zero unit", "if (absmax == 0.0f)\n        return 1.0f;", 1, 0,
     "if (absmax == 0.0f)\n        return 0.5f;"),
    ("bf16 decode shift", "uint32_t u = (uint32_t)b << 16;", 1, 0, "uint32_t u = (uint32_t)b << 15;"),
    ("append quantises K with the V scale", "oracle_quantize(kx, ks);", 1, 0, "oracle_quantize(kx, vs);"),
    ("append opens a unit at the wrong slot", "if (slot == 0) {", 1, 0, "if (slot == 1) {"),
    ("append ignores the page bound", "if (phys < 0 || phys >= c->num_pages) {", 2, 0,
     "if (phys < 0 || phys > c->num_pages) {"),
    ("validation page bound off by one", "if (phys < 0 || phys >= c->num_pages) {", 2, 1,
     "if (phys < 0 || phys > c->num_pages) {"),
    ("validation drops the last partial page", "int32_t np = (n + ORC_PAGE - 1) / ORC_PAGE;", 1, 0,
     "int32_t np = n / ORC_PAGE;"),
    ("validation reads head 0's tag", "c->page_tags[unit_index(c, phys, h)] != pg->expected_tags[bi]", 1, 0,
     "c->page_tags[unit_index(c, phys, 0)] != pg->expected_tags[bi]"),
    ("dequant transposes two dims", "int64_t idx = (u * ORC_PAGE + slot) * c->head_dim + d;", 1, 0,
     "int64_t idx = (u * ORC_PAGE + slot) * c->head_dim + (d ^ 1);"),
    ("dequant drops the unit scale", "* (double)scale[u];", 1, 0, ";"),
    ("decode: interleaved GQA mapping", "int h = hq / G;", 2, 0, "int h = hq % H;"),
    ("decode: softmax sign", "double p = exp(s[j] - m);", 2, 0, "double p = exp(m - s[j]);"),
    ("decode: no sm_scale", "s[j] = sm_scale * acc;", 3, 0, "s[j] = acc;"),
    ("decode: no normalisation", "            o[d] /= l;\n        free(qv);", 1, 0,
     "            o[d] /= 1.0;\n        free(qv);"),
    ("mass: no normalisation", "mrow[j] += exp(s[j] - m) / l;", 1, 0, "mrow[j] += exp(s[j] - m);"),
    ("mass: query head of kv head 0", "q + ((int64_t)b * Hq + (int64_t)h * G + g) * D", 1, 0,
     "q + ((int64_t)b * Hq + g) * D"),
    ("multi: causal window one short", "int64_t seen = (int64_t)n - kq + 1 + i;", 1, 0,
     "int64_t seen = (int64_t)n - kq + i;"),
    ("multi: interleaved GQA mapping", "int h = hq / G;", 2, 1, "int h = hq % H;"),
    ("multi: no sm_scale", "s[j] = sm_scale * acc;", 3, 2, "s[j] = acc;"),
]

PIN_FILES = sorted(f for f in os.listdir(os.path.join(ROOT, "tests"))
                   if f.startswith("test_oracle_") and f.endswith(".py")
                   and f != os.path.basename(__file__))


def _mutate(src, text, count, which, new):
    assert src.count(text) == count, (text, src.count(text))
    at = -1
    for _ in range(which + 1):
        at = src.index(text, at + 1)
    return src[:at] + new + src[at + len(text):]


def _scratch_copy(dst):
    """The oracle, the oracle pins and the input generators, nothing else."""
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "build.py", "oracle.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    os.makedirs(os.path.join(dst, "paged_fp8_kv_decode_gb300"))
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "paged_fp8_kv_decode_gb300", f),
                    os.path.join(dst, "paged_fp8_kv_decode_gb300", f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ["conftest.py", "oracle_cases.py"] + PIN_FILES:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _run_pins(dst):
    env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *[os.path.join("tests", f) for f in PIN_FILES]],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, (r.stdout + r.stderr)[-2000:]


def test_every_mutation_applies_to_the_current_oracle():
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    for name, text, count, which, new in MUTATIONS:
        assert _mutate(src, text, count, which, new) != src, name


def test_unmutated_copy_passes_the_pins(tmp_path):
    _scratch_copy(str(tmp_path))
    rc, log = _run_pins(str(tmp_path))
    assert rc == 0, log


def test_every_planted_mistake_fails_a_pin(tmp_path):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    jobs = []
    for i, (name, text, count, which, new) in enumerate(MUTATIONS):
        dst = str(tmp_path / f"m{i}")
        _scratch_copy(dst)
        with open(os.path.join(dst, "oracle", "oracle.c"), "w") as f:
            f.write(_mutate(src, text, count, which, new))
        jobs.append((name, dst))
    workers = max(1, min(len(jobs), (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda j: (j[0],) + _run_pins(j[1]), jobs))
    survivors = [(name, log) for name, rc, log in results if rc == 0]
    assert not survivors, "mutants that passed every pin: " + ", ".join(n for n, _ in survivors)
    # a mutant must fail a pin, not the build or the collection
    broken = [(name, log) for name, rc, log in results
              if rc != 1 or "FAILED" not in log or "CalledProcessError" in log]
    assert not broken, broken[0]
