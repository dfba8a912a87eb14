"""The oracle's pins catch plausible slips.

Each case below plants one mistake in a copy of oracle/oracle.c, compiles it
with the oracle's own flags and runs tests/test_oracle_pins.py against it (the
oracle loads the copy named by ORACLE_LIB_UNDER_TEST).  The pins must fail for
every mutant and pass for an unmodified copy built the same way.  All of this
runs on the CPU."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (slip, text in oracle.c, replacement); each text occurs exactly once
MUTANTS = [
    ("RoPE rotation sign", "v[i] = a * c - b * s;", "v[i] = a * c + b * s;"),
    ("RoPE frequency exponent", "double w = pow(theta, -2.0 * (double)i / (double)hd);",
     "double w = pow(theta, -1.0 * (double)i / (double)hd);"),
    ("RMSNorm eps outside the root", "double inv = 1.0 / sqrt(ss / (double)n + eps);",
     "double inv = 1.0 / (sqrt(ss / (double)n) + eps);"),
    ("RMSNorm gain dropped", "out[i] = x[i] * inv * rd(g, gdt, i);", "out[i] = x[i] * inv;"),
    ("attention scale missing", "s[j] = acc * scale;", "s[j] = acc;"),
    ("GQA head map", "int g = i / G;\n            const char *kb", "int g = i % Hkv;\n            const char *kb"),
    ("mask drops the current position", "pos + 1, hd, o + (size_t)i * hd);", "pos, hd, o + (size_t)i * hd);"),
    ("SiLU sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("FFN residual dropped", "x[i] += dx[i];\n    free(dx);", "x[i] = dx[i];\n    free(dx);"),
    ("argmax ties to the highest index", "if (v[i] > v[best]) best = i;", "if (v[i] >= v[best]) best = i;"),
    ("bf16 ties away from zero", "frac == 0.5 && fmod(fl, 2.0) != 0.0", "frac == 0.5"),
    ("matvec reads W transposed", "acc += rd(W, wdt, base + c) * h[c];",
     "acc += rd(W, wdt, (int64_t)c * rows + r) * h[c];"),
]


def _compile(src_text: str, out_dir: str) -> str:
    c = os.path.join(out_dir, "oracle.c")
    with open(c, "w") as f:
        f.write(src_text)
    lib = os.path.join(out_dir, "liboracle.so")
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                           "-o", lib, c, "-lm"])
    return lib


def _run_pins(lib: str):
    """(pytest exit code, the first failing pin or None)."""
    env = dict(os.environ, ORACLE_LIB_UNDER_TEST=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-rf", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    failed = [l.split("::", 1)[1].split(" ")[0] for l in r.stdout.splitlines() if l.startswith("FAILED ")]
    return r.returncode, (failed[0] if failed else None)


@pytest.fixture(scope="module")
def workdir():
    if shutil.which("gcc") is None:
        pytest.skip("no gcc on this machine")
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_pins_reject_every_planted_slip(workdir):
    src = open(SRC).read()
    jobs = [("unmodified copy", src)]
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, f"{name}: the text to mutate must occur once in oracle.c"
        jobs.append((name, src.replace(old, new)))

    def run(i_job):
        i, (name, text) = i_job
        d = os.path.join(workdir, f"m{i}")
        os.makedirs(d)
        return name, _run_pins(_compile(text, d))

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = dict(ex.map(run, enumerate(jobs)))
    assert results.pop("unmodified copy")[0] == 0, "the pins must pass on an unmodified copy"
    # exit code 1: a pin failed (not a crash or a collection error)
    missed = {name: rc for name, (rc, pin) in results.items() if rc != 1 or pin is None}
    assert not missed, f"slips no pin caught by failing: {missed}"
    for name, (_, pin) in sorted(results.items()):
        print(f"{name}: caught by {pin}")


# slips in the sampling suffix's oracle (Python): (slip, function, text, replacement)
PY_MUTANTS = [
    ("top-p cut takes the prefix before reaching top_p", "sample", "S >= min(top_p, 1.0) * S[-1]",
     "S > min(top_p, 1.0) * S[-1]"),
    ("min-p relative to the total instead of the largest", "sample", "np.count_nonzero(q >= min_p)",
     "np.count_nonzero(q / S[-1] >= min_p)"),
    ("temperature multiplies", "sample", "(l[order] - l[order[0]]) / temperature",
     "(l[order] - l[order[0]]) * temperature"),
    ("ties go to the higher index", "sample", "np.lexsort((np.arange(l.size), -l))",
     "np.lexsort((-np.arange(l.size), -l))"),
    ("uniform from 52 bits", "uniform", ">> 11) * 2.0 ** -53", ">> 12) * 2.0 ** -53"),
    ("splitmix64 increment", "splitmix64_at", "(counter + 1) * 0x9E3779B97F4A7C15", "counter * 0x9E3779B97F4A7C15"),
    ("log-sum-exp loses the shift", "top_logprobs", "lse = m + np.log(", "lse = np.log("),
]

_PY_RUNNER = """
import inspect, sys
sys.path.insert(0, {root!r})
import pytest
import oracle
src = inspect.getsource(getattr(oracle, {fn!r}))
assert src.count({old!r}) == 1, "the text to mutate must occur once"
ns = {{}}
exec(src.replace({old!r}, {new!r}), oracle.__dict__, ns)
setattr(oracle, {fn!r}, ns[{fn!r}])
sys.exit(pytest.main([{pins!r}, "-x", "-q", "-rf", "-p", "no:cacheprovider"]))
"""


def _run_pins_patched(fn: str, old: str, new: str):
    code = _PY_RUNNER.format(root=ROOT, fn=fn, old=old, new=new, pins=PINS)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    failed = [l.split("::", 1)[1].split(" ")[0] for l in r.stdout.splitlines() if l.startswith("FAILED ")]
    return r.returncode, (failed[0] if failed else None), r.stdout + r.stderr


def test_pins_reject_every_planted_sampling_slip():
    # control: the same patching path with an identity replacement passes
    rc, _, log = _run_pins_patched("sample", "S = np.cumsum(q)", "S = np.cumsum(q)")
    assert rc == 0, log[-2000:]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda m: (m[0],) + _run_pins_patched(*m[1:]), PY_MUTANTS))
    missed = {name: (rc, log[-400:]) for name, rc, pin, log in results if rc != 1 or pin is None}
    assert not missed, f"slips no pin caught by failing: {missed}"
    for name, _, pin, _ in results:
        print(f"{name}: caught by {pin}")
