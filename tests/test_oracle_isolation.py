"""The oracle side never maps the CUDA product: the seeded input generator,
the oracle and the bench's reference arm (the oracle timed on host cores)
load neither the package nor libkvgqa.so."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
import sys
sys.path.insert(0, {root!r})
import bench, oracle, workloads
tokens, secs, steps = bench.oracle_decode_sample(0.0)
assert tokens == workloads.LLAMA_DECODE.A and steps == 1
sys.path.insert(0, {golden!r})
import make_golden
maps = open("/proc/self/maps").read()
print("package" if "kv_cached_gqa_rope_gb300" in sys.modules else "no-package")
print("mapped" if "libkvgqa" in maps else "not-mapped")
"""


def test_reference_arm_does_not_load_the_product():
    code = PROBE.format(root=ROOT, golden=os.path.join(ROOT, "tests", "golden"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split() == ["no-package", "not-mapped"], r.stdout
