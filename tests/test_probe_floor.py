"""The GEMM floor microbenchmarks (libbi_probe.so, run by `bench.py --floor`) are built with the library, export
their two entry points, and reject arguments they cannot run before any CUDA call.  The calls run in a child
process that sees no GPU (CUDA_VISIBLE_DEVICES empty), so a check that let one through would fail with a CUDA
error rather than launch anything."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from invariant_fixed_order_gb300 import build
build.build()
lib = ctypes.CDLL(build.PROBE_LIB)
assert hasattr(lib, "bip_mma_ns") and hasattr(lib, "bip_ingest")
dp = ctypes.POINTER(ctypes.c_double)
lib.bip_mma_ns.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
lib.bip_ingest.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp]
v, w = ctypes.c_double(), ctypes.c_double()
bad_mma = [
    (1, 128, 8, 1),     # M = 128 needs N a multiple of 16
    (1, 128, 256, 1),   # a single CTA holds 128 rows of B
    (1, 96, 16, 1),     # M is 64 or 128 for one CTA
    (2, 64, 64, 1),     # the pair form is M = 128 or 256
    (2, 128, 48, 1),    # M = 128 in a pair needs N a multiple of 32
    (2, 256, 264, 1),   # N at most 256
    (1, 128, 128, 8),   # 1, 2 or 4 accumulators
    (1, 128, 128, 4 + 1),
    (2, 256, 256, 4),   # 4 x 256 columns exceed the 512 of tensor memory
    (3, 256, 64, 1),
]
for args in bad_mma:
    assert lib.bip_mma_ns(*args, ctypes.byref(v)) == -1, args
assert lib.bip_mma_ns(1, 128, 64, 1, None) == -1
for mode, ctas in ((3, 1), (-1, 1), (0, 0), (0, 153), (2, -4)):
    assert lib.bip_ingest(mode, ctas, ctypes.byref(v), ctypes.byref(w)) == -1, (mode, ctas)
assert lib.bip_ingest(0, 1, None, ctypes.byref(w)) == -1
print("ok")
"""


def test_probe_library_exports_and_rejects_bad_arguments():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
