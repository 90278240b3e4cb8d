"""Calls from several host threads at once, each on its own stream.

Run in a fresh process so that the library's per-device caches (device
properties, occupancy, tensor-map encoder, kernel attributes) are filled by
the threads racing on first use.  Every thread's results must equal the
same calls made serially afterwards.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
sys.path.insert(0, ROOT)
import torch
import dense_gemm_09_gb300 as dg
from tests import parity

jobs = [("f16_tn", (1024, 2048, 512)), ("tf32", (768, 1536, 1000)), ("f32", (300, 520, 1000)),
        ("bf16_nn", (100, 1000, 2048)), ("f16_nn", (8192, 512, 256)), ("tf32", (129, 257, 301))]
ops = []
for i, (path, (M, N, K)) in enumerate(jobs):
    A, B, C = parity.host_operands(path, M, N, K, seed=40 + i)
    ops.append((path, A.cuda(), B.cuda(), C.cuda()))
torch.cuda.synchronize()
results = [None] * len(jobs)
errors = []
start = threading.Barrier(len(jobs))

def work(i):
    try:
        path, dA, dB, C0 = ops[i]
        s = torch.cuda.Stream()
        outs = []
        start.wait()
        with torch.cuda.stream(s):
            for rep in range(4):
                out = C0.clone()
                parity.fn(path)(dA, dB, out, 1.5, -0.25)
                outs.append(out)
        s.synchronize()
        results[i] = outs
    except Exception as e:  # reported by the main thread
        errors.append("%d: %r" % (i, e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
for i, (path, dA, dB, C0) in enumerate(ops):
    want = C0.clone()
    parity.fn(path)(dA, dB, want, 1.5, -0.25)
    torch.cuda.synchronize()
    for out in results[i]:
        assert torch.equal(out, want), (i, path)
assert dg.device_status() == dg.OK
print("threads ok")
"""


def test_concurrent_first_use_from_threads():
    code = "ROOT = %r\n" % ROOT + SCRIPT
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
