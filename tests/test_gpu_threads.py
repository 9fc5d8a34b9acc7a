"""Several host threads making their first library calls at the same time.

Each kernel's shared-memory limit and occupancy are set up once per
(device, kernel) in a table under a mutex. This test runs in a fresh process
(so every kernel's first use happens here): four threads, each on its own
stream, wait at a barrier and then pack weights and run forwards through
every contraction kernel (dp4a GEMV, mma.sync, tensor cores) at once. Every
output must match the oracle bit for bit, and no bounded wait may give up.
"""

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect -m gpu
    pytest.skip("needs a CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import numpy as np
import torch
import bit_ternary_forward_b300 as blt
import oracle
from gpu_common import bits, x_to_oracle
from workloads import gaussian_activations, gaussian_weights

cases = [(1, 2560, 1024), (8, 1024, 512), (40, 1536, 768), (3, 4096, 640)]
inputs = [(gaussian_weights(n, k, seed=10 + i), gaussian_activations(m, k, seed=20 + i))
          for i, (m, k, n) in enumerate(cases)]
start = threading.Barrier(len(cases))
results = [None] * len(cases)
errors = []

def work(i):
    try:
        w, x = inputs[i]
        s = torch.cuda.Stream()
        wd, xd = w.cuda(), x.cuda()
        torch.cuda.synchronize()
        start.wait()
        with torch.cuda.stream(s):
            packed = blt.pack_weights(wd)
            y = blt.forward(xd, packed)
        s.synchronize()
        results[i] = (packed.gamma.cpu().numpy()[0], packed.wp.cpu().numpy(), y.cpu().numpy())
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
for t in threads: t.start()
for t in threads: t.join()
assert not errors, errors
for (w, x), (g, wp, y) in zip(inputs, results):
    ref = oracle.bitlinear_forward(x_to_oracle(x), w.numpy())
    assert bits(g) == bits(ref["gamma"])
    np.testing.assert_array_equal(wp, ref["packed"])
    np.testing.assert_array_equal(bits(y), bits(ref["y"]))
assert blt.device_error() == 0
print("threads ok")
"""


def test_concurrent_first_calls_from_four_threads():
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    assert "threads ok" in p.stdout
