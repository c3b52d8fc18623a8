"""The bounds-checked build of the library on the parity shapes.

compute-sanitizer is closed on the GPU pool, so race and range errors are
caught by other means: bitwise determinism and odd shapes in the parity
tests, and this run of the same small, ragged and degenerate cases against
libmxq_debug.so, whose kernels check every global index they compute and
report MXQ_ERR_BOUNDS (skipping the access) instead of touching memory out of
range.  Runs in a subprocess because the library variant is chosen when the
binding first loads.
"""

import json
import os
import subprocess
import sys

import pytest
import torch

from precision_mx_quantize_gb300 import build as _build
from tests.libutil import ensure_built

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_cases_report_no_bounds_error():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    assert os.path.exists(_build.LIB_DEBUG), "the bounds-checked library was not built"
    env = dict(os.environ, MXQ_BOUNDS_CHECKED="1")
    p = subprocess.run([sys.executable, "-m", "tests.bounds_checked_cases"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stdout[-3000:] + p.stderr[-3000:]
    res = json.loads(p.stdout.strip().splitlines()[-1])
    assert res["errors"] == [] and res["cases"] >= 60, res
