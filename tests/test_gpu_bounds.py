"""The GPU parity suite under the bounds-checked build (libexl3_bounds.so).

The bounds-checked build stands in for a memory checker that cannot run
here. It is the same kernels compiled with EXL3_DEBUG_BOUNDS=1. Each kernel
checks, against the extents its launch arguments imply:
  - every global and shared-memory index it computes;
  - every mbarrier address;
  - every TMA coordinate and bulk-copy span;
  - every TMEM column.
A failed check skips the access and records EXL3_ERR_OUT_OF_BOUNDS in the
device error word. These tests run in a child process that loads that
build:
  - its reporting self-test, in which every kernel translation unit must
    report;
  - the whole GPU parity suite (the same cases and sizes, ragged tails and
    full-size geometries included), with every test required to leave the
    error word clear.
"""
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(args, timeout):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, EXL3_BOUNDS_CHECKED="1")
    return subprocess.run([sys.executable] + args, cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


SELFTEST = """
import torch
import trellis_quantized_linear_gb300 as tql
assert tql.BOUNDS_CHECKED
tql.build()
torch.cuda.set_device(0)
tql.exl3_init(0)
assert tql.exl3_bounds_checked()
rep, tot = tql.exl3_selftest_bounds()
assert (rep, tot) == (7, 7), (rep, tot)
assert tql.exl3_get_device_status() == 0
print("bounds selftest ok")
"""


def test_bounds_checked_selftest_every_unit_reports():
    r = _child(["-c", SELFTEST], timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert "bounds selftest ok" in r.stdout


def test_gpu_parity_suite_under_bounds_checks():
    r = _child(["-m", "pytest", "tests/test_gpu_parity.py", "tests/test_zz_no_alloc.py", "-m", "gpu", "-x", "-q",
                "-p", "no:cacheprovider"], timeout=1800)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-4000:]
    assert "exl3 bounds check failed" not in r.stdout + r.stderr
    summary = r.stdout.strip().splitlines()[-1]
    m = re.search(r"(\d+) passed", summary)
    assert m and int(m.group(1)) >= 200 and "skipped" not in summary and "failed" not in summary, summary
