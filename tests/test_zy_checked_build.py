"""The checked build (reducescatter_reduction_gb300.build.build_checked:
every kernel tests each global access it computes against its rank buffer,
records a violation and skips the access) runs the seeded random cases, the
order-revealing parity cases of the main kernel paths, the fused RMSNorm
tests and the bounds-record tests, in a child process that loads
libccl_checked.so: every result must still equal the oracle's and no
violation may be recorded.  This is the
race-and-bounds check that stands in for a memory sanitizer."""
import os
import subprocess
import sys

import pytest
import torch

from reducescatter_reduction_gb300 import build as ccl_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_checked_build_passes_the_parity_cases():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = ccl_build.build_checked()
    env = dict(os.environ, CCL_LIBRARY=lib)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_bounds_record.py"),
           os.path.join(HERE, "test_fuzz.py"),
           os.path.join(HERE, "test_fuzz_tma.py"),
           os.path.join(HERE, "test_order_gpu.py") + "::test_sum_order_every_path",
           os.path.join(HERE, "test_tma.py") + "::test_tma_wide_ranks_match_oracle",
           os.path.join(HERE, "test_rmsnorm.py")]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (res.stdout + res.stderr)[-3000:]
    assert res.returncode == 0, tail
    assert " passed" in res.stdout and "skipped" not in res.stdout.splitlines()[-1], tail
