"""The range-checked build (LORA_CHECK) on valid inputs: the tiny workload and ragged
shapes (d_in, d_out not multiples of the tiles, ranks not multiples of 8, T around the
tile and decode limits) through the decode kernels and both prefill GEMM kernels, every
call LORA_OK (no gathered index out of range) and within the layer's tolerance of the
oracle. It runs in a child process, which loads liblora_linear_check.so in place of
the library the other tests use. (compute-sanitizer is closed on this machine; these
checks stand in for it.)"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_runs_clean():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = os.path.join(os.path.dirname(al.__file__), "liblora_linear_check.so")
    assert os.path.exists(lib), "the checked build is missing: run adapter_linear_gb300.build"
    env = dict(os.environ, ADAPTER_LINEAR_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "_checked_cases.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "all ok" in r.stdout
