"""Failure detection without a GPU fault: every mbarrier wait in the kernels is
bounded; a wait that runs out raises the pool's timeout bit and returns, so the host
reads an error status and the context stays usable.

The test makes one wait run out on purpose through the library's test hook (the same
bounded-wait code, on an mbarrier that nothing arrives on, with a 20 ms limit), then
checks the reported status and that the next layer call is still correct.
"""
import time

import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import assert_parity, load_pool, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


def test_bounded_wait_runs_out_and_reports():
    prob = L.tiny()
    pool = load_pool(al, prob)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pool.selftest_wait(20000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 1.0, elapsed           # it waited about its limit, then returned
    assert pool.check_errors() == al.LORA_ERR_TIMEOUT
    assert pool.check_errors() == al.LORA_OK        # reading the status clears it
    # the context is still usable: a layer call afterwards is correct
    Y = to_host_f64(pool.linear(to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids)))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    ref = oracle.lora_linear(prob.X, prob.W, prob.ids, oracle.problem_adapters(prob),
                             prob.max_adapters)
    assert_parity(Y, ref, "after a timed-out wait")
    with pytest.raises(al.LoraError) as e:
        pool.selftest_wait(0)
    assert e.value.status == al.LORA_ERR_ARG
    pool.close()
