"""Stream order under programmatic dependent launch (no GPU fault involved).

The decode kernels start before the kernel ahead of them in the stream has finished
(their weight loads and table reads overlap it); whatever they read that belongs to
the stream's order must still be taken after their wait on that kernel. The test hook
lora_test_delayed_copy is such a kernel: it lets the next kernel launch at once and
writes the token ids only ~200 us later. The layer must then use the new ids, on
both paths; a read of the ids before the wait would mix in the old ones.
"""
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


@pytest.mark.parametrize("path", [al.LORA_PATH_DECODE, al.LORA_PATH_PREFILL])
def test_ids_written_late_by_the_previous_kernel(path):
    d, T, seed = 512, 64, 71
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 32)
    ads = {i: L.make_adapter(seed, i, d, d, 16, 32.0, std=0.05) for i in range(8)}
    g = L.rng_for(seed, L.ROLE_IDS)
    ids_old = g.integers(0, 8, size=T).astype(np.int32)
    ids_new = ((ids_old + 1 + g.integers(0, 7, size=T)) % 8).astype(np.int32)  # differs everywhere
    assert np.all(ids_old != ids_new)
    prob = L.Problem("stream_order", d, d, X, W, ids_new, ads, 8, 16, seed)
    pool = load_pool(al, prob)
    pool.set_path(path)
    Xd, Wd = to_dev(X), to_dev(W)
    ids_dev = to_dev(ids_old)
    src = to_dev(ids_new)
    ref = oracle.lora_linear(X, W, ids_new, oracle.problem_adapters(prob), prob.max_adapters)
    for _ in range(3):
        ids_dev.copy_(to_dev(ids_old))
        torch.cuda.synchronize()
        al.delayed_copy(src, ids_dev, T, 200)
        Y = pool.linear(Xd, Wd, ids_dev)
        torch.cuda.synchronize()
        assert pool.check_errors() == al.LORA_OK
        assert_parity(to_host_f64(Y), ref, f"ids written late (path {path})")
    pool.close()


def test_delayed_copy_rejects_bad_arguments():
    a = torch.zeros(4, dtype=torch.int32, device="cuda")
    for n, delay in ((-1, 10), (4, 0), (4, 100001)):
        assert al.load_library().lora_test_delayed_copy(a.data_ptr(), a.data_ptr(), n, delay, None) == al.LORA_ERR_ARG
