"""The pool's cache of TMA descriptors (a small ring per pool) across many calls with
different buffers: a lookup that hits an entry must not lose it to a later lookup of
the same call. With the same W and a fresh X buffer per call, the ring's victim comes
round to W's own entry within a few calls; every call must still give the first
call's output bit for bit, with no error reported.
"""
import numpy as np
import pytest

import lora_inputs as L
from _helpers import load_pool, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("path,T", [("decode", 16), ("prefill", 200)])
def test_many_buffers_same_result(path, T):
    d, seed = 256, 97
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 16)
    ids = np.repeat(np.arange(4, dtype=np.int32), T // 4 + 1)[:T]
    ads = {i: L.make_adapter(seed, i, d, d, 8, 16.0) for i in range(4)}
    prob = L.Problem("tmap_cache", d, d, X, W, ids, ads, 4, 8, seed)
    pool = load_pool(al, prob)
    pool.set_path(al.LORA_PATH_DECODE if path == "decode" else al.LORA_PATH_PREFILL)
    Wd, idsd = to_dev(W), to_dev(ids)
    keep, outs = [], []
    for _ in range(10):  # more calls than the ring has entries, each with a new X and Y
        Xd = to_dev(X)
        keep.append(Xd)
        outs.append(pool.linear(Xd, Wd, idsd))
        torch.cuda.synchronize()
        assert pool.check_errors() == al.LORA_OK
    for i, Y in enumerate(outs[1:], 1):
        assert torch.equal(Y, outs[0]), f"call {i} differs"
    pool.close()
