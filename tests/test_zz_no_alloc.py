"""The allocation-free entry point, lora_base_linear_noalloc.

It serves callers that may not call cudaMalloc (code inside another
framework's memory arena, plugins whose host forbids device allocation): it
takes its scratch from a fixed array compiled into the library. Its output
must match the fp64 oracle's base product (every token id -1) and the
pool-based lora_base_linear (same kernels, pool-owned scratch) within the
layer's tolerance, on two calls in a row (the second call finds the first
call's leftovers in the shared array). This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import ATOL, RTOL, assert_parity, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


ARRAY_FLOATS = 4 << 20   # the fixed array: 16 MiB of fp32 partial sums


def test_the_largest_case_runs_with_fewer_ctas():
    """(256, 4096, 16384): the full stream-K split's partial sums exceed the array, so the
    call takes the reduced-CTA branch, and its plan at the reduced count fits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    full = al.decode_plan_info(256, [4096], [16384], [0], sms)
    assert full["partials_floats"] > ARRAY_FLOATS
    plan = full
    while plan["partials_floats"] > ARRAY_FLOATS:   # the entry point's own reduction rule
        assert plan["G"] > 1
        fit = ARRAY_FLOATS // (plan["max_seg"] * 256 * 128)
        plan = al.decode_plan_info(256, [4096], [16384], [0],
                                   max(fit, 1) if fit < plan["G"] else plan["G"] - 1)
    assert 1 <= plan["G"] < full["G"]


# (256, 4096, 16384) takes the reduced-CTA branch (see the test above)
@pytest.mark.parametrize("T,d_in,d_out", [(64, 4096, 4096), (37, 72, 136), (256, 4096, 8192),
                                          (256, 4096, 16384)])
def test_noalloc_matches_pool_entry_twice(T, d_in, d_out):
    seed = 41
    Wh = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 1.0 / 64)
    W = to_dev(Wh)
    pool = al.LoraPool(1, 8, d_in, d_out)
    for call in range(2):
        Xh = L.normal_bf16(seed, L.ROLE_X, call, (T, d_in), 1.0)
        X = to_dev(Xh)
        ref = to_host_f64(pool.base_linear(X, W))
        Y = torch.full((T, d_out), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = al.lora_base_linear_noalloc(X, W, T, d_in, d_out, Y)
        assert st == al.LORA_OK, al.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        got = to_host_f64(Y)
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)), f"call {call}"
        exact = oracle.lora_linear(Xh, Wh, np.full(T, -1, np.int32), {}, 1)
        assert_parity(got, exact, f"noalloc vs oracle, call {call}")
    pool.close()


def test_noalloc_rejects_what_does_not_fit():
    # 512 tiles of 128 output rows x 256 tokens of fp32 partials exceed the array
    # whatever the number of CTAs
    Ww = torch.zeros((65536, 64), dtype=torch.bfloat16, device="cuda")
    Xw = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    Yw = torch.empty((256, 65536), dtype=torch.bfloat16, device="cuda")
    assert al.lora_base_linear_noalloc(Xw, Ww, 256, 64, 65536, Yw) == al.LORA_ERR_SHAPE
    W = torch.zeros((16384, 4096), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((256, 4096), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((256, 16384), dtype=torch.bfloat16, device="cuda")
    assert al.lora_base_linear_noalloc(X, W, 257, 4096, 16384, Y) == al.LORA_ERR_ARG
    assert al.lora_base_linear_noalloc(X, W, 8, 4090, 16384, Y) == al.LORA_ERR_SHAPE
    assert al.lora_base_linear_noalloc(None, W, 8, 4096, 16384, Y) == al.LORA_ERR_ARG
