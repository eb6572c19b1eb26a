"""The cases the range-checked build runs (child process of test_gpu_checked_build.py).

Started with ADAPTER_LINEAR_CHECKED=1, so the binding loads liblora_linear_check.so
(LORA_CHECK: every index a kernel gathers through a table is range-checked first).
Valid inputs only: every call must report LORA_OK (no index out of range) and match the
fp64 oracle. Prints one line per case and exits non-zero on the first failure.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import torch  # noqa: E402

import adapter_linear_gb300 as al  # noqa: E402
import lora_inputs as L  # noqa: E402
import oracle  # noqa: E402
from _helpers import assert_parity, load_pool, to_dev, to_host_f64  # noqa: E402


def check(pool, prob, path, kernel, what):
    pool.set_path(path)
    pool.set_prefill_kernel(kernel)
    Y = pool.linear(to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids))
    torch.cuda.synchronize()
    st = pool.check_errors()
    assert st == al.LORA_OK, f"{what}: {al.STATUS_NAMES.get(st, st)}"
    ref = oracle.lora_linear(prob.X, prob.W, prob.ids, oracle.problem_adapters(prob), prob.max_adapters)
    assert_parity(to_host_f64(Y), ref, what)
    print("ok", what, flush=True)


def main():
    assert al.CHECKED and al.LIB_PATH.endswith("liblora_linear_check.so"), al.LIB_PATH
    al.load_library()
    torch.cuda.set_device(0)
    runs = [(al.LORA_PATH_DECODE, al.LORA_PREFILL_AUTO, "decode"),
            (al.LORA_PATH_PREFILL, al.LORA_PREFILL_SINGLE, "prefill/single"),
            (al.LORA_PATH_PREFILL, al.LORA_PREFILL_PAIR, "prefill/pair")]
    prob = L.tiny()
    pool = load_pool(al, prob)
    for path, kernel, name in runs:
        check(pool, prob, path, kernel, f"tiny {name}")
    pool.close()
    d_in, d_out, seed = 72, 136, 31
    ranks = [1, 5, 13, 24, 40]
    for T in (1, 37, 256, 300):
        X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
        W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
        ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 1.5 * r, std=0.2) for i, r in enumerate(ranks)}
        ids = L.rng_for(seed, L.ROLE_IDS, T).integers(-1, len(ranks), size=T).astype(np.int32)
        ids[: T // 3] = 3                          # a single-adapter stretch (tensor-core expand)
        prob = L.Problem("ragged", d_in, d_out, X, W, ids, ads, len(ranks), 40, seed)
        pool = load_pool(al, prob)
        for path, kernel, name in runs:
            if path == al.LORA_PATH_DECODE and T > 256:
                continue
            check(pool, prob, path, kernel, f"ragged T={T} {name}")
        pool.close()
    print("all ok", flush=True)


if __name__ == "__main__":
    main()
