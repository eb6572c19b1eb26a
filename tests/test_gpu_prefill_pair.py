"""The prefill path's two GEMM kernels on the same inputs, against the oracle: one CTA per
128-token x 256-column tile, and a CTA pair (cluster of two, tcgen05 MMAs spanning both
SMs) per 256 x 256 tile. The pair kernel decides per 256-token tile whether the expand
runs on the tensor cores (every adapter token of the 256 uses one adapter) or in each
CTA's epilogue (the halves use different adapters, or a half is mixed); the cases below
put each combination of halves in its own tile, with a d_out tail that leaves the second
CTA's column half empty and a ragged last tile whose second half has no tokens.
"""
import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import assert_parity, assert_routing, load_pool, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")

KERNELS = {"single": 1, "pair": 2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


def run(pool, prob, kernel):
    pool.set_path(al.LORA_PATH_PREFILL)
    pool.set_prefill_kernel(KERNELS[kernel])
    Y = pool.linear(to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    return Y


def tile_mode_problem():
    d_in, d_out, seed = 136, 520, 61
    T = 5 * 256 + 77
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
    ranks = [5, 40, 13, 64]        # rank 64: two expand k-blocks
    ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 2.0 * r, std=0.2) for i, r in enumerate(ranks)}
    g = L.rng_for(seed, L.ROLE_IDS)
    ids = np.full(T, -1, np.int32)
    ids[0:256] = 3                 # one adapter over both halves (tensor-core expand) ...
    ids[40:44] = -1                # ... with base rows inside
    ids[256:384] = 1               # halves with different adapters: epilogue expand
    ids[384:512] = 2
    ids[300] = -1
    ids[512:640] = 0               # one adapter and a base-only half: tensor-core expand
    ids[768:896] = -1              # a base-only half beside a mixed half
    ids[896:1024] = g.integers(-1, 4, size=128)
    ids[1024:1280] = -1            # all base
    ids[1280:] = g.integers(-1, 4, size=T - 1280)   # mixed, ragged (second half empty)
    return L.Problem("pair_tile_modes", d_in, d_out, X, W, ids, ads, 4, 64, seed)


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_tile_modes(kernel):
    prob = tile_mode_problem()
    pool = load_pool(al, prob)
    got = to_host_f64(run(pool, prob, kernel))
    ads = oracle.problem_adapters(prob)
    ref = oracle.lora_linear(prob.X, prob.W, prob.ids, ads, prob.max_adapters)
    base = oracle.lora_linear(prob.X, prob.W, np.full_like(prob.ids, -1), {}, prob.max_adapters)
    assert_parity(got, ref, f"prefill tile modes ({kernel})")
    assert_routing(got, ref, base, prob.ids, f"prefill tile modes ({kernel})")
    pool.close()


@pytest.mark.parametrize("T", [129, 255, 256, 257, 511, 640])
def test_pair_ragged_token_counts(T):
    """Token counts around the pair tile: a second half with a few rows, exactly one tile,
    one row past it, and several tiles of random ids."""
    d_in, d_out, seed = 72, 264, 67
    X = L.normal_bf16(seed, L.ROLE_X, T, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
    ranks = [8, 24, 3]
    ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 1.5 * r, std=0.2) for i, r in enumerate(ranks)}
    ids = L.rng_for(seed, L.ROLE_IDS, T).integers(-1, len(ranks), size=T).astype(np.int32)
    ids[: T // 2] = 1              # a single-adapter stretch as well
    prob = L.Problem("pair_ragged", d_in, d_out, X, W, ids, ads, len(ranks), 24, seed)
    pool = load_pool(al, prob)
    got = to_host_f64(run(pool, prob, "pair"))
    ref = oracle.lora_linear(prob.X, prob.W, prob.ids, oracle.problem_adapters(prob), prob.max_adapters)
    assert_parity(got, ref, f"pair kernel T={T}")
    pool.close()


def test_prefill_kernel_setter():
    prob = L.tiny()
    pool = load_pool(al, prob)
    for bad in (-1, 3):
        assert al.lora_pool_set_prefill_kernel(pool.handle, bad) == al.LORA_ERR_ARG
    # T <= 128 under AUTO takes the single-CTA kernel; PAIR forced runs the pair kernel
    # on a tile whose second half is empty
    for kernel in ("single", "pair"):
        got = to_host_f64(run(pool, prob, kernel))
        ref = oracle.lora_linear(prob.X, prob.W, prob.ids, oracle.problem_adapters(prob), prob.max_adapters)
        assert_parity(got, ref, f"tiny, {kernel} kernel")
    pool.set_prefill_kernel(al.LORA_PREFILL_AUTO)
    pool.close()


def test_pair_random_shapes():
    """Seeded random shapes (d_in, d_out multiples of 8 that are not multiples of the
    tiles; T past one pair tile), ranks and id mixes, each against the oracle."""
    g = np.random.default_rng(97)
    for case in range(12):
        d_in = int(8 * g.integers(1, 160))
        d_out = int(8 * g.integers(1, 200))
        T = int(g.integers(129, 1400))
        n_ad = int(g.integers(1, 6))
        ranks = [int(r) for r in g.integers(1, 65, size=n_ad)]
        seed = 200 + case
        X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
        W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
        ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 2.0 * r, std=0.1) for i, r in enumerate(ranks)}
        ids = g.integers(-1, n_ad, size=T).astype(np.int32)
        if case % 3 == 0:              # long single-adapter runs (tensor-core expand)
            ids = np.repeat(g.integers(-1, n_ad, size=-(-T // 300)), 300)[:T].astype(np.int32)
        prob = L.Problem("pair_random", d_in, d_out, X, W, ids, ads, n_ad, max(ranks), seed)
        pool = load_pool(al, prob)
        got = to_host_f64(run(pool, prob, "pair"))
        ref = oracle.lora_linear(X, W, ids, oracle.problem_adapters(prob), prob.max_adapters)
        assert_parity(got, ref, f"pair kernel, case {case}: T={T} {d_in}->{d_out} ranks {ranks}")
        pool.close()


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_shrink_rows_left_by_an_earlier_call(kernel):
    """The shrink output is not cleared between calls: a row of a token without an
    adapter is zeroed by the segment builder, and the columns past an adapter's own
    32-column groups are never read. Call 1 writes every row at rank 64; call 2 puts
    base-only tokens (and a rank-8 adapter) where those rows were."""
    d_in, d_out, seed, T = 136, 264, 83, 512
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
    ads = {0: L.make_adapter(seed, 0, d_in, d_out, 64, 128.0, std=0.2),
           1: L.make_adapter(seed, 1, d_in, d_out, 8, 16.0, std=0.2)}
    ids1 = np.zeros(T, np.int32)                       # every row at rank 64
    ids2 = np.full(T, 1, np.int32)
    ids2[3:40] = -1                                    # base rows inside single-adapter tiles
    ids2[300:310] = -1
    ids2[384:] = -1                                    # a base-only tile
    pool = None
    for ids in (ids1, ids2):
        prob = L.Problem("stale_rows", d_in, d_out, X, W, ids, ads, 2, 64, seed)
        if pool is None:
            pool = load_pool(al, prob)
        got = to_host_f64(run(pool, prob, kernel))
        ref = oracle.lora_linear(X, W, ids, oracle.problem_adapters(prob), prob.max_adapters)
        assert_parity(got, ref, f"rows left by an earlier call ({kernel})")
    pool.close()
