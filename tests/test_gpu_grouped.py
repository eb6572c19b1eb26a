"""GPU parity of lora_linear_grouped (several layers sharing one batch of ids in one
decode launch chain) against the fp64 CPU oracle, layer by layer, through the C ABI.

Same tolerance as the single-layer tests. The grouped call's stream-K split runs over
all layers' weights at once, so a CTA's range can cross layers and cover more tiles
than the TMEM accumulator ring holds; the shapes below exercise both.
"""
import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import assert_parity, assert_routing, load_pool, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


def ref_of(prob):
    ads = oracle.problem_adapters(prob)
    Y = oracle.lora_linear(prob.X, prob.W, prob.ids, ads, prob.max_adapters)
    Yb = oracle.lora_linear(prob.X, prob.W, np.full_like(prob.ids, -1), {}, prob.max_adapters)
    return Y, Yb


def grouped(pools, probs, ids):
    Ys = al.LoraPool.linear_grouped(pools, [to_dev(p.X) for p in probs],
                                    [to_dev(p.W) for p in probs], to_dev(ids))
    torch.cuda.synchronize()
    for pool in pools:
        assert pool.check_errors() == al.LORA_OK
    return Ys


def small_layers(T, seed=11):
    """Ragged layer shapes (not multiples of 128), mixed ranks, one id vector."""
    shapes = [(136, 200, 8), (64, 8, 16), (264, 1000, 24), (4096, 384, 64), (8, 136, 1)]
    g = L.rng_for(seed, L.ROLE_IDS)
    n_ad = 6
    ids = g.integers(-1, n_ad, size=T).astype(np.int32)
    probs = []
    for i, (d_in, d_out, rank) in enumerate(shapes):
        s = seed * 100 + i
        X = L.normal_bf16(s, L.ROLE_X, 0, (T, d_in), 1.0)
        W = L.normal_bf16(s, L.ROLE_W, 0, (d_out, d_in), 1.0 / 16)
        ads = {a: L.make_adapter(s, a, d_in, d_out, rank, 2.0 * rank, std=0.1)
               for a in range(n_ad)}
        probs.append(L.Problem(f"small{i}", d_in, d_out, X, W, ids.copy(), ads,
                               max_adapters=n_ad, max_rank=rank, seed=s))
    return probs, ids


def test_grouped_llama3_layer():
    """The seven target modules of a Llama-3-8B layer (T = 32, shared ids) in one call."""
    probs = L.llama3_7mod()
    pools = [load_pool(al, p) for p in probs]
    Ys = grouped(pools, probs, probs[0].ids)
    for p, pool, Y in zip(probs, pools, Ys):
        got = to_host_f64(Y)
        ref, base = ref_of(p)
        assert_parity(got, ref, f"grouped/{p.name}")
        assert_routing(got, ref, base, p.ids, f"grouped/{p.name}")
        # the single-layer call computes the same thing (up to the split-K sum order)
        single = to_host_f64(pool.linear(to_dev(p.X), to_dev(p.W), to_dev(p.ids)))
        assert_parity(single, ref, f"single/{p.name}")
    for pool in pools:
        pool.close()


@pytest.mark.parametrize("T", [1, 37, 256])
def test_grouped_ragged_layers(T):
    probs, ids = small_layers(T)
    pools = [load_pool(al, p) for p in probs]
    Ys = grouped(pools, probs, ids)
    for p, Y in zip(probs, Ys):
        got = to_host_f64(Y)
        ref, base = ref_of(p)
        assert_parity(got, ref, f"grouped T={T}/{p.name}")
        assert_routing(got, ref, base, p.ids, f"grouped T={T}/{p.name}")
    for pool in pools:
        pool.close()


def test_grouped_one_layer_equals_linear_bitwise():
    """n = 1 runs exactly the single-layer plan: bit-identical to lora_linear."""
    (prob,) = L.llama3_7mod(modules=["q_proj"])
    pool = load_pool(al, prob)
    (Yg,) = grouped([pool], [prob], prob.ids)
    Ys = pool.linear(to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids))
    torch.cuda.synchronize()
    assert torch.equal(Yg.view(torch.int16), Ys.view(torch.int16))
    again = grouped([pool], [prob], prob.ids)[0]
    assert torch.equal(Yg.view(torch.int16), again.view(torch.int16))  # deterministic
    pool.close()


def test_accumulator_ring_wraps():
    """A wide layer at T = 200: each CTA range covers ~4 tiles of 128 rows while the
    TMEM ring holds 2 accumulators of 208 columns, so slots are recycled."""
    T, d_in, d_out = 200, 128, 65536
    s = 9001
    g = L.rng_for(s, L.ROLE_IDS)
    ids = g.integers(-1, 3, size=T).astype(np.int32)
    X = L.normal_bf16(s, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(s, L.ROLE_W, 0, (d_out, d_in), 1.0 / 16)
    ads = {a: L.make_adapter(s, a, d_in, d_out, 16, 32.0, std=0.1) for a in range(3)}
    prob = L.Problem("wide", d_in, d_out, X, W, ids, ads, max_adapters=3, max_rank=16, seed=s)
    pool = load_pool(al, prob)
    (Y,) = grouped([pool], [prob], ids)
    got = to_host_f64(Y)
    ref, base = ref_of(prob)
    assert_parity(got, ref, "ring wrap")
    assert_routing(got, ref, base, ids, "ring wrap")
    pool.close()


def test_grouped_prefill_sized_batch_runs_per_layer():
    probs, ids = small_layers(300, seed=12)
    pools = [load_pool(al, p) for p in probs]
    Ys = grouped(pools, probs, ids)
    for p, Y in zip(probs, Ys):
        assert_parity(to_host_f64(Y), ref_of(p)[0], f"grouped prefill/{p.name}")
    for pool in pools:
        pool.close()


def test_grouped_errors():
    probs, ids = small_layers(16, seed=13)
    pools = [load_pool(al, p) for p in probs[:2]]
    Xs = [to_dev(p.X) for p in probs[:2]]
    Ws = [to_dev(p.W) for p in probs[:2]]
    Ys = [torch.empty((16, p.d_out), dtype=torch.bfloat16, device="cuda") for p in probs[:2]]
    d_ids = to_dev(ids)
    h = [p.handle for p in pools]
    assert al.lora_linear_grouped([], [], [], d_ids, 16, []) == al.LORA_ERR_ARG
    assert al.lora_linear_grouped(h * 5, Xs * 5, Ws * 5, d_ids, 16, Ys * 5) == al.LORA_ERR_ARG
    assert al.lora_linear_grouped([h[0], h[0]], Xs, Ws, d_ids, 16, Ys) == al.LORA_ERR_ARG
    assert al.lora_linear_grouped(h, [Xs[0], None], Ws, d_ids, 16, Ys) == al.LORA_ERR_ARG
    assert al.lora_linear_grouped(h, Xs, Ws, None, 16, Ys) == al.LORA_ERR_ARG
    assert al.lora_linear_grouped(h, Xs, Ws, d_ids, -1, Ys) == al.LORA_ERR_ARG
    assert al.lora_linear_grouped(h, Xs, Ws, d_ids, 0, Ys) == al.LORA_OK
    # strict mode: an id no pool holds is reported by every layer's pool
    bad = ids.copy()
    bad[3] = 5000
    assert al.lora_linear_grouped(h, Xs, Ws, to_dev(bad), 16, Ys) == al.LORA_OK
    torch.cuda.synchronize()
    for pool in pools:
        assert pool.check_errors() == al.LORA_ERR_BAD_ADAPTER_ID
        assert pool.check_errors() == al.LORA_OK
    for pool in pools:
        pool.close()
