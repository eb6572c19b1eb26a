"""GPU parity of adapter chains (lora_define_chain) against the fp64 oracle's chain
definition, on both kernel families, plus the chain management rules.

A chain slot stands for its members applied together: a token with that id gets the
sum of the members' low-rank branches. Same tolerance as the single-adapter tests.
"""
import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import assert_parity, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")

PATHS = {"decode": 1, "prefill": 2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


def make(seed, T, d_in, d_out, ranks, chains, max_rank, n_slots=16, std=0.1):
    """Adapters in slots 0..len(ranks)-1, chains in the given slots; ids over
    -1, the adapters and the chains."""
    ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 2.0 * r + i, std=std)
           for i, r in enumerate(ranks)}
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 1.0 / 16)
    choices = [-1] + list(ads) + list(chains)
    ids = np.array(L.rng_for(seed, L.ROLE_IDS).choice(choices, size=T), np.int32)
    pool = al.LoraPool(n_slots, max_rank, d_in, d_out)
    for s, a in ads.items():
        pool.load_adapter(s, to_dev(a.A), to_dev(a.B), a.rank, a.alpha)
    for c, members in chains.items():
        pool.define_chain(c, members)
    tup = {s: (a.A, a.B, a.rank, a.alpha) for s, a in ads.items()}
    return pool, X, W, ids, tup


def run(pool, X, W, ids, path):
    pool.set_path(PATHS[path])
    Y = pool.linear(to_dev(X), to_dev(W), to_dev(ids))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    return Y


@pytest.mark.parametrize("path,T", [("decode", 1), ("decode", 100), ("decode", 256),
                                    ("prefill", 100), ("prefill", 700)])
def test_chains_mixed_ranks(path, T):
    chains = {10: [0, 1], 11: [2, 3, 4], 12: [4], 13: [1, 3]}
    pool, X, W, ids, ads = make(31, T, 264, 200, [3, 8, 13, 16, 5], chains, max_rank=64)
    got = to_host_f64(run(pool, X, W, ids, path))
    ref = oracle.lora_linear_chains(X, W, oracle.chain_lists(ids, chains), ads, 16)
    assert_parity(got, ref, f"chains/{path}/T={T}")
    # the branches themselves are reproduced, not hidden in the tolerance
    base = oracle.lora_linear(X, W, np.full_like(ids, -1), {}, 16)
    rows = np.array([i in chains for i in ids.tolist()])
    if rows.any():
        d_ref, d_got = (ref - base)[rows], (got - base)[rows]
        assert np.mean(np.abs(d_got - d_ref)) < 0.25 * np.mean(np.abs(d_ref))
    pool.close()


def test_chain_q_proj_decode():
    """Llama-2-7B q_proj shapes: 200 x r16 adapters, chains of two (rank 32)."""
    prob = L.q_proj_decode()
    chains = {200 + k: [2 * k, 2 * k + 1] for k in range(20)}
    pool = al.LoraPool(prob.max_adapters + 20, 32, prob.d_in, prob.d_out)
    for s, a in prob.adapters.items():
        pool.load_adapter(s, to_dev(a.A), to_dev(a.B), a.rank, a.alpha)
    for c, m in chains.items():
        pool.define_chain(c, m)
    ids = prob.ids.copy()
    ids[::3] = 200 + (np.arange(len(ids[::3])) % 20)
    got = to_host_f64(run(pool, prob.X, prob.W, ids, "decode"))
    ads = oracle.problem_adapters(prob)
    ref = oracle.lora_linear_chains(prob.X, prob.W, oracle.chain_lists(ids, chains), ads,
                                    prob.max_adapters + 20)
    assert_parity(got, ref, "q_proj chains")
    pool.close()


@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_chain_of_one_is_its_member_bitwise(path):
    pool, X, W, ids, _ = make(32, 300 if path == "prefill" else 64, 136, 72, [5, 16], {9: [1]},
                              max_rank=16)
    ids_member = np.where(ids == 9, 1, ids).astype(np.int32)
    ids_chain = np.where(ids == 1, 9, ids_member).astype(np.int32)
    a = run(pool, X, W, ids_member, path)
    b = run(pool, X, W, ids_chain, path)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    pool.close()


def test_chain_management():
    # three pages a slot: adapters of 1, 2 and 1 pages
    pool, X, W, ids, _ = make(33, 8, 64, 64, [8, 16, 8], {}, max_rank=24, n_slots=8)
    E = al.LoraError
    with pytest.raises(E) as e:
        pool.define_chain(0, [1, 2])                  # slot 0 holds an adapter
    assert e.value.status == al.LORA_ERR_SLOT_OCCUPIED
    with pytest.raises(E) as e:
        pool.define_chain(5, [1, 6])                  # slot 6 is empty
    assert e.value.status == al.LORA_ERR_SLOT_EMPTY
    with pytest.raises(E) as e:
        pool.define_chain(5, [1, 1])                  # a repeated member
    assert e.value.status == al.LORA_ERR_ARG
    with pytest.raises(E) as e:
        pool.define_chain(5, [0, 1, 2])               # 1 + 2 + 1 pages > 3
    assert e.value.status == al.LORA_ERR_RANK
    with pytest.raises(E) as e:
        pool.define_chain(8, [0])
    assert e.value.status == al.LORA_ERR_SLOT_RANGE
    with pytest.raises(E) as e:
        pool.define_chain(5, [])
    assert e.value.status == al.LORA_ERR_ARG
    pool.define_chain(5, [0, 1])
    with pytest.raises(E) as e:
        pool.define_chain(6, [5])                     # a chain is not a member
    assert e.value.status == al.LORA_ERR_ARG
    with pytest.raises(E) as e:
        pool.unload_adapter(1)                        # listed by chain 5
    assert e.value.status == al.LORA_ERR_IN_USE
    free_before = pool.stats()["free_pages"]
    pool.unload_adapter(5)                            # the chain owns no pages
    assert pool.stats()["free_pages"] == free_before
    pool.unload_adapter(1)
    assert pool.stats()["free_pages"] == free_before + 2
    # a chain over a reloaded member computes with the new weights
    new = L.make_adapter(34, 1, 64, 64, 16, 8.0, std=0.1)
    pool.load_adapter(1, to_dev(new.A), to_dev(new.B), 16, 8.0)
    pool.define_chain(5, [1, 2])
    two = L.make_adapter(33, 2, 64, 64, 8, 2.0 * 8 + 2, std=0.1)  # as make() loaded it
    ads = {1: (new.A, new.B, 16, 8.0), 2: (two.A, two.B, 8, 2.0 * 8 + 2)}
    ids = np.array([5, -1, 5, 2, 1, 5, 5, -1], np.int32)
    got = to_host_f64(run(pool, X, W, ids, "decode"))
    ref = oracle.lora_linear_chains(X, W, oracle.chain_lists(ids, {5: [1, 2]}), ads, 8)
    assert_parity(got, ref, "chain after member reload")
    pool.close()
