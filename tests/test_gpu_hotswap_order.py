"""Hot swap without a device-wide stall (icman.com.cn Multi-LoRA article, section 4.2:
a cold adapter load must not hold up the requests already running).

A bounded 50 ms kernel (the stream-order test hook, copying into an unrelated buffer)
runs on a second stream while the pool is used on a first one. An unload + load of one
of the pool's slots must return while that kernel still runs; the call enqueued before
the swap must still use the old adapter and the call enqueued after it the new one
(oracle parity on both); the caller may overwrite the A and B it passed as soon as the
load returns. On an ordinary stream the error-word read returns while the other kernel
runs as well. On the legacy default stream it may not: CUDA completes an event recorded
there only after all earlier work of the context, other streams included, and the pool
learns that its calls have finished from such an event.
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

DELAY_US = 50000


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("stream_kind", ["side", "legacy"])
@pytest.mark.parametrize("path", [al.LORA_PATH_DECODE, al.LORA_PATH_PREFILL])
def test_swap_does_not_wait_for_other_streams(path, stream_kind):
    d, T, seed, slot = 512, 64, 73, 3
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 32)
    ads = {i: L.make_adapter(seed, i, d, d, 16, 32.0, std=0.05) for i in range(8)}
    ids = L.rng_for(seed, L.ROLE_IDS).integers(0, 8, size=T).astype(np.int32)
    ids[::4] = slot                                   # the swapped slot is well used
    old = L.Problem("swap_old", d, d, X, W, ids, ads, 8, 16, seed)
    fresh = L.make_adapter(seed, slot, d, d, 16, 32.0, std=0.05, generation=1)
    new_ads = dict(ads)
    new_ads[slot] = fresh
    new = L.Problem("swap_new", d, d, X, W, ids, new_ads, 8, 16, seed)

    pool = load_pool(al, old)
    pool.set_path(path)
    pool.reserve(T)
    Xd, Wd, idsd = to_dev(X), to_dev(W), to_dev(ids)
    A_new, B_new = to_dev(fresh.A), to_dev(fresh.B)
    main = torch.cuda.Stream() if stream_kind == "side" else torch.cuda.default_stream()
    pool.linear(Xd, Wd, idsd, stream=main)            # warm (modules, tensor maps)
    torch.empty(8, dtype=torch.bfloat16, device="cuda").fill_(float("nan"))  # torch's fill kernel
    torch.cuda.synchronize()                          # loaded now, not behind the long kernel

    other = torch.cuda.Stream()
    src = torch.arange(16, dtype=torch.int32, device="cuda")
    dst = torch.zeros(16, dtype=torch.int32, device="cuda")
    done_other = torch.cuda.Event()
    al.delayed_copy(src, dst, 16, DELAY_US, stream=other)
    done_other.record(other)

    Y_before = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    Y_after = torch.empty_like(Y_before)
    pool.linear(Xd, Wd, idsd, Y_before, stream=main)
    t0 = time.perf_counter()
    pool.unload_adapter(slot)
    pool.load_adapter(slot, A_new, B_new, 16, 32.0)
    swap_s = time.perf_counter() - t0
    swapped_while_running = not done_other.query()
    with torch.cuda.stream(main):
        A_new.fill_(float("nan"))                     # the caller's copies are free again
        B_new.fill_(float("nan"))
    pool.linear(Xd, Wd, idsd, Y_after, stream=main)
    st = pool.check_errors()
    checked_while_running = not done_other.query()
    torch.cuda.synchronize()

    assert st == al.LORA_OK
    assert swapped_while_running, f"the swap waited for another stream ({swap_s * 1e3:.1f} ms)"
    assert swap_s < 0.5 * DELAY_US * 1e-6
    if stream_kind == "side":
        assert checked_while_running, "the error-word read waited for another stream"
    assert torch.equal(dst, src)
    for Y, prob, what in ((Y_before, old, "call before the swap"), (Y_after, new, "call after the swap")):
        ref = oracle.lora_linear(X, W, ids, oracle.problem_adapters(prob), prob.max_adapters)
        assert_parity(to_host_f64(Y), ref, what)
    pool.close()


def test_unload_then_bad_id_is_reported():
    """A call enqueued after an unload sees the slot empty: its id is a strict error."""
    d, T, seed = 256, 32, 79
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 16)
    ads = {i: L.make_adapter(seed, i, d, d, 8, 16.0) for i in range(2)}
    ids = np.zeros(T, np.int32)
    prob = L.Problem("unload_bad_id", d, d, X, W, ids, ads, 2, 8, seed)
    pool = load_pool(al, prob)
    Xd, Wd, idsd = to_dev(X), to_dev(W), to_dev(ids)
    pool.linear(Xd, Wd, idsd)
    pool.unload_adapter(0)
    pool.linear(Xd, Wd, idsd)
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_ERR_BAD_ADAPTER_ID
    assert pool.check_errors() == al.LORA_OK        # read and cleared
    pool.close()


def test_back_to_back_swaps_on_a_full_pool():
    """Four unload + reload swaps of one slot of a full pool, each followed by a call,
    while every call is held back behind a bounded 50 ms kernel on the calls' stream: the
    first two swaps write the pool's reserve pages at once (no enqueued call can read
    them); the next two find only pages freed by the earlier swaps, whose calls have not
    run yet, and must write those on the copy stream after them. Every call sees the
    adapter generation loaded when it was enqueued (oracle parity on each)."""
    d, T, seed, slot, n = 256, 64, 83, 2, 4
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 16)
    ads = {i: L.make_adapter(seed, i, d, d, 16, 32.0, std=0.05) for i in range(n)}
    ids = L.rng_for(seed, L.ROLE_IDS).integers(-1, n, size=T).astype(np.int32)
    ids[::3] = slot
    prob = L.Problem("full_pool_swaps", d, d, X, W, ids, ads, n, 16, seed)
    gens = [ads[slot]] + [L.make_adapter(seed, slot, d, d, 16, 32.0, std=0.05, generation=g)
                          for g in range(1, 5)]

    pool = load_pool(al, prob)
    pool.set_path(al.LORA_PATH_DECODE)
    pool.reserve(T)
    st = pool.stats()
    assert st["total_pages"] == 2 * n and st["free_pages"] == 0     # full
    Xd, Wd, idsd = to_dev(X), to_dev(W), to_dev(ids)
    main = torch.cuda.Stream()
    pool.linear(Xd, Wd, idsd, stream=main)            # warm
    new_AB = [(to_dev(a.A), to_dev(a.B)) for a in gens]
    torch.cuda.synchronize()

    src = torch.arange(16, dtype=torch.int32, device="cuda")
    dst = torch.zeros(16, dtype=torch.int32, device="cuda")
    al.delayed_copy(src, dst, 16, DELAY_US, stream=main)  # holds back every call below
    Ys = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for _ in gens]
    pool.linear(Xd, Wd, idsd, Ys[0], stream=main)
    for g in range(1, len(gens)):
        pool.unload_adapter(slot)
        pool.load_adapter(slot, new_AB[g][0], new_AB[g][1], 16, 32.0)
        pool.linear(Xd, Wd, idsd, Ys[g], stream=main)
    torch.cuda.synchronize()

    assert pool.check_errors() == al.LORA_OK
    assert torch.equal(dst, src)
    st = pool.stats()
    assert st["total_pages"] == 2 * n and st["free_pages"] == 0
    for g, Y in enumerate(Ys):
        tup = {s: (a.A, a.B, a.rank, a.alpha) for s, a in ads.items()}
        tup[slot] = (gens[g].A, gens[g].B, 16, 32.0)
        ref = oracle.lora_linear(X, W, ids, tup, n)
        assert_parity(to_host_f64(Y), ref, f"call after swap {g}")
    pool.close()
