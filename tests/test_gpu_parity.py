"""GPU parity of lora_linear against the fp64 CPU oracle, through the C ABI.

Floating point: |Y_gpu - Y_ref| <= 1e-2 + 1e-2 |Y_ref| elementwise, plus a
check that the low-rank delta itself is reproduced (the tolerance alone would
hide a misrouted adapter on the small workload). Segment tables: bit-exact.
Both kernel families (decode: stream-K tcgen05 base GEMM + CUDA-core branch;
prefill: tcgen05 shrink + persistent tcgen05 GEMM with the expand in its
epilogue) are checked on the same inputs.
"""
import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import (assert_parity, assert_routing, load_pool, to_dev, to_host_f64)

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


def run_dev(pool, prob, path):
    pool.set_path(path)
    Y = pool.linear(to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    return Y


def run(pool, prob, path):
    return to_host_f64(run_dev(pool, prob, path))


def ref_of(prob, rows=None):
    ads = oracle.problem_adapters(prob)
    X, ids = prob.X, prob.ids
    if rows is not None:
        X, ids = X[rows], ids[rows]
    Y = oracle.lora_linear(X, prob.W, ids, ads, prob.max_adapters)
    Yb = oracle.lora_linear(X, prob.W, np.full_like(ids, -1), {}, prob.max_adapters)
    return Y, Yb


# ------------------------------------------------------------- the 5 workloads

@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_tiny(path):
    prob = L.tiny()
    pool = load_pool(al, prob)
    got = run(pool, prob, PATHS[path])
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"tiny/{path}")
    assert_routing(got, ref, base, prob.ids, f"tiny/{path}")


def test_tiny_routing_discriminates():
    """With B ~ N(0,1) the delta dwarfs the tolerance: swapping two adapters must fail."""
    prob = L.tiny()
    for s, ad in prob.adapters.items():
        ad.B = L.normal_bf16(77, L.ROLE_B, s, ad.B.shape, 1.0)
    pool = load_pool(al, prob)
    got = run(pool, prob, PATHS["decode"])
    ref, _ = ref_of(prob)
    assert_parity(got, ref, "tiny big-B")
    swapped = dict(prob.adapters)
    swapped[0], swapped[1] = prob.adapters[1], prob.adapters[0]
    prob_sw = L.Problem(prob.name, prob.d_in, prob.d_out, prob.X, prob.W, prob.ids, swapped,
                        prob.max_adapters, prob.max_rank, prob.seed)
    ref_sw, _ = ref_of(prob_sw)
    with pytest.raises(AssertionError):
        assert_parity(got, ref_sw, "swapped adapters must not match")


@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_q_proj_decode(path):
    prob = L.q_proj_decode()
    pool = load_pool(al, prob)
    got = run(pool, prob, PATHS[path])
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"q_proj/{path}")
    assert_routing(got, ref, base, prob.ids, f"q_proj/{path}")


@pytest.mark.parametrize("module", [m for m, _, _ in L.LLAMA3_MODULES])
def test_llama3_modules(module):
    (prob,) = L.llama3_7mod(modules=[module])
    pool = load_pool(al, prob)
    got = run(pool, prob, PATHS["decode"])
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"llama3/{module}")
    assert_routing(got, ref, base, prob.ids, f"llama3/{module}")
    if module in ("k_proj", "down_proj"):
        got_p = run(pool, prob, PATHS["prefill"])
        assert_parity(got_p, ref, f"llama3/{module}/prefill")


def test_hotswap_stream():
    prob, sched = L.hotswap()
    pool = load_pool(al, prob)
    X, W = to_dev(prob.X), to_dev(prob.W)
    current = dict(prob.adapters)
    swaps = {c: (slot, gen) for c, slot, gen in sched.swaps}
    check = {0, sched.calls - 1} | {c + 1 for c in swaps} | set(range(0, sched.calls, 100))
    pool.set_path(1)
    outs, states = {}, {}
    for c in range(sched.calls):
        Y = pool.linear(X, W, to_dev(sched.ids[c]))
        if c in check:
            outs[c] = Y
            states[c] = dict(current)
        if c in swaps:
            slot, gen = swaps[c]
            pool.unload_adapter(slot)
            ad = L.make_adapter(prob.seed, slot, prob.d_in, prob.d_out, 16, 32.0, generation=gen)
            pool.load_adapter(slot, to_dev(ad.A), to_dev(ad.B), ad.rank, ad.alpha)
            current[slot] = ad
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    for c in sorted(outs):
        p = L.Problem("hs", prob.d_in, prob.d_out, prob.X, prob.W, sched.ids[c], states[c],
                      prob.max_adapters, prob.max_rank, prob.seed)
        ref, _ = ref_of(p)
        assert_parity(to_host_f64(outs[c]), ref, f"hotswap call {c}")
    assert pool.stats()["loads"] == 2000 + len(sched.swaps)


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_short_requests_prefill(kernel):
    """Requests of 40 contiguous tokens, each with its own adapter (mixed ranks, one
    request without): every GEMM tile mixes adapters, most epilogue warps' 32 rows share
    one (the shared-B expand), the others straddle two."""
    d, n, ln, seed = 512, 12, 40, 95
    T = n * ln
    ranks = [8, 16, 24, 40]
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 32)
    ids = np.repeat(np.arange(n, dtype=np.int32), ln)
    ids[ids == 5] = -1
    ads = {i: L.make_adapter(seed, i, d, d, ranks[i % 4], 2.0 * ranks[i % 4]) for i in range(n)}
    prob = L.Problem("short_requests", d, d, X, W, ids, ads, n, 40, seed)
    pool = load_pool(al, prob)
    pool.set_prefill_kernel({"single": al.LORA_PREFILL_SINGLE, "pair": al.LORA_PREFILL_PAIR}[kernel])
    got = run(pool, prob, PATHS["prefill"])
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"short requests/{kernel}")
    assert_routing(got, ref, base, prob.ids, f"short requests/{kernel}")


@pytest.mark.parametrize("T", [300, 512])
def test_auto_decode_slices(T):
    """AUTO runs 257..512 tokens as decode calls over 256-token slices (the last one
    ragged at T = 300): the oracle's result, and the prefill kernels' within tolerance."""
    d, n, seed = 512, 40, 93
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 32)
    ids = L.zipf_ids(seed, T, n, 1.0)
    ids[L.rng_for(seed, L.ROLE_IDS, 6).random(T) < 0.1] = -1
    ads = {i: L.make_adapter(seed, i, d, d, 16, 32.0) for i in range(n)}
    prob = L.Problem("auto_slices", d, d, X, W, ids, ads, n, 16, seed)
    pool = load_pool(al, prob)
    got = run(pool, prob, al.LORA_PATH_AUTO)
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"auto T={T}")
    assert_routing(got, ref, base, prob.ids, f"auto T={T}")
    assert_parity(got, run(pool, prob, PATHS["prefill"]), f"auto vs prefill T={T}")
    pool.close()


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_scattered_prefill(kernel):
    """A prefill-sized batch spread over many adapters of mixed ranks (1, 2, 3 and 5
    pages): most segments hold a few tokens, a Zipf head holds many scattered ones (both
    on the warp-level shrink, the head in several 16-token chunks), some tokens have no
    adapter; every 128-token tile of the GEMM mixes adapters (the epilogue expand)."""
    d, T, n, seed = 512, 300, 120, 91
    ranks = [8, 16, 24, 40]
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 32)
    ids = L.zipf_ids(seed, T, n, 1.0)
    ids[L.rng_for(seed, L.ROLE_IDS, 5).random(T) < 0.1] = -1
    ads = {i: L.make_adapter(seed, i, d, d, ranks[i % 4], 2.0 * ranks[i % 4]) for i in range(n)}
    prob = L.Problem("scattered", d, d, X, W, ids, ads, n, 40, seed)
    sizes = np.bincount(ids[ids >= 0], minlength=n)
    assert (sizes[sizes > 0] <= 16).sum() > 20 and sizes.max() > 32  # one-chunk and multi-chunk segments
    pool = load_pool(al, prob)
    pool.set_prefill_kernel({"single": al.LORA_PREFILL_SINGLE, "pair": al.LORA_PREFILL_PAIR}[kernel])
    got = run(pool, prob, PATHS["prefill"])
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"scattered/{kernel}")
    assert_routing(got, ref, base, prob.ids, f"scattered/{kernel}")


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_many_adapter_prefill_full_size(kernel):
    """The large-pool prefill at its benchmarked size: 4096 tokens over 2000 rank-16
    adapters with Zipf ids (~1100 segments; every GEMM tile mixes adapters, every segment
    goes to the warp-level shrink, in one pass of work items). 128 sampled rows (the
    largest segment's, singletons', others) against the oracle, element by element."""
    prob = L.prefill_zipf()
    pool = load_pool(al, prob)
    pool.set_prefill_kernel({"single": al.LORA_PREFILL_SINGLE, "pair": al.LORA_PREFILL_PAIR}[kernel])
    got = run(pool, prob, PATHS["prefill"])
    assert pool.check_errors() == al.LORA_OK
    ids = prob.ids
    sizes = np.bincount(ids[ids >= 0], minlength=prob.max_adapters)
    g = L.rng_for(77, 9)
    head = np.flatnonzero(ids == int(np.argmax(sizes)))
    single = np.flatnonzero(sizes[np.maximum(ids, 0)] == 1)
    rows = np.unique(np.concatenate([g.choice(head, 32, replace=False), g.choice(single, 32, replace=False),
                                     g.choice(prob.T, 64, replace=False)]))
    used = {int(s) for s in ids[rows] if s >= 0}
    ads = {s: (a.A, a.B, a.rank, a.alpha) for s, a in prob.adapters.items() if s in used}
    ref = oracle.lora_linear(prob.X[rows], prob.W, ids[rows], ads, prob.max_adapters)
    base = oracle.lora_linear(prob.X[rows], prob.W, np.full(len(rows), -1, np.int32), {}, prob.max_adapters)
    assert_parity(got[rows], ref, f"many adapters/{kernel}")
    assert_routing(got[rows], ref, base, ids[rows], f"many adapters/{kernel}")
    pool.close()


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_many_small_segments_more_items_than_warps(kernel):
    """16384 tokens uniform over 4000 rank-16 adapters at d = 256: more (chunk, page) work
    items for the warp-level shrink than its grid has warps, so warps take several items;
    256 sampled rows against the oracle."""
    d, T, n, seed = 256, 16384, 4000, 97
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d, d), 1.0 / 16)
    ids = L.rng_for(seed, L.ROLE_IDS, 0).integers(0, n, T).astype(np.int32)
    ids[L.rng_for(seed, L.ROLE_IDS, 3).random(T) < 0.05] = -1
    ads = {i: L.make_adapter(seed, i, d, d, 16, 32.0) for i in range(n)}
    prob = L.Problem("many_small", d, d, X, W, ids, ads, n, 16, seed)
    sizes = np.bincount(ids[ids >= 0], minlength=n)
    chunks = int(((sizes + 15) // 16).sum())
    assert chunks * 2 > 8 * 152 * 4  # (chunk, page) items beyond one per warp of the largest grid
    pool = load_pool(al, prob)
    pool.set_prefill_kernel({"single": al.LORA_PREFILL_SINGLE, "pair": al.LORA_PREFILL_PAIR}[kernel])
    got = run(pool, prob, PATHS["prefill"])
    assert pool.check_errors() == al.LORA_OK
    rows = np.sort(L.rng_for(seed, 9).choice(T, 256, replace=False))
    used = {int(s) for s in ids[rows] if s >= 0}
    sub = {s: (a.A, a.B, a.rank, a.alpha) for s, a in ads.items() if s in used}
    ref = oracle.lora_linear(X[rows], W, ids[rows], sub, n)
    base = oracle.lora_linear(X[rows], W, np.full(len(rows), -1, np.int32), {}, n)
    assert_parity(got[rows], ref, f"many small segments/{kernel}")
    assert_routing(got[rows], ref, base, ids[rows], f"many small segments/{kernel}")
    pool.close()


# ------------------------------------------------------------------ segments

def seg_cases():
    g = L.rng_for(123, 9)
    cases = []
    for T in (1, 31, 32, 33, 64, 256, 1000, 16384):
        cases.append((f"rand{T}", g.integers(-1, 50, size=T).astype(np.int32), 50))
    cases.append(("all_base", np.full(300, -1, np.int32), 50))
    cases.append(("one_id", np.full(257, 7, np.int32), 50))
    cases.append(("max_slot", np.array([49, -1, 49, 0, 49] * 20, np.int32), 50))
    cases.append(("zipf", L.zipf_ids(5, 4096, 2000), 2000))
    cases.append(("sorted_runs", np.repeat(np.arange(8, dtype=np.int32), 2048), 8))
    # many chunks of the multi-CTA builder (235 x 256 tokens)
    cases.append(("rand60000", g.integers(-1, 50, size=60000).astype(np.int32), 50))
    # more keys than the multi-CTA builder takes (1101 > 1024): one CTA of 32 warps;
    # the Zipf case above (2001 keys) runs the 8-warp single-CTA builder
    cases.append(("wide_pool", g.integers(-1, 1100, size=3000).astype(np.int32), 1100))
    return cases


@pytest.mark.parametrize("name,ids,n_slots", seg_cases(), ids=[c[0] for c in seg_cases()])
def test_segments_bit_exact(name, ids, n_slots):
    d = 64
    pool = al.LoraPool(n_slots, 8, d, d)
    A = torch.zeros((d, 8), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((8, d), dtype=torch.bfloat16, device="cuda")
    for s in np.unique(ids[ids >= 0]):
        pool.load_adapter(int(s), A, B, 8, 16.0)
    order, hdr, seg_start, seg_slot = pool.build_segments(to_dev(ids))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    ref = oracle.segments(ids, n_slots)
    ns = ref["num_seg"]
    assert hdr.cpu().tolist() == [ref["n_base"], ns]
    assert np.array_equal(order.cpu().numpy(), ref["order"])
    assert np.array_equal(seg_start.cpu().numpy()[:ns + 1], ref["seg_start"])
    assert np.array_equal(seg_slot.cpu().numpy()[:ns], ref["seg_slot"])


# ----------------------------------------------------------- ragged and edges

@pytest.mark.parametrize("T,path", [(1, "decode"), (37, "decode"), (256, "decode"),
                                    (1, "prefill"), (300, "prefill"), (257, "prefill")])
def test_ragged_shapes_and_ranks(T, path):
    """d_in, d_out multiples of 8 but not of the tiles; ranks not multiples of 8."""
    d_in, d_out, seed = 72, 136, 31
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
    ranks = [1, 5, 13, 24, 40]
    ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 1.5 * r, std=0.2) for i, r in enumerate(ranks)}
    ids = L.rng_for(seed, L.ROLE_IDS).integers(-1, len(ranks), size=T).astype(np.int32)
    prob = L.Problem("ragged", d_in, d_out, X, W, ids, ads, len(ranks), 40, seed)
    pool = load_pool(al, prob)
    got = run(pool, prob, PATHS[path])
    ref, base = ref_of(prob)
    assert_parity(got, ref, f"ragged T={T} {path}")


@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_base_linear_and_all_base_ids(path):
    prob = L.q_proj_decode(T=48, n_adapters=4)
    pool = load_pool(al, prob)
    pool.set_path(PATHS[path])
    X, W = to_dev(prob.X), to_dev(prob.W)
    Yb = to_host_f64(pool.base_linear(X, W))
    ids = np.full(prob.T, -1, np.int32)
    Yl = to_host_f64(pool.linear(X, W, to_dev(ids)))
    torch.cuda.synchronize()
    _, base = ref_of(prob)
    assert_parity(Yb, base, "base_linear")
    assert np.array_equal(Yl, Yb)  # id -1 rows: bit-identical to the base product


def test_deterministic_and_host_entry():
    prob = L.q_proj_decode(T=64, n_adapters=16)
    pool = load_pool(al, prob)
    X, W, ids = to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids)
    Y1 = pool.linear(X, W, ids).clone()
    Y2 = pool.linear(X, W, ids).clone()
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    Xh = torch.from_numpy(prob.X.view(np.int16)).view(torch.bfloat16).pin_memory()
    idh = torch.from_numpy(prob.ids).pin_memory()
    Yh = torch.empty((prob.T, prob.d_out), dtype=torch.bfloat16).pin_memory()
    pool.linear_host(Xh, W, idh, Yh)
    assert torch.equal(Yh, Y1.cpu())


def test_zero_tokens_is_a_noop():
    prob = L.tiny()
    pool = load_pool(al, prob)
    X = torch.empty((0, prob.d_in), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((0,), dtype=torch.int32, device="cuda")
    Y = torch.empty((0, prob.d_out), dtype=torch.bfloat16, device="cuda")
    assert al.lora_linear(pool.handle, X.data_ptr() or 16, to_dev(prob.W), ids.data_ptr() or 16, 0,
                          Y.data_ptr() or 16) == al.LORA_OK


def test_strict_mode_bad_ids():
    prob = L.tiny()
    pool = load_pool(al, prob)
    pool.unload_adapter(2)
    X, W = to_dev(prob.X), to_dev(prob.W)
    for bad in (2, 4, -2, 1 << 20):     # unloaded, out of range, negative, huge
        ids = prob.ids.copy()
        ids[5] = bad
        for path in (1, 2):
            pool.set_path(path)
            pool.linear(X, W, to_dev(ids))
            assert pool.check_errors() == al.LORA_ERR_BAD_ADAPTER_ID
    assert pool.check_errors() == al.LORA_OK   # cleared
    # rows without the bad id stay correct
    ids = prob.ids.copy()
    ids[5] = 2
    got = to_host_f64(pool.linear(X, W, to_dev(ids)))
    assert pool.check_errors() == al.LORA_ERR_BAD_ADAPTER_ID
    keep = ids != 2
    ads = {k: v for k, v in oracle.problem_adapters(prob).items() if k != 2}
    ref = oracle.lora_linear(prob.X[keep], prob.W, ids[keep], ads, 4)
    assert_parity(got[keep], ref, "rows beside a bad id")


def test_pool_management_errors():
    prob = L.tiny()
    pool = load_pool(al, prob)
    A, B = to_dev(prob.adapters[0].A), to_dev(prob.adapters[0].B)
    h = pool.handle
    assert al.lora_load_adapter(h, 0, A, B, 8, 16.0) == al.LORA_ERR_SLOT_OCCUPIED
    assert al.lora_load_adapter(h, 4, A, B, 8, 16.0) == al.LORA_ERR_SLOT_RANGE
    assert al.lora_load_adapter(h, -1, A, B, 8, 16.0) == al.LORA_ERR_SLOT_RANGE
    assert al.lora_unload_adapter(h, 3) == al.LORA_OK
    assert al.lora_unload_adapter(h, 3) == al.LORA_ERR_SLOT_EMPTY
    assert al.lora_load_adapter(h, 3, A, B, 9, 16.0) == al.LORA_ERR_RANK
    assert al.lora_load_adapter(h, 3, A, B, 0, 16.0) == al.LORA_ERR_RANK
    assert al.lora_pool_set_path(h, 7) == al.LORA_ERR_ARG
    pool.set_path(1)
    X = torch.zeros((300, prob.d_in), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(300, dtype=torch.int32, device="cuda")
    Y = torch.empty((300, prob.d_out), dtype=torch.bfloat16, device="cuda")
    assert al.lora_linear(h, X, to_dev(prob.W), ids, 300, Y) == al.LORA_ERR_ARG  # decode: T <= 256
    st = pool.stats()
    assert st["loaded"] == 3 and st["total_pages"] == 4 and st["free_pages"] == 1
    # load from host memory too
    ad = prob.adapters[3]
    Ah = torch.from_numpy(ad.A.view(np.int16)).view(torch.bfloat16)
    Bh = torch.from_numpy(ad.B.view(np.int16)).view(torch.bfloat16)
    pool.load_adapter(3, Ah, Bh, 8, 16.0)
    pool.set_path(0)
    got = run(pool, prob, 0)
    ref, _ = ref_of(prob)
    assert_parity(got, ref, "host-loaded adapter")


def test_prefill_expand_tile_modes():
    """Tiles with one adapter (the tensor-core expand, incl. base-only rows inside them),
    a tile with several adapters (the CUDA-core expand), ranks that are not multiples
    of 32, a d_out tail shorter than the 256-column tile and a ragged last token tile."""
    d_in, d_out, seed, T = 136, 200, 57, 350
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.1)
    ranks = [5, 40, 13, 8]
    ads = {i: L.make_adapter(seed, i, d_in, d_out, r, 2.0 * r, std=0.2) for i, r in enumerate(ranks)}
    ids = np.full(T, -1, np.int32)
    ids[0:128] = 0
    ids[5:9] = -1                  # base rows inside a single-adapter tile
    ids[128:256] = 1
    g = L.rng_for(seed, L.ROLE_IDS)
    ids[256:] = g.integers(-1, 4, size=T - 256)   # mixed, ragged tile
    prob = L.Problem("tile_modes", d_in, d_out, X, W, ids, ads, 4, 40, seed)
    pool = load_pool(al, prob)
    got = run(pool, prob, PATHS["prefill"])
    ref, base = ref_of(prob)
    assert_parity(got, ref, "prefill tile modes")
    assert_routing(got, ref, base, ids, "prefill tile modes")
    got_d = run(pool, prob, PATHS["decode"]) if T <= 256 else None
    assert got_d is None
