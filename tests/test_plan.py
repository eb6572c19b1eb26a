"""Host logic of the decode path, on the CPU (no GPU): the stream-K plan that
lora_linear and lora_linear_grouped compute.

The units of a call are its layers' (128-row tile, 128-column k-block) pairs
concatenated in layer order and cut into G equal contiguous ranges, one per CTA.
Checked against a brute-force walk of those ranges: every unit belongs to exactly
one range, the number of tiles a range touches (which sizes the TMEM accumulator ring
and the split-K partials), and the resource limits of the kernels (shared memory per
CTA, TMEM columns, 32-bit index arithmetic).
"""
import numpy as np
import pytest

al = pytest.importorskip("adapter_linear_gb300")

SMEM_PER_CTA = 227 * 1024


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        al.load_library()
    except al.LibraryMissing:
        pytest.skip("library not built")


def brute_force(T, d_in, d_out, G):
    kb = [-(-d // 128) for d in d_in]
    tiles = [-(-d // 128) for d in d_out]
    unit_tile = []          # global tile index of every unit, in unit order
    g = 0
    for m in range(len(d_in)):
        for t in range(tiles[m]):
            unit_tile += [g + t] * kb[m]
        g += tiles[m]
    U = len(unit_tile)
    starts = [(c * U) // G for c in range(G + 1)]
    covered = np.zeros(U, np.int32)
    max_seg = 1
    for c in range(G):
        u0, u1 = starts[c], starts[c + 1]
        assert u1 > u0, "a range without units"
        covered[u0:u1] += 1
        max_seg = max(max_seg, unit_tile[u1 - 1] - unit_tile[u0] + 1)
    assert np.all(covered == 1)
    return U, max_seg


def check(T, d_in, d_out, pages, sms=152):
    info = al.decode_plan_info(T, d_in, d_out, pages, sms)
    U, max_seg = brute_force(T, d_in, d_out, info["G"])
    assert info["units"] == U
    assert info["G"] == min(sms, U)
    assert info["max_seg"] == max_seg
    ntok = -(-T // 16) * 16
    assert info["ntok"] == ntok
    assert 1 <= info["n_acc"] <= max_seg and info["n_acc"] * ntok <= 512
    cols = info["tmem_cols"]
    assert cols & (cols - 1) == 0 and 32 <= cols <= 512 and cols >= info["n_acc"] * ntok
    assert 2 <= info["stages"] <= 8 and info["smem_bytes"] <= SMEM_PER_CTA
    pairs = T * sum(pages)
    assert info["pairs"] == pairs
    assert info["col_blocks"] == sum(-(-d // 1024) for d in d_out)
    assert info["G"] <= info["grid"] <= max(info["G"], sms)
    if pairs > info["G"]:
        assert info["grid"] == min(pairs, sms)
    assert info["partials_floats"] == info["G"] * max_seg * T * 128
    # A-page prefetch (one bulk request per page) whenever there are shrink pairs
    assert info["prefetch_a"] == int(pairs > 0)
    assert U * info["G"] < 2 ** 31
    return info


def test_plan_of_the_benchmarked_shapes():
    q = check(64, [4096], [4096], [2])
    assert (q["G"], q["max_seg"], q["tight"]) == (152, 2, 1)
    layer = check(32, [4096, 4096, 4096, 4096, 4096, 4096, 14336],
                  [4096, 1024, 1024, 4096, 14336, 14336, 4096], [2] * 7)
    assert layer["units"] == 13312 and layer["col_blocks"] == 42
    hs = check(256, [4096], [4096], [2])
    assert hs["tight"] == 0 and hs["n_acc"] == 2       # 256 columns per accumulator
    assert (q["prefetch_a"], layer["prefetch_a"], hs["prefetch_a"]) == (1, 1, 1)
    tiny = check(64, [256], [256], [1])
    assert tiny["G"] == 4 and tiny["grid"] == 64       # extra CTAs run shrink pairs only
    base = check(64, [4096], [4096], [0])
    assert base["pairs"] == 0 and base["tight"] == 0


def test_plan_random_shapes():
    g = np.random.default_rng(7)
    for _ in range(300):
        n = int(g.integers(1, 9))
        T = int(g.integers(1, 257))
        d_in = [int(8 * g.integers(1, 2048)) for _ in range(n)]
        d_out = [int(8 * g.integers(1, 4096)) for _ in range(n)]
        pages = [int(g.integers(0, 9)) for _ in range(n)]
        sms = int(g.choice([1, 7, 64, 148, 152]))
        check(T, d_in, d_out, pages, sms)


def test_plan_rings_wrap_when_ranges_cover_many_tiles():
    # 512 tiles of one k-block each over 152 ranges at T = 256: 4 tiles per range,
    # 2 accumulators of 256 columns, so the ring is reused
    info = check(256, [128], [65536], [1])
    assert info["max_seg"] > info["n_acc"] == 2


def test_plan_rejects_out_of_range():
    for args in [(0, [64], [64], [1]), (257, [64], [64], [1])]:
        with pytest.raises(al.LoraError):
            al.decode_plan_info(*args)
    with pytest.raises(al.LoraError):
        al.decode_plan_info(16, [64] * 9, [64] * 9, [1] * 9)
    with pytest.raises(al.LoraError):
        al.decode_plan_info(16, [60], [64], [1])        # d_in not a multiple of 8
