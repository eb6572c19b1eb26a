"""Pins for the fp64 CPU oracle (no GPU).

The oracle is trusted only because these checks tie it to facts outside
itself. Nothing here re-types the oracle's formula; each check is one of:

* a hand-worked example (``tests/golden/hand_example.json``, derived with
  pencil from the pages' definition; cited inside the file);
* a closed form of a special case (X a basis row: the sums collapse to one
  entry of W plus s * A[k,:] B);
* an independent library route (numpy fp64 matmul of the base product, and of
  the "merge" mode X (W + s (A B)^T)^T that the icman.com.cn article's
  section 2.1 says computes the same thing as per-sample branches);
* invariants the method implies: id -1 rows are the base product, B = 0 gives
  the base output, zero-padding the rank (alpha scaled to keep alpha/rank)
  changes nothing (the vLLM tutorial's 性能注意事项 says mixed ranks get
  aligned to the largest one), permuting tokens permutes rows, linearity in X;
* strict mode (icman.com.cn article section 4.1): an unknown id is an error;
* adapter chains (LoRA-Land blog, 技术方案 item 3 and 3. 热插拔 API 与组合:
  set_adaptive_chain): a token's listed adapters equal the merged weight
  W + sum_c s_c (A_c B_c)^T applied with numpy, and a chain of two adapters
  with one scale equals the single adapter whose A and B are the members'
  concatenated; the order of the members does not matter;
* exhaustive brute force for the segment builder on every id vector of
  length <= 5 over {-1, 0, 1, 2}: the output must be a permutation, sorted by
  id, stable, with maximal segments.

``test_planted_mistakes_are_caught`` builds mutated copies of the oracle's C
source (a dropped term, a wrong sign, a transposed operand, an inverted scale,
an unstable tie-break ...) and checks that every one fails at least one pin.
"""
import itertools
import json
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import lora_inputs as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


def bits(a):
    return L.f32_to_bf16_bits(np.asarray(a, np.float32))


def val(b):
    return L.bf16_bits_to_f32(b).astype(np.float64)


def small_problem(seed, T=12, d_in=24, d_out=20, ranks=(3, 8, 5), std_ab=0.5):
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    W = L.normal_bf16(seed, L.ROLE_W, 0, (d_out, d_in), 0.3)
    ads = {}
    for i, r in enumerate(ranks):
        ad = L.make_adapter(seed, i, d_in, d_out, r, 2.0 * r + i, std=std_ab)
        ads[i] = (ad.A, ad.B, ad.rank, ad.alpha)
    ids = L.rng_for(seed, L.ROLE_IDS).integers(-1, len(ranks), size=T).astype(np.int32)
    return X, W, ids, ads


# ------------------------------------------------------------------ pins

def pin_golden(lib):
    g = json.load(open(GOLDEN))
    X = bits(g["X"])
    W = bits(g["W"])
    ids = np.array(g["ids"], np.int32)
    ads = {int(k): (bits(v["A"]), bits(v["B"]), v["rank"], v["alpha"])
           for k, v in g["adapters"].items()}
    # every fixture value is exact in bf16
    assert np.array_equal(val(X), np.array(g["X"], np.float64))
    Y = oracle.lora_linear(X, W, ids, ads, n_slots=2, lib=lib)
    assert np.array_equal(Y, np.array(g["Y"], np.float64)), Y
    seg = oracle.segments(ids, 2, lib=lib)
    exp = g["segments"]
    assert seg["order"].tolist() == exp["order"]
    assert seg["n_base"] == exp["n_base"] and seg["num_seg"] == exp["num_seg"]
    assert seg["seg_start"].tolist() == exp["seg_start"]
    assert seg["seg_slot"].tolist() == exp["seg_slot"]


def pin_basis_rows(lib):
    """X = e_k: Y[t,n] = W[n,k] + s * sum_j A[k,j] B[j,n] (one term of each sum survives)."""
    d_in, d_out, r = 7, 5, 3
    _, W, _, _ = small_problem(11, d_in=d_in, d_out=d_out)
    ad = L.make_adapter(11, 0, d_in, d_out, r, 6.0, std=0.5)
    X = np.zeros((2 * d_in, d_in), np.float32)
    ids = np.zeros(2 * d_in, np.int32)
    for k in range(d_in):
        X[k, k] = 1.0
        X[d_in + k, k] = 1.0
        ids[d_in + k] = -1
    Y = oracle.lora_linear(bits(X), W, ids, {0: (ad.A, ad.B, r, ad.alpha)}, 1, lib=lib)
    Wv, Av, Bv = val(W), val(ad.A), val(ad.B)
    s = ad.alpha / r
    for k in range(d_in):
        for n in range(d_out):
            lora_term = sum(Av[k, j] * Bv[j, n] for j in range(r))
            assert abs(Y[k, n] - (Wv[n, k] + s * lora_term)) <= 1e-15 * (1 + abs(Y[k, n]))
            assert Y[d_in + k, n] == Wv[n, k]


def pin_base_rows_match_numpy(lib):
    X, W, ids, ads = small_problem(1)
    Y = oracle.lora_linear(X, W, ids, ads, 3, lib=lib)
    ref = val(X) @ val(W).T
    base = ids == -1
    assert base.any()
    np.testing.assert_allclose(Y[base], ref[base], rtol=1e-12, atol=1e-12)


def pin_zero_B_is_base(lib):
    X, W, ids, ads = small_problem(2)
    zero = {k: (A, np.zeros_like(B), r, a) for k, (A, B, r, a) in ads.items()}
    Y = oracle.lora_linear(X, W, ids, zero, 3, lib=lib)
    Y_base = oracle.lora_linear(X, W, np.full_like(ids, -1), {}, 3, lib=lib)
    assert np.array_equal(Y, Y_base)


def pin_merge_mode(lib):
    """Per-token branches equal the merged weight W + s (A B)^T applied with numpy."""
    X, W, ids, ads = small_problem(3)
    Y = oracle.lora_linear(X, W, ids, ads, 3, lib=lib)
    Xv, Wv = val(X), val(W)
    for t in range(X.shape[0]):
        i = int(ids[t])
        Wm = Wv.copy()
        if i >= 0:
            A, B, r, alpha = ads[i]
            Wm = Wm + (alpha / r) * (val(A) @ val(B)).T
        ref = Xv[t] @ Wm.T
        np.testing.assert_allclose(Y[t], ref, rtol=1e-12, atol=1e-12)


def pin_rank_padding(lib):
    X, W, ids, ads = small_problem(4, ranks=(8, 8, 8))
    padded = {}
    for k, (A, B, r, a) in ads.items():
        p = L.pad_adapter(L.Adapter(A, B, r, a), 64)
        padded[k] = (p.A, p.B, p.rank, p.alpha)
    Y = oracle.lora_linear(X, W, ids, ads, 3, lib=lib)
    Yp = oracle.lora_linear(X, W, ids, padded, 3, lib=lib)
    assert np.array_equal(Y, Yp)


def pin_permutation(lib):
    X, W, ids, ads = small_problem(5)
    perm = L.rng_for(5, 99).permutation(X.shape[0])
    Y = oracle.lora_linear(X, W, ids, ads, 3, lib=lib)
    Yp = oracle.lora_linear(X[perm], W, ids[perm], ads, 3, lib=lib)
    assert np.array_equal(Yp, Y[perm])


def pin_linearity(lib):
    X, W, ids, ads = small_problem(6)
    g = L.rng_for(6, 98)
    X1 = g.integers(-8, 9, size=X.shape).astype(np.float32)
    X2 = g.integers(-8, 9, size=X.shape).astype(np.float32)   # X1 + X2 exact in bf16
    Y1 = oracle.lora_linear(bits(X1), W, ids, ads, 3, lib=lib)
    Y2 = oracle.lora_linear(bits(X2), W, ids, ads, 3, lib=lib)
    Y12 = oracle.lora_linear(bits(X1 + X2), W, ids, ads, 3, lib=lib)
    np.testing.assert_allclose(Y12, Y1 + Y2, rtol=1e-12, atol=1e-10)


def pin_scale(lib):
    """The branch scales with alpha and inversely with the rank the adapter is loaded with."""
    X, W, ids, ads = small_problem(7)
    ids = np.zeros_like(ids)
    A, B, r, a = ads[0]
    base = oracle.lora_linear(X, W, np.full_like(ids, -1), {}, 1, lib=lib)
    d1 = oracle.lora_linear(X, W, ids, {0: (A, B, r, a)}, 1, lib=lib) - base
    d2 = oracle.lora_linear(X, W, ids, {0: (A, B, r, 2 * a)}, 1, lib=lib) - base
    np.testing.assert_allclose(d2, 2 * d1, rtol=1e-9, atol=1e-12)
    # s = alpha / r: with alpha = r the branch is exactly (X A) B
    d_unit = oracle.lora_linear(X, W, ids, {0: (A, B, r, float(r))}, 1, lib=lib) - base
    np.testing.assert_allclose(d_unit, (val(X) @ val(A)) @ val(B), rtol=1e-9, atol=1e-10)


def pin_strict_ids(lib):
    X, W, ids, ads = small_problem(8)
    bad = ids.copy()
    bad[3] = 2                       # slot 2 is not loaded below
    with pytest.raises(oracle.OracleError) as e:
        oracle.lora_linear(X, W, bad, {0: ads[0], 1: ads[1]}, 3, lib=lib)
    assert e.value.code == oracle.ERR_BAD_ADAPTER_ID
    bad[3] = 3                       # out of range
    with pytest.raises(oracle.OracleError):
        oracle.lora_linear(X, W, bad, ads, 3, lib=lib)
    with pytest.raises(oracle.OracleError):
        oracle.segments(np.array([0, 5], np.int32), 3, lib=lib)
    with pytest.raises(oracle.OracleError):
        oracle.segments(np.array([0, -2], np.int32), 3, lib=lib)


def check_segments_properties(ids, seg):
    T = len(ids)
    order = seg["order"]
    assert sorted(order.tolist()) == list(range(T))                 # permutation
    keys = ids[order]
    assert all(keys[p] <= keys[p + 1] for p in range(T - 1))         # sorted by id
    for p in range(T - 1):                                           # stable
        if keys[p] == keys[p + 1]:
            assert order[p] < order[p + 1]
    nb = int(np.sum(ids == -1))
    assert seg["n_base"] == nb
    starts, slots = seg["seg_start"], seg["seg_slot"]
    assert seg["num_seg"] == len(set(ids.tolist()) - {-1})
    assert len(starts) == seg["num_seg"] + 1 and starts[-1] == T
    if seg["num_seg"]:
        assert starts[0] == nb
    for s in range(seg["num_seg"]):                                  # maximal runs
        a, b = starts[s], starts[s + 1]
        assert b > a and np.all(keys[a:b] == slots[s])
    assert np.all(np.diff(slots) > 0)


def pin_segments_bruteforce(lib):
    for T in range(0, 6):
        for combo in itertools.product([-1, 0, 1, 2], repeat=T):
            ids = np.array(combo, np.int32)
            check_segments_properties(ids, oracle.segments(ids, 3, lib=lib))
    g = L.rng_for(9, 97)
    for _ in range(20):
        ids = g.integers(-1, 50, size=int(g.integers(1, 3000))).astype(np.int32)
        check_segments_properties(ids, oracle.segments(ids, 50, lib=lib))


def chain_problem(seed, T=10, d_in=20, d_out=18):
    X, W, _, ads = small_problem(seed, T=T, d_in=d_in, d_out=d_out, ranks=(3, 8, 5, 4))
    g = L.rng_for(seed, 61)
    lists = []
    for t in range(T):
        n = int(g.integers(0, 4))
        lists.append([int(c) for c in g.choice(4, size=n, replace=False)])
    return X, W, lists, ads


def pin_chain_merge_mode(lib):
    """Each token's listed adapters equal the merged weight W + sum_c s_c (A_c B_c)^T."""
    X, W, lists, ads = chain_problem(21)
    assert any(len(lst) >= 2 for lst in lists) and any(len(lst) == 0 for lst in lists)
    Y = oracle.lora_linear_chains(X, W, lists, ads, 4, lib=lib)
    Xv, Wv = val(X), val(W)
    for t, lst in enumerate(lists):
        Wm = Wv.copy()
        for c in lst:
            A, B, r, alpha = ads[c]
            Wm = Wm + (alpha / r) * (val(A) @ val(B)).T
        np.testing.assert_allclose(Y[t], Xv[t] @ Wm.T, rtol=1e-12, atol=1e-12)


def pin_chain_concatenation(lib):
    """A chain of two adapters with one scale s is the rank r_a + r_b adapter with
    A = [A_a | A_b], B = [B_a ; B_b] and alpha = s (r_a + r_b), through the single-adapter
    entry point."""
    X, W, _, _ = small_problem(22)
    d_in, d_out = X.shape[1], W.shape[0]
    a = L.make_adapter(22, 0, d_in, d_out, 3, 6.0, std=0.5)    # s = 2
    b = L.make_adapter(22, 1, d_in, d_out, 5, 10.0, std=0.5)   # s = 2
    ads = {0: (a.A, a.B, 3, 6.0), 1: (b.A, b.B, 5, 10.0)}
    cat = {0: (np.concatenate([a.A, b.A], axis=1), np.concatenate([a.B, b.B], axis=0), 8, 16.0)}
    T = X.shape[0]
    Yc = oracle.lora_linear_chains(X, W, [[0, 1]] * T, ads, 2, lib=lib)
    Ys = oracle.lora_linear(X, W, np.zeros(T, np.int32), cat, 1, lib=lib)
    np.testing.assert_allclose(Yc, Ys, rtol=1e-12, atol=1e-12)


def pin_chain_order_and_reduction(lib):
    X, W, lists, ads = chain_problem(23)
    Y = oracle.lora_linear_chains(X, W, lists, ads, 4, lib=lib)
    Yr = oracle.lora_linear_chains(X, W, [lst[::-1] for lst in lists], ads, 4, lib=lib)
    np.testing.assert_allclose(Y, Yr, rtol=1e-12, atol=1e-12)
    # lists of at most one adapter: the single-adapter entry point
    ids = np.array([lst[0] if lst else -1 for lst in lists], np.int32)
    Y1 = oracle.lora_linear_chains(X, W, [[i] if i >= 0 else [] for i in ids], ads, 4, lib=lib)
    np.testing.assert_allclose(Y1, oracle.lora_linear(X, W, ids, ads, 4, lib=lib),
                               rtol=1e-12, atol=1e-12)
    with pytest.raises(oracle.OracleError):
        oracle.lora_linear_chains(X, W, [[0, 7]] + lists[1:], ads, 4, lib=lib)


# ------------------------------------------------ quantised base (4-bit codes)

GOLDEN_Q4 = os.path.join(os.path.dirname(__file__), "golden", "q4_hand_example.json")


def pin_q4_golden(lib):
    """The hand-worked example (tests/golden/q4_hand_example.json): codes, zero points
    and scales per group, a value that needs the rounding to bf16, and the layer."""
    g = json.load(open(GOLDEN_Q4))
    Wq = np.array(g["Wq_bytes"], np.uint8)
    codes = np.array(g["codes"])
    assert np.array_equal(Wq[:, ::1] & 0x0F, codes[:, 0::2]) and np.array_equal(Wq >> 4, codes[:, 1::2])
    W = oracle.dequant_q4(Wq, bits(g["scales"]), np.array(g["zeros"], np.uint8), g["d_in"],
                          group=g["group"], lib=lib)
    assert np.array_equal(val(W), np.array(g["W"], np.float64))
    ad = g["adapter"]
    ads = {0: (bits(ad["A"]), bits(ad["B"]), ad["rank"], ad["alpha"])}
    Y = oracle.lora_linear_q4(bits(g["X"]), Wq, bits(g["scales"]), np.array(g["zeros"], np.uint8),
                              np.array(g["ids"], np.int32), ads, 1, group=g["group"], lib=lib)
    assert np.array_equal(Y, np.array(g["Y"], np.float64))


def q4_random(seed, d_out=40, d_in=256, group=128, pow2=False):
    rng = np.random.default_rng(seed)
    Wq = rng.integers(0, 256, size=(d_out, d_in // 2), dtype=np.uint8)
    zeros = rng.integers(0, 16, size=(d_in // group, d_out), dtype=np.uint8)
    if pow2:
        s = np.ldexp(1.0, rng.integers(-9, -3, size=zeros.shape)) * rng.choice([-1, 1], size=zeros.shape)
    else:
        s = rng.normal(0.0, 0.01, size=zeros.shape)
    return Wq, bits(s), zeros


def pin_q4_numpy_route(lib):
    """An independent route: numpy unpacks the nibbles, forms s (q - z) in float32
    (exact: 8-bit significand times a 4-bit integer) and rounds it to bf16 with the
    input generator's round-to-nearest-even; the oracle must agree bit for bit."""
    Wq, sc, z = q4_random(31)
    d_out, d_in = Wq.shape[0], 2 * Wq.shape[1]
    q = np.empty((d_out, d_in), np.int32)
    q[:, 0::2] = Wq & 0x0F
    q[:, 1::2] = Wq >> 4
    g = np.arange(d_in) // 128
    s = L.bf16_bits_to_f32(sc)[g, :].T                     # [d_out, d_in]
    zz = z[g, :].T.astype(np.int32)
    ref = L.f32_to_bf16_bits((s * (q - zz).astype(np.float32)).astype(np.float32))
    assert np.array_equal(oracle.dequant_q4(Wq, sc, z, d_in, lib=lib), ref)


def pin_q4_exact_scales_layer(lib):
    """Power-of-two scales make s (q - z) exact: the layer over the 4-bit base equals
    numpy's fp64 product with that weight on base-only rows, and the bf16 layer with
    the same weight written out directly, adapters included."""
    Wq, sc, z = q4_random(32, pow2=True)
    d_out, d_in = Wq.shape[0], 2 * Wq.shape[1]
    q = np.empty((d_out, d_in), np.int64)
    q[:, 0::2] = Wq & 0x0F
    q[:, 1::2] = Wq >> 4
    g = np.arange(d_in) // 128
    Wexact = val(sc)[g, :].T * (q - z[g, :].T.astype(np.int64))
    X = L.normal_bf16(32, L.ROLE_X, 0, (9, d_in), 1.0)
    ads = {0: (L.normal_bf16(32, L.ROLE_A, 0, (d_in, 4), 0.1), L.normal_bf16(32, L.ROLE_B, 0, (4, d_out), 0.1),
               4, 8.0)}
    ids = np.array([-1, 0, -1, 0, 0, -1, 0, -1, 0], np.int32)
    Y = oracle.lora_linear_q4(X, Wq, sc, z, ids, ads, 1, lib=lib)
    base = ids < 0
    np.testing.assert_allclose(Y[base], val(X)[base] @ Wexact.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(Y, oracle.lora_linear(X, bits(Wexact), ids, ads, 1, lib=lib))


def pin_q4_strict(lib):
    Wq, sc, z = q4_random(33)
    z2 = z.copy()
    z2[0, 3] = 16                                           # not a 4-bit zero point
    with pytest.raises(oracle.OracleError):
        oracle.dequant_q4(Wq, sc, z2, 2 * Wq.shape[1], lib=lib)
    # groups that do not divide d_in (120 inputs, groups of 128): an error from the C side
    out = np.empty((Wq.shape[0], 120), np.uint16)
    assert lib.oracle_dequant_q4(Wq.ctypes.data, sc.ctypes.data, z.ctypes.data, Wq.shape[0], 120, 128,
                                 out.ctypes.data) == 1


PINS = [pin_golden, pin_basis_rows, pin_base_rows_match_numpy, pin_zero_B_is_base,
        pin_merge_mode, pin_rank_padding, pin_permutation, pin_linearity, pin_scale,
        pin_strict_ids, pin_segments_bruteforce, pin_chain_merge_mode, pin_chain_concatenation,
        pin_chain_order_and_reduction, pin_q4_golden, pin_q4_numpy_route, pin_q4_exact_scales_layer,
        pin_q4_strict]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.load())


# ------------------------------------------------------- planted mistakes

MUTATIONS = {
    "drop_base": ("Y[t * d_out + n] = base + s * delta;", "Y[t * d_out + n] = s * delta;"),
    "drop_branch": ("Y[t * d_out + n] = base + s * delta;", "Y[t * d_out + n] = base;"),
    "sign": ("Y[t * d_out + n] = base + s * delta;", "Y[t * d_out + n] = base - s * delta;"),
    "no_scale": ("Y[t * d_out + n] = base + s * delta;", "Y[t * d_out + n] = base + delta;"),
    "inverted_scale": ("s = alpha[i] / (double)r;", "s = (double)r / alpha[i];"),
    "W_transposed": ("base += bf16_value(x[k]) * bf16_value(w[k]);",
                     "base += bf16_value(x[k]) * bf16_value(W[k * d_out + n]);"),
    "A_transposed": ("bf16_value(A[i][k * r + j])", "bf16_value(A[i][j * d_in + k])"),
    "B_transposed": ("bf16_value(B[i][j * d_out + n])", "bf16_value(B[i][n * r + j])"),
    "rank_off_by_one": ("for (int64_t j = 0; j < r; ++j) {", "for (int64_t j = 1; j < r; ++j) {"),
    "unstable_ties": ("if (a->index != b->index) return a->index < b->index ? -1 : 1;",
                      "if (a->index != b->index) return a->index < b->index ? 1 : -1;"),
    "base_last": ("if (a->key != b->key) return a->key < b->key ? -1 : 1;",
                  "if (a->key != b->key) return (uint32_t)a->key < (uint32_t)b->key ? -1 : 1;"),
    "chain_last_member_only": ("yt[n] += sc * branch;",
                               "yt[n] = (e + 1 == off[t + 1]) ? yt[n] + sc * branch : yt[n];"),
    "chain_shared_scale": ("const double sc = alpha[c] / (double)rc;",
                           "const double sc = alpha[list[off[t]]] / (double)rank[list[off[t]]];"),
    "chain_B_transposed": ("branch += low[j] * bf16_value(B[c][j * d_out + n]);",
                           "branch += low[j] * bf16_value(B[c][n * rc + j]);"),
    "chain_W_transposed": ("acc += bf16_value(xt[k]) * bf16_value(W[n * d_in + k]);",
                           "acc += bf16_value(xt[k]) * bf16_value(W[k * d_out + n]);"),
    "q4_nibbles_swapped": ("const int q = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
                           "const int q = (k % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    "q4_zero_point_dropped": ("s * (double)(q - z)", "s * (double)q"),
    "q4_group_by_row": ("const int64_t g = k / group;", "const int64_t g = n % groups;"),
    "q4_truncated": ("return (uint16_t)((u + 0x7FFFu + lsb) >> 16);", "return (uint16_t)(u >> 16);"),
    "q4_scales_transposed": ("const double s = bf16_value(scales[g * d_out + n]);",
                             "const double s = bf16_value(scales[n * groups + g]);"),
    "lenient_segment_ids": ("if (ids[t] < -1 || ids[t] >= n_slots) return ORACLE_ERR_BAD_ADAPTER_ID;",
                            "if (ids[t] < -1) return ORACLE_ERR_BAD_ADAPTER_ID;"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name):
    src = open(oracle.SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mut.c")
        so = os.path.join(d, "libmut.so")
        open(c, "w").write(mutated)
        oracle.build(c, so)
        lib = oracle.load(so)
        failed = []
        for pin in PINS:
            try:
                pin(lib)
            except KeyboardInterrupt:
                raise
            except BaseException:  # noqa: BLE001  (pytest.raises failures are BaseException)
                failed.append(pin.__name__)
        assert failed, f"planted mistake {name!r} passed every pin"
