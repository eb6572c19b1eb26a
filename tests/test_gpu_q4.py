"""GPU parity of the layer over a 4-bit quantised base ("多 LoRA 热插拔: 一模型服多租户"
(vLLM tutorial), section 性能注意事项: an AWQ-INT4 base under bf16 adapters), through
the C ABI, against the oracle's dequant_q4 / lora_linear_q4.

The dequantisation is integer-decided per element (one bf16 rounding of s (q - z)), so
it is compared bit for bit; the layer's output with the usual bf16 tolerance
(|Y_gpu - Y_ref| <= 1e-2 + 1e-2 |Y_ref|), plus the check that the low-rank delta itself
is reproduced. The decode kernel dequantises its W tiles in shared memory; on the same
plan it must give exactly the output of the bf16 decode kernel fed the dequantised W.
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


def q4_problem(seed, d_in, d_out, T, n_adapters, rank, none_frac=0.25):
    X = L.normal_bf16(seed, L.ROLE_X, 0, (T, d_in), 1.0)
    Wq, S, Z = L.q4_weight(seed, d_out, d_in, 1.0 / np.sqrt(d_in))
    g = L.rng_for(seed, L.ROLE_IDS)
    ids = g.integers(0, n_adapters, size=T).astype(np.int32)
    ids[g.random(T) < none_frac] = -1
    ads = {i: L.make_adapter(seed, i, d_in, d_out, rank, 2.0 * rank) for i in range(n_adapters)}
    # W of the Problem is the oracle's dequantised base (used by the bf16 comparison only)
    W = oracle.dequant_q4(Wq, S, Z, d_in)
    prob = L.Problem(f"q4_{d_in}x{d_out}_T{T}", d_in, d_out, X, W, ids, ads, n_adapters, rank, seed)
    return prob, (Wq, S, Z)


def dev_q4(q):
    Wq, S, Z = q
    return to_dev(Wq), to_dev(S), to_dev(Z)


@pytest.mark.parametrize("d_out,d_in,seed", [(256, 256, 1), (400, 384, 2), (1024, 4096, 3)])
def test_dequant_bitwise(d_out, d_in, seed):
    Wq, S, Z = L.q4_weight(seed, d_out, d_in, 0.02)
    ref = oracle.dequant_q4(Wq, S, Z, d_in)
    Wd = torch.empty((d_out, d_in), dtype=torch.bfloat16, device="cuda")
    st = al.lora_dequant_q4(*dev_q4((Wq, S, Z)), d_out, d_in, Wd)
    torch.cuda.synchronize()
    assert st == al.LORA_OK
    got = Wd.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} of {ref.size} weights differ"


@pytest.mark.parametrize("d_in,d_out,T,n_ad,rank,path", [
    (256, 256, 16, 4, 8, "decode"),        # one tile, one K block pair
    (384, 400, 37, 5, 16, "decode"),       # ragged rows (d_out % 128 = 16), ragged tokens
    (4096, 4096, 64, 32, 16, "decode"),    # q_proj at decode size
    (512, 1024, 256, 8, 16, "decode"),     # the largest decode batch
    (512, 768, 300, 6, 16, "prefill"),     # dequantise once, then the bf16 prefill path
    (384, 400, 129, 5, 8, "prefill"),      # ragged on the prefill path
])
def test_q4_layer_parity(d_in, d_out, T, n_ad, rank, path):
    prob, q = q4_problem(10 + T, d_in, d_out, T, n_ad, rank)
    pool = load_pool(al, prob)
    pool.set_path({"decode": al.LORA_PATH_DECODE, "prefill": al.LORA_PATH_PREFILL}[path])
    Xd, idsd = to_dev(prob.X), to_dev(prob.ids)
    Y = pool.linear_q4(Xd, *dev_q4(q), idsd)
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    ads = oracle.problem_adapters(prob)
    ref = oracle.lora_linear_q4(prob.X, *q, prob.ids, ads, prob.max_adapters)
    got = to_host_f64(Y)
    assert_parity(got, ref, prob.name)
    ref_base = oracle.lora_linear_q4(prob.X, *q, np.full(T, -1, np.int32), {}, prob.max_adapters)
    assert_routing(got, ref, ref_base, prob.ids, prob.name)
    if path == "decode":
        # the same plan over the dequantised base in HBM: the same sums in the same order
        Yb = pool.linear(Xd, to_dev(prob.W), idsd)
        torch.cuda.synchronize()
        assert torch.equal(Y, Yb), "in-tile dequantisation differs from the bf16 path"
    pool.close()


@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_q4_base_only(path):
    d_in, d_out, T = 512, 384, 48
    prob, q = q4_problem(5, d_in, d_out, T, 2, 8)
    pool = load_pool(al, prob)
    pool.set_path({"decode": al.LORA_PATH_DECODE, "prefill": al.LORA_PATH_PREFILL}[path])
    Y = pool.base_linear_q4(to_dev(prob.X), *dev_q4(q))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    ref = oracle.lora_linear_q4(prob.X, *q, np.full(T, -1, np.int32), {}, 2)
    assert_parity(to_host_f64(Y), ref, f"base only ({path})")
    pool.close()


def test_q4_repeated_calls_and_empty_batch():
    """Two calls in a row give the same output; T = 0 is a no-op."""
    prob, q = q4_problem(6, 256, 256, 24, 3, 8)
    pool = load_pool(al, prob)
    Xd, idsd = to_dev(prob.X), to_dev(prob.ids)
    qd = dev_q4(q)
    Y1 = pool.linear_q4(Xd, *qd, idsd)
    Y2 = pool.linear_q4(Xd, *qd, idsd)
    Y0 = torch.full((1, 256), 7.0, dtype=torch.bfloat16, device="cuda")  # T = 0 writes nothing
    assert al.lora_linear_q4(pool.handle, Xd, *qd, idsd, 0, Y0) == al.LORA_OK
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    assert torch.equal(Y1, Y2)
    assert bool((Y0 == 7.0).all())
    pool.close()


def test_q4_argument_errors():
    """Shapes the 4-bit layout cannot hold and misaligned operands are refused before
    any launch."""
    prob, q = q4_problem(7, 256, 256, 8, 2, 8)
    pool = load_pool(al, prob)
    Xd, idsd = to_dev(prob.X), to_dev(prob.ids)
    Wq, S, Z = dev_q4(q)
    Y = torch.empty((8, 256), dtype=torch.bfloat16, device="cuda")
    h = pool.handle
    assert al.lora_linear_q4(h, Xd, None, S, Z, idsd, 8, Y) == al.LORA_ERR_ARG
    raw = torch.empty(Wq.numel() + 16, dtype=torch.uint8, device="cuda")
    assert al.lora_linear_q4(h, Xd, raw[1:], S, Z, idsd, 8, Y) == al.LORA_ERR_ARG
    pool.close()
    # d_in not a multiple of the group (128): refused by both entry points
    pool = al.LoraPool(2, 8, 200, 256)
    assert al.lora_linear_q4(pool.handle, Xd, Wq, S, Z, idsd, 8, Y) == al.LORA_ERR_SHAPE
    assert al.lora_base_linear_q4(pool.handle, Xd, Wq, S, Z, 8, Y) == al.LORA_ERR_SHAPE
    pool.close()
    W = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    assert al.lora_dequant_q4(Wq, S, Z, 256, 200, W) == al.LORA_ERR_SHAPE
    assert al.lora_dequant_q4(Wq, S, Z, 256, 256, None) == al.LORA_ERR_ARG
    assert al.lora_dequant_q4(raw[1:], S, Z, 256, 256, W) == al.LORA_ERR_ARG
    torch.cuda.synchronize()
