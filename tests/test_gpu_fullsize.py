"""Full-size parity: every output element of the prefill workload against the fp64 oracle.

gate_proj 4096 -> 14336, 8 sequences x 2048 contiguous tokens, one adapter per
sequence with ranks {8,8,16,16,32,32,64,64} and alpha = 2 * rank, run unpadded and
with every adapter zero-padded to rank 64 (the vLLM tutorial's 性能注意事项: mixed
ranks aligned to the largest must not change the result). Both prefill GEMM kernels
(one CTA per 128 x 256 tile; a CTA pair per 256 x 256 tile) are run on both
variants and all 16384 x 14336 outputs are compared with one oracle result, at
|Y_gpu - Y_ref| <= 1e-2 + 1e-2 |Y_ref|.

At this size the persistent kernels take several tiles per CTA (pair: ~47 tiles per
cluster), so the TMEM double-buffer flips, the grouped raster and the next-tile
adapter-table lookahead all run; the smaller cases of the other files give each
cluster one tile.

The oracle is computed once (about a minute on 16 cores). Its use for the padded run
rests on the padding invariance being exact in fp64 (the added rank columns contribute
exact zeros); that is pinned on the CPU and re-checked here bitwise on sampled rows.
"""
import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import assert_parity, assert_routing, load_pool, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")

KERNELS = {"single": al.LORA_PREFILL_SINGLE, "pair": al.LORA_PREFILL_PAIR}
SEQ = 2048


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


def sample_rows(T):
    rows = set()
    for s in range(0, T, SEQ):
        rows.update([s, s + 1, s + 127, s + 128, s + 255, s + 256, s + SEQ // 2, s + SEQ - 1])
    return np.array(sorted(r for r in rows if r < T))


@pytest.fixture(scope="module")
def prefill():
    prob = L.prefill_mixed()
    padded = L.prefill_mixed(padded=True)
    ref = oracle.lora_linear(prob.X, prob.W, prob.ids, oracle.problem_adapters(prob),
                             prob.max_adapters)
    rows = sample_rows(prob.T)
    ref_pad = oracle.lora_linear(padded.X[rows], padded.W, padded.ids[rows],
                                 oracle.problem_adapters(padded), padded.max_adapters)
    assert np.array_equal(ref_pad, ref[rows])  # zero padding adds exact zeros in fp64
    base = oracle.lora_linear(prob.X[rows], prob.W, np.full(len(rows), -1, np.int32), {},
                              prob.max_adapters)
    return {"plain": prob, "padded": padded, "ref": ref, "rows": rows, "base": base}


def compare_all(Y, ref, what, chunk=1024):
    """Every element, in row blocks (the host copies stay a few hundred MB)."""
    for r0 in range(0, ref.shape[0], chunk):
        got = to_host_f64(Y[r0:r0 + chunk])
        assert_parity(got, ref[r0:r0 + chunk], f"{what}, rows {r0}..{r0 + got.shape[0] - 1}")


@pytest.mark.parametrize("variant", ["plain", "padded"])
@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_prefill_every_element(prefill, kernel, variant):
    prob = prefill[variant]
    pool = load_pool(al, prob)
    pool.set_path(al.LORA_PATH_PREFILL)
    pool.set_prefill_kernel(KERNELS[kernel])
    Y = pool.linear(to_dev(prob.X), to_dev(prob.W), to_dev(prob.ids))
    torch.cuda.synchronize()
    assert pool.check_errors() == al.LORA_OK
    what = f"prefill {variant} ({kernel} kernel)"
    compare_all(Y, prefill["ref"], what)
    rows = prefill["rows"]
    got_rows = to_host_f64(Y[torch.from_numpy(rows).cuda()])
    assert_routing(got_rows, prefill["ref"][rows], prefill["base"], prob.ids[rows], what)
    pool.close()
