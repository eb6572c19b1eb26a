"""Shared helpers of the GPU tests: marshalling between the seeded numpy
inputs and torch device tensors, and the parity check against the oracle."""
from __future__ import annotations

import numpy as np

import lora_inputs as L

# |Y_gpu - Y_ref| <= ATOL + RTOL * |Y_ref|, elementwise (bf16 inputs and output,
# fp32 accumulation; the stated tolerance of the layer).
ATOL = 1e-2
RTOL = 1e-2


def to_dev(a: np.ndarray, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_round_f64(y: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 (via fp32; used only to express 'the base output in bf16')."""
    return L.bf16_bits_to_f32(L.f32_to_bf16_bits(y.astype(np.float32))).astype(np.float64)


def load_pool(al, prob, max_rank=None):
    pool = al.LoraPool(prob.max_adapters, max_rank or prob.max_rank, prob.d_in, prob.d_out)
    for slot, ad in prob.adapters.items():
        pool.load_adapter(slot, to_dev(ad.A), to_dev(ad.B), ad.rank, ad.alpha)
    return pool


def assert_parity(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {i}: "
            f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.4g} bound {bound[i]:.4g}")
    return float(err.max()) if err.size else 0.0


def assert_routing(got: np.ndarray, ref: np.ndarray, ref_base: np.ndarray, ids: np.ndarray,
                   what: str = ""):
    """The low-rank delta itself must be reproduced, not only hidden inside the tolerance:
    mean |(Y_gpu - bf16(base_ref)) - (Y_ref - base_ref)| < 25% of mean |Y_ref - base_ref|
    over adapter rows."""
    rows = ids >= 0
    if not rows.any():
        return
    d_ref = (ref - ref_base)[rows]
    d_got = (got - bf16_round_f64(ref_base))[rows]
    mean_ref = float(np.mean(np.abs(d_ref)))
    mean_err = float(np.mean(np.abs(d_got - d_ref)))
    assert mean_err < 0.25 * mean_ref, f"{what}: delta error {mean_err:.4g} vs delta {mean_ref:.4g}"
