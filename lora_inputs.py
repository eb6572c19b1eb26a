"""Seeded synthetic inputs for the heterogeneous multi-LoRA linear layer.

This module only draws random numbers and describes workload shapes. It holds
none of the layer's arithmetic: both the fp64 CPU oracle (``oracle/``) and the
CUDA path (``adapter_linear_gb300``) receive the same arrays from here, and
neither of them is imported by this file.

Every tensor is drawn from its own numpy PCG64 stream, keyed by
``SeedSequence(seed, spawn_key=(role, index))``, as fp32 normals scaled by the
stated standard deviation and rounded to bfloat16 (round-to-nearest-even).
bf16 values travel as ``uint16`` bit patterns.

Workloads (shapes and value distributions follow the five synthetic
configurations the layer is specified on; "N(0, c)" is read as a standard
deviation of c):

* ``tiny``           d_in=d_out=256, T=64, 4 adapters rank 8 alpha 16,
                     ids uniform over {-1,0,1,2,3}; X~N(0,1), W~N(0,1/16),
                     A,B~N(0,0.02); seed 0.
* ``q_proj_decode``  d_in=d_out=4096, T=64, 200 adapters rank 16 alpha 32,
                     ids uniform over 0..199; W~N(0,1/64); seed 1.
* ``llama3_7mod``    Llama-3-8B's seven target modules (q,o 4096x4096;
                     k,v 4096->1024; gate,up 4096->14336; down 14336->4096),
                     T=32, 32 adapters rank 16 alpha 32 per module, exactly
                     4 of 32 tokens base-only at seeded positions, the rest
                     uniform over 0..31; seed 2.
* ``prefill_mixed``  gate_proj 4096->14336, 8 sequences x 2048 contiguous
                     tokens, sequence i uses slot i, ranks {8,8,16,16,32,32,
                     64,64}, alpha = 2*rank; seed 3. The padded variant
                     zero-pads every adapter to rank 64 with alpha scaled so
                     alpha/rank is unchanged.
* ``hotswap``        q_proj 4096x4096, T=256, 2000 adapters rank 16 alpha 32,
                     ids Zipf(s=1) over 2000 slots by inverse CDF, 1000 calls
                     with one unload+reload cycle (a uniformly drawn slot
                     gets a freshly drawn adapter) inside every block of 20
                     calls, 50 cycles in all; seed 4.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

# roles for SeedSequence spawn keys
ROLE_X, ROLE_W, ROLE_IDS, ROLE_A, ROLE_B, ROLE_SWAP = 0, 1, 2, 3, 4, 5


def rng_for(seed: int, role: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(role, index)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, role: int, index: int, shape, std: float) -> np.ndarray:
    g = rng_for(seed, role, index)
    x = g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    return f32_to_bf16_bits(x)


@dataclasses.dataclass
class Adapter:
    A: np.ndarray  # uint16 bf16 bits, d_in x rank, row-major
    B: np.ndarray  # uint16 bf16 bits, rank x d_out, row-major
    rank: int
    alpha: float


@dataclasses.dataclass
class Problem:
    """One lora_linear call's worth of inputs (host arrays)."""
    name: str
    d_in: int
    d_out: int
    X: np.ndarray          # uint16 T x d_in
    W: np.ndarray          # uint16 d_out x d_in
    ids: np.ndarray        # int32 T
    adapters: Dict[int, Adapter]
    max_adapters: int
    max_rank: int
    seed: int

    @property
    def T(self) -> int:
        return int(self.ids.shape[0])


def make_adapter(seed: int, slot: int, d_in: int, d_out: int, rank: int, alpha: float,
                 std: float = 0.02, generation: int = 0) -> Adapter:
    idx = slot + 1_000_000 * generation
    A = normal_bf16(seed, ROLE_A, idx, (d_in, rank), std)
    B = normal_bf16(seed, ROLE_B, idx, (rank, d_out), std)
    return Adapter(A, B, rank, float(alpha))


def pad_adapter(ad: Adapter, new_rank: int) -> Adapter:
    """Zero-pad an adapter's rank; alpha is scaled so alpha/rank is unchanged."""
    d_in, r = ad.A.shape
    A = np.zeros((d_in, new_rank), np.uint16)
    A[:, :r] = ad.A
    B = np.zeros((new_rank, ad.B.shape[1]), np.uint16)
    B[:r, :] = ad.B
    return Adapter(A, B, new_rank, ad.alpha * new_rank / r)


def zipf_ids(seed: int, n: int, n_slots: int, s: float = 1.0, index: int = 0) -> np.ndarray:
    """Zipf(s) over ranks 1..n_slots (P(k) ~ 1/k^s) mapped to slot k-1, by inverse CDF."""
    k = np.arange(1, n_slots + 1, dtype=np.float64)
    p = 1.0 / k ** s
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    u = rng_for(seed, ROLE_IDS, index).random(n)
    return np.searchsorted(cdf, u, side="right").clip(0, n_slots - 1).astype(np.int32)


def q4_weight(seed: int, d_out: int, d_in: int, std: float, index: int = 0, group: int = 128):
    """A random 4-bit base of the layout lora_linear_q4 takes: codes uniform over
    0..15 packed two per byte (the even input in the low nibble), zero points 7 or 8,
    bf16 scales near std / 4.6 (the codes minus the zero point have a spread of ~4.6),
    so that the dequantised weights have about the standard deviation std.
    Returns (Wq uint8 [d_out, d_in/2], scales uint16 bf16 bits [d_in/group, d_out],
    zeros uint8 [d_in/group, d_out])."""
    g = rng_for(seed, ROLE_W, 1000 + index)
    codes = g.integers(0, 16, size=(d_out, d_in), dtype=np.uint8)
    Wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    zeros = g.integers(7, 9, size=(d_in // group, d_out), dtype=np.uint8)
    s = (std / 4.6) * (1.0 + 0.1 * g.standard_normal(size=zeros.shape))
    return Wq, f32_to_bf16_bits(s.astype(np.float32)), zeros


# ---------------------------------------------------------------- workloads

def tiny(seed: int = 0, T: int = 64) -> Problem:
    d = 256
    X = normal_bf16(seed, ROLE_X, 0, (T, d), 1.0)
    W = normal_bf16(seed, ROLE_W, 0, (d, d), 1.0 / 16)
    ids = rng_for(seed, ROLE_IDS).integers(-1, 4, size=T).astype(np.int32)
    ads = {i: make_adapter(seed, i, d, d, 8, 16.0) for i in range(4)}
    return Problem("tiny", d, d, X, W, ids, ads, max_adapters=4, max_rank=8, seed=seed)


def q_proj_decode(seed: int = 1, T: int = 64, n_adapters: int = 200, rank: int = 16,
                  d: int = 4096) -> Problem:
    X = normal_bf16(seed, ROLE_X, 0, (T, d), 1.0)
    W = normal_bf16(seed, ROLE_W, 0, (d, d), 1.0 / 64)
    ids = rng_for(seed, ROLE_IDS).integers(0, n_adapters, size=T).astype(np.int32)
    ads = {i: make_adapter(seed, i, d, d, rank, 2.0 * rank) for i in range(n_adapters)}
    return Problem("q_proj_decode", d, d, X, W, ids, ads, max_adapters=n_adapters,
                   max_rank=rank, seed=seed)


LLAMA3_MODULES: List[Tuple[str, int, int]] = [
    ("q_proj", 4096, 4096), ("k_proj", 4096, 1024), ("v_proj", 4096, 1024),
    ("o_proj", 4096, 4096), ("gate_proj", 4096, 14336), ("up_proj", 4096, 14336),
    ("down_proj", 14336, 4096),
]


def llama3_7mod(seed: int = 2, T: int = 32, n_adapters: int = 32, rank: int = 16,
                modules: Optional[List[str]] = None) -> List[Problem]:
    """One Problem per target module; all modules see the same ids, each its own X/W/adapters."""
    g = rng_for(seed, ROLE_IDS)
    ids = g.integers(0, n_adapters, size=T).astype(np.int32)
    base_pos = g.choice(T, size=T // 8, replace=False)
    ids[base_pos] = -1
    out = []
    for mi, (name, d_in, d_out) in enumerate(LLAMA3_MODULES):
        if modules is not None and name not in modules:
            continue
        s = seed * 1000 + mi
        X = normal_bf16(s, ROLE_X, 0, (T, d_in), 1.0)
        W = normal_bf16(s, ROLE_W, 0, (d_out, d_in), 1.0 / 64)
        ads = {i: make_adapter(s, i, d_in, d_out, rank, 2.0 * rank) for i in range(n_adapters)}
        out.append(Problem(f"llama3_7mod/{name}", d_in, d_out, X, W, ids.copy(), ads,
                           max_adapters=n_adapters, max_rank=rank, seed=s))
    return out


PREFILL_RANKS = [8, 8, 16, 16, 32, 32, 64, 64]


def prefill_mixed(seed: int = 3, seq_len: int = 2048, n_seq: int = 8, d_in: int = 4096,
                  d_out: int = 14336, padded: bool = False, ranks=None) -> Problem:
    """ranks: the adapters' ranks in turn (default PREFILL_RANKS); alpha = 2 * rank."""
    ranks = PREFILL_RANKS if ranks is None else ranks
    T = seq_len * n_seq
    X = normal_bf16(seed, ROLE_X, 0, (T, d_in), 1.0)
    W = normal_bf16(seed, ROLE_W, 0, (d_out, d_in), 1.0 / 64)
    ids = np.repeat(np.arange(n_seq, dtype=np.int32), seq_len)
    ads = {}
    for i in range(n_seq):
        r = ranks[i % len(ranks)]
        ad = make_adapter(seed, i, d_in, d_out, r, 2.0 * r)
        ads[i] = pad_adapter(ad, 64) if padded else ad
    return Problem("prefill_mixed" + ("_padded" if padded else ""), d_in, d_out, X, W, ids,
                   ads, max_adapters=n_seq, max_rank=max(64 if padded else 0, max(ranks)), seed=seed)


def prefill_zipf(seed: int = 5, T: int = 4096, n_adapters: int = 2000, rank: int = 16,
                 d: int = 4096) -> Problem:
    """A prefill-sized batch whose tokens are spread over a large pool: ids Zipf(s=1)
    over n_adapters (a few adapters hold many tokens, most hold one or two)."""
    X = normal_bf16(seed, ROLE_X, 0, (T, d), 1.0)
    W = normal_bf16(seed, ROLE_W, 0, (d, d), 1.0 / 64)
    ids = zipf_ids(seed, T, n_adapters, 1.0)
    ads = {i: make_adapter(seed, i, d, d, rank, 2.0 * rank) for i in range(n_adapters)}
    return Problem("prefill_zipf", d, d, X, W, ids, ads, max_adapters=n_adapters, max_rank=rank, seed=seed)


@dataclasses.dataclass
class HotswapSchedule:
    calls: int
    ids: np.ndarray                 # int32 [calls, T]
    swaps: List[Tuple[int, int, int]]  # (after_call, slot, generation)


def hotswap(seed: int = 4, T: int = 256, n_adapters: int = 2000, rank: int = 16,
            d: int = 4096, calls: int = 1000, swap_every: int = 20,
            build_adapters: bool = True) -> Tuple[Problem, HotswapSchedule]:
    X = normal_bf16(seed, ROLE_X, 0, (T, d), 1.0)
    W = normal_bf16(seed, ROLE_W, 0, (d, d), 1.0 / 64)
    ids_all = np.stack([zipf_ids(seed, T, n_adapters, 1.0, index=c) for c in range(calls)])
    g = rng_for(seed, ROLE_SWAP)
    swaps = []
    # one cycle in the middle of every block of `swap_every` calls, so all cycles
    # fall strictly between calls (50 cycles for 1000 calls)
    for k, c in enumerate(range(swap_every // 2 - 1, calls - 1, swap_every)):
        swaps.append((c, int(g.integers(0, n_adapters)), k + 1))
    ads = {}
    if build_adapters:
        ads = {i: make_adapter(seed, i, d, d, rank, 2.0 * rank) for i in range(n_adapters)}
    p = Problem("hotswap", d, d, X, W, ids_all[0].copy(), ads, max_adapters=n_adapters,
                max_rank=rank, seed=seed)
    return p, HotswapSchedule(calls, ids_all, swaps)
