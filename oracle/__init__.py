"""fp64 CPU oracle for the heterogeneous multi-LoRA linear layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg use it; the product path never imports it. It
shares no code with the CUDA implementation. The arithmetic lives in
``lora_oracle.c`` (plain loops in double precision); this wrapper only
marshals numpy arrays and builds the C file with gcc when needed.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
the pages and the mathematics fix (see that file's docstring).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lora_oracle.c")
LIB = os.path.join(HERE, "liblora_oracle.so")

OK = 0
ERR_BAD_ADAPTER_ID = 7


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle returned status {code}")
        self.code = code


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile the oracle (gcc, OpenMP, no -march flags so it builds on x86 and Arm)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", *extra_flags, src, "-o",
           out + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if it is missing or stale)."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        path = LIB
    lib = ctypes.CDLL(path)
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    vp = ctypes.c_void_p
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_segments.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp]
    lib.oracle_segments.restype = ctypes.c_int
    lib.oracle_lora_linear.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, vp, vp, vp, vp]
    lib.oracle_lora_linear.restype = ctypes.c_int
    lib.oracle_lora_linear_chains.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp, vp, vp, vp,
                                              vp]
    lib.oracle_lora_linear_chains.restype = ctypes.c_int
    lib.oracle_dequant_q4.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    lib.oracle_dequant_q4.restype = ctypes.c_int
    if path == LIB:
        _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())


def segments(ids: np.ndarray, n_slots: int, lib=None) -> Dict[str, np.ndarray]:
    """Stable grouping of tokens by adapter id. Returns order, n_base, num_seg,
    seg_start[num_seg+1], seg_slot[num_seg]."""
    lib = lib or load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T = ids.shape[0]
    cap = min(T, max(n_slots, 0)) + 1
    order = np.zeros(max(T, 1), np.int32)
    n_base = np.zeros(1, np.int32)
    num_seg = np.zeros(1, np.int32)
    seg_start = np.zeros(cap, np.int32)
    seg_slot = np.zeros(cap, np.int32)
    rc = lib.oracle_segments(_ptr(ids), T, n_slots, _ptr(order), _ptr(n_base), _ptr(num_seg),
                             _ptr(seg_start), _ptr(seg_slot))
    if rc != OK:
        raise OracleError(rc)
    ns = int(num_seg[0])
    return {"order": order[:T].copy(), "n_base": int(n_base[0]), "num_seg": ns,
            "seg_start": seg_start[:ns + 1].copy(), "seg_slot": seg_slot[:ns].copy()}


def lora_linear(X: np.ndarray, W: np.ndarray, ids: np.ndarray,
                adapters: Dict[int, Tuple[np.ndarray, np.ndarray, int, float]],
                n_slots: int, lib=None) -> np.ndarray:
    """Y (float64, T x d_out) = X W^T + s_i (X A_i) B_i per token, s_i = alpha_i / r_i.

    X: uint16 bf16 bits [T, d_in]; W: uint16 [d_out, d_in]; ids: int32 [T];
    adapters: slot -> (A uint16 [d_in, r], B uint16 [r, d_out], r, alpha).
    """
    lib = lib or load()
    X = np.ascontiguousarray(X, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, d_in = X.shape
    d_out = W.shape[0]
    assert W.shape[1] == d_in and ids.shape[0] == T
    A_ptrs, B_ptrs, ranks, alphas, keep = _slot_arrays(adapters, n_slots, d_in, d_out)
    Y = np.empty((T, d_out), np.float64)
    rc = lib.oracle_lora_linear(_ptr(X), _ptr(W), _ptr(ids), T, d_in, d_out, n_slots,
                                ctypes.cast(A_ptrs, ctypes.c_void_p),
                                ctypes.cast(B_ptrs, ctypes.c_void_p), _ptr(ranks), _ptr(alphas),
                                _ptr(Y))
    if rc != OK:
        raise OracleError(rc)
    return Y


def _slot_arrays(adapters, n_slots, d_in, d_out):
    n = max(n_slots, 1)
    A_ptrs = (ctypes.c_void_p * n)()
    B_ptrs = (ctypes.c_void_p * n)()
    ranks = np.zeros(n, np.int32)
    alphas = np.zeros(n, np.float64)
    keep = []
    for slot, ad in adapters.items():
        A, B, r, alpha = ad
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        assert A.shape == (d_in, r) and B.shape == (r, d_out)
        keep += [A, B]
        A_ptrs[slot] = A.ctypes.data
        B_ptrs[slot] = B.ctypes.data
        ranks[slot] = r
        alphas[slot] = alpha
    return A_ptrs, B_ptrs, ranks, alphas, keep


def lora_linear_chains(X: np.ndarray, W: np.ndarray, token_lists: Sequence[Sequence[int]],
                       adapters: Dict[int, Tuple[np.ndarray, np.ndarray, int, float]],
                       n_slots: int, lib=None) -> np.ndarray:
    """Y (float64) = X W^T + sum over token t's listed adapters c of s_c (X A_c) B_c.

    token_lists[t]: the adapter slots applied to token t (empty: base only). Same
    adapter tuples as ``lora_linear``.
    """
    lib = lib or load()
    X = np.ascontiguousarray(X, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    T, d_in = X.shape
    d_out = W.shape[0]
    assert W.shape[1] == d_in and len(token_lists) == T
    off = np.zeros(T + 1, np.int32)
    off[1:] = np.cumsum([len(lst) for lst in token_lists])
    flat = np.array([c for lst in token_lists for c in lst] or [0], np.int32)
    A_ptrs, B_ptrs, ranks, alphas, keep = _slot_arrays(adapters, n_slots, d_in, d_out)
    Y = np.empty((T, d_out), np.float64)
    rc = lib.oracle_lora_linear_chains(_ptr(X), _ptr(W), _ptr(off), _ptr(flat), T, d_in, d_out,
                                       n_slots, ctypes.cast(A_ptrs, ctypes.c_void_p),
                                       ctypes.cast(B_ptrs, ctypes.c_void_p), _ptr(ranks),
                                       _ptr(alphas), _ptr(Y))
    if rc != OK:
        raise OracleError(rc)
    return Y


def chain_lists(ids: np.ndarray, chains: Dict[int, Sequence[int]]) -> List[List[int]]:
    """Per-token adapter lists for ids that may name chain slots: a chain slot stands for
    its members, a plain slot for itself, -1 for nothing."""
    out = []
    for i in np.asarray(ids).tolist():
        if i == -1:
            out.append([])
        elif i in chains:
            out.append(list(chains[i]))
        else:
            out.append([i])
    return out


def dequant_q4(Wq: np.ndarray, scales: np.ndarray, zeros: np.ndarray, d_in: int,
               group: int = 128, lib=None) -> np.ndarray:
    """The 4-bit base weight as bf16 bits [d_out, d_in]: bf16(s (q - z)) per group.

    Wq: uint8 [d_out, d_in / 2] (even k in the low nibble); scales: uint16 bf16 bits
    [d_in / group, d_out]; zeros: uint8 [d_in / group, d_out] in 0..15.
    """
    lib = lib or load()
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    zeros = np.ascontiguousarray(zeros, dtype=np.uint8)
    d_out = Wq.shape[0]
    assert Wq.shape == (d_out, d_in // 2) and scales.shape == zeros.shape == (d_in // group, d_out)
    W = np.empty((d_out, d_in), np.uint16)
    rc = lib.oracle_dequant_q4(_ptr(Wq), _ptr(scales), _ptr(zeros), d_out, d_in, group, _ptr(W))
    if rc != OK:
        raise OracleError(rc)
    return W


def lora_linear_q4(X: np.ndarray, Wq: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                   ids: np.ndarray, adapters, n_slots: int, group: int = 128, lib=None) -> np.ndarray:
    """The layer over the dequantised 4-bit base: lora_linear(X, dequant_q4(...), ...)."""
    W = dequant_q4(Wq, scales, zeros, X.shape[1], group, lib=lib)
    return lora_linear(X, W, ids, adapters, n_slots, lib=lib)


def problem_adapters(problem) -> Dict[int, Tuple[np.ndarray, np.ndarray, int, float]]:
    """Adapters of a ``lora_inputs.Problem`` in the tuple form ``lora_linear`` takes."""
    return {s: (a.A, a.B, a.rank, a.alpha) for s, a in problem.adapters.items()}
