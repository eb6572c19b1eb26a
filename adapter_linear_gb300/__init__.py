"""Python binding of the GB300 multi-LoRA linear library (``include/lora_linear.h``).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of ``liblora_linear.so``; torch tensors are used for device memory and
streams. There is no CPU fall-back: if the library has not been built (see
``adapter_linear_gb300.build``) every call raises ``LibraryMissing``.

The functions keep the C names (``lora_pool_create``, ``lora_load_adapter``,
``lora_linear`` ...); ``LoraPool`` wraps a handle for convenience.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
# ADAPTER_LINEAR_CHECKED=1 selects the build with range checks in every kernel
# (liblora_linear_check.so, the same ABI; see LORA_ERR_RANGE)
CHECKED = os.environ.get("ADAPTER_LINEAR_CHECKED", "0") == "1"
LIB_PATH = os.path.join(HERE, "liblora_linear_check.so" if CHECKED else "liblora_linear.so")

LORA_OK = 0
STATUS_NAMES = {
    0: "LORA_OK", 1: "LORA_ERR_ARG", 2: "LORA_ERR_SHAPE", 3: "LORA_ERR_SLOT_RANGE",
    4: "LORA_ERR_SLOT_OCCUPIED", 5: "LORA_ERR_SLOT_EMPTY", 6: "LORA_ERR_RANK",
    7: "LORA_ERR_BAD_ADAPTER_ID", 8: "LORA_ERR_CUDA", 9: "LORA_ERR_OOM", 10: "LORA_ERR_TIMEOUT",
    11: "LORA_ERR_UNSUPPORTED",
    12: "LORA_ERR_IN_USE", 13: "LORA_ERR_RANGE",
}
globals().update({v: k for k, v in STATUS_NAMES.items()})
LORA_PATH_AUTO, LORA_PATH_DECODE, LORA_PATH_PREFILL = 0, 1, 2
LORA_PREFILL_AUTO, LORA_PREFILL_SINGLE, LORA_PREFILL_PAIR = 0, 1, 2
LORA_STATS_COUNT = 7
STATS_FIELDS = ("loaded", "free_pages", "total_pages", "loads", "unloads", "calls", "bytes_held")

# every symbol the header declares
EXPORTS = (
    "lora_pool_create", "lora_pool_destroy", "lora_pool_reserve", "lora_load_adapter",
    "lora_unload_adapter", "lora_linear", "lora_linear_host", "lora_base_linear",
    "lora_pool_check_errors", "lora_build_segments", "lora_pool_stats", "lora_pool_set_path", "lora_pool_set_prefill_kernel",
    "lora_status_string", "lora_abi_version", "lora_pool_enable_timing", "lora_pool_kernel_times",
    "lora_base_linear_noalloc", "lora_linear_grouped", "lora_define_chain",
    "lora_host_register", "lora_host_unregister", "lora_acquire", "lora_prefetch", "lora_release",
    "lora_cache_stats", "lora_pool_selftest_wait", "lora_decode_plan_info", "lora_test_delayed_copy",
    "lora_pool_set_trace", "lora_linear_q4", "lora_base_linear_q4", "lora_dequant_q4",
)
PLAN_INFO_FIELDS = ("units", "G", "grid", "max_seg", "n_acc", "stages", "tmem_cols", "smem_bytes",
                    "pairs", "col_blocks", "tight", "ntok", "partials_floats", "prefetch_a")
CACHE_STATS_FIELDS = ("registered", "resident", "hits", "misses", "evictions")
LORA_MAX_GROUP = 8
LORA_KERNEL_SLOTS = 4
KERNEL_SLOT_NAMES = ("segment_build", "shrink", "base_gemm", "finish_expand")


class LibraryMissing(RuntimeError):
    pass


class LoraError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and type the C ABI. Raises LibraryMissing if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise LibraryMissing(
            f"{path} is missing: build it with `python -m adapter_linear_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "lora_pool_create": [i32, i32, i32, i32, ctypes.POINTER(vp)],
        "lora_pool_destroy": [vp],
        "lora_pool_reserve": [vp, i32],
        "lora_load_adapter": [vp, i32, vp, vp, i32, f32],
        "lora_unload_adapter": [vp, i32],
        "lora_linear": [vp, vp, vp, vp, i32, vp, vp],
        "lora_linear_host": [vp, vp, vp, vp, i32, vp, vp],
        "lora_base_linear": [vp, vp, vp, i32, vp, vp],
        "lora_pool_check_errors": [vp],
        "lora_build_segments": [vp, vp, i32, vp, vp, vp, vp, vp, vp],
        "lora_pool_stats": [vp, vp],
        "lora_pool_set_path": [vp, i32],
        "lora_pool_set_prefill_kernel": [vp, i32],
        "lora_status_string": [i32],
        "lora_abi_version": [],
        "lora_pool_enable_timing": [vp, i32],
        "lora_pool_kernel_times": [vp, vp],
        "lora_base_linear_noalloc": [vp, vp, i32, i32, i32, vp, vp],
        "lora_linear_grouped": [i32, vp, vp, vp, vp, i32, vp, vp],
        "lora_define_chain": [vp, i32, vp, i32],
        "lora_host_register": [vp, ctypes.c_int64, vp, vp, i32, f32],
        "lora_host_unregister": [vp, ctypes.c_int64],
        "lora_acquire": [vp, ctypes.c_int64, vp, ctypes.POINTER(i32)],
        "lora_prefetch": [vp, ctypes.c_int64],
        "lora_release": [vp, i32],
        "lora_cache_stats": [vp, vp],
        "lora_pool_selftest_wait": [vp, i32, vp],
        "lora_decode_plan_info": [i32, i32, vp, vp, vp, i32, vp],
        "lora_test_delayed_copy": [vp, vp, i32, i32, vp],
        "lora_pool_set_trace": [vp, vp, i32],
        "lora_linear_q4": [vp, vp, vp, vp, vp, vp, i32, vp, vp],
        "lora_base_linear_q4": [vp, vp, vp, vp, vp, i32, vp, vp],
        "lora_dequant_q4": [vp, vp, vp, i32, i32, vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.lora_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != LORA_OK:
        raise LoraError(status, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------ C-named thin wrappers

def lora_pool_create(max_adapters: int, max_rank: int, d_in: int, d_out: int) -> int:
    h = ctypes.c_void_p()
    _check(load_library().lora_pool_create(max_adapters, max_rank, d_in, d_out, ctypes.byref(h)),
           "lora_pool_create")
    return h.value


def lora_pool_destroy(pool: int) -> None:
    _check(load_library().lora_pool_destroy(pool), "lora_pool_destroy")


def lora_pool_reserve(pool: int, max_tokens: int) -> None:
    _check(load_library().lora_pool_reserve(pool, max_tokens), "lora_pool_reserve")


def lora_load_adapter(pool: int, slot: int, A, B, rank: int, alpha: float) -> int:
    """A: bf16 d_in x rank, B: bf16 rank x d_out (contiguous; host or device). Returns status."""
    return load_library().lora_load_adapter(pool, slot, _ptr(A), _ptr(B), rank, float(alpha))


def lora_unload_adapter(pool: int, slot: int) -> int:
    return load_library().lora_unload_adapter(pool, slot)


def lora_linear(pool: int, X, W_base, ids, T: int, Y, stream=None) -> int:
    return load_library().lora_linear(pool, _ptr(X), _ptr(W_base), _ptr(ids), T, _ptr(Y),
                                      _stream(stream))


def lora_linear_host(pool: int, X_host, W_base, ids_host, T: int, Y_host, stream=None) -> int:
    return load_library().lora_linear_host(pool, _ptr(X_host), _ptr(W_base), _ptr(ids_host), T,
                                           _ptr(Y_host), _stream(stream))


def delayed_copy(src, dst, n: int, delay_us: int, stream=None):
    """Stream-order test hook: copy n int32 src -> dst (device tensors) after delay_us,
    letting the next kernel in the stream launch at once."""
    _check(load_library().lora_test_delayed_copy(_ptr(src), _ptr(dst), n, delay_us, _stream(stream)),
           "lora_test_delayed_copy")


def decode_plan_info(T: int, d_in, d_out, max_pages, num_sms: int = 152) -> Dict[str, int]:
    """The decode plan for len(d_in) layers of T tokens (host only, no GPU)."""
    import numpy as np
    n = len(d_in)
    a = np.ascontiguousarray(d_in, np.int32)
    b = np.ascontiguousarray(d_out, np.int32)
    c = np.ascontiguousarray(max_pages, np.int32)
    out = np.zeros(len(PLAN_INFO_FIELDS), np.int64)
    _check(load_library().lora_decode_plan_info(n, T, a.ctypes.data, b.ctypes.data, c.ctypes.data,
                                                num_sms, out.ctypes.data), "lora_decode_plan_info")
    return dict(zip(PLAN_INFO_FIELDS, (int(v) for v in out)))


def lora_define_chain(pool: int, chain_slot: int, member_slots) -> int:
    members = (ctypes.c_int * max(len(member_slots), 1))(*member_slots)
    return load_library().lora_define_chain(pool, chain_slot, members, len(member_slots))


def lora_linear_grouped(pools, X, W_base, ids, T: int, Y, stream=None) -> int:
    """n layers that share the token ids in one decode launch chain: pools, X, W_base and Y
    are equal-length sequences (pool handles and tensors / device pointers)."""
    n = len(pools)
    arr = ctypes.c_void_p * max(n, 1)
    ph = arr(*[int(p) if p else None for p in pools])
    xs = arr(*[_ptr(x) for x in X])
    ws = arr(*[_ptr(w) for w in W_base])
    ys = arr(*[_ptr(y) for y in Y])
    return load_library().lora_linear_grouped(n, ph, xs, ws, _ptr(ids), T, ys, _stream(stream))


def lora_base_linear(pool: int, X, W_base, T: int, Y, stream=None) -> int:
    return load_library().lora_base_linear(pool, _ptr(X), _ptr(W_base), T, _ptr(Y),
                                           _stream(stream))


def lora_base_linear_noalloc(X, W_base, T: int, d_in: int, d_out: int, Y, stream=None) -> int:
    """Base product through the entry point that allocates no device memory (no pool):
    for callers that may not call cudaMalloc."""
    return load_library().lora_base_linear_noalloc(_ptr(X), _ptr(W_base), T, d_in, d_out, _ptr(Y),
                                                   _stream(stream))


def lora_pool_check_errors(pool: int) -> int:
    return load_library().lora_pool_check_errors(pool)


def lora_build_segments(pool: int, ids, T: int, order, n_base, num_seg, seg_start, seg_slot,
                        stream=None) -> int:
    return load_library().lora_build_segments(pool, _ptr(ids), T, _ptr(order), _ptr(n_base),
                                              _ptr(num_seg), _ptr(seg_start), _ptr(seg_slot),
                                              _stream(stream))


def lora_pool_stats(pool: int) -> Dict[str, int]:
    out = (ctypes.c_int64 * LORA_STATS_COUNT)()
    _check(load_library().lora_pool_stats(pool, ctypes.cast(out, ctypes.c_void_p)),
           "lora_pool_stats")
    return dict(zip(STATS_FIELDS, list(out)))


def lora_pool_set_path(pool: int, path: int) -> int:
    return load_library().lora_pool_set_path(pool, path)


def lora_pool_set_prefill_kernel(pool: int, kernel: int) -> int:
    return load_library().lora_pool_set_prefill_kernel(pool, kernel)


def lora_pool_enable_timing(pool: int, enable: bool) -> int:
    return load_library().lora_pool_enable_timing(pool, int(bool(enable)))


def lora_pool_kernel_times(pool: int) -> Dict[str, float]:
    """Device milliseconds of each kernel of the pool's last call (timing must be enabled)."""
    out = (ctypes.c_float * LORA_KERNEL_SLOTS)()
    _check(load_library().lora_pool_kernel_times(pool, ctypes.cast(out, ctypes.c_void_p)),
           "lora_pool_kernel_times")
    return dict(zip(KERNEL_SLOT_NAMES, list(out)))


def lora_pool_set_trace(pool: int, buf, n_calls: int) -> int:
    """Span trace of the pool's next calls into a device buffer (see the header)."""
    return load_library().lora_pool_set_trace(pool, _ptr(buf), n_calls)


def lora_linear_q4(pool: int, X, Wq, scales, zeros, ids, T: int, Y, stream=None) -> int:
    return load_library().lora_linear_q4(pool, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zeros), _ptr(ids), T,
                                         _ptr(Y), _stream(stream))


def lora_base_linear_q4(pool: int, X, Wq, scales, zeros, T: int, Y, stream=None) -> int:
    return load_library().lora_base_linear_q4(pool, _ptr(X), _ptr(Wq), _ptr(scales), _ptr(zeros), T,
                                              _ptr(Y), _stream(stream))


def lora_dequant_q4(Wq, scales, zeros, d_out: int, d_in: int, W, stream=None) -> int:
    return load_library().lora_dequant_q4(_ptr(Wq), _ptr(scales), _ptr(zeros), d_out, d_in, _ptr(W),
                                          _stream(stream))


def lora_status_string(status: int) -> str:
    return load_library().lora_status_string(status).decode()


def lora_abi_version() -> int:
    return load_library().lora_abi_version()


# --------------------------------------------------------------- convenience

class LoraPool:
    """Owns one pool handle; torch tensors in, torch tensors out."""

    def __init__(self, max_adapters: int, max_rank: int, d_in: int, d_out: int):
        self.max_adapters, self.max_rank, self.d_in, self.d_out = max_adapters, max_rank, d_in, d_out
        self.handle = lora_pool_create(max_adapters, max_rank, d_in, d_out)

    def close(self):
        if self.handle:
            lora_pool_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass

    def reserve(self, max_tokens: int):
        lora_pool_reserve(self.handle, max_tokens)

    def load_adapter(self, slot: int, A, B, rank: int, alpha: float):
        A = A.contiguous()
        B = B.contiguous()
        _check(lora_load_adapter(self.handle, slot, A, B, rank, alpha), "lora_load_adapter")

    def unload_adapter(self, slot: int):
        _check(lora_unload_adapter(self.handle, slot), "lora_unload_adapter")

    # ---- host tier
    def host_register(self, key: int, A, B, rank: int, alpha: float):
        _check(load_library().lora_host_register(self.handle, key, _ptr(A), _ptr(B), rank,
                                                 float(alpha)), "lora_host_register")

    def host_unregister(self, key: int):
        _check(load_library().lora_host_unregister(self.handle, key), "lora_host_unregister")

    def acquire(self, key: int, stream=None) -> int:
        slot = ctypes.c_int(-1)
        _check(load_library().lora_acquire(self.handle, key, _stream(stream), ctypes.byref(slot)),
               "lora_acquire")
        return slot.value

    def prefetch(self, key: int):
        _check(load_library().lora_prefetch(self.handle, key), "lora_prefetch")

    def release(self, slot: int):
        _check(load_library().lora_release(self.handle, slot), "lora_release")

    def cache_stats(self) -> Dict[str, int]:
        import numpy as np
        out = np.zeros(len(CACHE_STATS_FIELDS), np.int64)
        _check(load_library().lora_cache_stats(self.handle, out.ctypes.data), "lora_cache_stats")
        return dict(zip(CACHE_STATS_FIELDS, (int(v) for v in out)))

    def define_chain(self, chain_slot: int, member_slots):
        _check(lora_define_chain(self.handle, chain_slot, list(member_slots)), "lora_define_chain")

    def set_path(self, path: int):
        _check(lora_pool_set_path(self.handle, path), "lora_pool_set_path")

    def set_prefill_kernel(self, kernel: int):
        _check(lora_pool_set_prefill_kernel(self.handle, kernel), "lora_pool_set_prefill_kernel")

    def linear(self, X, W, ids, Y=None, stream=None):
        import torch
        T = X.shape[0]
        if Y is None:
            Y = torch.empty((T, self.d_out), dtype=torch.bfloat16, device=X.device)
        _check(lora_linear(self.handle, X, W, ids, T, Y, stream), "lora_linear")
        return Y

    def linear_host(self, X_host, W, ids_host, Y_host, stream=None):
        _check(lora_linear_host(self.handle, X_host, W, ids_host, X_host.shape[0], Y_host, stream),
               "lora_linear_host")
        return Y_host

    @staticmethod
    def linear_grouped(pools, Xs, Ws, ids, Ys=None, stream=None):
        """Y_m = lora_linear of pools[m] on (Xs[m], Ws[m]) for all m, with one set of ids,
        in one launch chain on the decode path (one call per layer above 256 tokens)."""
        import torch
        T = ids.shape[0]
        if Ys is None:
            Ys = [torch.empty((T, p.d_out), dtype=torch.bfloat16, device=ids.device) for p in pools]
        _check(lora_linear_grouped([p.handle for p in pools], Xs, Ws, ids, T, Ys, stream),
               "lora_linear_grouped")
        return Ys

    def linear_q4(self, X, Wq, scales, zeros, ids, Y=None, stream=None):
        """The layer over a 4-bit base (codes, bf16 scales, 4-bit zero points per 128 inputs)."""
        import torch
        T = X.shape[0]
        if Y is None:
            Y = torch.empty((T, self.d_out), dtype=torch.bfloat16, device=X.device)
        _check(lora_linear_q4(self.handle, X, Wq, scales, zeros, ids, T, Y, stream), "lora_linear_q4")
        return Y

    def base_linear_q4(self, X, Wq, scales, zeros, Y=None, stream=None):
        import torch
        T = X.shape[0]
        if Y is None:
            Y = torch.empty((T, self.d_out), dtype=torch.bfloat16, device=X.device)
        _check(lora_base_linear_q4(self.handle, X, Wq, scales, zeros, T, Y, stream), "lora_base_linear_q4")
        return Y

    def base_linear(self, X, W, Y=None, stream=None):
        import torch
        T = X.shape[0]
        if Y is None:
            Y = torch.empty((T, self.d_out), dtype=torch.bfloat16, device=X.device)
        _check(lora_base_linear(self.handle, X, W, T, Y, stream), "lora_base_linear")
        return Y

    def selftest_wait(self, limit_us: int, stream=None):
        _check(load_library().lora_pool_selftest_wait(self.handle, limit_us, _stream(stream)),
               "lora_pool_selftest_wait")

    def check_errors(self) -> int:
        return lora_pool_check_errors(self.handle)

    def build_segments(self, ids, stream=None):
        import torch
        T = ids.shape[0]
        cap = min(T, self.max_adapters) + 1
        dev = ids.device
        order = torch.empty(max(T, 1), dtype=torch.int32, device=dev)
        hdr = torch.zeros(2, dtype=torch.int32, device=dev)
        seg_start = torch.zeros(cap, dtype=torch.int32, device=dev)
        seg_slot = torch.zeros(cap, dtype=torch.int32, device=dev)
        _check(lora_build_segments(self.handle, ids, T, order, hdr[0:1], hdr[1:2], seg_start,
                                   seg_slot, stream), "lora_build_segments")
        return order[:T], hdr, seg_start, seg_slot

    def stats(self) -> Dict[str, int]:
        return lora_pool_stats(self.handle)

    def enable_timing(self, enable: bool = True):
        _check(lora_pool_enable_timing(self.handle, enable), "lora_pool_enable_timing")

    def kernel_times(self) -> Dict[str, float]:
        return lora_pool_kernel_times(self.handle)

    def set_trace(self, buf, n_calls: int = 1):
        """buf: device int64/uint64 tensor of n_calls * LORA_KERNEL_SLOTS * 4 entries, or None."""
        _check(lora_pool_set_trace(self.handle, buf, n_calls), "lora_pool_set_trace")
