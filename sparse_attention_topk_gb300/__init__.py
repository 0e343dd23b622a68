"""GB300 top-k index selector for sparse-attention indexer logits.

A thin ctypes binding over ``libtks.so`` (``include/tks.h``): argument
marshalling only.  Every step of the selection runs in the library's CUDA
kernel; there is no CPU fallback, and calls fail loudly when the library is
missing or the device is unsupported.

    import torch, sparse_attention_topk_gb300 as tks
    idx = tks.topk_indices(logits, k=2048)            # logits: cuda fp32/bf16 [batch, n]
    idx = tks.topk_indices(logits, 2048, row_len=lens)  # ragged rows (int32 cuda tensor)
"""

from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build, up_to_date

TKS_F32 = 0
TKS_BF16 = 1

TKS_OK = 0
TKS_E_INVAL = 1
TKS_E_UNSUPPORTED = 2
TKS_E_CUDA = 3
TKS_E_TIMEOUT = 4
TKS_E_INTERNAL = 5
TKS_E_ROW_LEN = 6
TKS_E_TOO_LARGE = 7
TKS_NOALLOC_MAX_ROWS = 8

TKS_K_MAX = 1 << 24
TKS_SORTED_K_MAX = 16384

TKS_OPT_FORCE_GROUP = 1
TKS_OPT_SPIN_LIMIT_NS = 2
TKS_OPT_MIN_PER_BLOCK = 3
TKS_OPT_TEST_SKIP_ARRIVE = 4
TKS_OPT_FORCE_THREADS = 5
TKS_OPT_CLUSTER = 6

# Every entry point include/tks.h declares, with its ctypes signature.
_I32, _I64, _VP = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
SIGNATURES = {
    "tks_topk_indices": (ctypes.c_int, [_VP, _VP, _I32, _I64, _I32, _I32, _VP, _VP]),
    "tks_device_status": (ctypes.c_int, [_VP]),
    "tks_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tks_version": (ctypes.c_int, []),
    "tks_release": (ctypes.c_int, []),
    "tks_set_option": (ctypes.c_int, [ctypes.c_int, _I64]),
    "tks_plan": (ctypes.c_int, [_I32, _I64, _I32, _I32, _VP, _VP]),
    "tks_topk_indices_noalloc": (ctypes.c_int, [_VP, _VP, _I32, _I64, _I32, _I32, _VP, _VP]),
    "tks_topk_indices_sorted": (ctypes.c_int, [_VP, _VP, _I32, _I64, _I32, _I32, _VP, _VP]),
    "tks_topk_indices_host": (ctypes.c_int, [_VP, _VP, _I32, _I64, _I32, _I32, _VP, _VP]),
}

_lock = threading.Lock()
_lib = None


class TksError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_string(status) if _lib is not None else f"status {status}"
        super().__init__(f"{what}: {msg}" if what else msg)


def lib_path() -> str:
    return LIB_PATH


def load(path: str | None = None):
    """Load libtks.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if path is None and not up_to_date(p):
            build()
        if not os.path.exists(p):
            raise RuntimeError(f"libtks.so not found at {p}; build it with "
                               "sparse_attention_topk_gb300._build.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def use(path: str):
    """Make the library at `path` (a build of libtks.so, e.g. the measurement
    build with warp-aggregated first-round adds) the one every call uses."""
    global _lib
    lib = load(path)
    with _lock:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().tks_status_string(int(status)).decode()


def version() -> int:
    return int(load().tks_version())


def set_option(option: int, value: int) -> None:
    rc = load().tks_set_option(int(option), int(value))
    if rc != TKS_OK:
        raise TksError(rc, "tks_set_option")


def plan(batch: int, row_stride: int, k: int, dtype: int = TKS_F32) -> tuple[int, int]:
    """(thread blocks per row, grid size) the next call with these sizes would use."""
    g, gr = ctypes.c_int32(0), ctypes.c_int32(0)
    rc = load().tks_plan(int(batch), int(row_stride), int(k), int(dtype),
                         ctypes.byref(g), ctypes.byref(gr))
    if rc != TKS_OK:
        raise TksError(rc, "tks_plan")
    return g.value, gr.value


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) its device-side status."""
    return int(load().tks_device_status(_stream_handle(stream)))


def release() -> None:
    rc = load().tks_release()
    if rc != TKS_OK:
        raise TksError(rc, "tks_release")


def topk_indices_raw(logits_ptr: int, row_len_ptr: int | None, batch: int, row_stride: int,
                     k: int, dtype: int, out_ptr: int, stream_handle: int | None = None) -> int:
    """Direct call of tks_topk_indices with raw device pointers; returns the status."""
    return int(load().tks_topk_indices(
        ctypes.c_void_p(logits_ptr), ctypes.c_void_p(row_len_ptr or 0), int(batch),
        int(row_stride), int(k), int(dtype), ctypes.c_void_p(out_ptr),
        ctypes.c_void_p(stream_handle or 0)))


def topk_indices_sorted_raw(logits_ptr: int, row_len_ptr: int | None, batch: int,
                            row_stride: int, k: int, dtype: int, out_ptr: int,
                            stream_handle: int | None = None) -> int:
    """Direct call of tks_topk_indices_sorted (rank-ordered output, k <= TKS_SORTED_K_MAX)."""
    return int(load().tks_topk_indices_sorted(
        ctypes.c_void_p(logits_ptr), ctypes.c_void_p(row_len_ptr or 0), int(batch),
        int(row_stride), int(k), int(dtype), ctypes.c_void_p(out_ptr),
        ctypes.c_void_p(stream_handle or 0)))


def topk_indices_host_raw(logits_ptr: int, row_len_ptr: int | None, batch: int, row_stride: int,
                          k: int, dtype: int, out_ptr: int, stream_handle: int | None = None) -> int:
    """Direct call of tks_topk_indices_host (page-locked host buffers)."""
    return int(load().tks_topk_indices_host(
        ctypes.c_void_p(logits_ptr), ctypes.c_void_p(row_len_ptr or 0), int(batch),
        int(row_stride), int(k), int(dtype), ctypes.c_void_p(out_ptr),
        ctypes.c_void_p(stream_handle or 0)))


def topk_indices_noalloc_raw(logits_ptr: int, row_len_ptr: int | None, batch: int,
                             row_stride: int, k: int, dtype: int, out_ptr: int,
                             stream_handle: int | None = None) -> int:
    """Direct call of tks_topk_indices_noalloc (no device allocation; at most
    TKS_NOALLOC_MAX_ROWS rows; calls must not overlap on the GPU)."""
    return int(load().tks_topk_indices_noalloc(
        ctypes.c_void_p(logits_ptr), ctypes.c_void_p(row_len_ptr or 0), int(batch),
        int(row_stride), int(k), int(dtype), ctypes.c_void_p(out_ptr),
        ctypes.c_void_p(stream_handle or 0)))


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def topk_indices(logits, k: int, row_len=None, out=None, stream=None, sorted: bool = False):
    """Top-k positions of every row of a CUDA tensor (or of a page-locked CPU tensor).

    ``logits``: float32 or bfloat16 CUDA tensor [batch, n] (or [n]) whose last
    dimension is contiguous; rows may be padded (row stride = ``logits.stride(0)``).
    ``row_len``: optional int32 CUDA tensor [batch] of valid lengths (<= n).
    ``out``: optional int32 CUDA tensor [batch, k] (contiguous) to fill.
    ``sorted``: rank order (largest value first, ties by lower position;
    tks_topk_indices_sorted, k <= TKS_SORTED_K_MAX) instead of unspecified order.
    Returns int32 [batch, k] (or [k]): each row holds its selected positions,
    then -1 where the row has fewer than k elements.

    With a page-locked (pinned) CPU ``logits`` tensor, ``row_len`` and ``out``
    are pinned CPU tensors too, the kernel reads and writes them across the
    host link (tks_topk_indices_host, unsorted only), and the result is
    complete once the stream has synchronised (``device_status(stream)``).
    """
    import torch

    squeeze = logits.dim() == 1
    x = logits.unsqueeze(0) if squeeze else logits
    host = x.dim() == 2 and not x.is_cuda
    if host:
        if sorted:
            raise ValueError("rank-ordered output needs CUDA tensors")
        if not x.is_pinned():
            raise ValueError("CPU logits must be page-locked (tensor.pin_memory())")
    if x.dim() != 2:
        raise ValueError("logits must be a 1-D or 2-D CUDA tensor")
    if x.dtype == torch.float32:
        dt = TKS_F32
    elif x.dtype == torch.bfloat16:
        dt = TKS_BF16
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    if x.size(1) > 0 and x.stride(1) != 1:
        if host:
            raise ValueError("CPU logits must have a contiguous last dimension")
        x = x.contiguous()
    batch, n = x.shape
    row_stride = x.stride(0) if batch > 1 else n
    if row_stride < n:
        if host:
            raise ValueError("CPU logits rows must not overlap")
        x = x.contiguous()
        row_stride = n
    where = "a pinned CPU" if host else "a CUDA"

    def placed(t):
        return t.is_pinned() if host else t.is_cuda

    rl_ptr = None
    if row_len is not None:
        if not (placed(row_len) and row_len.dtype == torch.int32 and row_len.numel() == batch
                and row_len.is_contiguous()):
            raise ValueError(f"row_len must be {where} int32 tensor with one entry per row")
        rl_ptr = row_len.data_ptr()
    if out is None:
        out = (torch.empty((batch, k), dtype=torch.int32, pin_memory=True) if host
               else torch.empty((batch, k), dtype=torch.int32, device=x.device))
    elif not (placed(out) and out.dtype == torch.int32 and out.is_contiguous()
              and tuple(out.shape) == (batch, k)):
        raise ValueError(f"out must be {where} contiguous int32 tensor [batch, k]")
    device = torch.cuda.current_device() if host else x.device
    with torch.cuda.device(device):
        call = (topk_indices_host_raw if host else
                topk_indices_sorted_raw if sorted else topk_indices_raw)
        rc = call(x.data_ptr() if x.numel() else 0, rl_ptr, batch,
                  row_stride if n > 0 else 0, k, dt, out.data_ptr(), _stream_handle(stream))
    if rc != TKS_OK:
        raise TksError(rc, "tks_topk_indices_host" if host else
                       "tks_topk_indices_sorted" if sorted else "tks_topk_indices")
    return out[0] if squeeze else out


__all__ = [
    "use", "topk_indices", "topk_indices_raw", "topk_indices_host_raw", "topk_indices_noalloc_raw", "topk_indices_sorted_raw", "device_status", "set_option", "plan", "release",
    "status_string", "version", "load", "lib_path", "build", "TksError", "SIGNATURES",
    "TKS_F32", "TKS_BF16", "TKS_OK", "TKS_E_INVAL", "TKS_E_UNSUPPORTED", "TKS_E_CUDA",
    "TKS_E_TIMEOUT", "TKS_E_INTERNAL", "TKS_E_ROW_LEN", "TKS_E_TOO_LARGE", "TKS_NOALLOC_MAX_ROWS",
    "TKS_K_MAX", "TKS_SORTED_K_MAX", "TKS_OPT_FORCE_GROUP",
    "TKS_OPT_SPIN_LIMIT_NS", "TKS_OPT_MIN_PER_BLOCK", "TKS_OPT_TEST_SKIP_ARRIVE", "TKS_OPT_FORCE_THREADS", "TKS_OPT_CLUSTER",
]
