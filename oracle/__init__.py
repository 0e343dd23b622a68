"""CPU oracle for the DSA TopK selector.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The selection library never does.

The arithmetic is in ``tks_oracle.c`` (plain C, single thread); this module
compiles it with gcc into ``oracle/_build/`` and calls it through ctypes.
See ``tks_oracle.c`` for what is computed and which readings of the
"Technical Deep Dive ... TopK Selector" page it takes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tks_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_NAME = "libtks_oracle.so"

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None

F32 = "f32"
BF16 = "bf16"


class OracleError(RuntimeError):
    pass


def build(out_dir: str | None = None, mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle; returns the path of the shared library.

    ``mutant`` > 0 builds a deliberately wrong variant (tests of the pins only).
    """
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = _LIB_NAME if mutant == 0 else f"libtks_oracle_mutant{mutant}.so"
    path = os.path.join(out_dir, name)
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, f"-DTKS_ORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.tks_oracle_topk_batch.argtypes = [vp, i32, i64, i64, vp, i64, vp]
    lib.tks_oracle_topk_batch.restype = ctypes.c_int
    lib.tks_oracle_topk_batch_order.argtypes = [vp, i32, i64, i64, vp, i64, i32, vp]
    lib.tks_oracle_topk_batch_order.restype = ctypes.c_int
    lib.tks_oracle_topk_f32.argtypes = [vp, i64, i64, vp]
    lib.tks_oracle_topk_f32.restype = ctypes.c_int
    lib.tks_oracle_selftest.argtypes = []
    lib.tks_oracle_selftest.restype = ctypes.c_int
    lib.tks_oracle_mutant.argtypes = []
    lib.tks_oracle_mutant.restype = ctypes.c_int
    rc = lib.tks_oracle_selftest()
    if rc != 0:
        raise OracleError(f"oracle build flushes subnormals or loses the sign of zero (code {rc})")
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use)."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def topk_indices(values: np.ndarray, k: int, row_len=None, dtype: str | None = None,
                 lib=None, ordered: bool = False) -> np.ndarray:
    """Top-k index set of every row.

    ``values``: [batch, row_stride] (or 1-D for one row) float32, or uint16 holding
    bf16 bit patterns (``dtype="bf16"``).  ``row_len``: valid length per row
    (default: the whole stride).  Returns int32 [batch, k]: each row's selected
    positions in ascending order (``ordered``: in rank order, largest value
    first, ties by lower position), then -1 where the row has fewer than k values.
    """
    v = np.asarray(values)
    squeeze = v.ndim == 1
    if squeeze:
        v = v[None, :]
    if dtype is None:
        dtype = BF16 if v.dtype == np.uint16 else F32
    if dtype == F32:
        v = np.ascontiguousarray(v, dtype=np.float32)
        code = 0
    elif dtype == BF16:
        v = np.ascontiguousarray(v, dtype=np.uint16)
        code = 1
    else:
        raise ValueError(f"dtype {dtype!r}")
    batch, stride = v.shape
    if row_len is None:
        rl = np.full(batch, stride, np.int32)
    else:
        rl = np.ascontiguousarray(np.broadcast_to(np.asarray(row_len, np.int32), (batch,)))
    out = np.empty((batch, int(k)), np.int32)
    lib = lib or load()
    rc = lib.tks_oracle_topk_batch_order(v.ctypes.data, code, batch, stride, rl.ctypes.data,
                                         int(k), 1 if ordered else 0, out.ctypes.data)
    if rc != 0:
        raise OracleError({1: "invalid argument", 2: "NaN in a valid position",
                           3: "out of memory"}.get(rc, f"error {rc}"))
    return out[0] if squeeze else out


def topk_workload(w, lib=None, ordered: bool = False) -> np.ndarray:
    """Top-k of a ``workloads.Workload``."""
    return topk_indices(w.values, w.k, w.row_len, w.dtype, lib=lib, ordered=ordered)


__all__ = ["build", "load", "topk_indices", "topk_workload", "OracleError", "F32", "BF16"]
