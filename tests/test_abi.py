"""The C-ABI library builds, loads and exports every entry point include/tks.h
declares; host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re

import pytest

import sparse_attention_topk_gb300 as tks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(tks_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_function():
    lib = tks.load()
    declared = declared_functions()
    assert "tks_topk_indices" in declared
    for name in declared:
        assert hasattr(lib, name), name
    # and the binding knows the signature of each
    assert declared == set(tks.SIGNATURES)


def test_status_strings_and_version():
    assert tks.version() >= 100
    for s in range(0, 7):
        assert tks.status_string(s)
    assert tks.status_string(999) == "unknown status"


@pytest.mark.parametrize("args", [
    # logits, row_len, batch, row_stride, k, dtype, out
    (16, None, -1, 8, 1, 0, 16),       # negative batch
    (16, None, 1, -8, 1, 0, 16),       # negative stride
    (16, None, 1, 1 << 31, 1, 0, 16),  # stride beyond int32
    (16, None, 1, 8, 0, 0, 16),        # k < 1
    (16, None, 1, 8, tks.TKS_K_MAX + 1, 0, 16),
    (16, None, 1, 8, 1, 7, 16),        # bad dtype
    (16, None, 1, 8, 1, 0, 0),         # null output
    (16, None, 1, 8, 1, 0, 18),        # misaligned output
    (0, None, 1, 8, 1, 0, 16),         # null logits
    (18, None, 1, 8, 1, 0, 16),        # fp32 logits not 4-byte aligned
])
def test_invalid_arguments_rejected_before_any_cuda_call(args):
    logits, row_len, batch, stride, k, dtype, out = args
    assert tks.topk_indices_raw(logits, row_len, batch, stride, k, dtype, out, 0) == tks.TKS_E_INVAL


@pytest.mark.parametrize("args", [
    # logits, row_len, batch, row_stride, k, dtype, out -- a few rows and k <= 4096 (the
    # many-block ordering path) and more rows (the one-block path) alike
    (16, None, 1, 8, 0, 0, 16),
    (16, None, 2, 8, 1, 7, 16),
    (16, None, 3, 8, 1, 0, 0),
    (16, None, 3, 8, 1, 0, 18),
    (0, None, 1, 8, 1, 0, 16),
    (18, None, 1, 8, 1, 0, 16),
    (16, None, 9, -8, 1, 0, 16),
    (16, None, 20, 8, 0, 0, 16),
])
def test_sorted_entry_rejects_bad_arguments_before_any_cuda_call(args):
    logits, row_len, batch, stride, k, dtype, out = args
    assert tks.topk_indices_sorted_raw(logits, row_len, batch, stride, k, dtype, out, 0) == \
        tks.TKS_E_INVAL


def test_sorted_entry_validates_like_the_plain_one():
    assert tks.topk_indices_sorted_raw(16, None, 1, 8, tks.TKS_SORTED_K_MAX + 1, 0, 16, 0) == tks.TKS_E_INVAL
    assert tks.topk_indices_sorted_raw(16, None, 1, 8, 0, 0, 16, 0) == tks.TKS_E_INVAL
    assert tks.topk_indices_sorted_raw(16, None, 1, 8, 1, 7, 16, 0) == tks.TKS_E_INVAL
    assert tks.topk_indices_sorted_raw(0, None, 0, 8, 1, 0, 16, 0) == tks.TKS_OK


def test_empty_batch_is_a_no_op():
    assert tks.topk_indices_raw(0, None, 0, 8, 1, 0, 16, 0) == tks.TKS_OK


def test_options():
    lib = tks.load()
    assert lib.tks_set_option(12345, 1) == tks.TKS_E_INVAL
    assert lib.tks_set_option(tks.TKS_OPT_FORCE_GROUP, -1) == tks.TKS_E_INVAL
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)
    tks.set_option(tks.TKS_OPT_SPIN_LIMIT_NS, 1_000_000_000)
    assert lib.tks_set_option(tks.TKS_OPT_FORCE_THREADS, 384) == tks.TKS_E_INVAL
    for t in (256, 512, 0):
        tks.set_option(tks.TKS_OPT_FORCE_THREADS, t)


def test_no_device_is_reported_not_faked():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid-looking arguments, no GPU: the library must not pretend to have run
    rc = tks.topk_indices_raw(16, None, 1, 8, 1, 0, 16, 0)
    assert rc in (tks.TKS_E_UNSUPPORTED, tks.TKS_E_CUDA)


def test_host_entry_validates_before_any_launch():
    assert tks.topk_indices_host_raw(16, None, -1, 8, 1, 0, 16, 0) == tks.TKS_E_INVAL
    assert tks.topk_indices_host_raw(16, None, 1, 8, 1, 0, 0, 0) == tks.TKS_E_INVAL
    assert tks.topk_indices_host_raw(0, None, 0, 8, 0, 0, 16, 0) == tks.TKS_E_INVAL
    assert tks.topk_indices_host_raw(0, None, 0, 8, 1, 0, 16, 0) == tks.TKS_OK
    # without a GPU (or with a pointer that is not page-locked host memory)
    # nothing can be translated: refused, never run
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert tks.topk_indices_host_raw(16, None, 1, 8, 1, 0, 16, 0) == tks.TKS_E_INVAL


def test_noalloc_entry_checks_arguments_before_its_row_limit():
    # argument errors are those of tks_topk_indices, whatever the batch size
    for args in [(16, None, 9, 8, 1, 0, 0), (16, None, 9, 8, 0, 0, 16), (18, None, 9, 8, 1, 0, 16),
                 (16, None, 1, 8, 1, 7, 16), (16, None, -1, 8, 1, 0, 16)]:
        assert tks.topk_indices_noalloc_raw(*args, 0) == tks.TKS_E_INVAL, args
    # then the array's row limit, still before any CUDA call
    assert tks.topk_indices_noalloc_raw(16, None, tks.TKS_NOALLOC_MAX_ROWS + 1, 8, 1, 0, 16, 0) == \
        tks.TKS_E_TOO_LARGE
    assert tks.topk_indices_noalloc_raw(0, None, 0, 8, 1, 0, 16, 0) == tks.TKS_OK
