"""tks_topk_indices_host against the oracle: page-locked host buffers read and
written by the kernel itself, on the named workloads and on rows that take
the non-resident (plain global load) path."""

import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_parity_gpu import _defaults, assert_matches_oracle  # noqa: F401
from tests.test_prefill_gpu import _mixed_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


def run_host(w, with_row_len=True):
    x = torch.from_numpy(w.values.copy()).pin_memory()
    if w.dtype == W.BF16:
        x = x.view(torch.bfloat16)
    rl = torch.from_numpy(w.row_len.copy()).pin_memory() if with_row_len else None
    s = torch.cuda.Stream()
    out = tks.topk_indices(x, w.k, row_len=rl, stream=s)
    assert out.is_pinned() and not out.is_cuda
    st = tks.device_status(s)
    assert st == tks.TKS_OK, tks.status_string(st)
    return out.numpy().copy()


@pytest.mark.parametrize("name", sorted(W.NAMED) + ["prefill_causal"])
def test_host_buffers_match_oracle(name):
    w = W.named(name)
    assert_matches_oracle(w, run_host(w), check_invariants=False)


def test_host_full_rows_without_row_len():
    w = W.named("decode_128k")
    assert_matches_oracle(w, run_host(w, with_row_len=False), check_invariants=False)


@pytest.mark.parametrize("dtype,stride", [(W.F32, 60001), (W.BF16, 100003)])
def test_host_rows_larger_than_on_chip_copy(dtype, stride):
    """Whole rows per block, some longer than the on-chip copy: those are read
    from host memory on every pass."""
    w = _mixed_rows(dtype, stride, 50, seed=77)
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 1)
    try:
        assert_matches_oracle(w, run_host(w), check_invariants=False)
    finally:
        tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)


def test_host_split_rows_through_clusters():
    w = W.named("decode_128k")
    tks.set_option(tks.TKS_OPT_CLUSTER, 1)
    try:
        assert_matches_oracle(w, run_host(w), check_invariants=False)
    finally:
        tks.set_option(tks.TKS_OPT_CLUSTER, 0)


def test_host_entry_rejects_memory_that_is_not_page_locked():
    """Pageable host memory and device memory are refused before any launch."""
    n, k = 4096, 16
    pageable = np.zeros(n, np.float32)
    out_pageable = np.zeros(k, np.int32)
    x_pin = torch.zeros(n, dtype=torch.float32).pin_memory()
    out_pin = torch.zeros(k, dtype=torch.int32).pin_memory()
    x_dev = torch.zeros(n, dtype=torch.float32, device="cuda")
    out_dev = torch.zeros(k, dtype=torch.int32, device="cuda")
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p).value  # noqa: E731
    cases = [
        (ptr(pageable), out_pin.data_ptr()),
        (x_pin.data_ptr(), ptr(out_pageable)),
        (x_dev.data_ptr(), out_pin.data_ptr()),
        (x_pin.data_ptr(), out_dev.data_ptr()),
    ]
    for xp, op in cases:
        assert tks.topk_indices_host_raw(xp, None, 1, n, k, tks.TKS_F32, op) == tks.TKS_E_INVAL
    with pytest.raises(ValueError):
        tks.topk_indices(torch.zeros(n), k)  # not pinned
    with pytest.raises(ValueError):
        tks.topk_indices(x_pin, k, sorted=True)
    assert tks.device_status(None) == tks.TKS_OK


def test_host_and_device_entries_agree_on_fuzz_rows():
    for w in W.fuzz_cases():
        if w.batch == 0 or w.row_stride == 0:
            continue
        want = oracle.topk_workload(w)
        assert_matches_oracle(w, run_host(w), want, check_invariants=False)
