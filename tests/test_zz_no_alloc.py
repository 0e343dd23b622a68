"""The allocation-free entry point, for callers that cannot allocate device
memory, gives the same index sets as the allocating entry point.

Collected last on purpose (its file name sorts after the others), so a run
that stops at the first failure has run every other test before it.  It
passes alone in a fresh process and after the rest of the suite."""

import ctypes

import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


def _call(fn, x, w, out, rl):
    return fn(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(rl.data_ptr() if rl is not None else 0),
              int(w.batch), int(w.row_stride), int(w.k), 0 if w.dtype == W.F32 else 1,
              ctypes.c_void_p(out.data_ptr()),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["decode_4k", "decode_1m_masked", "batch4_1m_bf16"])
def test_noalloc_matches_allocating_entry_point_on_two_calls(name):
    lib = tks.load()
    w = W.named(name)
    assert w.batch <= tks.TKS_NOALLOC_MAX_ROWS
    x = torch.from_numpy(w.values.copy()).cuda()
    rl = torch.from_numpy(w.row_len.copy()).cuda()
    ref = torch.full((w.batch, w.k), -7, dtype=torch.int32, device="cuda")
    assert _call(lib.tks_topk_indices, x, w, ref, rl) == tks.TKS_OK
    torch.cuda.synchronize()
    assert tks.device_status() == tks.TKS_OK
    want = np.sort(ref.cpu().numpy(), axis=1)
    for _ in range(2):  # two calls in a row share the fixed scratch
        got = torch.full((w.batch, w.k), -7, dtype=torch.int32, device="cuda")
        assert _call(lib.tks_topk_indices_noalloc, x, w, got, rl) == tks.TKS_OK
        torch.cuda.synchronize()
        # index sets: tolerance is exact equality
        assert np.array_equal(np.sort(got.cpu().numpy(), axis=1), want), name


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    lib = tks.load()
    n = tks.TKS_NOALLOC_MAX_ROWS + 1
    x = torch.zeros((n, 64), dtype=torch.float32, device="cuda")
    out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    rc = lib.tks_topk_indices_noalloc(ctypes.c_void_p(x.data_ptr()), None, n, 64, 4, 0,
                                      ctypes.c_void_p(out.data_ptr()), None)
    assert rc == tks.TKS_E_TOO_LARGE
    assert "fixed scratch" in tks.status_string(rc)
