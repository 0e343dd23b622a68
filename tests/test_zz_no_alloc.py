"""The allocation-free entry point, for callers that cannot allocate device
memory, against the CPU oracle (and the allocating entry point beside it).

Collected last on purpose (its file name sorts after the others), so a run
that stops at the first failure has run every other test before it.  It
passes alone in a fresh process and after the rest of the suite."""

import ctypes

import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import sparse_attention_topk_gb300 as tks  # noqa: E402


def _device_input(w):
    x = torch.from_numpy(w.values.copy()).cuda()
    rl = torch.from_numpy(w.row_len.astype(np.int32)).cuda()
    return x, rl


def _call(fn, x, w, out, rl):
    return fn(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(rl.data_ptr() if rl is not None else 0),
              int(w.batch), int(w.row_stride), int(w.k), 0 if w.dtype == W.F32 else 1,
              ctypes.c_void_p(out.data_ptr()),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_sets(got, want, lens, k, what):
    """Index sets compared exactly: the first min(k, L) slots of a row hold the
    oracle's positions in any order, the rest hold -1."""
    for r in range(got.shape[0]):
        take = min(k, max(0, int(lens[r])))
        assert np.array_equal(np.sort(got[r][got[r] >= 0]), want[r, :take]), f"{what}: row {r}"
        assert int(np.sum(got[r] < 0)) == k - take, f"{what}: row {r} padding"


def _ragged8():
    """Eight ragged fp32 rows (the array's whole capacity) on an odd row
    stride, each split over several blocks; row 7 is the longest."""
    rng = np.random.Generator(np.random.PCG64(71))
    lens = [20011, 65536, 131071, 5000, 99999, 40000, 150001, 199999]
    rows = [(rng.standard_normal(n) * 2.0 + rng.uniform(-3, 3)).astype(np.float32) for n in lens]
    return W.from_rows("ragged8", rows, 1000, W.F32, row_stride=200003)


def _bf16_k777():
    """Three bf16 rows, k=777: N(0,1), a few levels (heavy ties), and signed
    zeros with subnormals."""
    rng = np.random.Generator(np.random.PCG64(72))
    rows = [W.f32_to_bf16_bits(rng.standard_normal(300000)),
            W.f32_to_bf16_bits(rng.integers(0, 5, size=250000).astype(np.float32)),
            W.bf16_mixed_zeros_subnormals(rng, 280000, 0.2, 0.2, 0.2)]
    return W.from_rows("bf16_k777", rows, 777, W.BF16, row_stride=300000)


CASES = {
    "decode_4k": W.decode_4k, "decode_128k": W.decode_128k,
    "decode_1m_masked": W.decode_1m_masked, "batch4_1m_bf16": W.batch4_1m_bf16,
    "ragged8": _ragged8, "bf16_k777": _bf16_k777,
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle_on_two_calls(name):
    lib = tks.load()
    w = CASES[name]()
    assert w.batch <= tks.TKS_NOALLOC_MAX_ROWS
    want = oracle.topk_workload(w)
    x, rl = _device_input(w)
    for call in range(2):  # two calls in a row share the fixed scratch
        got = torch.full((w.batch, w.k), -7, dtype=torch.int32, device="cuda")
        assert _call(lib.tks_topk_indices_noalloc, x, w, got, rl) == tks.TKS_OK
        torch.cuda.synchronize()
        # index sets: the tolerance is exact equality
        _check_sets(got.cpu().numpy(), want, w.row_len, w.k, f"{name} call {call}")
    # the allocating entry point on the same input gives the same sets
    ref = torch.full((w.batch, w.k), -7, dtype=torch.int32, device="cuda")
    assert _call(lib.tks_topk_indices, x, w, ref, rl) == tks.TKS_OK
    assert tks.device_status() == tks.TKS_OK
    _check_sets(ref.cpu().numpy(), want, w.row_len, w.k, f"{name} allocating")


def test_noalloc_clamps_out_of_range_row_lengths_like_the_allocating_entry():
    """Row lengths below 0 and above row_stride are clamped to [0, row_stride];
    the allocating entry point reports TKS_E_ROW_LEN for them, this one does not
    report, and both give the oracle's sets for the clamped lengths."""
    lib = tks.load()
    rng = np.random.Generator(np.random.PCG64(73))
    stride = 150000
    base = W.from_rows("clamp", [rng.standard_normal(stride).astype(np.float32) for _ in range(3)],
                       512, W.F32, row_stride=stride)
    bad_len = np.array([-5, stride + 7, 70001], np.int32)
    clamped = np.clip(bad_len, 0, stride).astype(np.int32)
    want = oracle.topk_indices(base.values, base.k, clamped, W.F32)
    x = torch.from_numpy(base.values.copy()).cuda()
    rl = torch.from_numpy(bad_len).cuda()
    for call in range(2):
        got = torch.full((base.batch, base.k), -7, dtype=torch.int32, device="cuda")
        assert _call(lib.tks_topk_indices_noalloc, x, base, got, rl) == tks.TKS_OK
        torch.cuda.synchronize()
        _check_sets(got.cpu().numpy(), want, clamped, base.k, f"noalloc call {call}")
    ref = torch.full((base.batch, base.k), -7, dtype=torch.int32, device="cuda")
    assert _call(lib.tks_topk_indices, x, base, ref, rl) == tks.TKS_OK
    assert tks.device_status() == tks.TKS_E_ROW_LEN
    _check_sets(ref.cpu().numpy(), want, clamped, base.k, "allocating")


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    lib = tks.load()
    n = tks.TKS_NOALLOC_MAX_ROWS + 1
    x = torch.zeros((n, 64), dtype=torch.float32, device="cuda")
    out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    rc = lib.tks_topk_indices_noalloc(ctypes.c_void_p(x.data_ptr()), None, n, 64, 4, 0,
                                      ctypes.c_void_p(out.data_ptr()), None)
    assert rc == tks.TKS_E_TOO_LARGE
    assert "fixed scratch" in tks.status_string(rc)
    # argument errors come first, as for tks_topk_indices
    rc = lib.tks_topk_indices_noalloc(ctypes.c_void_p(x.data_ptr()), None, n, 64, 4, 0, None, None)
    assert rc == tks.TKS_E_INVAL
