"""The largest shapes, against the CPU oracle: rows far longer than all SMs'
shared memory holds (each block's slice is streamed from HBM in every round),
positions that need 24-25 bits, k up to the row length.  Index sets must
match exactly."""

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_parity_gpu import _defaults, assert_matches_oracle, run_gpu  # noqa: F401

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


def test_16m_fp32_row_default_plan():
    """One 64 MB fp32 row: 151 blocks whose 444 KB slices do not fit on chip."""
    n = 1 << 24
    rng = np.random.Generator(np.random.PCG64(91))
    row = rng.standard_normal(n).astype(np.float32)
    row[rng.integers(0, n, size=5000)] = np.float32(2.5)  # a tie straddling the threshold region
    w = W.from_rows("row_16m", [row], 2048)
    group, _ = tks.plan(1, n, 2048, tks.TKS_F32)
    assert group > 1
    assert_matches_oracle(w, run_gpu(w), oracle.topk_workload(w))


def test_32m_bf16_row_large_k():
    """One 64 MB bf16 row (heavy duplicates: 16-bit values), k = 65536."""
    n = 1 << 25
    rng = np.random.Generator(np.random.PCG64(92))
    w = W.from_rows("row_32m_bf16", [W.f32_to_bf16_bits(rng.standard_normal(n))], 65536, W.BF16)
    assert_matches_oracle(w, run_gpu(w), oracle.topk_workload(w))


def test_ragged_8m_rows_512_threads():
    """Two ragged rows on a 8M stride with 512-thread blocks, k = 16384."""
    n = 1 << 23
    rng = np.random.Generator(np.random.PCG64(93))
    rows = [rng.standard_normal(n - 1).astype(np.float32),
            (rng.integers(-3, 4, size=n // 3) * 0.5).astype(np.float32)]
    w = W.from_rows("ragged_8m", rows, 16384, row_stride=n)
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, 512)
    assert_matches_oracle(w, run_gpu(w), oracle.topk_workload(w))


@pytest.mark.parametrize("k_from_end", [1, 0])
def test_k_up_to_the_row_length(k_from_end):
    """k = N - 1 (the threshold is the row's minimum: almost every element is
    selected) and k = N (every position), on a 1M row with a masked tail."""
    n = 1 << 20
    rng = np.random.Generator(np.random.PCG64(94))
    row = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal(n))).copy()
    row[n - n // 10:] = -np.inf
    w = W.from_rows(f"k_near_n_{k_from_end}", [row], n - k_from_end)
    assert_matches_oracle(w, run_gpu(w), oracle.topk_workload(w))
