"""The large-batch (prefill-like) path against the oracle: 512 causal rows.

Rows of at most k positions take the short path (every position, then -1);
longer ones are spread over the persistent grid, one block per row.
"""

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_parity_gpu import _defaults, assert_matches_oracle, run_gpu  # noqa: F401
from tests.test_sorted_gpu import assert_same_order, run_sorted

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


@pytest.fixture(scope="module")
def prefill():
    return W.named("prefill_causal")


def test_prefill_plan_is_one_block_per_row(prefill):
    group, grid = tks.plan(prefill.batch, prefill.row_stride, prefill.k, tks.TKS_F32)
    assert group == 1 and grid >= 1


def test_prefill_causal_sets(prefill):
    assert_matches_oracle(prefill, run_gpu(prefill), check_invariants=False)


def test_prefill_causal_rank_order(prefill):
    assert_same_order(prefill, run_sorted(prefill))


def test_prefill_bf16_subset():
    w = W.named("prefill_causal")
    rows = [W.f32_to_bf16_bits(w.values[r, : w.row_len[r]]) for r in range(0, w.batch, 3)]
    wb = W.from_rows("prefill_bf16", rows, w.k, W.BF16, row_stride=w.row_stride)
    assert_matches_oracle(wb, run_gpu(wb), check_invariants=False)
