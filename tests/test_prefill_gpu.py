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


def _mixed_rows(dtype, stride, levels, seed):
    """Rows whose lengths cycle through: empty, at most k, just above k, short,
    resident on chip, and longer than a block's on-chip copy -- so that one
    block's consecutive rows take every path in turn; an odd row stride gives
    every row its own alignment."""
    rng = np.random.default_rng(seed)
    k = 2048
    lens = [0, k, k + 1, 5000, stride // 3, stride, 20001, stride - 3, 77, stride // 2 + 1]
    rows = []
    for r in range(3 * 152 + 7):
        n = lens[(r * 7 + r // 10) % len(lens)]
        x = (rng.integers(0, levels, size=n).astype(np.float32) - levels / 2 if levels
             else rng.standard_normal(n).astype(np.float32))
        rows.append(x if dtype == W.F32 else W.f32_to_bf16_bits(x))
    return W.from_rows(f"mixed_{dtype}_{levels}", rows, k, dtype, row_stride=stride)


@pytest.mark.parametrize("threads", [256, 512])
@pytest.mark.parametrize("dtype,stride", [(W.F32, 60001), (W.BF16, 100003)])
@pytest.mark.parametrize("levels", [0, 50])
def test_many_rows_per_block_mixed_lengths(dtype, stride, levels, threads):
    """Each block owns several rows and starts the next row's on-chip copy
    before finishing the current one: every combination of neighbouring row
    kinds must still give the oracle's sets."""
    w = _mixed_rows(dtype, stride, levels, seed=31 + levels)
    want = oracle.topk_workload(w)
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 1)
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, threads)
    try:
        assert_matches_oracle(w, run_gpu(w), want, check_invariants=False)
        assert_matches_oracle(w, run_gpu(w, offset_elems=1), want, check_invariants=False)
    finally:
        tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)
        tks.set_option(tks.TKS_OPT_FORCE_THREADS, 0)


def test_back_to_back_batches_and_graph_replays(prefill):
    """Blocks that own several rows each carry state from row to row (the next
    row's length and on-chip copy): back-to-back calls of different batch
    sizes on one stream, and replays of a captured graph, must all match."""
    want = oracle.topk_workload(prefill)
    s = torch.cuda.Stream()
    x = torch.from_numpy(prefill.values.copy()).cuda()
    rl = torch.from_numpy(prefill.row_len.copy()).cuda()
    for batch in (prefill.batch, 153, prefill.batch, 300):
        out = tks.topk_indices(x[:batch], prefill.k, row_len=rl[:batch], stream=s)
        assert tks.device_status(s) == tks.TKS_OK
        sub = W.Workload(prefill.name, prefill.values[:batch], prefill.row_len[:batch], prefill.k,
                         prefill.dtype, "")
        assert_matches_oracle(sub, out.cpu().numpy(), want[:batch], check_invariants=False)
    out = torch.empty((prefill.batch, prefill.k), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        tks.topk_indices(x, prefill.k, row_len=rl, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            tks.topk_indices(x, prefill.k, row_len=rl, out=out, stream=s)
    for _ in range(4):
        out.fill_(-7)
        with torch.cuda.stream(s):
            g.replay()
        assert tks.device_status(s) == tks.TKS_OK
        assert_matches_oracle(prefill, out.cpu().numpy(), want, check_invariants=False)
