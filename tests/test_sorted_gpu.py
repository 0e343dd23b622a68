"""Rank-ordered output (tks_topk_indices_sorted) against the oracle's rank order.

The comparison is exact, slot by slot: each row holds the selected positions
largest value first (+0.0 before -0.0, equal values by lower position), then -1.
"""

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_parity_gpu import _defaults, _device_values  # noqa: F401

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


def run_sorted(w, stream=None, offset_elems=0):
    x = _device_values(w, offset_elems)
    rl = torch.from_numpy(w.row_len.copy()).cuda()
    out = tks.topk_indices(x, w.k, row_len=rl, stream=stream, sorted=True)
    st = tks.device_status(stream)
    assert st == tks.TKS_OK, tks.status_string(st)
    return out.cpu().numpy()


def assert_same_order(w, got):
    want = oracle.topk_workload(w, ordered=True)
    for r in range(w.batch):
        if not np.array_equal(got[r], want[r]):
            bad = np.nonzero(got[r] != want[r])[0]
            raise AssertionError(f"{w.name}[{r}]: {bad.size} slots differ, first at {bad[0]}: "
                                 f"got {got[r][bad[0]]}, want {want[r][bad[0]]}")


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_named_workloads_sorted(name):
    w = W.named(name)
    assert_same_order(w, run_sorted(w))


def test_fuzz_sorted():
    for w in W.fuzz_cases():
        if w.k > tks.TKS_SORTED_K_MAX:
            continue
        assert_same_order(w, run_sorted(w))


@pytest.mark.parametrize("k", [1, 3, 255, 1000, 4096, 16384])
def test_sizes_of_k(k):
    rng = np.random.Generator(np.random.PCG64(100 + k))
    n = 1 << 17
    v = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32)))  # many ties
    w = W.from_rows(f"k{k}", [v, v[: n // 3]], k)
    assert_same_order(w, run_sorted(w))


def test_bf16_and_short_rows():
    rng = np.random.Generator(np.random.PCG64(77))
    rows = [W.bf16_mixed_zeros_subnormals(rng, 5000, 0.3, 0.3, 0.2), np.zeros(0, np.uint16),
            W.f32_to_bf16_bits(rng.standard_normal(100).astype(np.float32))]
    w = W.from_rows("bf16_short", rows, 512, W.BF16)
    assert_same_order(w, run_sorted(w))


def test_unaligned_rows_sorted():
    w = W.named("batch64_ragged")
    assert_same_order(w, run_sorted(w, offset_elems=3))


def test_back_to_back_calls_on_one_stream():
    """Selections and orderings chained on one stream (each kernel waits for the
    one ahead of it) give each call its own answer."""
    s = torch.cuda.Stream()
    ws = [W.named("decode_128k"), W.named("decode_1m_masked"), W.named("decode_4k")]
    xs = [_device_values(w) for w in ws]
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            for w, x in zip(ws, xs):
                outs.append((w, tks.topk_indices(x, w.k, stream=s, sorted=True)))
                outs.append((w, tks.topk_indices(x, w.k, stream=s)))
    assert tks.device_status(s) == tks.TKS_OK
    for i, (w, o) in enumerate(outs):
        got = o.cpu().numpy()
        if i % 2 == 0:
            assert_same_order(w, got)
        else:
            want = oracle.topk_workload(w)
            assert np.array_equal(np.sort(got, axis=1), want)


def test_k_above_the_sorted_limit_is_rejected():
    x = torch.zeros(1 << 16, device="cuda")
    out = torch.empty((1, tks.TKS_SORTED_K_MAX + 1), dtype=torch.int32, device="cuda")
    rc = tks.topk_indices_sorted_raw(x.data_ptr(), None, 1, 1 << 16, tks.TKS_SORTED_K_MAX + 1,
                                     tks.TKS_F32, out.data_ptr(), 0)
    assert rc == tks.TKS_E_INVAL


@pytest.mark.parametrize("batch,k", [(1, 2048), (8, 4096), (9, 4096), (3, 4097), (5, 33)])
def test_few_rows_over_many_blocks_and_many_rows(batch, k):
    """Up to 8 rows with k <= 4096 are ordered over many blocks from a scratch
    copy of the selection; more rows, or a larger k, by one block per row in
    place.  Both sides of each limit, with ties, short rows and -inf."""
    rng = np.random.Generator(np.random.PCG64(500 + batch * 7 + k))
    rows = []
    for r in range(batch):
        n = [k // 2, k, 3 * k + 17, 20000][r % 4]
        v = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32)))
        if r % 3 == 2:
            v[rng.integers(0, n, size=n // 5)] = -np.inf
        rows.append(v)
    w = W.from_rows(f"rank_{batch}_{k}", rows, k, row_stride=20011)
    assert_same_order(w, run_sorted(w))
    assert_same_order(w, run_sorted(w, offset_elems=1))
