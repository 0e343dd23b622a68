"""The launch plan the library chooses, and both ways the first round finds its
threshold bin (every warp on a window of at most 32 bins; a block-wide scan on
wider windows), against the CPU oracle."""

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_parity_gpu import assert_matches_oracle, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


@pytest.fixture(autouse=True)
def _defaults():
    for opt in (tks.TKS_OPT_FORCE_GROUP, tks.TKS_OPT_FORCE_THREADS, tks.TKS_OPT_CLUSTER):
        tks.set_option(opt, 0)
    yield
    for opt in (tks.TKS_OPT_FORCE_GROUP, tks.TKS_OPT_FORCE_THREADS, tks.TKS_OPT_CLUSTER):
        tks.set_option(opt, 0)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("batch, stride, dtype, want", [
    (1, 4096, tks.TKS_F32, lambda sms: (1, 1)),             # short rows stay on one block
    (1, 131072, tks.TKS_F32, lambda sms: (32, 32)),         # one block per 4096 elements
    (1, 262144, tks.TKS_F32, lambda sms: (64, 64)),
    (1, 1 << 20, tks.TKS_F32, lambda sms: (sms - 1, sms - 1)),  # capped, one SM left free
    (4, 1 << 20, tks.TKS_BF16, lambda sms: ((sms - 1) // 4, 4 * ((sms - 1) // 4))),
    (64, 65536, tks.TKS_F32, lambda sms: ((sms - 1) // 64, 64 * ((sms - 1) // 64))),
    (512, 32768, tks.TKS_F32, lambda sms: (1, sms)),        # many rows: one block per row
])
def test_default_plan(batch, stride, dtype, want):
    assert tks.plan(batch, stride, 2048, dtype) == want(_sms())


def test_clusters_only_on_request():
    assert tks.plan(1, 131072, 2048, tks.TKS_F32) == (32, 32)
    tks.set_option(tks.TKS_OPT_CLUSTER, 1)
    assert tks.plan(1, 131072, 2048, tks.TKS_F32) == (32, 32)
    tks.set_option(tks.TKS_OPT_CLUSTER, 8)
    assert tks.plan(1, 131072, 2048, tks.TKS_F32) == (8, 8)


def _wide(rng, n):
    """Values over many binades and both signs: a block's first-round window
    (its floor to the row's top) spans far more than 32 bins."""
    return (rng.choice([-1.0, 1.0], size=n) * np.exp(rng.uniform(-80.0, 80.0, size=n))).astype(np.float32)


@pytest.mark.parametrize("threads", [256, 512])
@pytest.mark.parametrize("kind", ["narrow", "wide"])
def test_split_row_first_round_pick(kind, threads):
    rng = np.random.Generator(np.random.PCG64(81))
    n = 1 << 20
    row = rng.standard_normal(n).astype(np.float32) if kind == "narrow" else _wide(rng, n)
    w = W.from_rows(f"split_{kind}", [row], 2048)
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, threads)
    assert tks.plan(1, n, 2048, tks.TKS_F32)[0] > 1
    assert_matches_oracle(w, run_gpu(w), oracle.topk_workload(w))


@pytest.mark.parametrize("n, kind", [(4096, "narrow"), (4096, "wide"), (40900, "narrow")])
def test_whole_row_first_round_pick(n, kind):
    """A row on one block: the warps' suffix sums go to the slice buffer's
    tail when the slice leaves it free (4096 elements), else (a 40,900-element
    row fills the buffer) the block-wide scan runs."""
    rng = np.random.Generator(np.random.PCG64(82))
    row = rng.standard_normal(n).astype(np.float32) if kind == "narrow" else _wide(rng, n)
    w = W.from_rows(f"whole_{kind}_{n}", [row], 256)
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 1)
    assert_matches_oracle(w, run_gpu(w), oracle.topk_workload(w))
