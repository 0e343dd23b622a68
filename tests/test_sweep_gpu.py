"""A seeded random sweep against the oracle: shapes, row lengths, k, dtypes and
value kinds drawn at random (workloads.sweep_cases), each run through one
entry point (device buffers, rank order, or page-locked host buffers) with a
drawn alignment offset, block size, cluster setting and forced split.  Index
sets must match the oracle exactly; rank order slot by slot."""

import numpy as np
import pytest

import oracle
import workloads as W
from tests.test_parity_gpu import _defaults, _device_values, assert_matches_oracle  # noqa: F401
from tests.test_sorted_gpu import assert_same_order

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


def _host_values(w, offset):
    v = w.values
    pad = np.zeros((v.shape[0], v.shape[1] + offset), v.dtype)
    pad[:, offset:] = v
    flat = torch.from_numpy(pad.reshape(-1).copy()).pin_memory()
    t = flat[offset:].as_strided((v.shape[0], v.shape[1]), (v.shape[1] + offset, 1)) if offset \
        else flat.view(v.shape[0], v.shape[1])
    return t.view(torch.bfloat16) if w.dtype == W.BF16 else t


def _run(w, draw):
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, draw["threads"])
    tks.set_option(tks.TKS_OPT_CLUSTER, draw["cluster"])
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, draw["group"])
    s = torch.cuda.Stream()
    if draw["host"]:
        x = _host_values(w, draw["offset"])
        rl = torch.from_numpy(w.row_len.copy()).pin_memory()
        out = tks.topk_indices(x, w.k, row_len=rl, stream=s)
    else:
        x = _device_values(w, draw["offset"])
        rl = torch.from_numpy(w.row_len.copy()).cuda()
        out = tks.topk_indices(x, w.k, row_len=rl, stream=s, sorted=draw["sorted"])
    st = tks.device_status(s)
    assert st == tks.TKS_OK, f"{w.name} {draw}: {tks.status_string(st)}"
    return out.cpu().numpy()


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5, 6])
def test_random_sweep(seed):
    for w, draw in W.sweep_cases(seed, 40):
        got = _run(w, draw)
        try:
            if draw["sorted"] and not draw["host"]:
                assert_same_order(w, got)
            else:
                assert_matches_oracle(w, got, oracle.topk_workload(w), check_invariants=False)
        except AssertionError as e:
            raise AssertionError(f"{w.name} ({w.note}, k={w.k}, {w.dtype}) {draw}: {e}") from None
