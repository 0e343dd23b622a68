"""CUDA path against the CPU oracle: bit-exact index sets.

Every case goes through the C ABI (``tks_topk_indices`` via the ctypes binding)
and is compared, row by row, with the oracle on the same seeded inputs:
the first min(k, len) output slots must hold exactly the oracle's set, the
rest -1.
"""

import numpy as np
import pytest

import oracle
import workloads as W
from tests import pins

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_topk_gb300 as tks  # noqa: E402


def _device_values(w, offset_elems=0):
    """Upload a workload; with offset_elems > 0 the rows start that many elements
    into a larger buffer (unaligned base pointer)."""
    v = w.values
    if offset_elems:
        pad = np.zeros((v.shape[0], v.shape[1] + offset_elems), v.dtype)
        pad[:, offset_elems:] = v
        flat = torch.from_numpy(pad.reshape(-1).copy()).cuda()
        base = flat[offset_elems:]
        t = base.as_strided((v.shape[0], v.shape[1]), (v.shape[1] + offset_elems, 1))
    else:
        t = torch.from_numpy(v.copy()).cuda()
    if w.dtype == W.BF16:
        t = t.view(torch.bfloat16)
    return t


def run_gpu(w, offset_elems=0, stream=None):
    x = _device_values(w, offset_elems)
    rl = torch.from_numpy(w.row_len.copy()).cuda()
    out = tks.topk_indices(x, w.k, row_len=rl, stream=stream)
    st = tks.device_status(stream)
    assert st == tks.TKS_OK, tks.status_string(st)
    return out.cpu().numpy()


def assert_matches_oracle(w, got, want=None, check_invariants=True):
    if want is None:
        want = oracle.topk_workload(w)
    vals = W.as_float32(w)
    for r in range(w.batch):
        L = int(w.row_len[r])
        take = min(w.k, L)
        g = got[r]
        assert np.all(g[take:] == -1), f"{w.name}[{r}]: padding"
        gs = np.sort(g[:take])
        assert np.array_equal(gs, want[r][:take]), \
            f"{w.name}[{r}]: {np.setdiff1d(gs, want[r][:take]).size} positions differ"
        if check_invariants and take < 20000:
            pins.check_invariants(vals[r], L, w.k, g, f"{w.name}[{r}]")


@pytest.fixture(autouse=True)
def _defaults():
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, 0)
    tks.set_option(tks.TKS_OPT_CLUSTER, 0)
    tks.set_option(tks.TKS_OPT_TEST_SKIP_ARRIVE, 0)
    tks.set_option(tks.TKS_OPT_SPIN_LIMIT_NS, 1_000_000_000)
    yield
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, 0)
    tks.set_option(tks.TKS_OPT_CLUSTER, 0)
    tks.set_option(tks.TKS_OPT_TEST_SKIP_ARRIVE, 0)
    tks.set_option(tks.TKS_OPT_SPIN_LIMIT_NS, 1_000_000_000)


_ORACLE_CACHE = {}


def oracle_of(w):
    key = w.name
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle.topk_workload(w)
    return _ORACLE_CACHE[key]


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_named_workloads_default_plan(name):
    """The five workloads, in the launch configuration the benchmark uses."""
    w = W.named(name)
    assert_matches_oracle(w, run_gpu(w), oracle_of(w))


@pytest.mark.parametrize("name", ["decode_4k", "decode_128k", "decode_1m_masked", "batch4_1m_bf16"])
@pytest.mark.parametrize("group", [1, 2, 3, 16, 1000])
def test_named_workloads_forced_split(name, group):
    """Every split of a row over thread blocks gives the same set (1000 is
    clamped to what the GPU co-schedules)."""
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
    w = W.named(name)
    assert_matches_oracle(w, run_gpu(w), oracle_of(w))


@pytest.mark.parametrize("group", [0, 1, 2, 5, 64])
def test_fuzz_cases(group):
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
    for w in W.fuzz_cases():
        assert_matches_oracle(w, run_gpu(w))


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_random_ragged_batches(seed, dtype):
    levels = [None, 3, 50][seed % 3]
    for batch, max_len, k in [(5, 20000, 777), (40, 3000, 64), (300, 2500, 100)]:
        w = W.random_rows(100 * seed + batch, batch, max_len, k, dtype, levels)
        assert_matches_oracle(w, run_gpu(w))


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("group", [0, 1, 7])
def test_unaligned_base_pointer(offset, group):
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
    rng = np.random.Generator(np.random.PCG64(offset))
    rows = [rng.standard_normal(n).astype(np.float32) for n in (50001, 4099, 77)]
    w = W.from_rows(f"unaligned{offset}", rows, 300, row_stride=50003)
    assert_matches_oracle(w, run_gpu(w, offset_elems=offset))
    wb = W.from_rows(f"unaligned_bf16_{offset}", [W.f32_to_bf16_bits(r) for r in rows], 300,
                     W.BF16, row_stride=50003)
    assert_matches_oracle(wb, run_gpu(wb, offset_elems=offset))


def test_long_row_streamed_past_on_chip_capacity():
    """A lone block whose slice does not fit in shared memory re-reads it."""
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 1)
    rng = np.random.Generator(np.random.PCG64(21))
    w = W.from_rows("long_row", [rng.standard_normal(300001).astype(np.float32),
                                 np.full(200000, 1.5, np.float32)], 2048)
    assert_matches_oracle(w, run_gpu(w))


def test_candidate_overflow_rows():
    """The threshold bin holds far more than fits on chip (the failure mode the
    page reports for an 8-bit first screen at long rows): still exact."""
    rng = np.random.Generator(np.random.PCG64(22))
    rows = [np.full(600000, 0.25, np.float32),
            rng.integers(0, 2, size=600000).astype(np.float32),
            W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal(600000) * 1e-3))]
    w = W.from_rows("overflow", rows, 4096)
    for group in (0, 1, 3, 40):
        tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
        assert_matches_oracle(w, run_gpu(w))


def test_row_len_out_of_range_is_clamped_and_reported():
    x = torch.randn(2, 1000, device="cuda")
    rl = torch.tensor([1200, -5], dtype=torch.int32, device="cuda")
    out = tks.topk_indices(x, 10, row_len=rl)
    assert tks.device_status() == tks.TKS_E_ROW_LEN
    want = oracle.topk_indices(x.cpu().numpy(), 10, [1000, 0])
    got = out.cpu().numpy()
    assert np.array_equal(np.sort(got[0]), want[0])
    assert np.all(got[1] == -1)
    # the status was cleared
    tks.topk_indices(x, 10)
    assert tks.device_status() == tks.TKS_OK


def test_barrier_timeout_reports_and_recovers():
    """One block never arrives: the others give up after the spin limit, the
    status says so, and the next call is correct again."""
    w = W.decode_128k()
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 8)
    tks.set_option(tks.TKS_OPT_SPIN_LIMIT_NS, 20_000_000)
    tks.set_option(tks.TKS_OPT_TEST_SKIP_ARRIVE, 1)
    x = _device_values(w)
    tks.topk_indices(x, w.k)
    assert tks.device_status() == tks.TKS_E_TIMEOUT
    tks.set_option(tks.TKS_OPT_TEST_SKIP_ARRIVE, 0)
    assert_matches_oracle(w, run_gpu(w), oracle_of(w))


def test_cuda_graph_capture_and_replay():
    w = W.decode_1m_masked()
    x = _device_values(w)
    s = torch.cuda.Stream()
    out = torch.empty((1, w.k), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        tks.topk_indices(x, w.k, out=out, stream=s)  # first call on s: workspace set-up
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            tks.topk_indices(x, w.k, out=out, stream=s)
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert tks.device_status(s) == tks.TKS_OK
    assert_matches_oracle(w, out.cpu().numpy(), oracle_of(w))


def test_two_streams_concurrently():
    w1, w2 = W.decode_128k(), W.decode_1m_masked()
    x1, x2 = _device_values(w1), _device_values(w2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 8)  # leave room for both grids
    outs = []
    for _ in range(4):
        with torch.cuda.stream(s1):
            o1 = tks.topk_indices(x1, w1.k, stream=s1)
        with torch.cuda.stream(s2):
            o2 = tks.topk_indices(x2, w2.k, stream=s2)
        outs.append((o1, o2))
    torch.cuda.synchronize()
    assert tks.device_status(s1) == tks.TKS_OK and tks.device_status(s2) == tks.TKS_OK
    for o1, o2 in outs:
        assert_matches_oracle(w1, o1.cpu().numpy(), oracle_of(w1))
        assert_matches_oracle(w2, o2.cpu().numpy(), oracle_of(w2))


def test_repeated_calls_reuse_workspace_cleanly():
    w = W.batch64_ragged()
    want = oracle_of(w)
    x = _device_values(w)
    rl = torch.from_numpy(w.row_len.copy()).cuda()
    outs = [tks.topk_indices(x, w.k, row_len=rl) for _ in range(20)]
    assert tks.device_status() == tks.TKS_OK
    for o in outs:
        assert_matches_oracle(w, o.cpu().numpy(), want, check_invariants=False)


def test_k_larger_than_every_row_and_one_element_rows():
    w = W.from_rows("tiny", [np.array([1.0], np.float32), np.array([], np.float32),
                             np.array([2.0, -1.0], np.float32)], 5, row_stride=3)
    assert_matches_oracle(w, run_gpu(w))
    w1 = W.from_rows("k1", [np.array([1.0, 3.0, 3.0, -0.0], np.float32)], 1)
    assert_matches_oracle(w1, run_gpu(w1))


@pytest.mark.parametrize("threads", [256, 512])
@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_both_block_sizes_named(threads, name):
    """Each block size on every named workload (the automatic choice uses 512
    only for large slices)."""
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, threads)
    w = W.named(name)
    assert_matches_oracle(w, run_gpu(w), oracle_of(w))


@pytest.mark.parametrize("threads", [256, 512])
def test_both_block_sizes_fuzz_and_splits(threads):
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, threads)
    for w in W.fuzz_cases():
        assert_matches_oracle(w, run_gpu(w), check_invariants=False)
    w = W.named("decode_128k")
    for g in (2, 3, 16, 100):
        tks.set_option(tks.TKS_OPT_FORCE_GROUP, g)
        assert_matches_oracle(w, run_gpu(w), oracle_of(w))
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)
    for seed in (31, 32):
        w = W.random_rows(seed, 40, 30000, 700, levels=5)
        assert_matches_oracle(w, run_gpu(w), check_invariants=False)


@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
def test_cluster_rows(cluster):
    """Rows split over one thread-block cluster (merge through distributed
    shared memory) for every cluster size, and with clusters switched off."""
    tks.set_option(tks.TKS_OPT_CLUSTER, cluster)
    for name in ("decode_128k", "decode_4k"):
        w = W.named(name)
        assert_matches_oracle(w, run_gpu(w), oracle_of(w))
    for w in W.fuzz_cases():
        assert_matches_oracle(w, run_gpu(w), check_invariants=False)
    for seed in (41, 42):
        w = W.random_rows(seed, 6, 60000, 900, levels=4)
        assert_matches_oracle(w, run_gpu(w), check_invariants=False)


@pytest.mark.parametrize("threads", [256, 512])
def test_cluster_rows_both_block_sizes_bf16(threads):
    tks.set_option(tks.TKS_OPT_FORCE_THREADS, threads)
    tks.set_option(tks.TKS_OPT_CLUSTER, 8)
    rng = np.random.Generator(np.random.PCG64(43))
    rows = [W.bf16_mixed_zeros_subnormals(rng, 150000, 0.2, 0.2, 0.2),
            W.f32_to_bf16_bits(rng.standard_normal(70001).astype(np.float32)), W.bf16_ramp(131072)]
    w = W.from_rows("cluster_bf16", rows, 3000, W.BF16)
    assert_matches_oracle(w, run_gpu(w), check_invariants=False)


@pytest.mark.parametrize("group", [2, 3, 4])
def test_large_slices_on_chip_finish(group):
    """Few blocks per row, many candidates (k = 15000 among heavy ties at zero):
    the finishing block reuses its slice buffer for the candidates, which must
    wait until every thread has finished its emission pass over that slice."""
    w = [x for x in W.fuzz_cases() if x.name == "bf16_zeros_subnormals"][0]
    for threads in (256, 512):
        tks.set_option(tks.TKS_OPT_FORCE_THREADS, threads)
        tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
        for _ in range(3):
            assert_matches_oracle(w, run_gpu(w), check_invariants=False)


@pytest.mark.parametrize("group", [0, 1, 9])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_all_equal_rows_and_near_misses(group, dtype):
    """A row whose keys are all equal is answered with its k lowest positions
    right after the first round; a single differing element anywhere (higher
    at the end, lower at the start, a -0.0 among +0.0, one ulp apart) must
    still be found."""
    n, k = 70001, 1500
    base = np.full(n, 1.0, np.float32)
    rows = [base.copy(), np.full(n, -np.inf, np.float32), np.zeros(n, np.float32)]
    hi_end = base.copy()
    hi_end[-1] = 2.0
    lo_start = base.copy()
    lo_start[0] = 0.5
    negz = np.zeros(n, np.float32)
    negz[123] = -0.0
    ulp = base.copy()
    ulp[n // 2] = np.nextafter(np.float32(1.0), np.float32(2.0)) if dtype == W.F32 else 1.0078125
    rows += [hi_end, lo_start, negz, ulp]
    rows = rows if dtype == W.F32 else [W.f32_to_bf16_bits(r) for r in rows]
    w = W.from_rows(f"all_equal_{dtype}", rows, k, dtype, row_stride=n + 3)
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
    assert_matches_oracle(w, run_gpu(w), check_invariants=False)
    assert_matches_oracle(w, run_gpu(w, offset_elems=1), check_invariants=False)
    tks.set_option(tks.TKS_OPT_CLUSTER, 1)
    assert_matches_oracle(w, run_gpu(w), check_invariants=False)


def test_mixed_shapes_back_to_back_on_one_stream():
    """One stream's workspace serves calls of different shapes and entry
    points queued back to back: row slots are reused with other block counts,
    other digit-round counts and other candidate counts, and each call cleans
    up only what the one before it on the slot left.  Every call must still
    give the oracle's sets (rank-ordered calls: the oracle's order)."""
    rng = np.random.Generator(np.random.PCG64(31))
    overflow = W.from_rows("mixed_overflow",
                           [np.full(300000, 0.25, np.float32),
                            rng.integers(0, 2, size=300000).astype(np.float32)], 4096)
    equal = W.from_rows("mixed_equal", [np.full(500000, -3.0, np.float32)], 2048)
    bf16 = W.from_rows("mixed_bf16", [W.f32_to_bf16_bits(rng.standard_normal(200000)) for _ in range(3)],
                       777, W.BF16)
    # (workload, forced blocks per row, entry point)
    cases = [(W.decode_1m_masked(), 0, "device"), (W.batch64_ragged(), 0, "device"),
             (overflow, 0, "device"), (W.decode_128k(), 0, "host"), (equal, 0, "device"),
             (W.batch4_1m_bf16(), 0, "device"), (bf16, 5, "sorted"), (W.decode_1m_masked(), 40, "device"),
             (W.decode_4k(), 0, "sorted"), (overflow, 17, "device"), (W.decode_1m_masked(), 0, "host"),
             (W.decode_1m_masked(), 0, "sorted")]
    inputs = {}
    for w, _, entry in cases:
        key = (w.name, entry == "host")
        if key not in inputs:
            if entry == "host":
                x = torch.from_numpy(w.values.copy()).pin_memory()
                x = x.view(torch.bfloat16) if w.dtype == W.BF16 else x
                rl = torch.from_numpy(w.row_len.copy()).pin_memory()
            else:
                x = _device_values(w)
                rl = torch.from_numpy(w.row_len.copy()).cuda()
            inputs[key] = (x, rl)
    s = torch.cuda.Stream()
    order = [i for _ in range(3) for i in rng.permutation(len(cases))]
    outs = []
    for i in order:
        w, group, entry = cases[i]
        tks.set_option(tks.TKS_OPT_FORCE_GROUP, group)
        x, rl = inputs[(w.name, entry == "host")]
        outs.append((w, entry, tks.topk_indices(x, w.k, row_len=rl, stream=s, sorted=entry == "sorted")))
    tks.set_option(tks.TKS_OPT_FORCE_GROUP, 0)
    assert tks.device_status(s) == tks.TKS_OK
    for n, (w, entry, o) in enumerate(outs):
        try:
            if entry == "sorted":
                assert np.array_equal(o.cpu().numpy(), oracle.topk_workload(w, ordered=True))
            else:
                assert_matches_oracle(w, o.cpu().numpy(), oracle_of(w), check_invariants=False)
        except AssertionError as e:
            raise AssertionError(f"call {n} ({w.name}, {entry}): {e}") from None
