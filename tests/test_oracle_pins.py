"""The CPU oracle against its pins (no GPU)."""

import os

import numpy as np
import pytest

import oracle
import workloads as W
from tests import pins


def _topk_with(lib):
    def topk(values, k, row_len, dtype):
        return oracle.topk_indices(np.atleast_2d(values), k, row_len, dtype, lib=lib)
    return topk


def _topk_ordered_with(lib):
    def topk(values, k, row_len, dtype):
        return oracle.topk_indices(np.atleast_2d(values), k, row_len, dtype, lib=lib, ordered=True)
    return topk


@pytest.fixture(scope="module")
def topk(oracle_lib):
    return _topk_with(oracle_lib)


@pytest.fixture(scope="module")
def topk_ordered(oracle_lib):
    return _topk_ordered_with(oracle_lib)


def test_rank_order_closed_form_and_brute_force(topk_ordered):
    pins.pin_rank_order(topk_ordered)


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_rank_order_is_the_set_in_order(topk, topk_ordered, name):
    """Rank-ordered output: the same set as the plain output, each entry ranked
    before the next, -1 padding last."""
    w = W.named(name)
    plain = topk(w.values, w.k, w.row_len, w.dtype)
    ordered = topk_ordered(w.values, w.k, w.row_len, w.dtype)
    vals = w.values if w.dtype == W.F32 else W.bf16_bits_to_f32(w.values)
    for r in range(w.batch):
        assert np.array_equal(np.sort(ordered[r]), np.sort(plain[r]))
        sel = ordered[r][ordered[r] >= 0]
        v = vals[r]
        for a, b in zip(sel[:-1], sel[1:]):
            assert pins._ranks_before(float(v[a]), int(a), float(v[b]), int(b))


def test_build_keeps_subnormals_and_signed_zero(oracle_lib):
    assert oracle_lib.tks_oracle_selftest() == 0
    assert oracle_lib.tks_oracle_mutant() == 0


def test_golden_base10_worked_examples(topk):
    pins.pin_golden_base10(topk)


def test_base10_procedure_on_random_integer_rows(topk):
    pins.pin_base10_random(topk)


def test_brute_force_tiny_rows(topk):
    pins.pin_brute_force(topk)


def test_rank_count_closed_form(topk):
    pins.pin_rank_count(topk)


def test_closed_forms(topk):
    pins.pin_closed_forms(topk)


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_bitkey_radix_full_size(topk, name):
    pins.pin_bitkey_radix(topk, W.named(name))


def test_bitkey_radix_fuzz(topk):
    for w in W.fuzz_cases():
        pins.pin_bitkey_radix(topk, w)


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_invariants_named(topk, name):
    w = W.named(name)
    got = topk(w.values, w.k, w.row_len, w.dtype)
    vals = W.as_float32(w)
    for r in range(w.batch):
        pins.check_invariants(vals[r], int(w.row_len[r]), w.k, got[r], f"{name}[{r}]")


def test_named_closed_forms(topk):
    """Rows whose answer is known without any selection."""
    w = W.batch4_1m_bf16()
    got = topk(w.values, w.k, w.row_len, w.dtype)
    assert np.array_equal(got[0], np.arange(2048))  # constant row
    first, size = W.expected_top_plateau(1 << 20)
    assert size == 2048
    assert np.array_equal(got[1], np.arange(first, 1 << 20))  # ramp: its top plateau
    w3 = W.decode_1m_masked()
    g3 = topk(w3.values, w3.k, w3.row_len, w3.dtype)[0]
    assert g3.max() < (1 << 20) - (1 << 20) // 10  # no masked (-inf) position selected


def test_values_match_library_topk(topk):
    """Values only (a library's tie choice is unspecified): the multiset of selected
    values equals torch.topk's on the CPU."""
    torch = pytest.importorskip("torch")
    for name in ("decode_128k", "decode_1m_masked", "batch64_ragged"):
        w = W.named(name)
        got = topk(w.values, w.k, w.row_len, w.dtype)
        vals = W.as_float32(w)
        for r in range(min(w.batch, 8)):
            L = int(w.row_len[r])
            ref = torch.topk(torch.from_numpy(vals[r, :L].copy()), min(w.k, L)).values.numpy()
            mine = vals[r, got[r][got[r] >= 0]]
            assert np.array_equal(np.sort(mine), np.sort(ref)), (name, r)


def test_nan_rejected(topk):
    with pytest.raises(oracle.OracleError):
        topk(np.array([1.0, np.nan, 2.0], np.float32), 1, None, W.F32)
    # NaN beyond the valid length is never looked at
    got = topk(np.array([[1.0, 3.0, np.nan]], np.float32), 1, [2], W.F32)
    assert list(got[0]) == [1]


MUTANTS = {1: "ascending order", 2: "-0.0 above +0.0", 3: "sign rule dropped",
           4: "ties to the highest position", 5: "one element short", 6: "bf16 widened from the wrong half",
           7: "rank order with ties reversed"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(tmp_path, mutant):
    """Each plausible mistake planted in the oracle fails at least one pin."""
    lib = oracle.load(oracle.build(out_dir=str(tmp_path), mutant=mutant))
    assert lib.tks_oracle_mutant() == mutant
    t = _topk_with(lib)
    checks = [
        lambda: pins.pin_golden_base10(t),
        lambda: pins.pin_brute_force(t, n_rows=150),
        lambda: pins.pin_closed_forms(t),
        lambda: pins.pin_bitkey_radix(t, W.fuzz_cases()[-4]),  # bf16 odd-stride rows
        lambda: pins.pin_rank_count(t),
        lambda: pins.pin_rank_order(_topk_ordered_with(lib)),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, oracle.OracleError):
            failed += 1
    assert failed >= 1, f"no pin caught mutant {mutant}: {MUTANTS[mutant]}"
