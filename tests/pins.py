"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes ``topk(values, k, row_len, dtype) -> int32 [batch, k]``
(the oracle, or a deliberately broken build of it) and raises AssertionError on a
mismatch.  They are also reused, as invariants, on the CUDA path's output.

What pins what:
  * ``pin_golden_base10``   - hand traces of the page's base-10 digit selection and its
                              collection step ("Technical Deep Dive ... TopK Selector",
                              section "02. Traditional GPU Approach: Radix Selection");
  * ``pin_base10_random``   - that procedure, restated here, on random nonnegative
                              integer rows with many ties;
  * ``pin_brute_force``     - every subset of tiny rows: exactly one subset has each
                              member ranked before each non-member, and it is the output;
  * ``pin_rank_count``      - closed form: position i is selected iff fewer than k
                              positions rank before it (O(L^2), L <= 2048);
  * ``pin_bitkey_radix``    - an independent selection at full size: the page's
                              "Mapping" step (floats to order-preserving unsigned keys),
                              extended by the inverted position so keys are unique, then
                              byte-wise digit selection with numpy histograms;
  * ``pin_closed_forms``    - constant rows, ramps, k >= L, k = 1 (first argmax),
                              signed zeros, -inf;
  * ``check_invariants``    - count, range, value separation, lowest-index ties.
"""

from __future__ import annotations

import functools
import itertools
import math
import os

import numpy as np

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# golden fixtures
# ----------------------------------------------------------------------------

def load_golden(name: str):
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                if cur and not line:
                    cases.append(cur)
                    cur = {}
                continue
            key, val = line.split(":", 1)
            val = val.strip()
            if key in ("values", "expect"):
                cur[key] = [int(t) for t in val.split()]
            elif key in ("k", "kth"):
                cur[key] = int(val)
            else:
                cur[key] = val
    if cur:
        cases.append(cur)
    return cases


# ----------------------------------------------------------------------------
# the page's base-10 digit selection, restated for nonnegative integers
# ----------------------------------------------------------------------------

def base10_kth_largest(a, k):
    """k-th largest (1-based) by selecting one decimal digit at a time, most
    significant first, keeping only the survivors whose digit holds the rank."""
    survivors = list(a)
    rank = k - 1
    top = max(a)
    exp = 1
    while exp * 10 <= top:
        exp *= 10
    while exp > 0:
        digit_of = [(x // exp) % 10 for x in survivors]
        hist = [digit_of.count(d) for d in range(10)]
        seen = 0
        for d in range(9, -1, -1):
            if rank < seen + hist[d]:
                chosen, rank = d, rank - seen
                break
            seen += hist[d]
        survivors = [x for x, dg in zip(survivors, digit_of) if dg == chosen]
        exp //= 10
    return survivors[0]


def base10_collect(a, k):
    """Positions: everything above the k-th value, then equal ones in scan order."""
    t = base10_kth_largest(a, k)
    picked = [i for i, x in enumerate(a) if x > t]
    for i, x in enumerate(a):
        if x == t and len(picked) < k:
            picked.append(i)
    return t, sorted(picked)


def pin_golden_base10(topk):
    for case in load_golden("base10_radix_select.txt"):
        a, k = case["values"], case["k"]
        t, picked = base10_collect(a, k)
        assert t == case["kth"], (case["name"], t)
        assert picked == case["expect"], (case["name"], picked)
        got = topk(np.array(a, np.float32), k, None, W.F32)[0]
        assert list(got) == case["expect"], (case["name"], list(got))


def pin_base10_random(topk, n_rows=60, seed=7):
    rng = np.random.Generator(np.random.PCG64(seed))
    for _ in range(n_rows):
        n = int(rng.integers(1, 300))
        hi = int(rng.choice([5, 50, 1000, 100000]))
        a = rng.integers(0, hi, size=n)
        k = int(rng.integers(1, n + 1))
        _, picked = base10_collect([int(x) for x in a], k)
        got = topk(a.astype(np.float32), k, None, W.F32)[0]
        assert list(got) == picked, (n, hi, k)


# ----------------------------------------------------------------------------
# brute force and rank counting
# ----------------------------------------------------------------------------

def _ranks_before(x, i, y, j):
    """Does position i (value x) rank before position j (value y)?  The order the
    selector defines: larger value first; +0.0 before -0.0; lower position first."""
    if x != y:
        return x > y
    sx, sy = math.copysign(1.0, x) < 0, math.copysign(1.0, y) < 0
    if sx != sy:
        return not sx
    return i < j


def brute_force_topk(v, k):
    L = len(v)
    take = min(k, L)
    found = []
    for subset in itertools.combinations(range(L), take):
        inside = set(subset)
        if all(_ranks_before(float(v[i]), i, float(v[j]), j)
               for i in inside for j in range(L) if j not in inside):
            found.append(list(subset))
    assert len(found) == 1, f"{len(found)} subsets satisfy the definition"
    return found[0] + [-1] * (k - take)


def pin_brute_force(topk, n_rows=400, seed=3):
    rng = np.random.Generator(np.random.PCG64(seed))
    pool = W.tiny_special_values()
    for _ in range(n_rows):
        L = int(rng.integers(0, 8))
        v = pool[rng.integers(0, pool.size, size=L)]
        k = int(rng.integers(1, L + 2))
        want = brute_force_topk(v, k)
        got = topk(v, k, None, W.F32)[0] if L > 0 else topk(np.zeros(1, np.float32), k, [0], W.F32)[0]
        assert list(got) == want, (v.tolist(), k, list(got), want)


def rank_count_topk(v, k):
    """i is selected iff #{j : j ranks before i} < k  (vectorised, O(L^2))."""
    v = np.asarray(v, np.float32)
    L = v.size
    neg = np.signbit(v)
    idx = np.arange(L)
    vj, vi = v[:, None], v[None, :]
    eq = vj == vi
    before = (vj > vi) | (eq & (~neg[:, None] & neg[None, :])) | \
             (eq & (neg[:, None] == neg[None, :]) & (idx[:, None] < idx[None, :]))
    sel = np.nonzero(before.sum(axis=0) < k)[0]
    out = np.full(k, -1, np.int64)
    out[:sel.size] = sel
    return out


def pin_rank_count(topk, seed=5):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = [
        rng.standard_normal(2048).astype(np.float32),
        rng.integers(0, 6, size=1500).astype(np.float32) - 3.0,
        W.straddle_row(rng, 2000),
        W.bf16_bits_to_f32(W.bf16_mixed_zeros_subnormals(rng, 1800, 0.2, 0.2, 0.2)),
        np.where(rng.random(1024) < 0.5, -np.inf, rng.standard_normal(1024)).astype(np.float32),
    ]
    for v in rows:
        for k in (1, 7, 100, v.size // 2, v.size - 1, v.size, v.size + 5):
            want = rank_count_topk(v, k)
            got = topk(v, k, None, W.F32)[0]
            assert np.array_equal(got, want), (v.size, k)


def rank_order_topk(v, k):
    """Rank-ordered top-k in closed form: the position whose count of positions
    ranking before it is r goes to output slot r (r < k)  (O(L^2))."""
    v = np.asarray(v, np.float32)
    L = v.size
    neg = np.signbit(v)
    idx = np.arange(L)
    vj, vi = v[:, None], v[None, :]
    eq = vj == vi
    before = (vj > vi) | (eq & (~neg[:, None] & neg[None, :])) | \
             (eq & (neg[:, None] == neg[None, :]) & (idx[:, None] < idx[None, :]))
    rank = before.sum(axis=0)
    out = np.full(k, -1, np.int64)
    sel = rank < k
    out[rank[sel]] = idx[sel]
    return out


def brute_force_ordered(v, k):
    """Rank order by pairwise comparison with the order's definition."""
    order = sorted(range(len(v)), key=functools.cmp_to_key(
        lambda i, j: -1 if _ranks_before(float(v[i]), i, float(v[j]), j) else 1))
    take = min(k, len(v))
    return order[:take] + [-1] * (k - take)


def pin_rank_order(topk_ordered, seed=15):
    """The rank-ordered oracle output against the closed form and, on tiny rows,
    against pairwise brute force."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = [
        rng.standard_normal(2048).astype(np.float32),
        rng.integers(0, 6, size=1500).astype(np.float32) - 3.0,
        W.straddle_row(rng, 2000),
        W.bf16_bits_to_f32(W.bf16_mixed_zeros_subnormals(rng, 1800, 0.2, 0.2, 0.2)),
        np.where(rng.random(1024) < 0.5, -np.inf, rng.standard_normal(1024)).astype(np.float32),
    ]
    for v in rows:
        for k in (1, 7, 100, v.size // 2, v.size, v.size + 5):
            got = topk_ordered(v, k, None, W.F32)[0]
            assert np.array_equal(got, rank_order_topk(v, k)), (v.size, k)
    pool = W.tiny_special_values()
    for _ in range(200):
        L = int(rng.integers(1, 9))
        v = pool[rng.integers(0, pool.size, size=L)]
        k = int(rng.integers(1, L + 2))
        got = topk_ordered(v, k, None, W.F32)[0]
        assert list(got) == brute_force_ordered(v, k), (v.tolist(), k, list(got))


# ----------------------------------------------------------------------------
# an independent selection over order-preserving bit keys
# ----------------------------------------------------------------------------

def order_key_u32(v):
    """The page's "Mapping" step: floats to unsigned integers with the same order
    (negative: all bits flipped; nonnegative: sign bit set)."""
    u = np.asarray(v, np.float32).view(np.uint32)
    return np.where((u >> 31) == 1, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def bitkey_radix_topk(v, k):
    v = np.asarray(v, np.float32)
    L = v.size
    take = min(k, L)
    out = np.full(k, -1, np.int64)
    if take == 0:
        return out
    pos = np.arange(L, dtype=np.uint64)
    # unique keys: value key in the high word, inverted position in the low word
    key = (order_key_u32(v).astype(np.uint64) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - pos)
    cand = key
    rank = take - 1
    prefix = np.uint64(0)
    for shift in range(56, -8, -8):
        digit = ((cand >> np.uint64(shift)) & np.uint64(0xFF)).astype(np.int64)
        hist = np.bincount(digit, minlength=256)
        above = np.cumsum(hist[::-1])[::-1] - hist  # count strictly above each bin
        d = int(np.nonzero((above <= rank) & (rank < above + hist))[0][0])
        rank -= int(above[d])
        prefix |= np.uint64(d) << np.uint64(shift)
        cand = cand[digit == d]
    kth = prefix
    sel = np.nonzero(key >= kth)[0]
    assert sel.size == take
    out[:take] = sel
    return out


def pin_bitkey_radix(topk, work):
    got = topk(work.values, work.k, work.row_len, work.dtype)
    vals = W.as_float32(work)
    for r in range(work.batch):
        want = bitkey_radix_topk(vals[r, :int(work.row_len[r])], work.k)
        assert np.array_equal(got[r], want), (work.name, r)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

def pin_closed_forms(topk):
    def one(v, k, dtype=W.F32):
        return topk(np.asarray(v), k, None, dtype)[0]

    ar = np.arange
    # constant row: the k lowest positions
    assert np.array_equal(one(np.full(5000, 2.5, np.float32), 300), ar(300))
    # strictly ascending / descending distinct values
    assert np.array_equal(one(ar(4000, dtype=np.float32), 123), ar(4000 - 123, 4000))
    assert np.array_equal(one(ar(4000, 0, -1).astype(np.float32), 123), ar(123))
    # k >= L: every position, then -1
    got = one(np.array([3.0, -1.0, 7.0], np.float32), 5)
    assert np.array_equal(got, [0, 1, 2, -1, -1])
    # k = 1: first position of the maximum (numpy's argmax returns the first one)
    rng = np.random.Generator(np.random.PCG64(9))
    for _ in range(20):
        v = rng.integers(1, 20, size=int(rng.integers(1, 500))).astype(np.float32)
        assert one(v, 1)[0] == int(np.argmax(v))
    # signed zeros: +0.0 ranks above -0.0 whatever the positions
    assert list(one(np.array([-0.0, 0.0], np.float32), 1)) == [1]
    assert list(one(np.array([0.0, -0.0], np.float32), 1)) == [0]
    assert list(one(np.array([-0.0, -0.0, 0.0, -1.0], np.float32), 2)) == [0, 2]
    # subnormals above zero, negative subnormals below -0.0
    tiny = np.float32(1.4e-45)
    assert list(one(np.array([0.0, tiny, -tiny, -0.0], np.float32), 1)) == [1]
    assert list(one(np.array([-tiny, -0.0], np.float32), 1)) == [1]
    # -inf is a value like any other, lowest of all
    assert list(one(np.array([-np.inf, -np.inf, 5.0], np.float32), 2)) == [0, 2]
    assert list(one(np.array([-np.inf, -3e38, -np.inf], np.float32), 2)) == [0, 1]
    # bf16: the ramp's top plateau (every i >= 2^20 - 2048 rounds to 2^20)
    n = 1 << 16
    first, size = W.expected_top_plateau(n)
    assert np.array_equal(one(W.bf16_ramp(n), size, W.BF16), ar(first, n))
    # bf16 widening: 0x3F80 is 1.0, 0x4000 is 2.0, 0xBF80 is -1.0
    got = one(np.array([0x3F80, 0x4000, 0xBF80, 0x0000], np.uint16), 2, W.BF16)
    assert list(got) == [0, 1]


# ----------------------------------------------------------------------------
# invariants (also applied to the CUDA path's output)
# ----------------------------------------------------------------------------

def check_invariants(v, L, k, got, where=""):
    """``got``: the selected positions of one row (any order, -1 padding)."""
    v = np.asarray(v, np.float32)[:L]
    got = np.asarray(got, np.int64)
    take = min(k, L)
    sel = got[:take]
    assert np.all(sel >= 0) and sel.size == take, f"{where}: {sel.size} selected, want {take}"
    assert got.size == k and np.all(got[take:] == -1), f"{where}: padding must fill slots take..k"
    assert np.unique(sel).size == take, f"{where}: duplicates"
    assert sel.size == 0 or (sel.min() >= 0 and sel.max() < L), f"{where}: out of range"
    if take == 0 or take == L:
        return
    mask = np.zeros(L, bool)
    mask[sel] = True
    key = order_key_u32(v)
    ks, ku = key[mask], key[~mask]
    assert ks.min() >= ku.max(), f"{where}: a larger value was left out"
    t = ks.min()
    if t == ku.max():
        tied = np.nonzero(key == t)[0]
        tsel = tied[mask[tied]]
        assert tsel.max() < tied[~mask[tied]].min(), f"{where}: ties not the lowest positions"
