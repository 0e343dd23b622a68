"""Seeded synthetic inputs for the DSA TopK selector.

This module only draws numbers. It holds none of the selection arithmetic, so
both the CPU oracle (``oracle/``) and the CUDA path can be fed from it without
sharing any of the method's code.

Every workload is a ``Workload``: a 2-D array ``values`` of shape
``[batch, row_stride]`` (``float32`` for fp32 logits, ``uint16`` holding the raw
bfloat16 bit patterns for bf16 logits), the valid length of each row, ``k`` and
a dtype tag. Positions at or beyond a row's valid length are filled with NaN, so
that any read of them shows up as a wrong answer.

The five named workloads follow the shapes the "Technical Deep Dive ... TopK
Selector" page talks about (single-query decode over 128K-1M tokens, and a
batched decode), with value recipes fixed here because the page gives none:

* ``decode_4k``          1 x 4096 fp32 ~ N(0,1), k=256
* ``decode_128k``        1 x 131072 fp32 ~ N(0,1), k=2048
* ``decode_1m_masked``   1 x 1048576 fp32, N(0,1) rounded to bf16 and widened
                         back (heavy duplicates), last 10% set to -inf, k=2048
* ``batch64_ragged``     64 rows, row_stride 65536 fp32, valid length uniform in
                         [4096, 65536], 3*N(0,1) + per-row offset U(-5,5), k=2048
* ``batch4_1m_bf16``     4 x 1048576 bf16, k=2048, rows: constant 1.0; ramp
                         bf16(i); N(0,1) with +-0 and subnormals mixed in;
                         Gumbel(0,1)
"""

from __future__ import annotations

import dataclasses

import numpy as np

F32 = "f32"
BF16 = "bf16"

# bit patterns of the bf16 NaN used to poison unused stride tails
_BF16_QNAN = np.uint16(0x7FC0)


@dataclasses.dataclass
class Workload:
    name: str
    values: np.ndarray  # [batch, row_stride]; float32, or uint16 bf16 bit patterns
    row_len: np.ndarray  # int32 [batch]
    k: int
    dtype: str  # F32 or BF16
    note: str = ""

    @property
    def batch(self) -> int:
        return int(self.values.shape[0])

    @property
    def row_stride(self) -> int:
        return int(self.values.shape[1])

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == F32 else 2

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes of valid logits: every one of them must be read once."""
        return int(self.row_len.astype(np.int64).sum()) * self.elem_size


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16, round-to-nearest-even, as bit patterns.

    Input generation only (the same rounding ``torch.Tensor.to(torch.bfloat16)``
    applies). NaN is never passed in here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _poison_tails(values: np.ndarray, row_len: np.ndarray, dtype: str) -> None:
    fill = np.float32(np.nan) if dtype == F32 else _BF16_QNAN
    for r, L in enumerate(row_len):
        values[r, int(L):] = fill


# ----------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------

def decode_4k(seed: int = 1) -> Workload:
    rng = _rng(seed)
    v = rng.standard_normal(4096).astype(np.float32)[None, :]
    return Workload("decode_4k", v, np.array([4096], np.int32), 256, F32,
                    "1 row, N=4096 fp32 ~ N(0,1), k=256")


def decode_128k(seed: int = 2) -> Workload:
    rng = _rng(seed)
    v = rng.standard_normal(131072).astype(np.float32)[None, :]
    return Workload("decode_128k", v, np.array([131072], np.int32), 2048, F32,
                    "batch=1, N=131072 fp32 ~ N(0,1), k=2048")


def decode_1m_masked(seed: int = 3) -> Workload:
    n = 1 << 20
    rng = _rng(seed)
    x = rng.standard_normal(n).astype(np.float32)
    v = bf16_bits_to_f32(f32_to_bf16_bits(x)).copy()
    v[n - n // 10:] = -np.inf  # masked positions: the last 10%
    return Workload("decode_1m_masked", v[None, :], np.array([n], np.int32), 2048, F32,
                    "batch=1, N=1048576 fp32 from bf16-rounded N(0,1), last 10% -inf, k=2048")


def batch64_ragged(seed: int = 4) -> Workload:
    rng = _rng(seed)
    batch, stride = 64, 65536
    lens = rng.integers(4096, 65536, size=batch, endpoint=True).astype(np.int32)
    offs = rng.uniform(-5.0, 5.0, size=batch)
    v = np.empty((batch, stride), np.float32)
    for r in range(batch):
        v[r, :] = (3.0 * rng.standard_normal(stride) + offs[r]).astype(np.float32)
    _poison_tails(v, lens, F32)
    return Workload("batch64_ragged", v, lens, 2048, F32,
                    "batch=64, row_stride=65536 fp32, ragged lengths U[4096,65536], "
                    "3*N(0,1)+U(-5,5) per row, k=2048")


def bf16_ramp(n: int) -> np.ndarray:
    """bf16(i) for i = 0..n-1: non-decreasing, with plateaus once i > 256."""
    return f32_to_bf16_bits(np.arange(n, dtype=np.float32))


def bf16_mixed_zeros_subnormals(rng: np.random.Generator, n: int,
                                frac_pz=0.05, frac_nz=0.05, frac_sub=0.05) -> np.ndarray:
    """N(0,1) rounded to bf16 with +0, -0 and subnormals planted at seeded positions."""
    b = f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    perm = rng.permutation(n)
    n_pz, n_nz, n_sub = int(n * frac_pz), int(n * frac_nz), int(n * frac_sub)
    b[perm[:n_pz]] = 0x0000
    b[perm[n_pz:n_pz + n_nz]] = 0x8000
    sub = perm[n_pz + n_nz:n_pz + n_nz + n_sub]
    mant = rng.integers(1, 128, size=sub.size).astype(np.uint16)
    sign = (rng.integers(0, 2, size=sub.size).astype(np.uint16) << 15).astype(np.uint16)
    b[sub] = sign | mant
    return b


def gumbel_open(rng: np.random.Generator, n: int) -> np.ndarray:
    """Gumbel(0,1) samples -ln(-ln U) with U drawn from the open interval (0,1)."""
    u = rng.integers(1, 1 << 53, size=n).astype(np.float64) / float(1 << 53)
    return -np.log(-np.log(u))


def batch4_1m_bf16(seed: int = 5) -> Workload:
    n = 1 << 20
    rng = _rng(seed)
    v = np.empty((4, n), np.uint16)
    v[0] = f32_to_bf16_bits(np.full(n, 1.0, np.float32))  # (a) all equal
    v[1] = bf16_ramp(n)  # (b) ascending ramp, top plateau has exactly 2048 members
    v[2] = bf16_mixed_zeros_subnormals(rng, n)  # (c)
    v[3] = f32_to_bf16_bits(gumbel_open(rng, n).astype(np.float32))  # (d)
    return Workload("batch4_1m_bf16", v, np.full(4, n, np.int32), 2048, BF16,
                    "batch=4, N=1048576 bf16, k=2048: constant, ramp, N(0,1)+zeros+subnormals, Gumbel")


NAMED = {
    "decode_4k": decode_4k,
    "decode_128k": decode_128k,
    "decode_1m_masked": decode_1m_masked,
    "batch64_ragged": batch64_ragged,
    "batch4_1m_bf16": batch4_1m_bf16,
}


def prefill_causal(seed: int = 6) -> Workload:
    """A prefill-like batch: 512 query rows over a 32K context with causal
    lengths (row r sees 64 (r + 1) tokens), N(0,1) fp32 logits, k=2048.  Not
    one of the five named configurations: the large-batch case that the
    page's batch=64 results point to, at the scale of a prefill chunk."""
    rng = _rng(seed)
    batch, stride = 512, 32768
    lens = (64 * (np.arange(batch) + 1)).astype(np.int32)
    v = rng.standard_normal((batch, stride)).astype(np.float32)
    _poison_tails(v, lens, F32)
    return Workload("prefill_causal", v, lens, 2048, F32,
                    "batch=512, row_stride=32768 fp32, causal lengths 64(r+1), N(0,1), k=2048")


EXTRA = {"prefill_causal": prefill_causal}


def named(name: str) -> Workload:
    return NAMED[name]() if name in NAMED else EXTRA[name]()


# ----------------------------------------------------------------------------
# Edge and fuzz rows
# ----------------------------------------------------------------------------

def from_rows(name: str, rows, k: int, dtype: str = F32, row_stride: int | None = None,
              note: str = "") -> Workload:
    """Pack a list of 1-D rows (float32 values, or uint16 bf16 bits) into a Workload."""
    lens = np.array([len(r) for r in rows], np.int32)
    stride = int(row_stride if row_stride is not None else max(1, int(lens.max(initial=1))))
    assert stride >= int(lens.max(initial=0))
    if dtype == F32:
        v = np.full((len(rows), stride), np.nan, np.float32)
    else:
        v = np.full((len(rows), stride), _BF16_QNAN, np.uint16)
    for r, row in enumerate(rows):
        v[r, :len(row)] = row
    return Workload(name, v, lens, int(k), dtype, note)


def tiny_special_values() -> np.ndarray:
    """A pool of float32 values that exercise every ordering rule."""
    return np.array([-np.inf, -1.0, -0.0, 0.0, np.float32(1.4e-45), np.float32(-1.4e-45),
                     1.0, 1.0, np.inf, 2.5, -2.5, np.float32(1.1754942e-38)], np.float32)


def straddle_row(rng: np.random.Generator, n: int) -> np.ndarray:
    """Values drawn from a handful of levels around zero (+-0, +-subnormal, +-tiny),
    so that the k-th value lands among signed zeros and subnormals for most k."""
    levels = np.array([0.0, -0.0, 1.4e-45, -1.4e-45, 2.8e-45, -2.8e-45, 1.0e-40,
                       -1.0e-40, 1.1754942e-38, -1.1754942e-38, 1e-3, -1e-3], np.float32)
    return levels[rng.integers(0, levels.size, size=n)]


def fuzz_cases(seed: int = 11):
    """Seeded edge and fuzz workloads (small enough for the oracle in well under a second)."""
    rng = _rng(seed)
    out = []
    out.append(from_rows("len_lt_k", [rng.standard_normal(100).astype(np.float32)], 256))
    out.append(from_rows("len_eq_k", [rng.standard_normal(256).astype(np.float32)], 256))
    out.append(from_rows("k_eq_1", [rng.standard_normal(5000).astype(np.float32)], 1))
    out.append(from_rows("k1_ties", [np.full(7001, 3.0, np.float32)], 1))
    out.append(from_rows("len_1", [np.array([0.5], np.float32)], 4))
    out.append(from_rows("odd_len", [rng.standard_normal(4099).astype(np.float32)], 300))
    out.append(from_rows("all_neg_inf", [np.full(3001, -np.inf, np.float32)], 100))
    out.append(from_rows("all_equal", [np.full(20000, -7.25, np.float32)], 1000))
    out.append(from_rows("straddle_zero_subnormal",
                         [straddle_row(rng, 9000), straddle_row(rng, 12345)], 1500))
    out.append(from_rows("ascending", [np.arange(30000, dtype=np.float32)], 777))
    out.append(from_rows("descending", [np.arange(30000, 0, -1).astype(np.float32)], 777))
    # many exact ties at the threshold, spread over the whole row
    few = rng.integers(0, 4, size=50000).astype(np.float32)
    out.append(from_rows("few_levels", [few], 20000))
    # odd row stride (rows start at unaligned addresses) and ragged lengths
    rows = [rng.standard_normal(int(n)).astype(np.float32)
            for n in rng.integers(1, 9000, size=9)]
    out.append(from_rows("odd_stride_ragged", rows, 513, row_stride=9001))
    # empty rows mixed in
    out.append(from_rows("with_empty_rows",
                         [np.zeros(0, np.float32), rng.standard_normal(3000).astype(np.float32),
                          np.zeros(0, np.float32)], 64, row_stride=3001))
    # bf16 edge rows
    out.append(from_rows("bf16_small", [f32_to_bf16_bits(rng.standard_normal(5003))], 129, BF16))
    out.append(from_rows("bf16_zeros_subnormals",
                         [bf16_mixed_zeros_subnormals(rng, 40000, 0.3, 0.3, 0.3)], 15000, BF16))
    out.append(from_rows("bf16_odd_stride",
                         [f32_to_bf16_bits(rng.standard_normal(int(n))) for n in (17, 4097, 1023)],
                         200, BF16, row_stride=4099))
    out.append(from_rows("bf16_ramp_64k", [bf16_ramp(65536)], 3000, BF16))
    # large k
    out.append(from_rows("large_k", [rng.standard_normal(100000).astype(np.float32)], 40000))
    return out


def random_rows(seed: int, batch: int, max_len: int, k: int, dtype: str = F32,
                levels: int | None = None) -> Workload:
    """Random ragged rows; ``levels`` draws values from that many distinct levels
    (to make ties), else N(0,1)."""
    rng = _rng(seed)
    rows = []
    for _ in range(batch):
        n = int(rng.integers(0, max_len + 1))
        if levels is None:
            x = rng.standard_normal(n).astype(np.float32)
        else:
            x = rng.integers(0, levels, size=n).astype(np.float32) - levels / 2
        rows.append(x if dtype == F32 else f32_to_bf16_bits(x))
    return from_rows(f"random_{seed}", rows, k, dtype, row_stride=max(1, max_len))


def _sweep_values(rng: np.random.Generator, n: int, kind: str) -> np.ndarray:
    """float32 values of one sweep row, by kind."""
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "levels":  # heavy ties
        return (rng.integers(0, 7, size=n).astype(np.float32) - 3.0)
    if kind == "wide":  # many exponents, both signs
        return (rng.choice([-1.0, 1.0], size=n) *
                np.exp(rng.uniform(-80.0, 80.0, size=n))).astype(np.float32)
    if kind == "specials":  # signed zeros, subnormals, -inf mixed with normals
        v = rng.standard_normal(n).astype(np.float32)
        m = rng.integers(0, 6, size=n)
        v[m == 0] = 0.0
        v[m == 1] = -0.0
        v[m == 2] = -np.inf
        v[m == 3] = np.float32(1e-42) * rng.integers(1, 100, size=int((m == 3).sum()))
        return v
    if kind == "ramp":  # sorted runs, ascending or descending
        v = np.arange(n, dtype=np.float32)
        return v if rng.integers(0, 2) else v[::-1].copy()
    raise ValueError(kind)


def sweep_cases(seed: int, count: int, max_elems: int = 2_000_000):
    """Seeded random shapes for a parity sweep: batch, row stride, row lengths,
    k, dtype and value kind all drawn, at most max_elems logits per case.
    Returns (workload, draw) pairs; draw also holds the non-value choices
    (alignment offset, block size, cluster, forced split) for the caller."""
    rng = _rng(seed)
    out = []
    for c in range(count):
        batch = int(rng.choice([1, 1, 2, 3, 5, 8, 9, 16, 64, 160, 300]))
        cap = max(64, max_elems // batch)
        stride = int(rng.integers(1, min(cap, 400_000) + 1))
        ragged = bool(rng.integers(0, 2))
        lens = rng.integers(0, stride + 1, size=batch) if ragged else np.full(batch, stride)
        kind = str(rng.choice(["normal", "levels", "wide", "specials", "ramp"]))
        dtype = F32 if rng.integers(0, 3) else BF16
        kmax = int(min(TKS_K_MAX_SWEEP, max(1, stride)))
        k = int(rng.choice([1, int(rng.integers(1, kmax + 1)), int(rng.integers(1, min(kmax, 4096) + 1)),
                            min(kmax, 2048)]))
        if rng.integers(0, 8) == 0:
            k = int(min(TKS_K_MAX_SWEEP, stride + int(rng.integers(1, 50))))  # k above every length
        rows = []
        for r in range(batch):
            v = _sweep_values(rng, int(lens[r]), kind)
            rows.append(v if dtype == F32 else f32_to_bf16_bits(v))
        w = from_rows(f"sweep{seed}_{c}", rows, max(1, k), dtype, row_stride=stride,
                      note=f"{kind}, batch {batch}, stride {stride}, ragged {ragged}")
        draw = {"offset": int(rng.choice([0, 0, 1, 3])), "threads": int(rng.choice([0, 256, 512])),
                "cluster": int(rng.integers(0, 2)), "group": int(rng.choice([0, 0, 0, 2, 5, 17])),
                "sorted": bool(rng.integers(0, 3) == 0), "host": bool(rng.integers(0, 4) == 0)}
        out.append((w, draw))
    return out


TKS_K_MAX_SWEEP = 16384


def as_float32(w: Workload) -> np.ndarray:
    """The values as float32 (bf16 widened exactly)."""
    return w.values if w.dtype == F32 else bf16_bits_to_f32(w.values)


def expected_top_plateau(n: int) -> tuple[int, int]:
    """First index and size of the top plateau of ``bf16_ramp(n)`` for n a power of two
    (every i >= n - n/512 rounds to n under bf16's 8 significant bits)."""
    assert n & (n - 1) == 0 and n >= 512
    spacing = n // 256  # ulp of bf16 just below n
    first = n - spacing // 2
    return first, n - first


__all__ = [
    "Workload", "F32", "BF16", "NAMED", "EXTRA", "named", "fuzz_cases", "random_rows", "from_rows",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "as_float32", "bf16_ramp", "tiny_special_values",
    "expected_top_plateau", "decode_4k", "decode_128k", "decode_1m_masked", "batch64_ragged",
    "batch4_1m_bf16", "gumbel_open", "bf16_mixed_zeros_subnormals", "straddle_row",
]
