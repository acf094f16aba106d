"""Seeded synthetic CTR batches for the sparse embedding training step.

This module is the only code shared by the CUDA path's tests/bench and by the
CPU oracle.  It produces *inputs* only -- table shapes, CSR batches of
categorical keys, upstream gradients and the initial table values -- and holds
none of the embedding arithmetic (no pooling, dedup, reduction or optimizer).

Workloads mimic the click-through-rate setting of the HugeCTR pages (GTC 2022
"Merlin HugeCTR" slides, "COMMON EMBEDDING PRIMITIVES": multi-hot categorical
features, one table per feature) and the Criteo-like 26 categorical features of
the Merlin overview article ("NVTabular" section).  The datasets themselves are
not available, so every batch is synthetic:

* bulk random draws use NumPy's PCG64, keyed by ``SeedSequence([seed, purpose,
  table])`` so every (workload, purpose, table) stream is independent;
* skewed keys follow a Zipf law ``P(k) ~ (k+1)**-alpha`` over ``[0, rows)``
  (rank 0 hottest, no scrambling), sampled with Hoermann & Derflinger's
  rejection-inversion method (ACM TOMACS 6(3), 1996);
* initial table values come from a counter-based generator: the n-th output of
  splitmix64 (Steele, Lea & Flood, OOPSLA 2014) with the workload seed as the
  state, ``n = t*2**44 + r*2**12 + c``.  The value is
  ``lo + (hi - lo) * ((h >> 40) * 2**-24)`` evaluated in fp32, one rounding
  per operation, then rounded to nearest-even into the table's storage type.
  The CUDA library's table initialiser implements the same published
  generator on the device, so untouched rows never need to be materialised on
  the host.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

__all__ = [
    "TableSpec", "Workload", "Batch", "WORKLOADS", "workload",
    "make_batch", "make_grad", "init_values", "stored_to_f64",
    "splitmix64_at", "zipf_keys", "dynamic_key", "init_values_dynamic",
]

# purposes for SeedSequence keys
_P_ROWS, _P_HOT, _P_KEYS, _P_GRAD = 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class TableSpec:
    rows: int
    dim: int
    dtype: str = "f32"          # storage type: "f32" | "f16" | "bf16"
    pooling: str = "sum"        # "sum" | "mean"
    opt: str = "sgd"            # "sgd" | "adagrad" | "rowwise_adagrad"
    lr: float = 0.01
    eps: float = 1e-8
    init_acc: float = 0.0
    master: bool = False        # keep an fp32 master copy (16-bit storage only)
    dynamic: bool = False       # keys are arbitrary int64 ids; rows is the hash-map capacity

    @property
    def key_space(self) -> int:
        """Distinct keys a batch draws from: rows, or half the capacity of a
        dynamic table (so its map stays at most half full)."""
        return max(1, self.rows // 2) if self.dynamic else self.rows


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tables: tuple               # tuple[TableSpec]
    batch: int
    hot_kind: str               # "fixed" | "per_bag_uniform" | "per_table_uniform"
    hot_lo: int
    hot_hi: int
    key_dist: str               # "uniform" | "zipf"
    alpha: float = 0.0
    seed: int = 0
    w_lo: float = -0.05
    w_hi: float = 0.05

    @property
    def num_tables(self) -> int:
        return len(self.tables)

    @property
    def total_dim(self) -> int:
        return sum(t.dim for t in self.tables)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def with_tables(self, **kw) -> "Workload":
        """Same workload with every table spec changed by ``kw``."""
        return dataclasses.replace(
            self, tables=tuple(dataclasses.replace(t, **kw) for t in self.tables))

    def hotness(self) -> np.ndarray:
        """Bag lengths, int64 [T, B] (bag j = t*B + b)."""
        T, B = self.num_tables, self.batch
        if self.hot_kind == "fixed":
            return np.full((T, B), self.hot_lo, dtype=np.int64)
        if self.hot_kind == "per_bag_uniform":
            out = np.empty((T, B), dtype=np.int64)
            for t in range(T):
                rng = _rng(self.seed, _P_HOT, t)
                out[t] = rng.integers(self.hot_lo, self.hot_hi + 1, size=B)
            return out
        if self.hot_kind == "per_table_uniform":
            rng = _rng(self.seed, _P_HOT, 0)
            h = rng.integers(self.hot_lo, self.hot_hi + 1, size=T)
            return np.repeat(h[:, None], B, axis=1).astype(np.int64)
        raise ValueError(self.hot_kind)


@dataclasses.dataclass
class Batch:
    keys: np.ndarray        # int64 [nnz]   local row ids, bag-major
    offsets: np.ndarray     # int64 [T*B+1] CSR bag boundaries, bag j = t*B + b
    table_ids: np.ndarray   # int32 [T*B]   table of each bag (== j // B)
    batch: int

    @property
    def nnz(self) -> int:
        return int(self.keys.shape[0])


def _rng(seed: int, purpose: int, table: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, purpose, table])))


def _log_uniform_rows(seed: int, n: int, lo: float, hi: float) -> List[int]:
    rng = _rng(seed, _P_ROWS, 0)
    u = rng.random(n)
    return [int(math.floor(math.exp(math.log(lo) + x * (math.log(hi) - math.log(lo))))) for x in u]


def _build_workloads() -> dict:
    w = {}
    w["tiny"] = Workload(
        name="tiny", tables=tuple(TableSpec(1000, 16, "f32", "sum", "sgd", 0.01) for _ in range(4)),
        batch=256, hot_kind="per_bag_uniform", hot_lo=1, hot_hi=4, key_dist="uniform")
    rows = _log_uniform_rows(0, 26, 1e3, 1e7)
    w["dlrm"] = Workload(
        name="dlrm", tables=tuple(TableSpec(r, 128, "f32", "sum", "adagrad", 0.01, 1e-8) for r in rows),
        batch=65536, hot_kind="fixed", hot_lo=1, hot_hi=1, key_dist="zipf", alpha=1.05)
    w["multihot"] = Workload(
        name="multihot",
        tables=tuple(TableSpec(1_000_000, 64, "f32", "mean", "adagrad", 0.01, 1e-8) for _ in range(100)),
        batch=16384, hot_kind="per_table_uniform", hot_lo=1, hot_hi=100, key_dist="zipf", alpha=1.2)
    w["huge"] = Workload(
        name="huge", tables=(TableSpec(200_000_000, 64, "f16", "sum", "adagrad", 0.01, 1e-8),),
        batch=131072, hot_kind="fixed", hot_lo=20, hot_hi=20, key_dist="zipf", alpha=1.1)
    w["skew"] = Workload(
        name="skew",
        tables=tuple(TableSpec(5_000_000, d, "f32", "sum", "sgd", 0.01) for d in (16, 32, 64, 128) * 2),
        batch=262144, hot_kind="fixed", hot_lo=50, hot_hi=50, key_dist="zipf", alpha=1.5)
    # the dlrm workload with one Adagrad accumulator per row instead of per element
    w["dlrm_rowwise"] = w["dlrm"].replace(name="dlrm_rowwise").with_tables(opt="rowwise_adagrad")
    # the dlrm workload with its tables behind hash maps: the same Zipf ranks,
    # drawn from the same key spaces, become scrambled int64 ids; each map has
    # twice as many rows as its key space
    w["dlrm_dynamic"] = w["dlrm"].replace(name="dlrm_dynamic", tables=tuple(
        dataclasses.replace(t, rows=2 * t.rows, dynamic=True) for t in w["dlrm"].tables))
    # the huge fp16 table with an fp32 master copy
    w["huge_master"] = w["huge"].replace(name="huge_master").with_tables(master=True)
    return w


WORKLOADS = _build_workloads()


def workload(name: str) -> Workload:
    return WORKLOADS[name]


# ----------------------------------------------------------------------------
# Zipf keys by rejection-inversion (Hoermann & Derflinger 1996)
# ----------------------------------------------------------------------------

def _expm1_over(x):
    x = np.asarray(x, dtype=np.float64)
    small = np.abs(x) < 1e-8
    safe = np.where(small, 1.0, x)
    return np.where(small, 1.0 + 0.5 * x * (1.0 + x / 3.0), np.expm1(safe) / safe)


def _log1p_over(x):
    x = np.asarray(x, dtype=np.float64)
    small = np.abs(x) < 1e-8
    safe = np.where(small, 1.0, x)
    return np.where(small, 1.0 - 0.5 * x * (1.0 - 2.0 * x / 3.0), np.log1p(safe) / safe)


class _ZipfRI:
    """Rejection-inversion sampler for P(k) ~ k**-s on k = 1..n."""

    def __init__(self, n: int, s: float):
        self.n, self.s = float(n), float(s)
        self.hx1 = self.H(1.5) - 1.0
        self.hn = self.H(self.n + 0.5)
        self.thr = 2.0 - self.Hinv(self.H(2.5) - self.h(2.0))

    def h(self, x):
        return np.exp(-self.s * np.log(x))

    def H(self, x):
        lx = np.log(x)
        return _expm1_over((1.0 - self.s) * lx) * lx

    def Hinv(self, y):
        t = np.maximum(y * (1.0 - self.s), -1.0)
        return np.exp(_log1p_over(t) * y)

    def sample(self, rng: np.random.Generator, m: int) -> np.ndarray:
        out = np.empty(m, dtype=np.int64)
        todo = np.arange(m)
        while todo.size:
            u = self.hn + rng.random(todo.size) * (self.hx1 - self.hn)
            x = self.Hinv(u)
            k = np.clip(np.floor(x + 0.5), 1.0, self.n)
            ok = (k - x <= self.thr) | (u >= self.H(k + 0.5) - self.h(k))
            out[todo[ok]] = k[ok].astype(np.int64)
            todo = todo[~ok]
        return out


def zipf_keys(rng: np.random.Generator, rows: int, alpha: float, m: int) -> np.ndarray:
    """m keys in [0, rows) with P(key) ~ (key+1)**-alpha."""
    return _ZipfRI(rows, alpha).sample(rng, m) - 1


def make_batch(w: Workload, seed: Optional[int] = None) -> Batch:
    """CSR batch: bag j = t*B + b holds hot[t,b] keys of table t."""
    seed = w.seed if seed is None else seed
    hot = w.replace(seed=seed).hotness()
    T, B = w.num_tables, w.batch
    lens = hot.reshape(-1)
    offsets = np.zeros(T * B + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    keys = np.empty(int(offsets[-1]), dtype=np.int64)
    for t, spec in enumerate(w.tables):
        lo, hi = int(offsets[t * B]), int(offsets[(t + 1) * B])
        rng = _rng(seed, _P_KEYS, t)
        if w.key_dist == "uniform":
            keys[lo:hi] = rng.integers(0, spec.key_space, size=hi - lo)
        elif w.key_dist == "zipf":
            keys[lo:hi] = zipf_keys(rng, spec.key_space, w.alpha, hi - lo)
        else:
            raise ValueError(w.key_dist)
        if spec.dynamic:
            keys[lo:hi] = dynamic_key(t, keys[lo:hi])
    table_ids = np.repeat(np.arange(T, dtype=np.int32), B)
    return Batch(keys=keys, offsets=offsets, table_ids=table_ids, batch=B)


def make_grad(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """Upstream gradient of the concatenated pooled output, fp32 [B, sum(dim)] ~ N(0,1)."""
    seed = w.seed if seed is None else seed
    rng = _rng(seed, _P_GRAD, 0)
    return rng.standard_normal((w.batch, w.total_dim), dtype=np.float32)


# ----------------------------------------------------------------------------
# counter-based initial values
# ----------------------------------------------------------------------------

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64_at(seed: int, n: np.ndarray) -> np.ndarray:
    """n-th output (0-based) of splitmix64 started from state ``seed``."""
    n = np.asarray(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (n + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def init_values(seed: int, table: int, rows: np.ndarray, dim: int, lo: float, hi: float,
                dtype: str = "f32") -> np.ndarray:
    """Initial values of rows ``rows`` of table ``table`` in the storage type.

    Returns float32 [n, dim] for "f32", float16 for "f16" and the raw uint16
    bit patterns for "bf16"."""
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    cols = np.arange(dim, dtype=np.uint64).reshape(1, -1)
    n = (np.uint64(table) << np.uint64(44)) | (rows << np.uint64(12)) | cols
    h = splitmix64_at(seed, n)
    f = (h >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    d = np.float32(hi) - np.float32(lo)
    w = np.float32(lo) + d * f
    w = w.astype(np.float32)
    if dtype == "f32":
        return w
    if dtype == "f16":
        return w.astype(np.float16)
    if dtype == "bf16":
        return _f32_to_bf16_bits(w)
    raise ValueError(dtype)


def dynamic_key(table: int, rank: np.ndarray) -> np.ndarray:
    """The int64 id of key rank ``rank`` of a dynamic table: splitmix64 output
    number rank of the stream seeded with the table index (a bijection of the
    rank for each table), so ids look like arbitrary 64-bit hashes.  The
    value -2^63 is reserved (empty map slot) and replaced by 2^63 - 1."""
    k = splitmix64_at(int(table), np.asarray(rank, dtype=np.uint64)).view(np.int64)
    return np.where(k == np.iinfo(np.int64).min, np.iinfo(np.int64).max, k)


def init_values_dynamic(seed: int, table: int, keys: np.ndarray, dim: int, lo: float, hi: float,
                        dtype: str = "f32") -> np.ndarray:
    """Initial values of the rows of keys ``keys`` of a dynamic table, like
    ``init_values`` but with splitmix64 output number
    (key << 8) ^ (table << 57) ^ c (64-bit wrap-around) for column c."""
    k = np.asarray(keys, dtype=np.int64).view(np.uint64).reshape(-1, 1)
    cols = np.arange(dim, dtype=np.uint64).reshape(1, -1)
    with np.errstate(over="ignore"):
        n = (k << np.uint64(8)) ^ (np.uint64(table) << np.uint64(57)) ^ cols
    h = splitmix64_at(seed, n)
    f = (h >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    w = (np.float32(lo) + (np.float32(hi) - np.float32(lo)) * f).astype(np.float32)
    if dtype == "f32":
        return w
    if dtype == "f16":
        return w.astype(np.float16)
    if dtype == "bf16":
        return _f32_to_bf16_bits(w)
    raise ValueError(dtype)


def stored_to_f64(v: np.ndarray, dtype: str) -> np.ndarray:
    """Stored table values (as returned by ``init_values``) to float64."""
    if dtype == "bf16":
        return (v.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return v.astype(np.float64)
