"""CPU oracle for the sparse embedding training step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package.  The product path (``dlrm_sparse_embedding_gb300``)
never does, and the two share no code: this wrapper loads its own C library
(``emb_oracle.c``, plain single-threaded C, binary64 accumulation) with its own
ctypes declarations.

The step it computes, by definition (see the C file for the passages):
  a1 lookup + pooling + concatenation, a2 global row ids, a3 unique keys with
  inverse index, counts and segment offsets, a4 per-unique-row gradient sums,
  a5 one SGD / Adagrad / row-wise Adagrad step per touched row, rounded once
  into the table's storage type.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, brute force and
independent library routines); the pages print no numeric worked example, so
no pin comes from the pages' own numbers.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Callable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "emb_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
_POOL_CODE = {"sum": 0, "mean": 1}
_OPT_CODE = {"sgd": 0, "adagrad": 1, "rowwise_adagrad": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FP contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None

_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        L.ora_round_f16.restype = ctypes.c_uint16
        L.ora_round_f16.argtypes = [ctypes.c_double]
        L.ora_round_bf16.restype = ctypes.c_uint16
        L.ora_round_bf16.argtypes = [ctypes.c_double]
        L.ora_f16_to_f64.restype = ctypes.c_double
        L.ora_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.ora_bf16_to_f64.restype = ctypes.c_double
        L.ora_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.ora_round_f16_array.argtypes = [_f64p, i64, _u16p]
        L.ora_round_bf16_array.argtypes = [_f64p, i64, _u16p]
        L.ora_global_ids.restype = i64
        L.ora_global_ids.argtypes = [i32, i32, _i64p, _i64p, _i32p, _i64p, _i64p, _i64p]
        L.ora_unique.restype = i64
        L.ora_unique.argtypes = [_i64p, i64, ctypes.c_int, _i64p, _vp, _vp, _vp]
        L.ora_forward.argtypes = [i32, i32, _i64p, _i32p, i64, _i64p, _f64p, _i32p, _i64p, _i32p, i64,
                                  _vp, i64, _f32p, _vp]
        L.ora_reduce.argtypes = [i32, i32, _i64p, _i32p, i64, _i64p, i64, _i32p, _i64p, _i32p, i64,
                                 _f32p, _f64p, _vp]
        L.ora_reduce_sampled.argtypes = [i32, i32, _i64p, _i64p, _i64p, i64, i32, _i32p, _i64p, _i32p,
                                         i64, _f32p, _f64p, _vp, _i64p]
        L.ora_update.argtypes = [i64, _i32p, _i64p, _i32p, _i32p, _i32p, _i32p, _f64p, _f64p,
                                 _f64p, _vp, _f64p, _f64p, _vp, _vp, _vp]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------

def round_f16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(-1)
    out = np.empty(x.size, dtype=np.uint16)
    lib().ora_round_f16_array(x, x.size, out)
    return out


def round_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(-1)
    out = np.empty(x.size, dtype=np.uint16)
    lib().ora_round_bf16_array(x, x.size, out)
    return out


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Stored 16-bit patterns (uint16) of an "f16"/"bf16" table to float64."""
    f = lib().ora_f16_to_f64 if dtype == "f16" else lib().ora_bf16_to_f64
    flat = np.asarray(bits, dtype=np.uint16).reshape(-1)
    return np.fromiter((f(int(b)) for b in flat), dtype=np.float64, count=flat.size).reshape(np.shape(bits))


def stored_to_f64(v: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(v, dtype=np.float32).astype(np.float64)
    if dtype == "f16":
        bits = np.asarray(v).view(np.uint16) if np.asarray(v).dtype == np.float16 else np.asarray(v, np.uint16)
        return _decode_fast(bits, 10, 5)
    return _decode_fast(np.asarray(v, np.uint16), 7, 8)


def _decode_fast(bits: np.ndarray, mbits: int, ebits: int) -> np.ndarray:
    # Same decoding as the C routine, vectorised for large row sets.
    b = bits.astype(np.int64)
    neg = (b >> 15) & 1
    ex = (b >> mbits) & ((1 << ebits) - 1)
    mant = b & ((1 << mbits) - 1)
    bias = (1 << (ebits - 1)) - 1
    sub = np.ldexp(mant.astype(np.float64), 1 - bias - mbits)
    nor = np.ldexp((mant | (1 << mbits)).astype(np.float64), (ex - bias - mbits).astype(np.int32))
    v = np.where(ex == 0, sub, nor)
    v = np.where(ex == (1 << ebits) - 1, np.where(mant != 0, np.nan, np.inf), v)
    return np.where(neg == 1, -v, v)


def store(v64: np.ndarray, dtype: str) -> np.ndarray:
    """binary64 values already representable in `dtype` to its storage array."""
    if dtype == "f32":
        return v64.astype(np.float32)
    if dtype == "f16":
        return round_f16(v64).reshape(v64.shape).view(np.float16)
    return round_bf16(v64).reshape(v64.shape)


# ---------------------------------------------------------------------------
# the steps
# ---------------------------------------------------------------------------

def row_base(rows: Sequence[int]) -> np.ndarray:
    rb = np.zeros(len(rows), dtype=np.int64)
    if len(rows) > 1:
        rb[1:] = np.cumsum(np.asarray(rows, dtype=np.int64))[:-1]
    return rb


def global_ids(tables, B: int, offsets: np.ndarray, keys: np.ndarray, table_ids: np.ndarray):
    """a2: global row ids (-1 for invalid positions) and the error count."""
    rows = np.array([t.rows for t in tables], dtype=np.int64)
    gids = np.empty(keys.shape[0], dtype=np.int64)
    bad = lib().ora_global_ids(len(tables), B, np.ascontiguousarray(offsets, np.int64),
                               np.ascontiguousarray(keys, np.int64),
                               np.ascontiguousarray(table_ids, np.int32), rows, row_base(rows), gids)
    return gids, int(bad)


def unique(keys: np.ndarray, skip_negative: bool = False):
    """a3: (unique int64[U], inverse int32[n], counts int32[U], seg_off int32[U+1])."""
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    n = keys.shape[0]
    uniq = np.empty(max(n, 1), dtype=np.int64)
    inv = np.empty(max(n, 1), dtype=np.int32)
    cnt = np.empty(max(n, 1), dtype=np.int32)
    seg = np.empty(n + 1, dtype=np.int32)
    U = lib().ora_unique(keys, n, int(skip_negative), uniq, _ptr(inv), _ptr(cnt), _ptr(seg))
    return uniq[:U].copy(), inv[:n].copy(), cnt[:U].copy(), seg[:U + 1].copy()


def _meta(tables):
    dims = np.array([t.dim for t in tables], dtype=np.int32)
    doff = np.zeros(len(tables), dtype=np.int64)
    if len(tables) > 1:
        doff[1:] = np.cumsum(dims.astype(np.int64))[:-1]
    pool = np.array([_POOL_CODE[t.pooling] for t in tables], dtype=np.int32)
    return dims, doff, pool, int(dims.sum())


@dataclasses.dataclass
class RowStore:
    """binary64 values of a set of rows, row k at vals[row_start[k]:+dim]."""
    table: np.ndarray       # int32 [U]
    row: np.ndarray         # int64 [U] local row id
    row_start: np.ndarray   # int64 [U]
    vals: np.ndarray        # float64 [sum dims]


def make_row_store(tables, gids_sorted: np.ndarray,
                   init_rows: Callable[[int, np.ndarray], np.ndarray],
                   state_init: bool = False, fp32_values: bool = False) -> RowStore:
    """Row store of the rows `gids_sorted` (ascending global ids), filled with
    their stored values from init_rows(t, local_rows) decoded to binary64, or
    with the tables' initial accumulator value when state_init is set.  With
    fp32_values, init_rows returns float32 values whatever the table's
    storage type (an fp32 master copy)."""
    rows = np.array([t.rows for t in tables], dtype=np.int64)
    rb = row_base(rows)
    tab = (np.searchsorted(rb, gids_sorted, side="right") - 1).astype(np.int32)
    loc = gids_sorted - rb[tab]
    dims = np.array([t.dim for t in tables], dtype=np.int64)[tab]
    start = np.zeros(gids_sorted.shape[0], dtype=np.int64)
    if start.size > 1:
        start[1:] = np.cumsum(dims)[:-1]
    vals = np.empty(int(dims.sum()), dtype=np.float64)
    for t, spec in enumerate(tables):
        sel = np.nonzero(tab == t)[0]
        if sel.size == 0:
            continue
        idx = (start[sel][:, None] + np.arange(spec.dim)[None, :]).reshape(-1)
        if state_init:
            vals[idx] = float(np.float32(spec.init_acc))
        else:
            vals[idx] = stored_to_f64(init_rows(t, loc[sel]), "f32" if fp32_values else spec.dtype).reshape(-1)
    return RowStore(tab, loc, start, vals)


def forward(tables, B: int, offsets: np.ndarray, inverse: np.ndarray, store_: RowStore,
            bags: Optional[np.ndarray] = None, want_scale: bool = False):
    """a1: pooled, concatenated fp32 output [B, sum dim] (only rows of `bags`
    are written when given; others stay zero) and optionally its scale."""
    dims, doff, pool, D = _meta(tables)
    out = np.zeros((B, D), dtype=np.float32)
    scale = np.zeros((B, D), dtype=np.float64) if want_scale else None
    bags_a = None if bags is None else np.ascontiguousarray(bags, dtype=np.int64)
    lib().ora_forward(len(tables), B, np.ascontiguousarray(offsets, np.int64),
                      np.ascontiguousarray(inverse, np.int32), store_.row_start.shape[0],
                      store_.row_start, store_.vals, dims, doff, pool, D,
                      _ptr(bags_a), 0 if bags_a is None else bags_a.shape[0], out, _ptr(scale))
    return (out, scale) if want_scale else out


def reduce(tables, B: int, offsets: np.ndarray, inverse: np.ndarray, store_: RowStore,
           grad_out: np.ndarray):
    """a4: per-unique-row gradient sums G and their magnitude sums (binary64)."""
    dims, doff, pool, D = _meta(tables)
    G = np.empty_like(store_.vals)
    Gabs = np.empty_like(store_.vals)
    lib().ora_reduce(len(tables), B, np.ascontiguousarray(offsets, np.int64),
                     np.ascontiguousarray(inverse, np.int32), store_.row_start.shape[0],
                     store_.row_start, store_.vals.shape[0], dims, doff, pool, D,
                     np.ascontiguousarray(grad_out, np.float32), G, _ptr(Gabs))
    return G, Gabs


def reduce_sampled(tables, B: int, offsets: np.ndarray, gids: np.ndarray, sample: np.ndarray,
                   grad_out: np.ndarray):
    """a4 restricted to the sorted global ids `sample`: (G [S, maxdim], Gabs, count)."""
    dims, doff, pool, D = _meta(tables)
    S, md = sample.shape[0], int(dims.max())
    G = np.empty((S, md), dtype=np.float64)
    Gabs = np.empty((S, md), dtype=np.float64)
    cnt = np.empty(S, dtype=np.int64)
    lib().ora_reduce_sampled(len(tables), B, np.ascontiguousarray(offsets, np.int64),
                             np.ascontiguousarray(gids, np.int64),
                             np.ascontiguousarray(sample, np.int64), S, md, dims, doff, pool, D,
                             np.ascontiguousarray(grad_out, np.float32), G, _ptr(Gabs), cnt)
    return G, Gabs, cnt


def update(tables, store_: RowStore, state: RowStore, G: np.ndarray, Gabs: Optional[np.ndarray]):
    """a5: updated weights and accumulators (binary64 of the rounded values),
    their magnitude scales, and the stored weights after the step.  For a
    table with an fp32 master copy (``master`` set, 16-bit storage) `store_`
    holds the master values, the returned weights are the new masters and
    the stored weights are them rounded to the storage type; otherwise the
    two are equal.  Inputs are not modified."""
    dims = np.array([t.dim for t in tables], dtype=np.int32)
    dt = np.array([_DTYPE_CODE[t.dtype] for t in tables], dtype=np.int32)
    opt = np.array([_OPT_CODE[t.opt] for t in tables], dtype=np.int32)
    master = np.array([int(bool(getattr(t, "master", False))) for t in tables], dtype=np.int32)
    lr = np.array([float(np.float32(t.lr)) for t in tables], dtype=np.float64)
    eps = np.array([float(np.float32(t.eps)) for t in tables], dtype=np.float64)
    W = store_.vals.copy()
    A = state.vals.copy()
    Ws = np.empty_like(W)
    As = np.empty_like(A)
    W16 = np.empty_like(W)
    lib().ora_update(store_.row_start.shape[0], store_.table, store_.row_start, dims, dt, opt, master, lr, eps,
                     np.ascontiguousarray(G, np.float64), _ptr(Gabs), W, A, _ptr(Ws), _ptr(As), _ptr(W16))
    return W, A, Ws, As, W16


@dataclasses.dataclass
class StepResult:
    gids: np.ndarray
    n_bad: int
    unique: np.ndarray
    inverse: np.ndarray
    counts: np.ndarray
    seg_off: np.ndarray
    out: np.ndarray
    out_scale: np.ndarray
    rows: RowStore          # initial values of the touched rows
    W: np.ndarray           # updated weights (binary64 of stored values), row store layout
    M: np.ndarray           # updated fp32 masters (tables with one; elsewhere equal to W)
    A: np.ndarray           # updated accumulators
    W_scale: np.ndarray
    A_scale: np.ndarray
    G: np.ndarray
    G_abs: np.ndarray


def step(tables, B: int, offsets, keys, table_ids, grad_out,
         init_rows: Callable[[int, np.ndarray], np.ndarray],
         init_master: Optional[Callable[[int, np.ndarray], np.ndarray]] = None) -> StepResult:
    """One full training step a1..a5 over a batch, on the touched rows only.
    Tables with an fp32 master copy take its initial values from
    init_master(t, local_rows) (float32); the forward reads the stored rows."""
    gids, bad = global_ids(tables, B, offsets, keys, table_ids)
    uniq, inv, cnt, seg = unique(gids, skip_negative=True)
    rows = make_row_store(tables, uniq, init_rows)
    has_master = [bool(getattr(t, "master", False)) and t.dtype != "f32" for t in tables]
    upd_rows = rows
    if any(has_master):
        if init_master is None:
            raise ValueError("tables with an fp32 master copy need init_master")
        upd_rows = make_row_store(tables, uniq, lambda t, r: init_master(t, r) if has_master[t] else
                                  stored_to_f64(init_rows(t, r), tables[t].dtype).astype(np.float32),
                                  fp32_values=True)
    state = make_row_store(tables, uniq, init_rows, state_init=True)
    out, oscale = forward(tables, B, offsets, inv, rows, want_scale=True)
    G, Gabs = reduce(tables, B, offsets, inv, rows, grad_out)
    M, A, Ws, As, W = update(tables, upd_rows, state, G, Gabs)
    return StepResult(gids, bad, uniq, inv, cnt, seg, out, oscale, rows, W, M, A, Ws, As, G, Gabs)


def step_dynamic(tables, B: int, offsets, keys, table_ids, grad_out,
                 init_rows: Callable[[int, np.ndarray], np.ndarray],
                 init_dynamic: Callable[[int, np.ndarray], np.ndarray],
                 init_master: Optional[Callable[[int, np.ndarray], np.ndarray]] = None,
                 init_dynamic_master: Optional[Callable[[int, np.ndarray], np.ndarray]] = None):
    """A step on a layer with dynamic tables (``dynamic`` set): such a table
    maps arbitrary int64 keys to rows, each row starting at
    init_dynamic(t, keys) when its key first appears.  By that definition it
    is a table over its distinct keys, so each dynamic table's keys are
    relabelled to dense ids (ascending key order; the reserved key -2^63 is
    skipped like an out-of-range key) and the plain step runs on the result.
    Returns (StepResult, key_of) with key_of[t] the keys of table t's dense
    ids (dynamic tables only)."""
    keys2 = np.array(keys, dtype=np.int64, copy=True)
    tables2 = list(tables)
    key_of = {}
    for t, spec in enumerate(tables):
        if not getattr(spec, "dynamic", False):
            continue
        lo, hi = int(offsets[t * B]), int(offsets[(t + 1) * B])
        k = keys2[lo:hi]
        valid = k != np.iinfo(np.int64).min
        uk, inv = np.unique(k[valid], return_inverse=True)
        dense = np.full(hi - lo, -1, dtype=np.int64)
        dense[valid] = inv
        keys2[lo:hi] = dense
        tables2[t] = dataclasses.replace(spec, rows=max(int(uk.size), 1), dynamic=False)
        key_of[t] = uk
    rows_fn = lambda t, r: init_dynamic(t, key_of[t][r]) if t in key_of else init_rows(t, r)
    master_fn = None
    if init_master is not None or init_dynamic_master is not None:
        master_fn = lambda t, r: (init_dynamic_master(t, key_of[t][r]) if t in key_of else init_master(t, r))
    return step(tables2, B, offsets, keys2, table_ids, grad_out, rows_fn, master_fn), key_of


def forward_with_cache(tables, B: int, offsets, keys, table_ids,
                       init_rows: Callable[[int, np.ndarray], np.ndarray], cached: dict):
    """Inference forward with fp16 caches: the pooled output (a1) over the
    tables with every row in cached[t] (row ids of table t) replaced by its
    nearest-even fp16 rounding (NumPy's conversion), as a cache of those rows
    would serve it.  Returns (out, out_scale)."""
    gids, _ = global_ids(tables, B, offsets, keys, table_ids)
    uniq, inv, _, _ = unique(gids, skip_negative=True)

    def values(t, r):
        v = stored_to_f64(init_rows(t, r), tables[t].dtype)
        hit = np.isin(np.asarray(r), np.asarray(cached.get(t, []), dtype=np.int64))
        v[hit] = v[hit].astype(np.float16).astype(np.float64)
        return v.astype(np.float32)

    rows = make_row_store(tables, uniq, values, fp32_values=True)
    return forward(tables, B, offsets, inv, rows, want_scale=True)
