"""Thin Python binding over the C ABI: argument marshalling only.

Tensors are torch CUDA tensors; every call runs on the current torch stream.
All computation happens in libemb.so's kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from ._lib import (DTYPES, OPTS, PHASES, POOLINGS, VARIANTS, EmbTableSpec, check, lib)

_TORCH_WDTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
_NP_WDTYPE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[ctypes.c_void_p]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, min_numel: Optional[int] = None,
           shape: Optional[tuple] = None, device: Optional[torch.device] = None) -> None:
    """Raises ValueError unless `t` is a tensor of `dtype` on `device` holding
    at least `min_numel` elements, or exactly `shape`.  The C ABI receives bare
    pointers, so sizes it reads past cannot be checked below this point."""
    if not isinstance(t, torch.Tensor):
        raise ValueError("%s must be a torch tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError("%s holds %d elements, needs at least %d" % (name, t.numel(), min_numel))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the batch on %s" % (name, t.device, device))


def _spec_field(s, name, default=None):
    v = getattr(s, name, default)
    return v if v is not None else default


def state_cols(spec) -> int:
    """fp32 optimizer state values per row: dim (Adagrad), 1 (row-wise Adagrad), 0 (SGD)."""
    opt = _spec_field(spec, "opt", "sgd")
    return int(spec.dim) if opt == "adagrad" else (1 if opt == "rowwise_adagrad" else 0)


class EmbeddingLayer:
    """Multi-table embedding layer resident on the current CUDA device.

    ``tables``: sequence of objects with ``rows, dim`` and optionally
    ``dtype`` ("f32"/"f16"/"bf16"), ``pooling`` ("sum"/"mean"), ``opt``
    ("sgd"/"adagrad"/"rowwise_adagrad"), ``lr``, ``eps``, ``init_acc``,
    ``master`` (keep an fp32 master copy of a 16-bit table), ``dynamic``
    (arbitrary int64 keys mapped to rows by a hash map of ``rows`` slots).
    """

    def __init__(self, tables: Sequence, max_batch: int, max_nnz: int):
        self.tables = list(tables)
        T = len(self.tables)
        arr = (EmbTableSpec * T)()
        for i, s in enumerate(self.tables):
            arr[i].rows = int(s.rows)
            arr[i].dim = int(s.dim)
            arr[i].dtype = DTYPES[_spec_field(s, "dtype", "f32")]
            arr[i].pooling = POOLINGS[_spec_field(s, "pooling", "sum")]
            arr[i].opt = OPTS[_spec_field(s, "opt", "sgd")]
            arr[i].lr = float(_spec_field(s, "lr", 0.01))
            arr[i].eps = float(_spec_field(s, "eps", 1e-8))
            arr[i].init_acc = float(_spec_field(s, "init_acc", 0.0))
            arr[i].master_fp32 = 1 if _spec_field(s, "master", False) else 0
            arr[i].dynamic = 1 if _spec_field(s, "dynamic", False) else 0
        h = ctypes.c_void_p()
        check(lib.emb_create(arr, T, int(max_batch), int(max_nnz), ctypes.byref(h)), "emb_create")
        self._h = h
        self.max_batch = int(max_batch)
        self.max_nnz = int(max_nnz)
        self.total_dim = sum(int(s.dim) for s in self.tables)
        self.doff = np.concatenate([[0], np.cumsum([int(s.dim) for s in self.tables])[:-1]]).astype(np.int64)
        self.row_base = np.concatenate([[0], np.cumsum([int(s.rows) for s in self.tables])[:-1]]).astype(np.int64)
        self.last_nnz = 0
        self.last_batch = None   # batch of the last training forward (None: no forward yet)

    # -- life cycle ---------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "_h", None):
            lib.emb_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- step ---------------------------------------------------------------
    def init_uniform(self, seed: int, lo: float, hi: float, stream=None) -> None:
        check(lib.emb_init_uniform(self._h, ctypes.c_uint64(seed & (2 ** 64 - 1)), lo, hi, _stream(stream)),
              "emb_init_uniform")

    def _check_batch(self, keys, offsets, table_ids, batch, out):
        batch = int(batch)
        bags = len(self.tables) * batch
        dev = offsets.device if isinstance(offsets, torch.Tensor) else None
        _check(keys, "keys", torch.int64, device=dev)
        _check(offsets, "offsets", torch.int64, min_numel=bags + 1)
        _check(table_ids, "table_ids", torch.int32, min_numel=bags, device=dev)
        if out is None:
            out = torch.empty((batch, self.total_dim), dtype=torch.float32, device=dev)
        _check(out, "out", torch.float32, shape=(batch, self.total_dim), device=dev)
        return batch, out

    def forward(self, keys: torch.Tensor, offsets: torch.Tensor, table_ids: torch.Tensor, batch: int,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        batch, out = self._check_batch(keys, offsets, table_ids, batch, out)
        nnz = int(keys.numel())
        check(lib.emb_forward(self._h, _ptr(keys) if nnz else None, _ptr(offsets), _ptr(table_ids), nnz,
                              batch, _ptr(out), _stream(stream)), "emb_forward")
        self.last_nnz = nnz
        self.last_batch = batch
        return out

    def backward_update(self, grad_out: torch.Tensor, variant: str = "reduction", stream=None) -> None:
        """grad_out: fp32 [batch, sum(dim)] of the last forward (extra rows are not read)."""
        if variant not in VARIANTS:
            raise ValueError("unknown backward variant %r" % (variant,))
        _check(grad_out, "grad_out", torch.float32)
        if self.last_batch is not None:   # before any forward the library reports the state error itself
            if grad_out.dim() != 2 or grad_out.shape[1] != self.total_dim or grad_out.shape[0] < self.last_batch:
                raise ValueError("grad_out must be [>= %d, %d], got %s"
                                 % (self.last_batch, self.total_dim, tuple(grad_out.shape)))
        check(lib.emb_backward_update(self._h, _ptr(grad_out), VARIANTS[variant], _stream(stream)),
              "emb_backward_update")

    # -- dedup by-products ----------------------------------------------------
    def set_keep_dedup(self, keep: bool) -> None:
        check(lib.emb_set_keep_dedup(self._h, 1 if keep else 0))

    def set_early_dedup(self, variant: Optional[str]) -> None:
        """Run the given backward variant's dedup inside forward(), on the
        layer's own stream, overlapping the pooling kernel (None: off)."""
        check(lib.emb_set_early_dedup(self._h, -1 if variant is None else VARIANTS[variant]), "emb_set_early_dedup")

    def dedup_result(self, with_inverse: bool = True, stream=None):
        """(unique int64[U], inverse int32[nnz] or None, counts int32[U],
        seg_offsets int32[U+1], sorted_bags int32[nnz]) of the last backward."""
        n = max(self.last_nnz, 1)
        dev = torch.device("cuda", torch.cuda.current_device())
        uniq = torch.empty(n, dtype=torch.int64, device=dev)
        inv = torch.empty(n, dtype=torch.int32, device=dev) if with_inverse else None
        cnt = torch.empty(n, dtype=torch.int32, device=dev)
        seg = torch.empty(n + 1, dtype=torch.int32, device=dev)
        bags = torch.empty(n, dtype=torch.int32, device=dev)
        U = ctypes.c_int64()
        check(lib.emb_dedup_result(self._h, _ptr(uniq), _ptr(inv), _ptr(cnt), _ptr(seg), _ptr(bags),
                                   ctypes.byref(U), _stream(stream)), "emb_dedup_result")
        u = U.value
        m = self.last_nnz
        return (uniq[:u], None if inv is None else inv[:m], cnt[:u], seg[:u + 1], bags[:m])

    # -- rows -----------------------------------------------------------------
    # State arrays have state_cols(spec) columns: dim (Adagrad), 1 (row-wise
    # Adagrad); SGD tables have none.
    def gather_rows(self, t: int, rows: torch.Tensor, with_state: bool = False, stream=None):
        _check(rows, "rows", torch.int64)
        spec = self.tables[t]
        dt = _spec_field(spec, "dtype", "f32")
        n = int(rows.numel())
        w = torch.empty((n, int(spec.dim)), dtype=_TORCH_WDTYPE[dt], device=rows.device)
        s = torch.empty((n, state_cols(spec)), dtype=torch.float32, device=rows.device) if with_state else None
        check(lib.emb_gather_rows(self._h, t, _ptr(rows), n, _ptr(w), _ptr(s), _stream(stream)), "emb_gather_rows")
        return w, s

    def get_rows(self, t: int, row0: int, n: int, with_state: bool = False, stream=None):
        spec = self.tables[t]
        dt = _spec_field(spec, "dtype", "f32")
        w = np.empty((n, int(spec.dim)), dtype=_NP_WDTYPE[dt])
        s = np.empty((n, state_cols(spec)), dtype=np.float32) if with_state else None
        check(lib.emb_get_rows(self._h, t, row0, n, w.ctypes.data_as(ctypes.c_void_p),
                               None if s is None else s.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
              "emb_get_rows")
        return w, s

    def set_rows(self, t: int, row0: int, weights: np.ndarray, state: Optional[np.ndarray] = None, stream=None):
        spec = self.tables[t]
        dt = _spec_field(spec, "dtype", "f32")
        w = np.ascontiguousarray(weights, dtype=_NP_WDTYPE[dt])
        s = None if state is None else np.ascontiguousarray(state, dtype=np.float32)
        if s is not None and s.size != w.shape[0] * state_cols(spec):
            raise ValueError("state must hold %d values per row" % state_cols(spec))
        check(lib.emb_set_rows(self._h, t, row0, w.shape[0], w.ctypes.data_as(ctypes.c_void_p),
                               None if s is None else s.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
              "emb_set_rows")

    # -- inference ------------------------------------------------------------------
    def cache_build(self, t: int, rows: torch.Tensor, stream=None) -> None:
        """fp16 inference cache of the given rows (int64, device) of table t (empty: none)."""
        _check(rows, "rows", torch.int64)
        n = int(rows.numel())
        check(lib.emb_cache_build(self._h, t, _ptr(rows) if n else None, n, _stream(stream)), "emb_cache_build")

    def forward_infer(self, keys: torch.Tensor, offsets: torch.Tensor, table_ids: torch.Tensor, batch: int,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """Pooled output reading cached rows from the fp16 caches; keeps nothing for a backward."""
        batch, out = self._check_batch(keys, offsets, table_ids, batch, out)
        nnz = int(keys.numel())
        check(lib.emb_forward_infer(self._h, _ptr(keys) if nnz else None, _ptr(offsets), _ptr(table_ids), nnz,
                                    batch, _ptr(out), _stream(stream)), "emb_forward_infer")
        return out

    # -- dynamic tables -----------------------------------------------------------
    def find_keys(self, t: int, keys: torch.Tensor, stream=None) -> torch.Tensor:
        """Rows (int64, -1 when absent) of int64 keys of dynamic table t; inserts nothing."""
        _check(keys, "keys", torch.int64)
        out = torch.empty(int(keys.numel()), dtype=torch.int64, device=keys.device)
        check(lib.emb_find_keys(self._h, t, _ptr(keys), int(keys.numel()), _ptr(out), _stream(stream)),
              "emb_find_keys")
        return out

    # -- fp32 master copies of 16-bit tables ------------------------------------
    def gather_master_rows(self, t: int, rows: torch.Tensor, stream=None) -> torch.Tensor:
        _check(rows, "rows", torch.int64)
        spec = self.tables[t]
        n = int(rows.numel())
        m = torch.empty((n, int(spec.dim)), dtype=torch.float32, device=rows.device)
        check(lib.emb_gather_master_rows(self._h, t, _ptr(rows), n, _ptr(m), _stream(stream)),
              "emb_gather_master_rows")
        return m

    def get_master_rows(self, t: int, row0: int, n: int, stream=None) -> np.ndarray:
        m = np.empty((n, int(self.tables[t].dim)), dtype=np.float32)
        check(lib.emb_get_master_rows(self._h, t, row0, n, m.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
              "emb_get_master_rows")
        return m

    def set_master_rows(self, t: int, row0: int, master: np.ndarray, stream=None) -> None:
        m = np.ascontiguousarray(master, dtype=np.float32).reshape(-1, int(self.tables[t].dim))
        check(lib.emb_set_master_rows(self._h, t, row0, m.shape[0], m.ctypes.data_as(ctypes.c_void_p),
                                      _stream(stream)), "emb_set_master_rows")

    # -- status ---------------------------------------------------------------
    def sync_status(self, stream=None) -> int:
        """Waits for the stream; returns and clears the sticky device status."""
        return int(lib.emb_sync_status(self._h, _stream(stream)))

    def set_timing(self, enable: bool) -> None:
        check(lib.emb_set_timing(self._h, 1 if enable else 0), "emb_set_timing")

    def phase_times(self, reset: bool = False):
        """({phase: accumulated ms}, steps) of the steps timed since the last reset."""
        arr = (ctypes.c_float * len(PHASES))()
        steps = ctypes.c_int64()
        check(lib.emb_phase_times(self._h, arr, len(PHASES), ctypes.byref(steps), 1 if reset else 0))
        return {p: float(arr[i]) for i, p in enumerate(PHASES)}, steps.value

    def launch_count(self, reset: bool = False) -> int:
        c = ctypes.c_int64()
        check(lib.emb_launch_count(self._h, ctypes.byref(c), 1 if reset else 0))
        return c.value


def unique_workspace_bytes(n: int) -> int:
    b = ctypes.c_size_t()
    check(lib.emb_unique_workspace(int(n), ctypes.byref(b)), "emb_unique_workspace")
    return b.value


def unique(keys: torch.Tensor, stream=None):
    """Sorted unique keys, inverse index, counts and segment offsets of int64 keys.

    Returns (unique[:U], inverse, counts[:U], seg_offsets[:U+1]); U is read
    back to the host (one synchronisation)."""
    _check(keys, "keys", torch.int64)
    n = int(keys.numel())
    dev = keys.device
    m = max(n, 1)
    uniq = torch.empty(m, dtype=torch.int64, device=dev)
    inv = torch.empty(m, dtype=torch.int32, device=dev)
    cnt = torch.empty(m, dtype=torch.int32, device=dev)
    seg = torch.empty(m + 1, dtype=torch.int32, device=dev)
    nu = torch.empty(1, dtype=torch.int64, device=dev)
    ws_bytes = unique_workspace_bytes(n)
    ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
    base = ws.data_ptr()
    aligned = (base + 255) & ~255
    check(lib.emb_unique(_ptr(keys) if n else None, n, _ptr(uniq), _ptr(inv), _ptr(cnt), _ptr(seg), _ptr(nu),
                         ctypes.c_void_p(aligned), ws_bytes, _stream(stream)), "emb_unique")
    U = int(nu.item())
    return uniq[:U], inv[:n], cnt[:U], seg[:U + 1]
