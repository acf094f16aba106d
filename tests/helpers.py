"""Shared test utilities: run the CUDA path and the oracle on the same seeded
inputs and compare them.

Float tolerance.  Results are judged by the maximum relative error
    |gpu - ref| / max(|ref|, A / 32)
where ref is the oracle's binary64 result rounded once to the stored type and
A is the sum of the magnitudes of the terms that form the element (for a
pooled output s_j * sum |W|; for an updated weight |W| + lr * sum |g| scaled
like the step; for an Adagrad accumulator A + (sum |g|)^2).  The bound is
1e-5 for fp32 storage and 1e-2 for fp16/bf16 storage.  Any fp32 evaluation
rounds intermediates as large as A a few times, each by up to 2^-24 * A, so
an element that cancels to below A/32 is held to an absolute error of
1e-5 * A/32 (about 5 fp32 ulps of A) instead of a relative one.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

import ctr_inputs as ci

FLOOR = 2.0 ** -5
TOL = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2}


def max_rel_err(got, ref, scale) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    if got.size == 0:
        return 0.0
    den = np.maximum(np.abs(ref), FLOOR * scale)
    diff = np.abs(got - ref)
    exact = den == 0
    if np.any(diff[exact] != 0):
        return float("inf")
    den = np.where(exact, 1.0, den)
    return float(np.max(diff / den))


def plain_rel_err(got, ref, rms_frac: float = 1e-3) -> float:
    """Plain maximum relative error |gpu - ref| / |ref| over the elements with
    |ref| >= rms_frac * rms(ref): the companion of max_rel_err that no floor
    softens, reported beside it.  0 when no element qualifies."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    sel = np.abs(ref) >= rms_frac * rms
    sel &= ref != 0
    if not np.any(sel):
        return 0.0
    return float(np.max(np.abs(got[sel] - ref[sel]) / np.abs(ref[sel])))


# (case, quantity, plain max relative error) of every GPU parity comparison in
# this session; conftest prints them at the end of the run
PLAIN_REPORT = []


def report_plain(case: str, quantity: str, got, ref) -> float:
    v = plain_rel_err(got, ref)
    PLAIN_REPORT.append((case, quantity, v))
    return v


def init_rows_fn(w: ci.Workload, seed: int):
    return lambda t, r: ci.init_values(seed, t, r, w.tables[t].dim, w.w_lo, w.w_hi, w.tables[t].dtype)


def to_f64(t, dtype: str) -> np.ndarray:
    """Stored table values (torch tensor of the table dtype) to float64."""
    import torch
    if dtype == "f32":
        return t.double().cpu().numpy()
    return t.float().double().cpu().numpy()   # fp16/bf16 -> fp32 is exact


@dataclasses.dataclass
class GpuStep:
    out: np.ndarray
    status_fwd: int
    status_bwd: int
    unique: np.ndarray
    inverse: Optional[np.ndarray]
    counts: np.ndarray
    seg_off: np.ndarray
    sorted_bags: np.ndarray
    layer: object


def run_gpu_step(w: ci.Workload, batch: ci.Batch, grad: np.ndarray, variant: str, seed: int = 0,
                 keep_layer: bool = False, max_nnz: Optional[int] = None, early: bool = False) -> GpuStep:
    """One step through the C ABI.  early: the dedup of `variant` runs inside
    the forward, on the layer's second stream."""
    import torch
    from dlrm_sparse_embedding_gb300 import EmbeddingLayer
    dev = torch.device("cuda", 0)
    layer = EmbeddingLayer(w.tables, w.batch, max(batch.nnz, 1) if max_nnz is None else max_nnz)
    layer.init_uniform(seed, w.w_lo, w.w_hi)
    # the dedup by-products are kept from the start: with early dedup the
    # forward already runs the dedup
    layer.set_keep_dedup(True)
    if early:
        layer.set_early_dedup(variant)
    keys = torch.from_numpy(batch.keys).to(dev)
    offsets = torch.from_numpy(batch.offsets).to(dev)
    tids = torch.from_numpy(batch.table_ids).to(dev)
    g = torch.from_numpy(grad).to(dev)
    out = layer.forward(keys, offsets, tids, batch.batch)
    st_f = layer.sync_status()
    out_np = out.cpu().numpy()
    layer.backward_update(g, variant)
    st_b = layer.sync_status()
    u, inv, cnt, seg, bags = layer.dedup_result(with_inverse=variant != "reduction")
    res = GpuStep(out_np, st_f, st_b, u.cpu().numpy(), None if inv is None else inv.cpu().numpy(),
                  cnt.cpu().numpy(), seg.cpu().numpy(), bags.cpu().numpy(), layer if keep_layer else None)
    if not keep_layer:
        layer.close()
    return res


def gather_rows(layer, w: ci.Workload, t: int, rows: np.ndarray):
    import torch
    spec = w.tables[t]
    r = torch.from_numpy(np.ascontiguousarray(rows, dtype=np.int64)).cuda()
    W, A = layer.gather_rows(t, r, with_state=spec.opt != "sgd")
    return to_f64(W, spec.dtype), None if A is None else A.double().cpu().numpy()


def expected_sorted_bags(gids: np.ndarray, bag_of_pos: np.ndarray) -> np.ndarray:
    valid = gids >= 0
    pos = np.nonzero(valid)[0]
    order = np.argsort(gids[pos], kind="stable")
    return bag_of_pos[pos[order]].astype(np.int32)


def bag_of_positions(offsets: np.ndarray) -> np.ndarray:
    lens = np.diff(offsets)
    return np.repeat(np.arange(lens.size, dtype=np.int64), lens)


def ref_state(spec, A: np.ndarray, A_scale: np.ndarray, idx: np.ndarray):
    """The oracle's accumulators (and scales) for the rows whose element
    indices are `idx` [n, dim], shaped like the layer's state: [n, dim] for
    Adagrad, [n, 1] for row-wise Adagrad (the oracle repeats the row's value
    in every column)."""
    if spec.opt == "rowwise_adagrad":
        return A[idx[:, :1]], A_scale[idx[:, :1]]
    return A[idx], A_scale[idx]
