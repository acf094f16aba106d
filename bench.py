"""Benchmark of one sparse-embedding training step on GB300.

A step is the whole hot path over one synthetic batch: forward lookup +
pooling + concatenation, backward dedup, segmented gradient reduction and the
optimizer update (emb_forward + emb_backward_update through the C ABI).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config multihot]
                    [--variant reduction|unique_sort|unique_hash] [--impl ours|reference]

Default workload: the multi-hot configuration (100 fp32 tables x 1e6 rows x
dim 64, batch 16,384, per-table hotness U[1,100], Zipf(1.2) keys, mean pooling,
Adagrad), the largest of the stated workloads in the bytes a step must move.
Its tables (25.6 GB plus 25.6 GB of Adagrad state) and its per-step tensors
(keys 0.6 GB, out and grad_out 0.42 GB each) are larger than L2, so no L2
flush is needed between steps.

Two timed regions of K steps each: the headline one with the library's phase
timing off, then one with it on (CUDA events around each phase, recorded on
the stream that runs it, read back only after the region) for the phase
breakdown and the roofline of the dominant phase.

--impl reference times the CPU oracle (test infrastructure, single-threaded C)
on a bounded sample of the same workload; it is a reported baseline only.
Under torchrun every rank runs a full replica (the path has no exchange step);
rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import ctr_inputs as ci  # noqa: E402

METRIC = "embedding lookups/sec (fwd+bwd+update) on 1 GB300; achieved HBM GB/s vs peak"
CONFIG_TEXT = {
    "tiny": "tiny: 4 fp32 tables x 1,000 rows x dim 16, batch 256, hotness U[1,4], uniform keys, sum, SGD",
    "dlrm": ("DLRM-style one-hot: 26 fp32 tables, rows log-uniform in [1e3,1e7], dim 128, batch 65,536, "
             "hotness 1, Zipf(1.05) keys, sum pooling, Adagrad lr=0.01 eps=1e-8"),
    "multihot": ("multi-hot: 100 fp32 tables x 1e6 rows x dim 64, batch 16,384, per-table hotness U[1,100], "
                 "Zipf(1.2), mean pooling, Adagrad"),
    "huge": ("single huge table: 1 fp16 table x 2e8 rows x dim 64, fp32 Adagrad state, batch 131,072, "
             "hotness 20, Zipf(1.1), sum pooling"),
    "huge_master": ("single huge table with an fp32 master copy: 1 fp16 table x 2e8 rows x dim 64 plus fp32 master "
                    "and fp32 Adagrad state, batch 131,072, hotness 20, Zipf(1.1), sum pooling"),
    "dlrm_dynamic": ("DLRM-style one-hot with dynamic tables: 26 fp32 tables of int64 ids (scrambled Zipf(1.05) "
                     "ranks, key spaces log-uniform in [1e3,1e7]) behind GPU hash maps of twice that many rows, "
                     "dim 128, batch 65,536, hotness 1, sum pooling, Adagrad"),
    "dlrm_rowwise": ("DLRM-style one-hot with row-wise Adagrad: 26 fp32 tables, rows log-uniform in [1e3,1e7], "
                     "dim 128, batch 65,536, hotness 1, Zipf(1.05) keys, sum pooling, one fp32 accumulator per row"),
    "skew": ("skewed dedup stress: 8 fp32 tables dims {16,32,64,128}x2 x 5e6 rows, batch 262,144, hotness 50, "
             "Zipf(1.5), sum pooling, SGD"),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _wbytes(dtype: str) -> int:
    return 4 if dtype == "f32" else 2


def _per_table_bytes(w: ci.Workload, U_per_table: np.ndarray):
    """Touched-row bytes of the step: rows in their storage type, optimizer
    state, and what an fp32 master copy adds to the update."""
    rows_bytes = sum(int(U_per_table[t]) * s.dim * _wbytes(s.dtype) for t, s in enumerate(w.tables))
    # an fp32 master copy: the update reads and writes the master (8 B) and
    # writes the stored row, instead of reading and writing the stored row
    master_bytes = sum(int(U_per_table[t]) * s.dim * (8 - _wbytes(s.dtype))
                       for t, s in enumerate(w.tables) if getattr(s, "master", False))
    state_cols = {"sgd": 0, "adagrad": None, "rowwise_adagrad": 1}
    state_bytes = sum(int(U_per_table[t]) * 4 * (s.dim if state_cols[s.opt] is None else state_cols[s.opt])
                      for t, s in enumerate(w.tables))
    return rows_bytes, master_bytes, state_bytes


def algorithmic_bytes(w: ci.Workload, batch: ci.Batch, U_per_table: np.ndarray) -> dict:
    """Compulsory bytes of each phase: what the method must move through HBM
    at least once, whatever the implementation.

    forward: keys (8 nnz) + offsets (8 (T B + 1)) + every touched row once +
    the pooled output (4 B sum(dim)); dedup: keys in (8 nnz), unique ids (8 U),
    inverse (4 nnz) and counts (4 U) out; reduce+update: grad_out once
    (4 B sum(dim)), one position per lookup (4 nnz), and every touched row
    and its optimizer state read and written once.  Dynamic tables add, per
    lookup, the key's map slot read and its resolved row written and read
    back (24 B)."""
    T, B, nnz = w.num_tables, w.batch, batch.nnz
    D = w.total_dim
    U = int(np.sum(U_per_table))
    rows_bytes, master_bytes, state_bytes = _per_table_bytes(w, U_per_table)
    fwd = 8 * nnz + 8 * (T * B + 1) + rows_bytes + 4 * B * D
    dyn_lookups = sum(int(batch.offsets[(t + 1) * B] - batch.offsets[t * B])
                      for t, s in enumerate(w.tables) if getattr(s, "dynamic", False))
    fwd += 24 * dyn_lookups
    dedup = 8 * nnz + 8 * U + 4 * nnz + 4 * U
    upd = 4 * B * D + 4 * nnz + 2 * rows_bytes + 2 * state_bytes + master_bytes
    return {"forward": fwd, "dedup": dedup, "reduce_update": upd, "step": fwd + dedup + upd}


def implementation_bytes(w: ci.Workload, batch: ci.Batch, U_per_table: np.ndarray, sort_passes: int) -> dict:
    """Bytes this implementation moves through HBM by design (each array
    touched once per pass, no L2 re-reads counted), next to the compulsory
    bytes: the forward also reads the table ids and writes a 32-bit global id
    and bag per lookup; the reduction-based dedup sorts those (id, bag) pairs
    (per pass: the histogram reads the ids, the ranking reads and writes both
    arrays); the reduction reads the sorted ids and bags."""
    T, B, nnz = w.num_tables, w.batch, batch.nnz
    D = w.total_dim
    rows_bytes, master_bytes, state_bytes = _per_table_bytes(w, U_per_table)
    comp = algorithmic_bytes(w, batch, U_per_table)
    fwd = comp["forward"] + 4 * T * B + 8 * nnz
    dedup = sort_passes * (4 * nnz + 16 * nnz)
    upd = 4 * B * D + 8 * nnz + 2 * rows_bytes + 2 * state_bytes + master_bytes
    return {"forward": fwd, "dedup": dedup, "reduce_update": upd, "step": fwd + dedup + upd}


def logical_row_bytes(w: ci.Workload, batch: ci.Batch) -> int:
    """Row bytes the forward reads when every lookup reads its row (one read
    per lookup): under skewed keys most of them are served by L2."""
    B = w.batch
    return sum(int(batch.offsets[(t + 1) * B] - batch.offsets[t * B]) * s.dim * _wbytes(s.dtype)
               for t, s in enumerate(w.tables))


def _bits_for(v: int) -> int:
    b = 1
    while b < 64 and (v >> b) != 0:
        b += 1
    return b


def table_sort_bits(rows_max: int) -> int:
    """Bits of the dedup sort's table-local keys: every row id of the largest
    table plus an all-ones key for skipped lookups in a top digit of its own
    (digits of at most 10 bits, passes balanced)."""
    b = _bits_for(rows_max)
    while True:
        passes = -(-b // 10)
        D = -(-b // passes)
        top_shift = (passes - 1) * D
        if ((rows_max - 1) >> top_shift) < (((1 << b) - 1) >> top_shift):
            return b
        b += 1


def sort_passes(w: ci.Workload, variant: str) -> int:
    """Radix-sort passes over the lookups in the dedup: the reduction-based and
    the sort-based variants sort each table's lookups on their table-local row
    id; the hash-based one sorts them on the unique index (at most the lookups
    or the rows, whichever is fewer)."""
    if variant == "unique_hash":
        total_rows = sum(s.rows for s in w.tables)
        return -(-_bits_for(total_rows) // 10)
    return -(-table_sort_bits(max(s.rows for s in w.tables)) // 10)


def recorded_traffic(config: str, variant: str, phase: str, root: str = ROOT):
    """DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) of one
    full-size launch of `phase`'s kernels, from
    profiles/traffic_<config>_<variant>.json -- or None when there is no
    record, or when any source file the record names no longer hashes to its
    recorded SHA-256 (the kernels changed since the counters were taken)."""
    import hashlib
    tpath = os.path.join(root, "profiles", "traffic_%s_%s.json" % (config, variant))
    try:
        with open(tpath) as f:
            rec = json.load(f).get(phase)
        if not rec or not rec.get("sources_sha256"):
            return None
        for src, sha in rec["sources_sha256"].items():
            with open(os.path.join(root, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != sha:
                    return None
        return int(rec["traffic_bytes"])
    except (OSError, ValueError, KeyError, TypeError):
        return None


def unique_per_table(w: ci.Workload, batch: ci.Batch) -> np.ndarray:
    B = w.batch
    U = np.zeros(w.num_tables, dtype=np.int64)
    for t in range(w.num_tables):
        k = batch.keys[batch.offsets[t * B]:batch.offsets[(t + 1) * B]]
        U[t] = np.unique(k).size
    return U


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.idx = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # the timed region starts once the sampler is producing samples
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def max_over_ranks(value: float, device) -> float:
    """Largest value over all ranks (each rank times its own replica)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world_size: int, ms_per_step_max: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return world_size * units_per_rank / (ms_per_step_max / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def oracle_step_timed(w: ci.Workload, batch: ci.Batch, grad: np.ndarray, seed: int) -> float:
    """Seconds the CPU oracle takes for a1..a5 on `batch` (initial rows prepared untimed)."""
    import oracle
    if any(getattr(s, "dynamic", False) for s in w.tables):
        # dynamic tables: the oracle relabels keys to rows and prepares the rows inside the timed step
        t0 = time.perf_counter()
        oracle.step_dynamic(
            w.tables, w.batch, batch.offsets, batch.keys, batch.table_ids, grad,
            lambda t, r: ci.init_values(seed, t, r, w.tables[t].dim, w.w_lo, w.w_hi, w.tables[t].dtype),
            lambda t, k: ci.init_values_dynamic(seed, t, k, w.tables[t].dim, w.w_lo, w.w_hi, w.tables[t].dtype))
        return time.perf_counter() - t0
    gids, _ = oracle.global_ids(w.tables, w.batch, batch.offsets, batch.keys, batch.table_ids)
    u, inv, _, _ = oracle.unique(gids, skip_negative=True)
    rows = oracle.make_row_store(w.tables, u, lambda t, r: ci.init_values(
        seed, t, r, w.tables[t].dim, w.w_lo, w.w_hi, w.tables[t].dtype))
    state = oracle.make_row_store(w.tables, u, None, state_init=True)
    t0 = time.perf_counter()
    gids, _ = oracle.global_ids(w.tables, w.batch, batch.offsets, batch.keys, batch.table_ids)
    u, inv, _, _ = oracle.unique(gids, skip_negative=True)
    oracle.forward(w.tables, w.batch, batch.offsets, inv, rows)
    G, Gabs = oracle.reduce(w.tables, w.batch, batch.offsets, inv, rows, grad)
    oracle.update(w.tables, rows, state, G, None)
    return time.perf_counter() - t0


def lookups_per_sample(w: ci.Workload) -> float:
    """Mean lookups of one sample (one bag per table) under the workload's hotness law."""
    h = w.replace(batch=min(w.batch, 4096)).hotness()
    return float(h.sum()) / h.shape[1]


def cpu_sample_batch(w: ci.Workload, target_lookups: int) -> int:
    """Samples whose lookups come to about target_lookups (at least one, at most the batch)."""
    n = int(round(target_lookups / max(lookups_per_sample(w), 1.0)))
    return max(1, min(w.batch, n))


def cpu_sample(w: ci.Workload, sample_batch: int):
    ws = w.replace(batch=sample_batch)
    b = ci.make_batch(ws)
    g = ci.make_grad(ws)
    return ws, b, g


def run_reference(args, w: ci.Workload):
    ws_, rank, _ = _dist()
    if rank != 0:
        return
    sb_n = cpu_sample_batch(w, args.cpu_sample_lookups)
    sw, sb, sg = cpu_sample(w, sb_n)
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle_step_timed(sw, sb, sg, w.seed)
    secs = [oracle_step_timed(sw, sb, sg, w.seed) for _ in range(args.steps)]
    per = sum(secs) / len(secs)
    v = sb.nnz / per
    sample = "%d of the %d samples (%d lookups) per step, full step a1..a5, %d timed steps" % (
        sb_n, w.batch, sb.nnz, args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "lookups/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": CONFIG_TEXT[args.config], "batch": sb_n, "nnz": int(sb.nnz),
                                        "sample_of_batch": w.batch,
                                        "variant": "definition (no dedup variant)"},
        "cpu_baseline": {"value": v, "unit": "lookups/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "lookups/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="multihot", choices=sorted(CONFIG_TEXT))
    ap.add_argument("--variant", default="reduction", choices=["reduction", "unique_sort", "unique_hash"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batches", type=int, default=2, help="distinct seeded batches cycled through")
    ap.add_argument("--cpu-sample-lookups", type=int, default=400000,
                    help="lookups in the oracle's sample of the workload (CPU baseline and reference arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--early-dedup", action="store_true",
                    help="run the dedup inside the forward on the layer's second stream (overlap)")
    ap.add_argument("--infer", action="store_true",
                    help="also time the inference-only forward with fp16 caches of each table's hottest rows")
    ap.add_argument("--cache-frac", type=float, default=0.01,
                    help="share of each static table's rows (the hottest ranks) held in its inference cache")
    ap.add_argument("--batch", type=int, default=0, help="override the batch size (small profiling cases)")
    ap.add_argument("--rows-cap", type=int, default=0, help="cap every table's rows (small profiling cases)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    w = ci.workload(args.config)
    if args.batch:
        w = w.replace(batch=args.batch)
    if args.rows_cap:
        w = w.replace(tables=tuple(dataclasses.replace(t, rows=min(t.rows, args.rows_cap)) for t in w.tables))

    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    if ws > 1:
        dist.barrier(device_ids=[local])
    from dlrm_sparse_embedding_gb300 import EMB_OK, EmbeddingLayer

    # inputs: a few seeded batches of the same workload, one grad_out
    batches = [ci.make_batch(w, seed=w.seed + i) for i in range(args.batches)]
    grad = ci.make_grad(w)
    max_nnz = max(b.nnz for b in batches)
    U_t = unique_per_table(w, batches[0])
    bytes_ = algorithmic_bytes(w, batches[0], U_t)

    dkeys = [torch.from_numpy(b.keys).to(dev) for b in batches]
    doffs = [torch.from_numpy(b.offsets).to(dev) for b in batches]
    dtids = [torch.from_numpy(b.table_ids).to(dev) for b in batches]
    dgrad = torch.from_numpy(grad).to(dev)
    out = torch.empty((w.batch, w.total_dim), dtype=torch.float32, device=dev)

    layer = EmbeddingLayer(w.tables, w.batch, max_nnz)
    layer.init_uniform(w.seed, w.w_lo, w.w_hi)
    if args.early_dedup:
        layer.set_early_dedup(args.variant)

    def step(i):
        k = i % args.batches
        layer.forward(dkeys[k], doffs[k], dtids[k], w.batch, out)
        layer.backward_update(dgrad, args.variant)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    status = layer.sync_status()
    if status != EMB_OK:
        raise SystemExit("device status %d after warm-up" % status)

    def timed_region(timing: bool):
        """Milliseconds per step over K steps (max over ranks), launches, and
        with timing on the per-phase totals of the library's CUDA events."""
        layer.set_timing(timing)
        layer.phase_times(reset=True)
        layer.launch_count(reset=True)
        if ws > 1:
            dist.barrier(device_ids=[local])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(args.steps):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier(device_ids=[local])
        ms_ = e0.elapsed_time(e1) / args.steps
        launches_ = layer.launch_count(reset=True)
        phases_, nsteps_ = layer.phase_times(reset=True)
        layer.set_timing(False)
        return max_over_ranks(ms_, dev), launches_, phases_, nsteps_

    # ---- device-resident timed regions: headline (phase timing off), then phases ----
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    ms, launches, _, _ = timed_region(False)
    ms_phased, _, phases, nsteps = timed_region(True)
    clk = clocks.stop() if rank == 0 else None
    status = layer.sync_status()

    # ---- inference-only forward with fp16 hot-row caches (optional) ----
    infer = None
    if args.infer:
        cached_rows = 0
        for t, s_ in enumerate(w.tables):
            if getattr(s_, "dynamic", False):
                continue
            n_c = max(1, int(s_.rows * args.cache_frac))        # Zipf rank 0 is the hottest row
            layer.cache_build(t, torch.arange(n_c, dtype=torch.int64, device=dev))
            cached_rows += n_c
        for i in range(args.warmup):
            layer.forward_infer(dkeys[i % args.batches], doffs[i % args.batches], dtids[i % args.batches], w.batch, out)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record()
        for i in range(args.steps):
            k_ = i % args.batches
            layer.forward_infer(dkeys[k_], doffs[k_], dtids[k_], w.batch, out)
        f1.record()
        torch.cuda.synchronize()
        ims = max_over_ranks(f0.elapsed_time(f1) / args.steps, dev)
        # compulsory bytes: keys, offsets, table ids, each touched row once, the output, a code per lookup
        ibytes = bytes_["forward"] - 8 * batches[0].nnz + 16 * batches[0].nnz
        infer = {"metric": "inference lookups/s (pooled forward, fp16 caches of the hottest rows)",
                 "value": whole_job_rate(batches[0].nnz, ws, ims), "unit": "lookups/s", "ms_per_step": ims,
                 "cache": "hottest %.2f%% of each static table's rows as fp16 (%d rows)" % (100 * args.cache_frac,
                                                                                          cached_rows),
                 "hbm": {"algorithmic_bytes": ibytes, "achieved_gbs": ibytes / (ims / 1e3) / 1e9},
                 "status": layer.sync_status()}

    # ---- end to end: host buffers, copies inside the timed region ----
    # Every step copies its inputs (keys, offsets, table ids, grad_out) from
    # pinned host memory and reads the pooled output back.  The copies run on
    # their own streams, double-buffered: while step i computes, the inputs of
    # step i+1 go up, and step i's output comes down as soon as its forward
    # is done.  The pipeline runs on from the warm-up into the timed steps, so
    # the timed region holds K uploads (those of the steps after the first
    # timed one, the first's having gone up during the last warm-up step) and
    # K downloads: the bytes of K steps, at the pipeline's steady rate.
    e2e = None
    if not args.no_e2e:
        hk = [torch.from_numpy(b.keys).pin_memory() for b in batches]
        ho = [torch.from_numpy(b.offsets).pin_memory() for b in batches]
        ht = [torch.from_numpy(b.table_ids).pin_memory() for b in batches]
        hg = torch.from_numpy(grad).pin_memory()
        hout = [torch.empty((w.batch, w.total_dim), dtype=torch.float32).pin_memory() for _ in range(2)]
        dbuf = [dict(k=torch.empty(max_nnz, dtype=torch.int64, device=dev), o=torch.empty_like(doffs[0]),
                     t=torch.empty_like(dtids[0]), g=torch.empty_like(dgrad),
                     out=torch.empty_like(out)) for _ in range(2)]
        comp = torch.cuda.current_stream()
        s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_fwd = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]

        def upload(i):
            b, k = i % 2, i % args.batches
            n = hk[k].numel()
            with torch.cuda.stream(s_up):
                s_up.wait_event(ev_comp[b])          # step i-2 is done with these buffers
                dbuf[b]["k"][:n].copy_(hk[k], non_blocking=True)
                dbuf[b]["o"].copy_(ho[k], non_blocking=True)
                dbuf[b]["t"].copy_(ht[k], non_blocking=True)
                dbuf[b]["g"].copy_(hg, non_blocking=True)
                ev_up[b].record(s_up)

        def e2e_step(i):
            b, k = i % 2, i % args.batches
            n = hk[k].numel()
            upload(i + 1)
            comp.wait_event(ev_up[b])
            comp.wait_event(ev_down[b])              # output buffer b has been read back
            layer.forward(dbuf[b]["k"][:n], dbuf[b]["o"], dbuf[b]["t"], w.batch, dbuf[b]["out"])
            ev_fwd[b].record(comp)
            layer.backward_update(dbuf[b]["g"], args.variant)
            ev_comp[b].record(comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_fwd[b])
                hout[b].copy_(dbuf[b]["out"], non_blocking=True)
                ev_down[b].record(s_down)

        # the host link's own rates on this machine, each way alone (best of 3
        # copies of grad_out up and of the output down): what the copies of a
        # step cost when nothing else runs
        def link_gbs(dst, src):
            best = float("inf")
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(comp)
                dst.copy_(src, non_blocking=True)
                e1.record(comp)
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1))
            return src.numel() * src.element_size() / (best * 1e6)

        h2d_gbs = link_gbs(dbuf[0]["g"], hg)
        d2h_gbs = link_gbs(hout[0], dbuf[0]["out"])
        upload(0)
        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier(device_ids=[local])
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(comp)
        for i in range(args.warmup, args.warmup + args.steps):
            e2e_step(i)
        comp.wait_stream(s_down)
        comp.wait_stream(s_up)
        f1.record(comp)
        torch.cuda.synchronize()
        ems = f0.elapsed_time(f1) / args.steps
        ems = max_over_ranks(ems, dev)
        h2d = batches[0].keys.nbytes + batches[0].offsets.nbytes + batches[0].table_ids.nbytes + grad.nbytes
        d2h = w.batch * w.total_dim * 4
        e2e = {"value": whole_job_rate(batches[0].nnz, ws, ems), "unit": "lookups/s", "ms_per_step": ems,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "copies": "pinned host <-> device, double-buffered on two copy streams overlapping compute; "
                         "steady state: K uploads and K downloads inside the K timed steps",
               "link_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs}}

    layer.close()
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return

    nnz = batches[0].nnz
    peak, peak_kind = _peaks()
    per_phase_ms = {p: phases[p] / max(nsteps, 1) for p in phases}
    dom = max(("forward", "dedup", "reduce_update"), key=lambda p: per_phase_ms[p])
    dom_kernel = {"forward": "fwd_pool", "dedup": "sort_upsweep+sort_scan+sort_downsweep (radix sort passes)",
                  "reduce_update": "reduce_update_chunks+combine"}[dom]
    dom_gbs = bytes_[dom] / (per_phase_ms[dom] / 1e3) / 1e9
    step_gbs = bytes_["step"] / (ms / 1e3) / 1e9
    impl = implementation_bytes(w, batches[0], U_t, sort_passes(w, args.variant))
    traffic = None if (args.batch or args.rows_cap) else recorded_traffic(args.config, args.variant, dom)

    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        sb_n = cpu_sample_batch(w, args.cpu_sample_lookups)
        sw, sb, sg = cpu_sample(w, sb_n)
        import oracle
        oracle.build()
        secs = []
        t_start = time.perf_counter()
        while not secs or (time.perf_counter() - t_start < 10.0 and len(secs) < 20):
            secs.append(oracle_step_timed(sw, sb, sg, w.seed))
        cpu = {"value": sb.nnz / (sum(secs) / len(secs)), "unit": "lookups/s", "cores": 1,
               "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": "%d of the %d samples (%d lookups), full step a1..a5, mean of %d runs" % (
                   sb_n, w.batch, sb.nnz, len(secs))}

    line = {
        "metric": METRIC,
        "value": whole_job_rate(nnz, ws, ms),
        "unit": "lookups/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if all(s.dtype == "f32" for s in w.tables) else "f32-accumulate/16-bit-storage",
        "data": "synthetic",
        "config": {"workload": CONFIG_TEXT[args.config] + (
                       " [batch overridden to %d]" % w.batch if args.batch else "") + (
                       " [rows capped at %d]" % args.rows_cap if args.rows_cap else ""),
                   "batch": w.batch, "nnz": nnz,
                   "unique_rows": int(U_t.sum()), "variant": args.variant, "batches_cycled": args.batches,
                   "dedup": "overlapped with the forward on the layer's second stream" if args.early_dedup
                            else "inside the backward",
                   "l2": "inputs larger than L2 (tables %.1f GB; out, grad_out %.0f MB each)" % (
                       sum(s.rows * (s.dim * _wbytes(s.dtype) + 4 * {"sgd": 0, "adagrad": s.dim,
                                                                       "rowwise_adagrad": 1}[s.opt]
                                     + (4 * s.dim if getattr(s, "master", False) else 0))
                           for s in w.tables) / 1e9, w.batch * w.total_dim * 4 / 1e6),
                   "parallelism": "replicas x%d" % ws,
                   "timing": "headline: %d steps with phase timing off; phases: %d further steps with "
                             "CUDA events around each phase" % (args.steps, args.steps)},
        "hbm": {"algorithmic_bytes_per_step": bytes_["step"], "achieved_gbs": step_gbs, "peak_gbs": peak,
                "frac": step_gbs / peak, "peak_kind": peak_kind,
                "algorithmic_bytes_per_phase": {p: bytes_[p] for p in ("forward", "dedup", "reduce_update")},
                "impl_bytes_per_phase": {p: impl[p] for p in ("forward", "dedup", "reduce_update")},
                "logical_forward_row_bytes": logical_row_bytes(w, batches[0])},
        "phases_ms": per_phase_ms,
        "ms_per_step_phase_timing_on": ms_phased,
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "achieved": dom_gbs, "peak": peak, "unit": "GB/s",
                     "frac": dom_gbs / peak, "traffic": traffic,
                     "algorithmic_bytes": bytes_[dom], "peak_kind": peak_kind},
        "cpu_baseline": cpu,
        "e2e": e2e,
        **({"infer": infer} if infer is not None else {}),
        "gpu_launches": launches,
        "clocks": clk,
        "status": status,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
