"""Host logic of bench.py on CPU: the algorithmic bytes behind every roofline
fraction, the validity check of a recorded ncu traffic figure, and the
reading of the clock samples that decide whether a run is kept."""
import hashlib
import json
import os

import numpy as np

import bench
import ctr_inputs as ci


def _two_table_case():
    # table 0: 10 rows x 8, fp32, Adagrad; table 1: 20 rows x 4, fp16 with an
    # fp32 master, SGD, mean pooling.  Three bags of two lookups per table.
    w = ci.Workload(name="hand", tables=(ci.TableSpec(10, 8, "f32", "sum", "adagrad"),
                                         ci.TableSpec(20, 4, "f16", "mean", "sgd", master=True)),
                    batch=3, hot_kind="fixed", hot_lo=2, hot_hi=2, key_dist="uniform")
    keys = np.array([1, 1, 2, 5, 1, 9,      # table 0: rows {1, 2, 5, 9}
                     0, 0, 0, 0, 3, 0],     # table 1: rows {0, 3}
                    dtype=np.int64)
    batch = ci.Batch(keys=keys, offsets=np.arange(0, 13, 2, dtype=np.int64),
                     table_ids=np.array([0, 0, 0, 1, 1, 1], dtype=np.int32), batch=3)
    return w, batch


def test_unique_rows_per_table():
    w, batch = _two_table_case()
    assert bench.unique_per_table(w, batch).tolist() == [4, 2]


def test_algorithmic_bytes_hand_count():
    """The compulsory bytes of each phase, counted by hand for the two-table case."""
    w, batch = _two_table_case()
    got = bench.algorithmic_bytes(w, batch, bench.unique_per_table(w, batch))
    nnz, bags, U, out = 12, 6, 6, 3 * 12 * 4    # out / grad_out: B x sum(dim) fp32
    rows = 4 * 8 * 4 + 2 * 4 * 2                # touched rows once, in their storage type
    fwd = 8 * nnz + 8 * (bags + 1) + rows + out
    dedup = 8 * nnz + 8 * U + 4 * nnz + 4 * U   # keys in; unique ids, inverse, counts out
    state = 4 * 8 * 4                           # Adagrad accumulators of table 0's touched rows
    master = 2 * 4 * 6                          # table 1: master read + written (8 B) minus the fp16 read (2 B)
    upd = out + 4 * nnz + 2 * rows + 2 * state + master
    assert got == {"forward": fwd, "dedup": dedup, "reduce_update": upd, "step": fwd + dedup + upd}
    assert (fwd, dedup, upd) == (440, 216, 784)


def test_implementation_bytes_hand_count():
    """What this implementation moves by design: table ids and 32-bit (id, bag)
    pairs from the forward, 20 B per element and sort pass, sorted pairs read
    by the reduction."""
    w, batch = _two_table_case()
    got = bench.implementation_bytes(w, batch, bench.unique_per_table(w, batch), sort_passes=2)
    assert got["forward"] == 440 + 4 * 6 + 8 * 12
    assert got["dedup"] == 2 * 20 * 12
    assert got["reduce_update"] == 784 + 4 * 12
    assert got["step"] == got["forward"] + got["dedup"] + got["reduce_update"]


def test_cpu_sample_is_bounded_by_lookups():
    w = ci.workload("multihot")
    per = bench.lookups_per_sample(w)
    assert 100 * 1 <= per <= 100 * 100
    n = bench.cpu_sample_batch(w, 400000)
    assert abs(n * per - 400000) <= per
    assert bench.cpu_sample_batch(ci.workload("tiny"), 10 ** 9) == 256
    assert bench.cpu_sample_batch(ci.workload("tiny"), 1) == 1


def test_logical_row_bytes():
    w, batch = _two_table_case()
    assert bench.logical_row_bytes(w, batch) == 6 * 8 * 4 + 6 * 4 * 2


def _write_record(root, text, sha=None):
    src = os.path.join(root, "k.cu")
    with open(src, "w") as f:
        f.write(text)
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    rec = {"reduce_update": {"traffic_bytes": 1234,
                             "sources_sha256": {"k.cu": sha or hashlib.sha256(text.encode()).hexdigest()}}}
    with open(os.path.join(root, "profiles", "traffic_cfg_reduction.json"), "w") as f:
        json.dump(rec, f)
    return src


def test_recorded_traffic_only_while_the_kernel_source_is_unchanged(tmp_path):
    root = str(tmp_path)
    src = _write_record(root, "kernel v1")
    assert bench.recorded_traffic("cfg", "reduction", "reduce_update", root=root) == 1234
    assert bench.recorded_traffic("cfg", "reduction", "forward", root=root) is None
    assert bench.recorded_traffic("cfg", "unique_sort", "reduce_update", root=root) is None
    with open(src, "w") as f:
        f.write("kernel v2")
    assert bench.recorded_traffic("cfg", "reduction", "reduce_update", root=root) is None
    os.remove(src)
    assert bench.recorded_traffic("cfg", "reduction", "reduce_update", root=root) is None


def test_committed_traffic_record_names_the_reduction_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic_multihot_reduction.json")) as f:
        rec = json.load(f)["reduce_update"]
    # the reduction's sources: the combine and launch, the chunk kernel, its
    # fp32 specialisations (the multi-hot layer is uniform fp32), shared helpers
    assert set(rec["sources_sha256"]) == {"dlrm_sparse_embedding_gb300/csrc/update.cu",
                                          "dlrm_sparse_embedding_gb300/csrc/reduce_chunks.cuh",
                                          "dlrm_sparse_embedding_gb300/csrc/update_f32.cu",
                                          "dlrm_sparse_embedding_gb300/csrc/emb_internal.cuh"}
    assert rec["traffic_bytes"] == sum(k["read"] + k["write"] for k in rec["per_kernel"].values())


class _DoneProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.f = open(s.path, "a")
    s.proc = _DoneProcess()
    return s


def test_clock_samples_median_and_active_reasons(tmp_path):
    na = "Not Active"
    s = _sampler_with(tmp_path, [
        "0, 2070, 2070, 180.5, 0x0000000000000004, %s, %s, %s, Active" % (na, na, na),
        "0, 2055, 2070, 190.1, 0x0000000000000004, %s, %s, %s, Active" % (na, na, na),
        "0, 2070, 2070, 175.0, 0x0000000000000000, %s, %s, %s, %s" % (na, na, na, na),
        "garbage line",
    ])
    r = s.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 190.1
    assert not os.path.exists(s.path)


def test_clock_samples_report_a_slowdown(tmp_path):
    na = "Not Active"
    s = _sampler_with(tmp_path, [
        "0, 1500, 2070, 300.0, 0x0000000000000008, Active, %s, Active, %s" % (na, na),
    ])
    r = s.stop()
    assert r["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and r["sm_mhz"] == 1500.0


def test_no_clock_samples(tmp_path):
    r = _sampler_with(tmp_path, []).stop()
    assert r["samples"] == 0 and r["reasons"] == ["no samples"]


def test_every_bench_config_is_a_workload():
    assert set(bench.CONFIG_TEXT) <= set(ci.WORKLOADS)
    assert {"tiny", "dlrm", "multihot", "huge", "skew"} <= set(bench.CONFIG_TEXT)
