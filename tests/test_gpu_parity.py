"""GPU vs oracle parity on small, several-tile workloads and edge cases.

Every test calls the CUDA path through the C ABI (via the thin binding) and
compares with the CPU oracle on the same seeded inputs: bit-exact for ids,
counts, offsets and bag order; the stated relative tolerance for floats.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import ctr_inputs as ci
import oracle
from helpers import (TOL, bag_of_positions, expected_sorted_bags, gather_rows, init_rows_fn, max_rel_err,
                     ref_state, report_plain, run_gpu_step)

pytestmark = pytest.mark.gpu

VARIANTS = ["reduction", "unique_sort", "unique_hash"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _small(name):
    base = ci.workload(name if name in ci.WORKLOADS else name.split("_")[0])
    if name == "tiny":
        return base
    if name in ("dlrm_small", "dlrm_small_rowwise"):
        opt = "rowwise_adagrad" if name.endswith("rowwise") else None
        tabs = tuple(ci.TableSpec(min(t.rows, 200_000), t.dim, t.dtype, t.pooling, opt or t.opt, t.lr, t.eps)
                     for t in base.tables)
        return base.replace(name=name, tables=tabs, batch=4096)
    if name == "multihot_small":
        return base.replace(name=name, tables=base.tables[:10], batch=512).with_tables(rows=10_000)
    if name == "multihot_bf16":
        return base.replace(name=name, tables=base.tables[:6], batch=300).with_tables(rows=5_000, dtype="bf16")
    if name == "huge_small":
        return base.replace(name=name, batch=4096).with_tables(rows=1_000_000)
    if name == "skew_small":
        return base.replace(name=name, batch=2048).with_tables(rows=50_000)
    raise KeyError(name)


def check_step(w, batch, grad, variant, seed=0, expect_status=0, sample_untouched=64, early=False):
    g = run_gpu_step(w, batch, grad, variant, seed, keep_layer=True, early=early)
    layer = g.layer
    case = "%s/%s%s" % (w.name, variant, "/early" if early else "")
    try:
        assert g.status_fwd == expect_status and g.status_bwd == 0
        ref = oracle.step(w.tables, w.batch, batch.offsets, batch.keys, batch.table_ids, grad, init_rows_fn(w, seed))
        # a1 forward
        assert max_rel_err(g.out, ref.out, ref.out_scale) <= 1e-5
        # every row is a compensated term, so the plain relative error holds too
        assert report_plain(case, "forward", g.out, ref.out) <= 1e-5
        # a3 dedup: bit-exact
        assert np.array_equal(g.unique, ref.unique)
        assert np.array_equal(g.counts, ref.counts)
        assert np.array_equal(g.seg_off, ref.seg_off)
        if g.inverse is not None:
            assert np.array_equal(g.inverse, ref.inverse)
        exp_bags = expected_sorted_bags(ref.gids, bag_of_positions(batch.offsets))
        assert np.array_equal(g.sorted_bags[:exp_bags.size], exp_bags)
        # a5 updated rows, all touched rows
        for t, spec in enumerate(w.tables):
            sel = np.nonzero(ref.rows.table == t)[0]
            if sel.size == 0:
                continue
            W, A = gather_rows(layer, w, t, ref.rows.row[sel])
            idx = (ref.rows.row_start[sel][:, None] + np.arange(spec.dim)[None, :])
            assert max_rel_err(W, ref.W[idx], ref.W_scale[idx]) <= TOL[spec.dtype], (t, spec)
            report_plain(case, "weights_" + spec.dtype, W, ref.W[idx])
            if spec.opt != "sgd":
                ra, rs = ref_state(spec, ref.A, ref.A_scale, idx)
                assert max_rel_err(A, ra, rs) <= 1e-5, t
                report_plain(case, "state", A, ra)
        # untouched rows keep their initial values exactly
        rng = np.random.default_rng(1)
        for t, spec in enumerate(w.tables):
            touched = set(ref.rows.row[ref.rows.table == t].tolist())
            cand = rng.integers(0, spec.rows, size=sample_untouched)
            rows = np.array([r for r in cand if r not in touched] + [spec.rows - 1] * (spec.rows - 1 not in touched),
                            dtype=np.int64)
            if rows.size == 0:
                continue
            W, A = gather_rows(layer, w, t, rows)
            init = ci.stored_to_f64(ci.init_values(seed, t, rows, spec.dim, w.w_lo, w.w_hi, spec.dtype), spec.dtype)
            assert np.array_equal(W, init)
            if A is not None:
                assert np.all(A == np.float32(spec.init_acc))
        return g, ref
    finally:
        layer.close()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "dlrm_small", "dlrm_small_rowwise", "multihot_small", "multihot_bf16",
                                  "huge_small", "skew_small"])
def test_step_parity(name, variant):
    w = _small(name)
    batch = ci.make_batch(w)
    grad = ci.make_grad(w)
    check_step(w, batch, grad, variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "multihot_small", "skew_small"])
def test_early_dedup_step_parity(name, variant):
    """The dedup run inside the forward (on the layer's second stream) against
    the oracle, element by element, like the default mode."""
    w = _small(name)
    batch = ci.make_batch(w)
    grad = ci.make_grad(w)
    check_step(w, batch, grad, variant, early=True)


def test_init_matches_counter_generator_bit_exactly():
    import torch
    from dlrm_sparse_embedding_gb300 import EmbeddingLayer
    tabs = [ci.TableSpec(3000, 16, "f32"), ci.TableSpec(777, 64, "f16", opt="adagrad", init_acc=0.1),
            ci.TableSpec(5000, 128, "bf16"), ci.TableSpec(901, 12, "f32", opt="rowwise_adagrad", init_acc=0.1),
            ci.TableSpec(640, 32, "bf16", opt="adagrad", init_acc=0.1, master=True)]
    layer = EmbeddingLayer(tabs, 8, 16)
    try:
        layer.init_uniform(12345, -0.05, 0.05)
        for t, s in enumerate(tabs):
            W, A = layer.get_rows(t, 0, s.rows, with_state=s.opt != "sgd")
            ref = ci.init_values(12345, t, np.arange(s.rows), s.dim, -0.05, 0.05, s.dtype)
            assert np.array_equal(W.view(np.uint16) if s.dtype != "f32" else W,
                                  ref.view(np.uint16) if s.dtype == "f16" else ref)
            if A is not None:
                assert A.shape == (s.rows, s.dim if s.opt == "adagrad" else 1)
                assert np.all(A == np.float32(0.1))
            if s.master:
                M = layer.get_master_rows(t, 0, s.rows)
                assert np.array_equal(M, ci.init_values(12345, t, np.arange(s.rows), s.dim, -0.05, 0.05, "f32"))
    finally:
        layer.close()


# ---------------------------------------------------------------------------
# unique primitive
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,lo,hi", [(0, 0, 1), (1, 5, 6), (7, -3, 3), (4096, 0, 100), (4097, -(1 << 40), 1 << 40),
                                     (100_003, -(1 << 62), 1 << 62), (300_000, 0, 1_000), (65_536, 7, 8)])
def test_unique_primitive_bit_exact(n, lo, hi):
    import torch
    from dlrm_sparse_embedding_gb300 import unique
    rng = np.random.default_rng(n)
    keys = rng.integers(lo, hi, size=n, dtype=np.int64)
    u, inv, cnt, seg = unique(torch.from_numpy(keys).cuda())
    ru, rinv, rcnt, rseg = oracle.unique(keys)
    assert np.array_equal(u.cpu().numpy(), ru)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(seg.cpu().numpy(), rseg)


def test_unique_extreme_int64_values():
    import torch
    from dlrm_sparse_embedding_gb300 import unique
    keys = np.array([np.iinfo(np.int64).max, np.iinfo(np.int64).min, 0, -1, np.iinfo(np.int64).max, 1],
                    dtype=np.int64)
    u, inv, cnt, seg = unique(torch.from_numpy(keys).cuda())
    ru, rinv, rcnt, rseg = oracle.unique(keys)
    assert np.array_equal(u.cpu().numpy(), ru) and np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(cnt.cpu().numpy(), rcnt) and np.array_equal(seg.cpu().numpy(), rseg)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def _custom(tables, B, lens, key_fn, seed=0, name="edge"):
    w = ci.Workload(name=name, tables=tuple(tables), batch=B, hot_kind="fixed", hot_lo=1, hot_hi=1,
                    key_dist="uniform", seed=seed)
    lens = np.asarray(lens, dtype=np.int64).reshape(-1)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    keys = np.empty(int(offsets[-1]), dtype=np.int64)
    rng = np.random.default_rng(seed)
    for j in range(len(tables) * B):
        t = j // B
        keys[offsets[j]:offsets[j + 1]] = key_fn(rng, t, tables[t], int(lens[j]))
    batch = ci.Batch(keys=keys, offsets=offsets, table_ids=np.repeat(np.arange(len(tables), dtype=np.int32), B),
                     batch=B)
    grad = np.random.default_rng(seed + 1).standard_normal((B, sum(t.dim for t in tables))).astype(np.float32)
    return w, batch, grad


@pytest.mark.parametrize("variant", VARIANTS)
def test_empty_bags_and_mean_pooling(variant):
    tabs = [ci.TableSpec(500, 16, pooling="mean", opt="adagrad"), ci.TableSpec(300, 32, pooling="sum")]
    lens = np.random.default_rng(3).integers(0, 4, size=2 * 200)
    lens[:17] = 0
    w, b, g = _custom(tabs, 200, lens, lambda rng, t, s, L: rng.integers(0, s.rows, L))
    check_step(w, b, g, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_lookups(variant):
    tabs = [ci.TableSpec(50, 8)]
    w, b, g = _custom(tabs, 16, np.zeros(16), lambda rng, t, s, L: np.zeros(0, np.int64))
    gs = run_gpu_step(w, b, g, variant)
    assert np.all(gs.out == 0) and gs.unique.size == 0 and gs.seg_off.tolist() == [0]


@pytest.mark.parametrize("variant", VARIANTS)
def test_one_key_everywhere_spans_many_chunks(variant):
    # every lookup hits row 7: one run crossing every chunk boundary
    tabs = [ci.TableSpec(1000, 64, opt="adagrad"), ci.TableSpec(10, 128)]
    w, b, g = _custom(tabs, 5000, np.full(2 * 5000, 30), lambda rng, t, s, L: np.full(L, 7 if t == 0 else s.rows - 1))
    check_step(w, b, g, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_odd_dims_and_last_rows(variant):
    dims = [4, 12, 48, 100, 128, 20]
    tabs = [ci.TableSpec(r, d, opt="adagrad" if i % 2 else "sgd", pooling="mean" if i % 3 == 0 else "sum")
            for i, (r, d) in enumerate(zip([3, 64, 1000, 17, 5, 2], dims))]
    lens = np.random.default_rng(5).integers(0, 9, size=len(tabs) * 333)
    w, b, g = _custom(tabs, 333, lens,
                      lambda rng, t, s, L: np.where(rng.random(L) < 0.3, s.rows - 1, rng.integers(0, s.rows, L)))
    check_step(w, b, g, variant)


# Layers whose tables share one storage type, optimizer and pooling run a
# reduction kernel specialised for that combination: every combination, with
# the chunk length small inputs get (32 lookups) and, forced through the
# library's test hook, the multi-hot one (256 lookups, key windows staged in
# shared memory).  A hot row spans several chunks (split runs and one-run
# chunks) and bags repeat rows (entries of multiplicity above one).
UNIFORM_SPECS = [(dt, opt, pool) for dt in ("f32", "f16", "bf16")
                 for opt in ("sgd", "adagrad", "rowwise_adagrad") for pool in ("sum", "mean")]


@pytest.mark.parametrize("chunk", [0, 256])
@pytest.mark.parametrize("variant", ["reduction", "unique_sort"])
@pytest.mark.parametrize("dt,opt,pool", UNIFORM_SPECS)
def test_uniform_layer_kernels(dt, opt, pool, variant, chunk, monkeypatch):
    if chunk:
        monkeypatch.setenv("EMB_TEST_REDUCE_CHUNK", str(chunk))
    else:
        monkeypatch.delenv("EMB_TEST_REDUCE_CHUNK", raising=False)
    tabs = [ci.TableSpec(r, d, dt, pool, opt) for r, d in ((1500, 16), (700, 64), (300, 128))]
    B = 300
    lens = np.random.default_rng(61).integers(0, 45, size=len(tabs) * B)

    def keys(rng, t, s, L):
        k = rng.integers(0, s.rows, L)
        k[rng.random(L) < 0.25] = 3                         # a row hit about 2 000 times per table
        return k

    w, b, g = _custom(tabs, B, lens, keys, seed=62, name="uniform_%s_%s_%s" % (dt, opt, pool))
    check_step(w, b, g, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_out_of_range_keys_are_skipped_and_reported(variant):
    from dlrm_sparse_embedding_gb300 import EMB_ERR_KEY_RANGE
    tabs = [ci.TableSpec(100, 16), ci.TableSpec(40, 32, opt="adagrad")]

    def keys(rng, t, s, L):
        k = rng.integers(0, s.rows, L)
        bad = rng.random(L) < 0.1
        k[bad] = rng.choice([-1, s.rows, s.rows + 5, -(1 << 40), 1 << 40], size=int(bad.sum()))
        return k

    w, b, g = _custom(tabs, 256, np.random.default_rng(2).integers(1, 6, 512), keys)
    check_step(w, b, g, variant, expect_status=EMB_ERR_KEY_RANGE)


def test_wrong_table_id_is_reported():
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_ERR_INVALID_ARG, EmbeddingLayer
    tabs = [ci.TableSpec(100, 16), ci.TableSpec(40, 16)]
    w, b, g = _custom(tabs, 64, np.ones(128), lambda rng, t, s, L: rng.integers(0, s.rows, L))
    b.table_ids[70] = 0
    layer = EmbeddingLayer(tabs, 64, b.nnz)
    try:
        layer.init_uniform(0, -0.05, 0.05)
        out = layer.forward(torch.from_numpy(b.keys).cuda(), torch.from_numpy(b.offsets).cuda(),
                            torch.from_numpy(b.table_ids).cuda(), 64)
        assert layer.sync_status() == EMB_ERR_INVALID_ARG
        ref = oracle.step(tabs, 64, b.offsets, b.keys, b.table_ids, g, init_rows_fn(w, 0))
        assert max_rel_err(out.cpu().numpy(), ref.out, ref.out_scale) <= 1e-5
    finally:
        layer.close()


@pytest.mark.parametrize("variant", VARIANTS)
def test_table_segments_with_skipped_ids_over_several_passes(variant):
    """The dedup sorts each table's lookups on their table-local row id.  Tables
    of very different sizes (one-pass and multi-pass local ids; 2^20 - 1 rows,
    whose largest id would share the top digit of the skipped-id key without
    one more bit), skipped ids in several tables moved behind every valid id,
    and an empty first table."""
    from dlrm_sparse_embedding_gb300 import EMB_ERR_KEY_RANGE
    tabs = [ci.TableSpec(50, 8), ci.TableSpec((1 << 20) - 1, 4, opt="adagrad"), ci.TableSpec(1023, 16),
            ci.TableSpec(300_000, 8, pooling="mean"), ci.TableSpec(1024, 4)]
    B = 3000
    rng0 = np.random.default_rng(11)
    lens = rng0.integers(0, 12, size=len(tabs) * B)
    lens[:B] = 0                      # table 0: no lookups at all

    def keys(rng, t, s, L):
        k = rng.integers(0, s.rows, L)
        top = rng.random(L) < 0.2
        k[top] = s.rows - 1 - rng.integers(0, 2, int(top.sum())).clip(0, s.rows - 1)
        bad = rng.random(L) < 0.05
        k[bad] = rng.choice([-1, s.rows, s.rows + 7], size=int(bad.sum()))
        return k

    w, b, g = _custom(tabs, B, lens, keys, seed=21)
    check_step(w, b, g, variant, expect_status=EMB_ERR_KEY_RANGE)


@pytest.mark.parametrize("variant", ["reduction", "unique_hash"])
def test_many_small_tables(variant):
    """1300 tables (more segments than the sort's set-up block has threads),
    a few bags each, some tables empty."""
    T, B = 1300, 8
    tabs = [ci.TableSpec(10 + (t * 37) % 200, 4 * (1 + t % 3)) for t in range(T)]
    lens = np.random.default_rng(4).integers(0, 4, size=T * B)
    lens[5 * B:6 * B] = 0
    w, b, g = _custom(tabs, B, lens, lambda rng, t, s, L: rng.integers(0, s.rows, L), seed=5)
    check_step(w, b, g, variant, sample_untouched=2)


@pytest.mark.parametrize("hot", [1, 7])
def test_bad_offsets_are_clamped_and_reported(hot):
    """Offsets past nnz or decreasing are clamped on the GPU and reported as a
    bad argument; the layer stays usable.  A valid step runs first, so every
    id the backward reads afterwards is one a forward wrote."""
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_ERR_INVALID_ARG, EMB_OK, EmbeddingLayer
    tabs = [ci.TableSpec(100, 16), ci.TableSpec(40, 64)]
    B = 64
    w, b, g = _custom(tabs, B, np.full(2 * B, hot), lambda rng, t, s, L: rng.integers(0, s.rows, L))
    dev = torch.device("cuda", 0)
    keys, tids, grad = (torch.from_numpy(x).to(dev) for x in (b.keys, b.table_ids, g))
    good = torch.from_numpy(b.offsets).to(dev)
    bad_np = b.offsets.copy()
    bad_np[10] = b.nnz + 1000          # past the end of the keys
    bad_np[40] = bad_np[39] - 2        # decreasing
    bad_np[B + 3] = -5                 # negative
    bad = torch.from_numpy(bad_np).to(dev)
    layer = EmbeddingLayer(tabs, B, b.nnz)
    try:
        layer.init_uniform(0, -0.05, 0.05)
        layer.forward(keys, good, tids, B)
        layer.backward_update(grad, "reduction")
        assert layer.sync_status() == EMB_OK
        layer.forward(keys, bad, tids, B)
        assert layer.sync_status() == EMB_ERR_INVALID_ARG
        layer.backward_update(grad, "reduction")
        layer.sync_status()
        layer.forward(keys, good, tids, B)
        layer.backward_update(grad, "unique_hash")
        assert layer.sync_status() == EMB_OK
    finally:
        layer.close()


@pytest.mark.parametrize("variant", VARIANTS)
def test_deterministic_bitwise(variant):
    w = _small("skew_small").replace(batch=512)
    batch = ci.make_batch(w)
    grad = ci.make_grad(w)
    outs = []
    for _ in range(2):
        gs = run_gpu_step(w, batch, grad, variant, keep_layer=True)
        rows = []
        for t in range(w.num_tables):
            W, _ = gs.layer.get_rows(t, 0, 64)
            rows.append(W.copy())
        gs.layer.close()
        outs.append((gs.out, rows))
    assert np.array_equal(outs[0][0], outs[1][0])
    for a, c in zip(outs[0][1], outs[1][1]):
        assert np.array_equal(a, c)


def test_variants_agree():
    w = _small("multihot_small")
    batch = ci.make_batch(w)
    grad = ci.make_grad(w)
    res = {}
    for v in VARIANTS:
        gs = run_gpu_step(w, batch, grad, v, keep_layer=True)
        res[v] = (gs.unique, gs.counts, gs.seg_off, gs.sorted_bags,
                  [gs.layer.get_rows(t, 0, 2000, with_state=True) for t in range(3)])
        gs.layer.close()
    for v in VARIANTS[1:]:
        for a, c in zip(res["reduction"][:4], res[v][:4]):
            assert np.array_equal(a, c)
        for (wa, sa), (wc, sc) in zip(res["reduction"][4], res[v][4]):
            assert np.array_equal(wa, wc) and np.array_equal(sa, sc)


def test_backward_before_forward_is_a_state_error():
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_ERR_STATE, EmbError, EmbeddingLayer
    layer = EmbeddingLayer([ci.TableSpec(10, 8)], 4, 4)
    try:
        with pytest.raises(EmbError) as e:
            layer.backward_update(torch.zeros((4, 8), device="cuda"))
        assert e.value.status == EMB_ERR_STATE
    finally:
        layer.close()


def test_allocation_failure_returns_oom_and_leaks_nothing():
    code = (
        "import ctypes, torch, sys; sys.path.insert(0, %r)\n"
        "from dlrm_sparse_embedding_gb300 import EmbeddingLayer, EmbError, EMB_ERR_OOM\n"
        "import ctr_inputs as ci\n"
        "torch.cuda.init()\n"
        "free0 = torch.cuda.mem_get_info()[0]\n"
        "try:\n"
        "    EmbeddingLayer([ci.TableSpec(1000000, 64)] * 4, 1024, 100000)\n"
        "    print('NO-ERROR')\n"
        "except EmbError as e:\n"
        "    assert e.status == EMB_ERR_OOM, e.status\n"
        "    torch.cuda.synchronize()\n"
        "    print('OOM', free0 - torch.cuda.mem_get_info()[0])\n"
    ) % os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, EMB_TEST_ALLOC_LIMIT_BYTES=str(600 << 20))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("OOM"), r.stdout
    leaked = int(r.stdout.split()[1])
    assert leaked < (64 << 20)


@pytest.mark.parametrize("early,bwd", [("reduction", "reduction"), ("unique_sort", "unique_sort"),
                                       ("unique_hash", "unique_hash"), ("reduction", "unique_hash"),
                                       ("unique_hash", "reduction")])
def test_early_dedup_is_bitwise_identical(early, bwd):
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_OK, EmbeddingLayer
    w = _small("skew_small").replace(batch=700)
    batch = ci.make_batch(w)
    grad = torch.from_numpy(ci.make_grad(w)).cuda()
    keys, offs, tids = (torch.from_numpy(x).cuda() for x in (batch.keys, batch.offsets, batch.table_ids))
    res = []
    for mode in (None, early):
        layer = EmbeddingLayer(w.tables, w.batch, batch.nnz)
        try:
            layer.init_uniform(3, w.w_lo, w.w_hi)
            layer.set_early_dedup(mode)
            layer.set_keep_dedup(True)
            outs = []
            for _ in range(2):                      # two steps: the second reuses the side stream
                outs.append(layer.forward(keys, offs, tids, w.batch).cpu().numpy())
                layer.backward_update(grad, bwd)
            assert layer.sync_status() == EMB_OK
            ded = [x.cpu().numpy() for x in layer.dedup_result(with_inverse=False) if x is not None]
            rows = [layer.get_rows(t, 0, 512)[0] for t in range(w.num_tables)]
            res.append((outs, ded, rows))
        finally:
            layer.close()
    (o0, d0, r0), (o1, d1, r1) = res
    for a, b in zip(o0 + d0 + r0, o1 + d1 + r1):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("variant", VARIANTS)
def test_rowwise_adagrad_dims_pooling_and_split_rows(variant):
    # row-wise Adagrad on narrow, odd and full-width rows (lanes past the row's
    # end take part in the row's sum of squares with zeros), mean pooling,
    # 16-bit storage, and one row hit by a third of the lookups, so it is split
    # over many chunks and finished by the combine kernel
    tabs = [ci.TableSpec(2000, 20, "f32", "mean", "rowwise_adagrad", 0.01, 1e-8, 0.05),
            ci.TableSpec(500, 100, "bf16", "sum", "rowwise_adagrad", 0.02, 1e-8, 0.0),
            ci.TableSpec(3000, 4, "f16", "sum", "rowwise_adagrad", 0.01, 1e-6, 0.0),
            ci.TableSpec(50, 128, "f32", "sum", "rowwise_adagrad", 0.01, 1e-8, 0.1)]
    B = 1500
    lens = np.random.default_rng(6).integers(0, 12, size=len(tabs) * B)

    def keys(rng, t, s, L):
        k = rng.integers(0, s.rows, L)
        k[rng.random(L) < 0.33] = s.rows // 2
        return k

    w, b, g = _custom(tabs, B, lens, keys, seed=8)
    check_step(w, b, g, variant)


def _round_stored(m32: np.ndarray, dtype: str) -> np.ndarray:
    """Nearest-even rounding of fp32 values to the storage type, as binary64
    (NumPy's fp16 conversion, torch's bf16 conversion)."""
    import torch
    if dtype == "f16":
        return m32.astype(np.float16).astype(np.float64)
    return torch.from_numpy(np.ascontiguousarray(m32)).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("variant", VARIANTS)
def test_master_copy_parity(variant):
    # 16-bit tables with an fp32 master next to one without: the stored rows
    # match the oracle's, the masters match the oracle's masters, and every
    # stored row is its GPU master rounded to nearest-even
    import torch
    tabs = [ci.TableSpec(3000, 16, "f16", "sum", "adagrad", 0.01, 1e-8, 0.0, master=True),
            ci.TableSpec(800, 64, "bf16", "mean", "rowwise_adagrad", 0.02, 1e-8, 0.1, master=True),
            ci.TableSpec(500, 8, "f16", "sum", "sgd", 0.01),
            ci.TableSpec(200, 128, "bf16", "sum", "sgd", 0.05, master=True)]
    B = 1200
    lens = np.random.default_rng(12).integers(0, 10, size=len(tabs) * B)

    def keys(rng, t, s, L):
        k = rng.integers(0, s.rows, L)
        k[rng.random(L) < 0.3] = 5
        return k

    w, b, g = _custom(tabs, B, lens, keys, seed=13)
    seed = 0
    gs = run_gpu_step(w, b, g, variant, seed, keep_layer=True)
    layer = gs.layer
    try:
        assert gs.status_fwd == 0 and gs.status_bwd == 0
        ref = oracle.step(w.tables, w.batch, b.offsets, b.keys, b.table_ids, g, init_rows_fn(w, seed),
                          lambda t, r: ci.init_values(seed, t, r, w.tables[t].dim, w.w_lo, w.w_hi, "f32"))
        assert max_rel_err(gs.out, ref.out, ref.out_scale) <= 1e-5
        for t, spec in enumerate(w.tables):
            sel = np.nonzero(ref.rows.table == t)[0]
            rows = ref.rows.row[sel]
            idx = ref.rows.row_start[sel][:, None] + np.arange(spec.dim)[None, :]
            W, A = gather_rows(layer, w, t, rows)
            assert max_rel_err(W, ref.W[idx], ref.W_scale[idx]) <= TOL[spec.dtype], t
            if spec.opt != "sgd":
                ra, rs = ref_state(spec, ref.A, ref.A_scale, idx)
                assert max_rel_err(A, ra, rs) <= 1e-5, t
            if spec.master:
                M = layer.gather_master_rows(t, torch.from_numpy(rows).cuda()).cpu().numpy()
                assert max_rel_err(M, ref.M[idx], ref.W_scale[idx]) <= 1e-5, t
                assert np.array_equal(W, _round_stored(M, spec.dtype)), t
            else:
                with pytest.raises(Exception):
                    layer.get_master_rows(t, 0, 1)
    finally:
        layer.close()


# ---------------------------------------------------------------------------
# dynamic tables (int64 keys behind a GPU hash map)
# ---------------------------------------------------------------------------

def _dynamic_inputs(B=900, seed=21):
    tabs = [ci.TableSpec(1000, 16, "f32", "sum", "adagrad", 0.01, 1e-8, 0.0),
            ci.TableSpec(4096, 32, "f32", "mean", "rowwise_adagrad", 0.01, 1e-8, 0.1, dynamic=True),
            ci.TableSpec(2048, 64, "bf16", "sum", "adagrad", 0.02, 1e-8, 0.0, master=True, dynamic=True),
            ci.TableSpec(1024, 8, "f16", "sum", "sgd", 0.01, dynamic=True)]
    lens = np.random.default_rng(seed).integers(0, 9, size=len(tabs) * B)

    def keys(rng, t, s, L):
        k = rng.integers(0, s.key_space, L)
        k[rng.random(L) < 0.25] = 3
        return ci.dynamic_key(t, k) if s.dynamic else k

    return _custom(tabs, B, lens, keys, seed=seed)


def _dynamic_reference(w, b, g, seed):
    lo, hi = w.w_lo, w.w_hi
    return oracle.step_dynamic(
        w.tables, w.batch, b.offsets, b.keys, b.table_ids, g, init_rows_fn(w, seed),
        lambda t, k: ci.init_values_dynamic(seed, t, k, w.tables[t].dim, lo, hi, w.tables[t].dtype),
        None, lambda t, k: ci.init_values_dynamic(seed, t, k, w.tables[t].dim, lo, hi, "f32"))


@pytest.mark.parametrize("variant", VARIANTS)
def test_dynamic_tables_parity(variant):
    import torch
    w, b, g = _dynamic_inputs()
    seed = 0
    gs = run_gpu_step(w, b, g, variant, seed, keep_layer=True)
    layer = gs.layer
    try:
        assert gs.status_fwd == 0 and gs.status_bwd == 0
        ref, key_of = _dynamic_reference(w, b, g, seed)
        assert max_rel_err(gs.out, ref.out, ref.out_scale) <= 1e-5
        # one unique row per distinct key of each table, with the same counts
        assert gs.unique.size == ref.unique.size
        assert np.array_equal(np.sort(gs.counts), np.sort(ref.counts))
        for t, spec in enumerate(w.tables):
            sel = np.nonzero(ref.rows.table == t)[0]
            idx = ref.rows.row_start[sel][:, None] + np.arange(spec.dim)[None, :]
            rows = ref.rows.row[sel]
            if spec.dynamic:
                rows = layer.find_keys(t, torch.from_numpy(key_of[t][rows]).cuda()).cpu().numpy()
                assert np.all(rows >= 0) and np.unique(rows).size == rows.size
            W, A = gather_rows(layer, w, t, rows)
            assert max_rel_err(W, ref.W[idx], ref.W_scale[idx]) <= TOL[spec.dtype], t
            if spec.opt != "sgd":
                ra, rs = ref_state(spec, ref.A, ref.A_scale, idx)
                assert max_rel_err(A, ra, rs) <= 1e-5, t
            if spec.master:
                M = layer.gather_master_rows(t, torch.from_numpy(rows).cuda()).cpu().numpy()
                assert max_rel_err(M, ref.M[idx], ref.W_scale[idx]) <= 1e-5, t
    finally:
        layer.close()


def test_dynamic_first_lookup_initializes_rows_once():
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_OK, EmbeddingLayer
    w, b, _ = _dynamic_inputs(B=400, seed=22)
    layer = EmbeddingLayer(w.tables, w.batch, b.nnz)
    try:
        layer.init_uniform(7, -0.05, 0.05)
        k, o, tid = (torch.from_numpy(x).cuda() for x in (b.keys, b.offsets, b.table_ids))
        layer.forward(k, o, tid, w.batch)
        assert layer.sync_status() == EMB_OK
        for t, spec in enumerate(w.tables):
            if not spec.dynamic:
                continue
            seg = b.keys[b.offsets[t * w.batch]:b.offsets[(t + 1) * w.batch]]
            uk = np.unique(seg)
            rows = layer.find_keys(t, torch.from_numpy(uk).cuda()).cpu().numpy()
            assert np.all(rows >= 0) and np.unique(rows).size == uk.size
            W, A = layer.gather_rows(t, torch.from_numpy(rows).cuda(), with_state=spec.opt != "sgd")
            want = ci.init_values_dynamic(7, t, uk, spec.dim, -0.05, 0.05, spec.dtype)
            got = W.view(torch.int16).cpu().numpy().view(np.uint16) if spec.dtype == "bf16" else W.cpu().numpy()
            assert np.array_equal(got.view(np.uint16) if spec.dtype != "f32" else got,
                                  want.view(np.uint16) if spec.dtype != "f32" else want)
            if A is not None:
                assert np.all(A.cpu().numpy() == np.float32(spec.init_acc))
            if spec.master:
                M = layer.gather_master_rows(t, torch.from_numpy(rows).cuda()).cpu().numpy()
                assert np.array_equal(M, ci.init_values_dynamic(7, t, uk, spec.dim, -0.05, 0.05, "f32"))
            # keys already held keep their rows; keys never seen have none
            layer.forward(k, o, tid, w.batch)
            again = layer.find_keys(t, torch.from_numpy(uk).cuda()).cpu().numpy()
            assert np.array_equal(again, rows)
            absent = ci.dynamic_key(t, np.arange(spec.key_space, spec.key_space + 50))
            assert np.all(layer.find_keys(t, torch.from_numpy(absent).cuda()).cpu().numpy() == -1)
    finally:
        layer.close()


def test_dynamic_table_full_and_reserved_key_are_reported():
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_ERR_CAPACITY, EMB_ERR_KEY_RANGE, EmbeddingLayer
    tabs = [ci.TableSpec(64, 8, "f32", "sum", "sgd", 0.01, dynamic=True)]
    B = 100
    keys = ci.dynamic_key(0, np.arange(B))              # 100 distinct keys, 64 rows
    offsets = np.arange(B + 1, dtype=np.int64)
    tid = np.zeros(B, np.int32)
    layer = EmbeddingLayer(tabs, B, B)
    try:
        layer.init_uniform(0, -0.05, 0.05)
        kt = torch.from_numpy(keys).cuda()
        out = layer.forward(kt, torch.from_numpy(offsets).cuda(), torch.from_numpy(tid).cuda(), B)
        assert layer.sync_status() == EMB_ERR_CAPACITY
        rows = layer.find_keys(0, kt).cpu().numpy()
        held = rows >= 0
        assert held.sum() == 64 and np.unique(rows[held]).size == 64
        assert np.all(out.cpu().numpy()[~held] == 0)          # lookups that found no row are skipped
        keys2 = keys.copy()
        keys2[5] = np.iinfo(np.int64).min                   # the reserved key
        layer.init_uniform(0, -0.05, 0.05)                   # empties the map
        layer.forward(torch.from_numpy(keys2[:60]).cuda(), torch.from_numpy(offsets[:61]).cuda(),
                      torch.from_numpy(tid[:60]).cuda(), 60)
        assert layer.sync_status() == EMB_ERR_KEY_RANGE
    finally:
        layer.close()


# ---------------------------------------------------------------------------
# inference forward with fp16 caches of hot rows
# ---------------------------------------------------------------------------

# "mixed": fp32 and 16-bit tables (16-byte ring slots), short bags;
# "rows16": 16-bit tables only (the 8-byte-slot kernel), bags of up to 74 keys
# (several key windows, cached rows in every batch of a window)
INFER_CASES = {
    "mixed": ([ci.TableSpec(3000, 128, "f32", "sum", "adagrad"), ci.TableSpec(900, 16, "bf16", "mean", "sgd"),
               ci.TableSpec(500, 64, "f16", "sum", "sgd"), ci.TableSpec(60, 20, "f32", "mean", "sgd")], 700, 7,
              {0: np.arange(30), 1: np.array([2, 2, 5, 899, 800, 3]), 3: np.arange(60)}),
    "rows16": ([ci.TableSpec(2000, 64, "f16", "sum", "sgd"), ci.TableSpec(700, 8, "bf16", "mean", "sgd"),
                ci.TableSpec(300, 128, "f16", "mean", "adagrad")], 300, 75,
               {0: np.arange(40), 2: np.array([2, 7, 299])}),
}


@pytest.mark.parametrize("case", sorted(INFER_CASES))
def test_forward_infer_with_caches(case):
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_ERR_KEY_RANGE, EMB_OK, EmbeddingLayer
    tabs, B, max_len, cached = INFER_CASES[case]
    lens = np.random.default_rng(31).integers(0, max_len, size=len(tabs) * B)

    def keys(rng, t, s, L):
        k = rng.integers(0, s.rows, L)
        k[rng.random(L) < 0.4] = 2                          # a hot row, cached in two tables
        return k

    w, b, _ = _custom(tabs, B, lens, keys, seed=32)
    seed = 0
    layer = EmbeddingLayer(w.tables, B, b.nnz)
    try:
        layer.init_uniform(seed, w.w_lo, w.w_hi)
        k, o, tid = (torch.from_numpy(x).cuda() for x in (b.keys, b.offsets, b.table_ids))
        for t, rows in cached.items():
            layer.cache_build(t, torch.from_numpy(rows.astype(np.int64)).cuda())
        got = layer.forward_infer(k, o, tid, B).cpu().numpy()
        assert layer.sync_status() == EMB_OK
        want, scale = oracle.forward_with_cache(w.tables, B, b.offsets, b.keys, b.table_ids, init_rows_fn(w, seed),
                                                cached)
        assert max_rel_err(got, want, scale) <= 1e-5
        # the training forward still reads the tables
        plain = layer.forward(k, o, tid, B).cpu().numpy()
        want0, scale0 = oracle.forward_with_cache(w.tables, B, b.offsets, b.keys, b.table_ids,
                                                  init_rows_fn(w, seed), {})
        assert max_rel_err(plain, want0, scale0) <= 1e-5
        # removing the caches: inference reads the tables too
        for t in cached:
            layer.cache_build(t, torch.zeros(0, dtype=torch.int64).cuda())
        assert max_rel_err(layer.forward_infer(k, o, tid, B).cpu().numpy(), want0, scale0) <= 1e-5
        # a row id outside the table is reported
        layer.cache_build(1, torch.tensor([1, tabs[1].rows], dtype=torch.int64).cuda())
        assert layer.sync_status() == EMB_ERR_KEY_RANGE
    finally:
        layer.close()


def test_forward_infer_on_dynamic_tables_skips_unseen_ids():
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_OK, EmbeddingLayer
    w, b, g = _dynamic_inputs(B=300, seed=33)
    seed = 0
    layer = EmbeddingLayer(w.tables, w.batch, b.nnz)
    try:
        layer.init_uniform(seed, w.w_lo, w.w_hi)
        k, o, tid = (torch.from_numpy(x).cuda() for x in (b.keys, b.offsets, b.table_ids))
        layer.forward(k, o, tid, w.batch)                   # inserts every key
        # a second batch whose dynamic keys are half new
        keys2 = b.keys.copy()
        for t, spec in enumerate(w.tables):
            if spec.dynamic:
                lo_, hi_ = b.offsets[t * w.batch], b.offsets[(t + 1) * w.batch]
                flip = np.random.default_rng(t).random(hi_ - lo_) < 0.5
                keys2[lo_:hi_][flip] = ci.dynamic_key(t, np.arange(spec.key_space, spec.key_space + flip.sum()))
        got = layer.forward_infer(torch.from_numpy(keys2).cuda(), o, tid, w.batch).cpu().numpy()
        assert layer.sync_status() == EMB_OK
        # reference: unseen ids contribute nothing (the reserved key stands in for them)
        keys_ref = keys2.copy()
        for t, spec in enumerate(w.tables):
            if spec.dynamic:
                lo_, hi_ = b.offsets[t * w.batch], b.offsets[(t + 1) * w.batch]
                seen = np.isin(keys2[lo_:hi_], b.keys[lo_:hi_])
                keys_ref[lo_:hi_][~seen] = np.iinfo(np.int64).min
        ref, _ = _dynamic_reference(w, ci.Batch(keys_ref, b.offsets, b.table_ids, w.batch), g, seed)
        assert max_rel_err(got, ref.out, ref.out_scale) <= 1e-5
    finally:
        layer.close()


def test_inference_between_forward_and_backward_changes_nothing():
    # with the dedup running early on the layer's second stream, an inference
    # forward (which rewrites the dynamic tables' resolved rows) between a
    # forward and its backward leaves the step bitwise unchanged
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_OK, EmbeddingLayer
    w, b, g = _dynamic_inputs(B=500, seed=41)
    _, b2, _ = _dynamic_inputs(B=500, seed=42)
    k, o, tid = (torch.from_numpy(x).cuda() for x in (b.keys, b.offsets, b.table_ids))
    k2, o2, tid2 = (torch.from_numpy(x).cuda() for x in (b2.keys, b2.offsets, b2.table_ids))
    grad = torch.from_numpy(g).cuda()
    res = []
    for early in (None, "reduction"):
        layer = EmbeddingLayer(w.tables, w.batch, max(b.nnz, b2.nnz))
        try:
            layer.init_uniform(5, w.w_lo, w.w_hi)
            layer.forward(k2, o2, tid2, w.batch)        # both layers hold the same keys
            layer.set_early_dedup(early)
            out = layer.forward(k, o, tid, w.batch).cpu().numpy()
            if early:
                layer.forward_infer(k2, o2, tid2, w.batch)
            layer.backward_update(grad, "reduction")
            assert layer.sync_status() == EMB_OK
            rows = []
            for t, s in enumerate(w.tables):
                if s.dynamic:   # rows are compared key by key: a key's row depends on insertion order
                    keys_t = np.unique(np.concatenate([x.keys[x.offsets[t * w.batch]:x.offsets[(t + 1) * w.batch]]
                                                       for x in (b, b2)]))
                    r = layer.find_keys(t, torch.from_numpy(keys_t).cuda())
                    W, A = layer.gather_rows(t, r, with_state=s.opt != "sgd")
                    W = W.view(torch.int16) if s.dtype == "bf16" else W
                    rows.append((W.cpu().numpy(), None if A is None else A.cpu().numpy()))
                else:
                    rows.append(layer.get_rows(t, 0, s.rows, with_state=s.opt != "sgd"))
            res.append((out, rows))
        finally:
            layer.close()
    assert np.array_equal(res[0][0], res[1][0])
    for (wa, sa), (wb, sb) in zip(res[0][1], res[1][1]):
        assert np.array_equal(wa, wb)
        assert (sa is None and sb is None) or np.array_equal(sa, sb)
