"""Pins of the seeded input generators (CPU only).

The synthetic batches stand in for the CTR datasets of the pages, so their
recipe is checked against what fixes it independently of the generator's own
code: the workload shapes against the stated workloads, the Zipf sampler
against the exact probability law (chi-square on a small support, head
frequencies from the Hurwitz zeta function on the largest supports), the
number of distinct rows of the full-size one-hot and single-table batches
against its exact expectation, and the CSR structure of every batch.
"""
import dataclasses

import numpy as np
import pytest

import ctr_inputs as ci

scipy_special = pytest.importorskip("scipy.special")
scipy_stats = pytest.importorskip("scipy.stats")


def _harmonic(n, s):
    """H(n, s) = sum_{k=1..n} k^-s, exactly through the Hurwitz zeta function."""
    return float(scipy_special.zeta(s, 1) - scipy_special.zeta(s, n + 1))


def test_workloads_have_the_stated_shapes():
    tiny = ci.workload("tiny")
    assert tiny.num_tables == 4 and tiny.batch == 256 and tiny.key_dist == "uniform"
    assert (tiny.hot_kind, tiny.hot_lo, tiny.hot_hi) == ("per_bag_uniform", 1, 4)
    assert all((t.rows, t.dim, t.dtype, t.pooling, t.opt, t.lr) == (1000, 16, "f32", "sum", "sgd", 0.01)
               for t in tiny.tables)

    dlrm = ci.workload("dlrm")
    assert dlrm.num_tables == 26 and dlrm.batch == 65536 and (dlrm.hot_lo, dlrm.hot_hi) == (1, 1)
    assert (dlrm.key_dist, dlrm.alpha, dlrm.w_lo, dlrm.w_hi) == ("zipf", 1.05, -0.05, 0.05)
    assert all(1000 <= t.rows <= 10_000_000 for t in dlrm.tables)
    assert all((t.dim, t.dtype, t.pooling, t.opt, t.lr, t.eps) == (128, "f32", "sum", "adagrad", 0.01, 1e-8)
               for t in dlrm.tables)
    # log-uniform rows: the seeded draw spans several decades
    assert min(t.rows for t in dlrm.tables) < 10_000 and max(t.rows for t in dlrm.tables) > 1_000_000

    mh = ci.workload("multihot")
    assert mh.num_tables == 100 and mh.batch == 16384 and (mh.key_dist, mh.alpha) == ("zipf", 1.2)
    assert (mh.hot_kind, mh.hot_lo, mh.hot_hi) == ("per_table_uniform", 1, 100)
    assert all((t.rows, t.dim, t.dtype, t.pooling, t.opt) == (1_000_000, 64, "f32", "mean", "adagrad")
               for t in mh.tables)

    huge = ci.workload("huge")
    assert huge.num_tables == 1 and huge.batch == 131072 and (huge.hot_lo, huge.hot_hi) == (20, 20)
    assert (huge.key_dist, huge.alpha) == ("zipf", 1.1)
    t = huge.tables[0]
    assert (t.rows, t.dim, t.dtype, t.pooling, t.opt) == (200_000_000, 64, "f16", "sum", "adagrad")

    skew = ci.workload("skew")
    assert skew.batch == 262144 and (skew.hot_lo, skew.hot_hi) == (50, 50) and skew.alpha == 1.5
    assert [t.dim for t in skew.tables] == [16, 32, 64, 128] * 2
    assert all((t.rows, t.dtype, t.pooling, t.opt) == (5_000_000, "f32", "sum", "sgd") for t in skew.tables)


@pytest.mark.parametrize("alpha", [0.8, 1.05, 1.5])
def test_zipf_sampler_follows_the_law_on_a_small_support(alpha):
    n, m = 12, 120_000
    keys = ci.zipf_keys(np.random.default_rng(7), n, alpha, m)
    assert keys.min() >= 0 and keys.max() < n
    p = np.arange(1, n + 1, dtype=np.float64) ** -alpha
    p /= p.sum()
    counts = np.bincount(keys, minlength=n)
    chi2 = float(((counts - m * p) ** 2 / (m * p)).sum())
    assert chi2 < scipy_stats.chi2.ppf(1 - 1e-6, n - 1), chi2


@pytest.mark.parametrize("rows,alpha", [(10_000_000, 1.05), (200_000_000, 1.1), (5_000_000, 1.5)])
def test_zipf_sampler_head_frequencies_on_large_supports(rows, alpha):
    m = 400_000
    keys = ci.zipf_keys(np.random.default_rng(11), rows, alpha, m)
    assert keys.min() >= 0 and keys.max() < rows
    H = _harmonic(rows, alpha)
    # key 0, key 1 and the mass of the first 1000 keys, each a binomial count
    for got, p in ((np.count_nonzero(keys == 0), 1.0 / H),
                   (np.count_nonzero(keys == 1), 2.0 ** -alpha / H),
                   (np.count_nonzero(keys < 1000), _harmonic(1000, alpha) / H)):
        sd = np.sqrt(m * p * (1 - p))
        assert abs(got - m * p) < 6 * sd, (got, m * p, sd)


def _expected_unique(rows, alpha, draws):
    """E[distinct keys] and an upper bound of its variance for `draws` Zipf
    draws over `rows` keys: sum_k q_k, q_k = 1 - (1 - p_k)^draws."""
    H = _harmonic(rows, alpha)
    e = v = 0.0
    step = 10_000_000
    for lo in range(1, rows + 1, step):
        r = np.arange(lo, min(rows, lo + step - 1) + 1, dtype=np.float64)
        q = -np.expm1(draws * np.log1p(-(r ** -alpha) / H))
        e += float(q.sum())
        v += float((q * (1 - q)).sum())
    return e, v


@pytest.mark.parametrize("name", ["dlrm", "huge"])
def test_full_size_batch_has_the_expected_number_of_distinct_rows(name):
    w = ci.workload(name)
    b = ci.make_batch(w)
    B = w.batch
    U, EU, V = 0, 0.0, 0.0
    for t, spec in enumerate(w.tables):
        lo, hi = int(b.offsets[t * B]), int(b.offsets[(t + 1) * B])
        U += np.unique(b.keys[lo:hi]).size
        e, v = _expected_unique(spec.rows, w.alpha, hi - lo)
        EU += e
        V += v
    assert abs(U - EU) < 6 * np.sqrt(V), (U, EU, np.sqrt(V))


@pytest.mark.parametrize("name,batch", [("tiny", 0), ("multihot", 64), ("skew", 32), ("dlrm_dynamic", 128)])
def test_batches_are_well_formed_and_reproducible(name, batch):
    w = ci.workload(name)
    if batch:
        w = w.replace(batch=batch)
    b = ci.make_batch(w)
    T, B = w.num_tables, w.batch
    off = b.offsets
    assert off.dtype == np.int64 and off.shape == (T * B + 1,) and off[0] == 0 and off[-1] == b.nnz
    lens = np.diff(off)
    assert np.array_equal(lens.reshape(T, B), w.hotness())
    assert lens.min() >= w.hot_lo and lens.max() <= w.hot_hi
    if w.hot_kind == "per_table_uniform":
        assert all(np.unique(lens.reshape(T, B)[t]).size == 1 for t in range(T))
    assert np.array_equal(b.table_ids, (np.arange(T * B) // B).astype(np.int32))
    # a dynamic table draws the same ranks as a static table of key_space
    # rows, then maps each rank to its int64 id
    static = ci.make_batch(w.replace(tables=tuple(
        dataclasses.replace(t, rows=t.key_space, dynamic=False) for t in w.tables)))
    for t, spec in enumerate(w.tables):
        k = b.keys[off[t * B]:off[(t + 1) * B]]
        if spec.dynamic:
            assert np.array_equal(k, ci.dynamic_key(t, static.keys[off[t * B]:off[(t + 1) * B]]))
            ids = ci.dynamic_key(t, np.arange(100_000))
            assert np.unique(ids).size == ids.size              # distinct ranks, distinct ids
            assert not (k == np.iinfo(np.int64).min).any()      # the reserved empty-slot id
        else:
            assert k.min() >= 0 and k.max() < spec.rows
    again = ci.make_batch(w)
    assert np.array_equal(again.keys, b.keys) and np.array_equal(again.offsets, b.offsets)
    other = ci.make_batch(w, seed=w.seed + 1)
    assert not np.array_equal(other.keys[:64], b.keys[:64])


def test_upstream_gradient_is_standard_normal():
    w = ci.workload("tiny")
    g = ci.make_grad(w)
    assert g.dtype == np.float32 and g.shape == (w.batch, w.total_dim)
    n = g.size
    assert abs(float(g.mean())) < 6 / np.sqrt(n)
    assert abs(float(g.std()) - 1.0) < 6 / np.sqrt(2 * n)
    assert np.array_equal(g, ci.make_grad(w))


def test_initial_values_are_uniform_on_the_stated_interval():
    w = ci.workload("dlrm")
    v = ci.init_values(w.seed, 3, np.arange(4096), 128, w.w_lo, w.w_hi)
    assert v.dtype == np.float32 and v.min() >= -0.05 and v.max() < 0.05
    # 2^24-point lattice: mean and variance of U(lo, hi) within sampling error
    n = v.size
    assert abs(float(v.mean())) < 6 * 0.1 / np.sqrt(12 * n)
    assert abs(float(v.var()) - 0.1 ** 2 / 12) < 6 * 0.1 ** 2 / np.sqrt(180 * n)
