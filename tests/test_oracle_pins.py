"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a fact fixed independently of its code:
a hand-worked example, closed forms, invariants, brute force on tiny inputs,
or an independent library routine (NumPy / PyTorch CPU in float64).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import ctr_inputs as ci
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spec(rows, dim, pooling="sum", opt="sgd", lr=0.01, eps=1e-8, dtype="f32"):
    return ci.TableSpec(rows, dim, dtype, pooling, opt, lr, eps)


def _dense_rows(weights):
    """init_rows callback over explicit per-table float32 weight arrays."""
    return lambda t, r: np.asarray(weights[t], dtype=np.float32)[np.asarray(r, dtype=np.int64)]


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------

def test_f16_decode_and_round_trip_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    dec = oracle.stored_to_f64(bits, "f16")
    fin = np.isfinite(ref)
    assert np.array_equal(dec[fin], ref[fin])
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    back = oracle.round_f16(dec[fin])
    assert np.array_equal(back, bits[fin])
    # the scalar C decoder agrees with the vectorised one
    some = bits[::257]
    assert np.array_equal(oracle.decode(some, "f16")[np.isfinite(ref[::257])],
                          ref[::257][np.isfinite(ref[::257])])


def test_f16_rounding_matches_numpy_on_random_doubles():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-8, 5, 200000),
        # exact midpoints between neighbouring halves (ties go to even)
        (np.arange(0, 65504, 0.5) + 0.25)[::37],
        np.array([65519.99, 65520.0, 65536.0, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -24 * 1.5]),
    ])
    ours = oracle.round_f16(x)
    with np.errstate(over="ignore"):             # values beyond the fp16 range become inf on purpose
        ref = x.astype(np.float16).view(np.uint16)   # numpy rounds binary64 -> binary16 directly, RNE
    assert np.array_equal(ours, ref)


def _bf16_exact(x: float) -> float:
    """RNE of a binary64 to bfloat16 by exact rational arithmetic."""
    if x == 0:
        return 0.0
    f = Fraction(x)
    s = -1 if f < 0 else 1
    f = abs(f)
    e = f.numerator.bit_length() - f.denominator.bit_length()
    while Fraction(2) ** e > f:
        e -= 1
    while Fraction(2) ** (e + 1) <= f:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    n = f / q
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    v = lo * q
    if v >= Fraction(2) ** 128:
        return s * float("inf")
    return s * float(v)


def test_bf16_round_trip_exhaustive_and_exact_rounding():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # the NaN patterns are among the 65536
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dec = oracle.stored_to_f64(bits, "bf16")
    fin = np.isfinite(ref)
    assert np.array_equal(dec[fin], ref[fin])
    assert np.array_equal(oracle.round_bf16(dec[fin]), bits[fin])
    rng = np.random.default_rng(7)
    x = rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000)
    mids = (ref[fin][:-1][::97] + ref[fin][1:][::97]) / 2.0          # exact ties
    x = np.concatenate([x, mids[np.isfinite(mids)]])
    ours = oracle.stored_to_f64(oracle.round_bf16(x), "bf16")
    exact = np.array([_bf16_exact(float(v)) for v in x])
    assert np.array_equal(ours, exact)
    # binary32 inputs: torch's conversion is a single RNE step there
    x32 = rng.standard_normal(100000).astype(np.float32)
    t = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(x32.astype(np.float64)), t)


# ---------------------------------------------------------------------------
# a2 / a3: global ids and unique
# ---------------------------------------------------------------------------

def test_global_ids_brute_force_and_invalid_positions():
    tables = [_spec(5, 4), _spec(3, 4), _spec(7, 4)]
    B = 4
    rng = np.random.default_rng(0)
    lens = rng.integers(0, 4, size=3 * B)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    keys = rng.integers(-1, 8, size=int(offsets[-1])).astype(np.int64)
    table_ids = np.repeat(np.arange(3, dtype=np.int32), B)
    table_ids[5] = 0           # bag 5 belongs to table 1: wrong id -> invalid bag
    gids, bad = oracle.global_ids(tables, B, offsets, keys, table_ids)
    base = [0, 5, 8]
    exp_bad = 0
    for j in range(3 * B):
        t = j // B
        if table_ids[j] != t:
            exp_bad += 1
        for i in range(offsets[j], offsets[j + 1]):
            ok = table_ids[j] == t and 0 <= keys[i] < tables[t].rows
            assert gids[i] == (base[t] + keys[i] if ok else -1)
            if table_ids[j] == t and not ok:
                exp_bad += 1
    assert bad == exp_bad


@pytest.mark.parametrize("n,hi", [(0, 5), (1, 5), (37, 4), (500, 50), (2000, 100000), (2000, 3)])
def test_unique_brute_force_and_library(n, hi):
    rng = np.random.default_rng(n + hi)
    keys = rng.integers(-hi, hi, size=n).astype(np.int64)
    u, inv, cnt, seg = oracle.unique(keys)
    # brute force, O(n^2)
    distinct = []
    for k in keys.tolist():
        if k not in distinct:
            distinct.append(k)
    distinct.sort()
    assert u.tolist() == distinct
    assert [sum(1 for x in keys.tolist() if x == d) for d in distinct] == cnt.tolist()
    assert all(distinct[inv[i]] == keys[i] for i in range(n))
    # invariants
    assert int(cnt.sum()) == n and seg[-1] == n and seg[0] == 0
    assert np.all(np.diff(u) > 0) and np.all(cnt > 0)
    assert np.array_equal(np.diff(seg), cnt)
    # independent library routines
    nu, ninv, ncnt = np.unique(keys, return_inverse=True, return_counts=True)
    assert np.array_equal(u, nu) and np.array_equal(inv, ninv.reshape(-1)) and np.array_equal(cnt, ncnt)
    tu, tinv, tcnt = torch.unique(torch.from_numpy(keys), sorted=True, return_inverse=True,
                                  return_counts=True)
    assert np.array_equal(u, tu.numpy()) and np.array_equal(inv, tinv.numpy())
    assert np.array_equal(cnt, tcnt.numpy())


def test_unique_skip_negative_maps_to_U():
    keys = np.array([5, -1, 3, 5, -1, 9], dtype=np.int64)
    u, inv, cnt, seg = oracle.unique(keys, skip_negative=True)
    assert u.tolist() == [3, 5, 9] and cnt.tolist() == [1, 2, 1] and seg.tolist() == [0, 1, 3, 4]
    assert inv.tolist() == [1, 3, 0, 1, 3, 2]


# ---------------------------------------------------------------------------
# hand-worked example
# ---------------------------------------------------------------------------

def _load_golden():
    with open(os.path.join(GOLDEN, "hand_worked_step.json")) as f:
        return json.load(f)


def _val(x):
    return float(Fraction(x)) if isinstance(x, str) else float(x)


@pytest.mark.parametrize("opt", ["sgd", "adagrad"])
def test_hand_worked_example(opt):
    g = _load_golden()
    lr = g["sgd_lr"] if opt == "sgd" else g["adagrad_lr"]
    eps = 0.0 if opt == "sgd" else g["adagrad_eps"]
    tables = [_spec(t["rows"], t["dim"], t["pooling"], opt, lr, eps) for t in g["tables"]]
    res = oracle.step(tables, g["batch"], np.array(g["offsets"]), np.array(g["keys"]),
                      np.array(g["table_ids"], dtype=np.int32), np.array(g["grad_out"], np.float32),
                      _dense_rows(g["weights"]))
    assert res.out.tolist() == g["out"]
    assert res.gids.tolist() == g["gids"]
    assert res.unique.tolist() == g["unique"] and res.inverse.tolist() == g["inverse"]
    assert res.counts.tolist() == g["counts"] and res.seg_off.tolist() == g["seg_off"]
    rs = res.rows.row_start
    dims = [tables[t].dim for t in res.rows.table]
    for k in range(len(g["unique"])):
        assert res.G[rs[k]:rs[k] + dims[k]].tolist() == g["G"][k]
        want_W = g["sgd_W"][k] if opt == "sgd" else [_val(v) for v in g["adagrad_W"][k]]
        want_W = np.float32(np.array(want_W, dtype=np.float64)).astype(np.float64)
        assert res.W[rs[k]:rs[k] + dims[k]].tolist() == want_W.tolist()
        if opt == "adagrad":
            assert res.A[rs[k]:rs[k] + dims[k]].tolist() == g["adagrad_A"][k]


# ---------------------------------------------------------------------------
# a1: forward
# ---------------------------------------------------------------------------

def _random_csr(T, B, rows, max_len, seed, allow_empty=True):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0 if allow_empty else 1, max_len + 1, size=T * B)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    keys = np.empty(int(offsets[-1]), dtype=np.int64)
    for j in range(T * B):
        t = j // B
        keys[offsets[j]:offsets[j + 1]] = rng.integers(0, rows[t], size=lens[j])
    return offsets, keys, np.repeat(np.arange(T, dtype=np.int32), B)


@pytest.mark.parametrize("pooling", ["sum", "mean"])
def test_forward_all_ones_gives_hotness(pooling):
    rows, dims, B = [10, 20, 5], [4, 8, 16], 9
    tables = [_spec(r, d, pooling) for r, d in zip(rows, dims)]
    offsets, keys, tid = _random_csr(3, B, rows, 6, 1)
    ones = [np.ones((r, d), np.float32) for r, d in zip(rows, dims)]
    gids, _ = oracle.global_ids(tables, B, offsets, keys, tid)
    u, inv, _, _ = oracle.unique(gids, skip_negative=True)
    out = oracle.forward(tables, B, offsets, inv, oracle.make_row_store(tables, u, _dense_rows(ones)))
    lens = np.diff(offsets).reshape(3, B)
    col = 0
    for t in range(3):
        expect = lens[t].astype(np.float32) if pooling == "sum" else (lens[t] > 0).astype(np.float32)
        assert np.array_equal(out[:, col:col + dims[t]], np.repeat(expect[:, None], dims[t], 1))
        col += dims[t]


def test_forward_one_hot_copies_rows_exactly():
    rows, dims, B = [50, 30], [8, 4], 16
    tables = [_spec(r, d) for r, d in zip(rows, dims)]
    offsets = np.arange(2 * B + 1, dtype=np.int64)
    rng = np.random.default_rng(3)
    keys = np.concatenate([rng.integers(0, 50, B), rng.integers(0, 30, B)]).astype(np.int64)
    W = [rng.standard_normal((r, d)).astype(np.float32) for r, d in zip(rows, dims)]
    gids, _ = oracle.global_ids(tables, B, offsets, keys, np.repeat(np.arange(2, dtype=np.int32), B))
    u, inv, _, _ = oracle.unique(gids, skip_negative=True)
    out = oracle.forward(tables, B, offsets, inv, oracle.make_row_store(tables, u, _dense_rows(W)))
    assert np.array_equal(out[:, :8], W[0][keys[:B]])
    assert np.array_equal(out[:, 8:], W[1][keys[B:]])


@pytest.mark.parametrize("pooling", ["sum", "mean"])
def test_forward_matches_torch_embedding_bag_f64(pooling):
    rows, dims, B = [100, 7, 1000], [16, 32, 4], 33
    tables = [_spec(r, d, pooling) for r, d in zip(rows, dims)]
    offsets, keys, tid = _random_csr(3, B, rows, 12, 4)
    rng = np.random.default_rng(8)
    W = [rng.uniform(-1, 1, (r, d)).astype(np.float32) for r, d in zip(rows, dims)]
    gids, _ = oracle.global_ids(tables, B, offsets, keys, tid)
    u, inv, _, _ = oracle.unique(gids, skip_negative=True)
    out = oracle.forward(tables, B, offsets, inv, oracle.make_row_store(tables, u, _dense_rows(W)))
    col = 0
    for t in range(3):
        o = offsets[t * B:(t + 1) * B + 1]
        ref = torch.nn.functional.embedding_bag(
            torch.from_numpy(keys[o[0]:o[-1]]), torch.from_numpy(W[t].astype(np.float64)),
            torch.from_numpy(o[:-1] - o[0]), mode=pooling).numpy()
        got = out[:, col:col + dims[t]].astype(np.float64)
        assert np.allclose(got, ref.astype(np.float32), rtol=0, atol=0) or \
            np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)) <= 2.0 ** -24
        col += dims[t]


# ---------------------------------------------------------------------------
# a4: reduction
# ---------------------------------------------------------------------------

def test_skipped_lookups_count_in_the_mean_and_pass_no_gradient():
    # one table of 3 rows x 4, mean pooling, SGD with lr 0.5; bags {0, 7, 2}
    # (7 is out of range), {} and {-1}.  Values chosen so every result is exact.
    tables = [_spec(3, 4, "mean", "sgd", lr=0.5)]
    offsets = np.array([0, 3, 3, 4], np.int64)
    keys = np.array([0, 7, 2, -1], np.int64)
    W = np.array([[3, 6, -9, 0], [1, 1, 1, 1], [0, 3, 3, 3]], np.float32)
    grad = np.array([[3, -3, 6, 0], [5, 5, 5, 5], [7, 7, 7, 7]], np.float32)
    res = oracle.step(tables, 3, offsets, keys, np.zeros(3, np.int32), grad, _dense_rows([W]))
    # the mean divides by the whole bag length; empty and all-skipped bags pool to 0
    assert np.array_equal(res.out, np.array([[1, 3, -2, 1], [0, 0, 0, 0], [0, 0, 0, 0]], np.float32))
    assert res.n_bad == 2
    assert res.unique.tolist() == [0, 2] and res.counts.tolist() == [1, 1]
    # rows 0 and 2 each take bag 0's gradient / 3; the skipped lookups touch no row
    assert res.rows.row.tolist() == [0, 2] and res.rows.row_start.tolist() == [0, 4]
    assert np.array_equal(res.W, np.array([2.5, 6.5, -10, 0, -0.5, 3.5, 2, 3], np.float64))


@pytest.mark.parametrize("pooling", ["sum", "mean"])
def test_reduce_broadcasts_to_every_member(pooling):
    # every key distinct: G of each position's row is exactly s_j * grad_out[b]
    rows, dims, B = [200, 300], [4, 8], 10
    tables = [_spec(r, d, pooling) for r, d in zip(rows, dims)]
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 5, size=2 * B)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    keys = np.concatenate([rng.permutation(rows[t])[:lens[t * B:(t + 1) * B].sum()] for t in range(2)])
    tid = np.repeat(np.arange(2, dtype=np.int32), B)
    grad = rng.standard_normal((B, 12)).astype(np.float32)
    gids, _ = oracle.global_ids(tables, B, offsets, keys.astype(np.int64), tid)
    u, inv, cnt, _ = oracle.unique(gids, skip_negative=True)
    assert np.all(cnt == 1)
    st = oracle.make_row_store(tables, u, _dense_rows([np.zeros((r, d), np.float32) for r, d in zip(rows, dims)]))
    G, _ = oracle.reduce(tables, B, offsets, inv, st, grad)
    for j in range(2 * B):
        t, b = divmod(j, B)
        col = 0 if t == 0 else 4
        for i in range(offsets[j], offsets[j + 1]):
            k = inv[i]
            g = grad[b, col:col + dims[t]].astype(np.float64)
            want = g if pooling == "sum" else g / lens[j]
            assert np.array_equal(G[st.row_start[k]:st.row_start[k] + dims[t]], want)


def test_reduce_column_sums_are_conserved():
    rows, dims, B = [13, 9], [4, 4], 40
    tables = [_spec(r, d, "mean") for r, d in zip(rows, dims)]
    offsets, keys, tid = _random_csr(2, B, rows, 7, 12)
    rng = np.random.default_rng(13)
    grad = rng.standard_normal((B, 8)).astype(np.float32)
    gids, _ = oracle.global_ids(tables, B, offsets, keys, tid)
    u, inv, _, _ = oracle.unique(gids, skip_negative=True)
    st = oracle.make_row_store(tables, u, _dense_rows([np.zeros((r, d), np.float32) for r, d in zip(rows, dims)]))
    G, _ = oracle.reduce(tables, B, offsets, inv, st, grad)
    lens = np.diff(offsets).reshape(2, B)
    for t in range(2):
        sel = np.nonzero(st.table == t)[0]
        got = sum(G[st.row_start[k]:st.row_start[k] + 4] for k in sel)
        # each bag passes grad/L to each of its L members: column total = sum over non-empty bags
        want = (grad[:, 4 * t:4 * t + 4].astype(np.float64) * (lens[t] > 0)[:, None]).sum(0)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_reduce_sampled_matches_full():
    rows, dims, B = [60, 40], [8, 16], 25
    tables = [_spec(r, d, p) for r, d, p in zip(rows, dims, ["sum", "mean"])]
    offsets, keys, tid = _random_csr(2, B, rows, 9, 21)
    grad = np.random.default_rng(22).standard_normal((B, 24)).astype(np.float32)
    gids, _ = oracle.global_ids(tables, B, offsets, keys, tid)
    u, inv, cnt, _ = oracle.unique(gids, skip_negative=True)
    st = oracle.make_row_store(tables, u, _dense_rows([np.zeros((r, d), np.float32) for r, d in zip(rows, dims)]))
    G, Gabs = oracle.reduce(tables, B, offsets, inv, st, grad)
    sample = u[::3]
    Gs, Gas, cs = oracle.reduce_sampled(tables, B, offsets, gids, sample, grad)
    for q, gid in enumerate(sample):
        k = int(np.searchsorted(u, gid))
        d = tables[st.table[k]].dim
        assert cs[q] == cnt[k]
        assert np.array_equal(Gs[q, :d], G[st.row_start[k]:st.row_start[k] + d])
        assert np.array_equal(Gas[q, :d], Gabs[st.row_start[k]:st.row_start[k] + d])


# ---------------------------------------------------------------------------
# a5: optimizer
# ---------------------------------------------------------------------------

def test_sgd_row_touched_k_times_moves_by_lr_times_sum():
    # row 3 of a single sum-pooled table appears in k one-hot bags
    B, k = 12, 5
    tables = [_spec(10, 8, "sum", "sgd", lr=0.01)]
    keys = np.array([3] * k + list(range(4, 4 + B - k)), dtype=np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    rng = np.random.default_rng(2)
    W0 = rng.uniform(-0.05, 0.05, (10, 8)).astype(np.float32)
    grad = rng.standard_normal((B, 8)).astype(np.float32)
    res = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad, _dense_rows([W0]))
    kk = int(np.searchsorted(res.unique, 3))
    s = res.rows.row_start[kk]
    lr = float(np.float32(0.01))
    want = np.float32(W0[3].astype(np.float64) - lr * grad[:k].astype(np.float64).sum(0))
    assert np.array_equal(res.W[s:s + 8], want.astype(np.float64))


def test_adagrad_single_touch_closed_form():
    B = 6
    tables = [_spec(50, 4, "sum", "adagrad", lr=0.01, eps=1e-8)]
    keys = np.array([1, 7, 9, 11, 20, 33], dtype=np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    rng = np.random.default_rng(9)
    W0 = rng.uniform(-0.05, 0.05, (50, 4)).astype(np.float32)
    grad = rng.standard_normal((B, 4)).astype(np.float32)
    res = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad, _dense_rows([W0]))
    lr, eps = float(np.float32(0.01)), float(np.float32(1e-8))
    for b, key in enumerate(keys):
        k = int(np.searchsorted(res.unique, key))
        s = res.rows.row_start[k]
        g = grad[b].astype(np.float64)
        want = np.float32(W0[key].astype(np.float64) - lr * g / (np.abs(g) + eps))
        assert np.array_equal(res.W[s:s + 4], want.astype(np.float64))
        assert np.array_equal(res.A[s:s + 4], np.float32(g * g).astype(np.float64))


def test_rowwise_adagrad_hand_example():
    # lr 1/2 and eps 0 keep every intermediate exact: row 1 gets G = (3, 4, 0, 0),
    # mean of squares 25/4, sqrt 5/2, step (3, 4, 0, 0) / 5 = (0.6, 0.8, 0, 0);
    # row 2 gets G = (2, 2, 2, 2), mean of squares 4, sqrt 2, step 1/2 per column
    B = 2
    tables = [_spec(5, 4, "sum", "rowwise_adagrad", lr=0.5, eps=0.0)]
    keys = np.array([1, 2], dtype=np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    W0 = np.ones((5, 4), dtype=np.float32)
    grad = np.array([[3, 4, 0, 0], [2, 2, 2, 2]], dtype=np.float32)
    res = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad, _dense_rows([W0]))
    s1, s2 = res.rows.row_start[0], res.rows.row_start[1]
    assert res.W[s1:s1 + 4].tolist() == [float(np.float32(0.4)), float(np.float32(0.2)), 1.0, 1.0]
    assert res.A[s1:s1 + 4].tolist() == [6.25] * 4
    assert res.W[s2:s2 + 4].tolist() == [0.5] * 4
    assert res.A[s2:s2 + 4].tolist() == [4.0] * 4


def test_rowwise_adagrad_equals_elementwise_when_a_row_has_one_magnitude():
    # when every column of a row's gradient has the same magnitude and the row
    # starts from one accumulator value, the mean of squares is that square, so
    # the row-wise step is the element-wise one (pinned against torch below)
    B, dim = 12, 8
    rng = np.random.default_rng(41)
    keys = np.concatenate([[7, 7, 7, 7], rng.choice(np.arange(8, 30), B - 4, replace=False)]).astype(np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    W0 = rng.uniform(-0.05, 0.05, (30, dim)).astype(np.float32)
    signs = rng.choice([-1.0, 1.0], size=(B, dim))
    # dyadic magnitudes keep the sums of squares exact in binary64
    grad = (signs * (rng.integers(1, 9, (B, 1)) / 4.0)).astype(np.float32)
    grad[:4] = np.abs(grad[:4]) * np.sign(grad[0])    # same signs within the row touched four times
    res = {}
    for opt in ("adagrad", "rowwise_adagrad"):
        tables = [_spec(30, dim, "sum", opt, lr=0.01, eps=1e-8)]
        res[opt] = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad, _dense_rows([W0]))
    assert np.array_equal(res["adagrad"].W, res["rowwise_adagrad"].W)
    assert np.array_equal(res["adagrad"].A, res["rowwise_adagrad"].A)


def test_rowwise_adagrad_accumulator_is_one_value_per_row_and_column_order_free():
    B, dim = 16, 12
    rng = np.random.default_rng(43)
    keys = rng.integers(0, 40, B).astype(np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    W0 = rng.uniform(-0.05, 0.05, (40, dim)).astype(np.float32)
    grad = rng.standard_normal((B, dim)).astype(np.float32)
    perm = rng.permutation(dim)
    tables = [_spec(40, dim, "sum", "rowwise_adagrad")]
    a = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad, _dense_rows([W0]))
    b = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad[:, perm],
                    _dense_rows([W0[:, perm]]))
    for k in range(a.unique.shape[0]):
        s = a.rows.row_start[k]
        row_a = a.A[s:s + dim]
        assert np.all(row_a == row_a[0]) and row_a[0] > 0
        # permuting the columns permutes the weights and leaves the accumulator alone
        assert np.array_equal(b.A[s:s + dim], row_a)
        assert np.array_equal(b.W[s:s + dim], a.W[s:s + dim][perm])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("opt", ["sgd", "adagrad", "rowwise_adagrad"])
def test_master_copy_follows_the_fp32_table(dtype, opt):
    # the gradient does not depend on the weights (grad_out is given), so a
    # 16-bit table's fp32 master must take exactly the fp32 table's steps, and
    # its stored copy is that master rounded to nearest-even (NumPy's fp16
    # conversion, torch's bf16 conversion)
    rows, dim, B = 60, 8, 40
    rng = np.random.default_rng(51)
    keys = rng.integers(0, rows, B).astype(np.int64)
    keys[:9] = 17
    offsets = np.arange(B + 1, dtype=np.int64)
    W0 = rng.uniform(-0.05, 0.05, (rows, dim)).astype(np.float32)
    grad = rng.standard_normal((B, dim)).astype(np.float32)
    tid = np.zeros(B, np.int32)
    ref = oracle.step([_spec(rows, dim, "sum", opt)], B, offsets, keys, tid, grad, _dense_rows([W0]))
    spec = ci.TableSpec(rows, dim, dtype, "sum", opt, 0.01, 1e-8, 0.0, master=True)
    if dtype == "f16":
        stored = W0.astype(np.float16)
    else:
        stored = torch.from_numpy(W0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    res = oracle.step([spec], B, offsets, keys, tid, grad, lambda t, r: stored[r], lambda t, r: W0[r])
    assert np.array_equal(res.M, ref.W)
    assert np.array_equal(res.A, ref.A)
    m32 = res.M.astype(np.float32)
    if dtype == "f16":
        want = m32.astype(np.float16).astype(np.float64)
    else:
        want = torch.from_numpy(m32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(res.W, want)


def test_master_copy_keeps_a_step_below_half_a_16bit_ulp():
    # fp16 spacing just below 1 is 2^-11.  A step of 2^-12 from 1.0 lands on the
    # tie 1 - 2^-12, which rounds to the even neighbour 1.0: without a master
    # the stored weight does not move; with one the master holds 1 - 2^-12 and
    # the stored copy is 1.0.  Row 2, hit twice, moves by 2^-11 to 1 - 2^-11.
    B = 3
    lr = 2.0 ** -12
    keys = np.array([1, 2, 2], dtype=np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    W0 = np.ones((4, 4), dtype=np.float32)
    grad = np.ones((B, 4), dtype=np.float32)
    tid = np.zeros(B, np.int32)
    plain = oracle.step([ci.TableSpec(4, 4, "f16", "sum", "sgd", lr)], B, offsets, keys, tid, grad,
                        lambda t, r: W0.astype(np.float16)[r])
    mast = oracle.step([ci.TableSpec(4, 4, "f16", "sum", "sgd", lr, master=True)], B, offsets, keys, tid, grad,
                       lambda t, r: W0.astype(np.float16)[r], lambda t, r: W0[r])
    assert plain.W.tolist() == [1.0] * 4 + [0.99951171875] * 4
    assert mast.W.tolist() == [1.0] * 4 + [0.99951171875] * 4
    assert mast.M.tolist() == [0.999755859375] * 4 + [0.99951171875] * 4


def test_dynamic_table_is_the_static_table_over_its_keys():
    # a dynamic table over scrambled 64-bit ids gives exactly the static
    # table's step over the ranks, row for row (each id's row starts at the
    # value the static table's row for its rank starts at)
    B, rows, dim = 300, 64, 8
    offsets, keys, tid = _random_csr(2, B, [rows, rows], 5, 61)
    rng = np.random.default_rng(62)
    grad = rng.standard_normal((B, 2 * dim)).astype(np.float32)
    ids = {t: ci.dynamic_key(t, np.arange(rows)) for t in range(2)}
    keys_dyn = keys.copy()
    lo = offsets[B]
    keys_dyn[lo:] = ids[1][keys[lo:]]                       # table 1 dynamic, table 0 static
    W0 = [rng.uniform(-0.05, 0.05, (rows, dim)).astype(np.float32) for _ in range(2)]
    static = [_spec(rows, dim, "sum", "adagrad"), _spec(rows, dim, "mean", "rowwise_adagrad")]
    ref = oracle.step(static, B, offsets, keys, tid, grad, _dense_rows(W0))
    rank_of = {int(k): r for r, k in enumerate(ids[1])}
    dyn_specs = [static[0], ci.TableSpec(2 * rows, dim, "f32", "mean", "rowwise_adagrad", 0.01, 1e-8, dynamic=True)]
    res, key_of = oracle.step_dynamic(dyn_specs, B, offsets, keys_dyn, tid, grad, _dense_rows(W0),
                                      lambda t, k: W0[t][[rank_of[int(x)] for x in k]])
    assert np.array_equal(res.out, ref.out)
    for k in range(res.unique.shape[0]):
        t, r = int(res.rows.table[k]), int(res.rows.row[k])
        rank = r if t == 0 else rank_of[int(key_of[1][r])]
        kr = int(np.nonzero((ref.rows.table == t) & (ref.rows.row == rank))[0][0])
        a, b = res.rows.row_start[k], ref.rows.row_start[kr]
        assert np.array_equal(res.W[a:a + dim], ref.W[b:b + dim])
        assert np.array_equal(res.A[a:a + dim], ref.A[b:b + dim])


def test_forward_with_cache_reduces_to_the_plain_forward():
    # no cached rows: the training forward's output exactly; every row cached
    # but the table already fp16: unchanged again; an fp32 table's cached row
    # contributes its fp16 rounding
    B, dim = 64, 8
    offsets, keys, tid = _random_csr(2, B, [40, 40], 4, 71)
    rng = np.random.default_rng(72)
    W32 = rng.uniform(-0.05, 0.05, (40, dim)).astype(np.float32)
    W16 = rng.uniform(-0.05, 0.05, (40, dim)).astype(np.float16)
    tables = [_spec(40, dim), _spec(40, dim, dtype="f16")]
    init = lambda t, r: (W32 if t == 0 else W16)[r]
    grad = np.zeros((B, 2 * dim), np.float32)
    plain = oracle.step(tables, B, offsets, keys, tid, grad, init).out
    out0, _ = oracle.forward_with_cache(tables, B, offsets, keys, tid, init, {})
    assert np.array_equal(out0, plain)
    out1, _ = oracle.forward_with_cache(tables, B, offsets, keys, tid, init, {1: np.arange(40)})
    assert np.array_equal(out1, plain)
    # one-hot bags of table 0 holding row 3 now pool its fp16 value
    one = np.arange(B + 1, dtype=np.int64)
    k1 = np.full(B, 3, np.int64)
    t1 = [_spec(40, dim)]
    out2, _ = oracle.forward_with_cache(t1, B, one, k1, np.zeros(B, np.int32), lambda t, r: W32[r], {0: [3, 7]})
    assert np.array_equal(out2, np.broadcast_to(W32[3].astype(np.float16).astype(np.float32), (B, dim)))


def _torch_reference_step(tables, B, offsets, keys, grad, W, opt_name):
    """Independent reference: torch embedding_bag (float64, sparse grads) + torch.optim."""
    outs, params = [], []
    for t, spec in enumerate(tables):
        p = torch.nn.Parameter(torch.from_numpy(W[t].astype(np.float64)))
        params.append(p)
        o = offsets[t * B:(t + 1) * B + 1]
        outs.append(torch.nn.functional.embedding_bag(
            torch.from_numpy(keys[o[0]:o[-1]]), p, torch.from_numpy(o[:-1] - o[0]),
            mode=spec.pooling, sparse=True))
    out = torch.cat(outs, dim=1)
    out.backward(torch.from_numpy(grad.astype(np.float64)))
    lr = float(np.float32(tables[0].lr))
    if opt_name == "sgd":
        opt = torch.optim.SGD(params, lr=lr)
    else:
        opt = torch.optim.Adagrad(params, lr=lr, eps=float(np.float32(tables[0].eps)),
                                  initial_accumulator_value=0.0)
    opt.step()
    state = [opt.state[p]["sum"].numpy() if opt_name == "adagrad" else None for p in params]
    return out.detach().numpy(), [p.detach().numpy() for p in params], state


@pytest.mark.parametrize("opt_name", ["sgd", "adagrad"])
@pytest.mark.parametrize("pooling", ["sum", "mean"])
def test_full_step_matches_torch_autograd_and_optim(opt_name, pooling):
    rows, dims, B = [30, 17, 64], [8, 4, 16], 20
    tables = [_spec(r, d, pooling, opt_name, lr=0.01, eps=1e-8) for r, d in zip(rows, dims)]
    offsets, keys, tid = _random_csr(3, B, rows, 6, 31)
    rng = np.random.default_rng(32)
    W = [rng.uniform(-0.05, 0.05, (r, d)).astype(np.float32) for r, d in zip(rows, dims)]
    grad = rng.standard_normal((B, sum(dims))).astype(np.float32)
    res = oracle.step(tables, B, offsets, keys, tid, grad, _dense_rows(W))
    ref_out, ref_W, ref_A = _torch_reference_step(tables, B, offsets, keys, grad, W, opt_name)
    assert np.max(np.abs(res.out - ref_out)) <= 2.0 ** -24 * np.max(np.abs(ref_out)) * 4
    for k, gid in enumerate(res.unique):
        t, r = int(res.rows.table[k]), int(res.rows.row[k])
        s, d = res.rows.row_start[k], dims[t]
        ref = ref_W[t][r]
        got = res.W[s:s + d]
        # oracle rounds once to fp32; torch keeps float64
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -24 + 1e-300)
        if opt_name == "adagrad":
            assert np.all(np.abs(res.A[s:s + d] - ref_A[t][r]) <= np.abs(ref_A[t][r]) * 2.0 ** -24)
    # untouched rows keep their values in torch as well (no momentum, no decay)
    for t in range(3):
        touched = set(res.rows.row[res.rows.table == t].tolist())
        for r in range(rows[t]):
            if r not in touched:
                assert np.array_equal(ref_W[t][r], W[t][r].astype(np.float64))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_update_rounds_once_into_16bit_storage(dtype):
    B = 8
    tables = [_spec(40, 8, "sum", "adagrad", dtype=dtype)]
    keys = np.array([0, 5, 5, 9, 12, 12, 12, 39], dtype=np.int64)
    offsets = np.arange(B + 1, dtype=np.int64)
    init = lambda t, r: ci.init_values(0, t, r, 8, -0.05, 0.05, dtype)
    grad = np.random.default_rng(4).standard_normal((B, 8)).astype(np.float32)
    res = oracle.step(tables, B, offsets, keys, np.zeros(B, np.int32), grad, init)
    lr, eps = float(np.float32(0.01)), float(np.float32(1e-8))
    for k, key in enumerate(res.unique):
        s = res.rows.row_start[k]
        w0 = oracle.stored_to_f64(init(0, np.array([key])), dtype).reshape(-1)
        g = grad[keys == key].astype(np.float64).sum(0)
        wn = w0 - lr * g / (np.sqrt(g * g) + eps)
        if dtype == "f16":
            want = wn.astype(np.float16).astype(np.float64)
        else:
            want = np.array([_bf16_exact(float(v)) for v in wn])
        assert np.array_equal(res.W[s:s + 8], want)


def test_init_values_are_the_published_splitmix64_stream():
    # splitmix64 from state 0: first outputs as published with the algorithm
    # (Steele, Lea & Flood 2014; the reference C by Vigna, prng.di.unimi.it)
    out = ci.splitmix64_at(0, np.arange(3))
    assert [hex(int(v)) for v in out] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4", "0x6c45d188009454f"]
