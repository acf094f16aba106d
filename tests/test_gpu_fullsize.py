"""Parity at the full workload sizes, in the launch configuration bench.py times.

The oracle cannot redo whole steps of this size in test time, so each run is
checked on
  * sampled forward rows, recomputed by the oracle from the sampled bags;
  * the dedup outputs as a whole, through properties that fix them uniquely
    (ascending unique ids, unique[inverse[i]] == global id of lookup i,
    counts == histogram of the inverse / run lengths of the sorted ids,
    seg_offsets == exclusive prefix of counts), plus sampled groups of the
    sorted bag list;
  * sampled updated rows -- the heaviest rows plus random ones -- whose
    gradient sums the oracle recomputes with one pass over all lookups;
  * sampled untouched rows, which must still hold their initial values.
"""
import numpy as np
import pytest

import ctr_inputs as ci
import oracle
from helpers import TOL, gather_rows, max_rel_err, ref_state, report_plain

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

_CACHE = {}


def _inputs(name):
    if name not in _CACHE:
        _CACHE.clear()
        w = ci.workload(name)
        batch = ci.make_batch(w)
        grad = ci.make_grad(w)
        gids, _ = oracle.global_ids(w.tables, w.batch, batch.offsets, batch.keys, batch.table_ids)
        _CACHE[name] = (w, batch, grad, gids)
    return _CACHE[name]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    torch.cuda.set_device(0)
    yield
    _CACHE.clear()


# grouped by workload, so each workload's inputs are generated once
CASES = [("dlrm", "reduction"), ("dlrm", "unique_hash"), ("dlrm_rowwise", "reduction"), ("huge_master", "reduction"),
         ("multihot", "reduction"), ("multihot", "unique_sort"), ("multihot", "unique_hash"),
         ("huge", "reduction"), ("huge", "unique_hash"),
         ("skew", "reduction"), ("skew", "unique_sort"), ("skew", "unique_hash")]


@pytest.mark.parametrize("name,variant", CASES)
def test_fullsize_sampled_parity(name, variant):
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_OK, EmbeddingLayer
    w, batch, grad, gids = _inputs(name)
    seed = w.seed
    dev = torch.device("cuda", 0)
    B, T = w.batch, w.num_tables
    rng = np.random.default_rng(123)
    layer = EmbeddingLayer(w.tables, B, batch.nnz)
    try:
        layer.init_uniform(seed, w.w_lo, w.w_hi)
        out = layer.forward(torch.from_numpy(batch.keys).to(dev), torch.from_numpy(batch.offsets).to(dev),
                            torch.from_numpy(batch.table_ids).to(dev), B)
        bsample = np.sort(rng.choice(B, size=min(B, 192), replace=False))
        out_s = out[torch.from_numpy(bsample).to(dev)].cpu().numpy()
        del out
        layer.set_keep_dedup(True)
        layer.backward_update(torch.from_numpy(grad).to(dev), variant)
        assert layer.sync_status() == EMB_OK
        u_t, inv_t, cnt_t, seg_t, bags_t = layer.dedup_result(with_inverse=variant != "reduction")
        uniq, cnt, seg = u_t.cpu().numpy(), cnt_t.cpu().numpy(), seg_t.cpu().numpy()
        inv = None if inv_t is None else inv_t.cpu().numpy()
        sbags = bags_t.cpu().numpy()
        del u_t, inv_t, cnt_t, seg_t, bags_t

        # ---- forward, sampled bags (all tables of the sampled samples) ----
        bags = (np.arange(T)[:, None] * B + bsample[None, :]).reshape(-1)
        pos = np.concatenate([np.arange(batch.offsets[j], batch.offsets[j + 1]) for j in bags])
        u_s, inv_s, _, _ = oracle.unique(gids[pos], skip_negative=True)
        store = oracle.make_row_store(w.tables, u_s, lambda t, r: ci.init_values(
            seed, t, r, w.tables[t].dim, w.w_lo, w.w_hi, w.tables[t].dtype))
        full_inv = np.full(batch.nnz, u_s.size, dtype=np.int32)
        full_inv[pos] = inv_s
        ref_out, ref_scale = oracle.forward(w.tables, B, batch.offsets, full_inv, store, bags=bags, want_scale=True)
        assert max_rel_err(out_s, ref_out[bsample], ref_scale[bsample]) <= 1e-5
        assert report_plain("%s/%s full size" % (name, variant), "forward", out_s, ref_out[bsample]) <= 1e-5

        # ---- dedup: properties that fix the result uniquely ----
        valid = gids >= 0
        nvalid = int(valid.sum())
        U = uniq.size
        assert np.all(np.diff(uniq) > 0)
        assert np.all(cnt > 0) and int(cnt.sum()) == nvalid
        assert seg[0] == 0 and np.array_equal(np.diff(seg), cnt)
        if inv is not None:
            assert np.array_equal(uniq[inv[valid]], gids[valid])
            assert np.all(inv[~valid] == U)
            assert np.array_equal(np.bincount(inv[valid], minlength=U), cnt)
        else:
            assert np.array_equal(np.repeat(uniq, cnt), np.sort(gids[valid]))
        lens = np.diff(batch.offsets)
        heavy = np.argsort(cnt)[-8:]
        for k in np.concatenate([heavy, rng.choice(U, size=min(U, 24), replace=False)]):
            where = np.nonzero(gids == uniq[k])[0]
            expect = np.searchsorted(batch.offsets, where, side="right") - 1
            assert np.array_equal(sbags[seg[k]:seg[k + 1]], expect.astype(np.int32))

        # ---- updated rows: heaviest + random sample ----
        pick = np.unique(np.concatenate([np.argsort(cnt)[-12:], rng.choice(U, size=min(U, 244), replace=False)]))
        sample = uniq[pick]
        G, Gabs, count = oracle.reduce_sampled(w.tables, B, batch.offsets, gids, sample, grad)
        assert np.array_equal(count, cnt[pick])
        # the update starts from the fp32 master where a table has one
        def start_values(t, r):
            spec = w.tables[t]
            if spec.master:
                return ci.init_values(seed, t, r, spec.dim, w.w_lo, w.w_hi, "f32")
            return ci.stored_to_f64(ci.init_values(seed, t, r, spec.dim, w.w_lo, w.w_hi, spec.dtype),
                                    spec.dtype).astype(np.float32)

        st = oracle.make_row_store(w.tables, sample, start_values, fp32_values=True)
        state = oracle.make_row_store(w.tables, sample, None, state_init=True)
        Gflat = np.concatenate([G[q, :w.tables[st.table[q]].dim] for q in range(sample.size)])
        Gaflat = np.concatenate([Gabs[q, :w.tables[st.table[q]].dim] for q in range(sample.size)])
        M, A, Ws, As, W = oracle.update(w.tables, st, state, Gflat, Gaflat)
        for t, spec in enumerate(w.tables):
            sel = np.nonzero(st.table == t)[0]
            if sel.size == 0:
                continue
            gw, ga = gather_rows(layer, w, t, st.row[sel])
            idx = st.row_start[sel][:, None] + np.arange(spec.dim)[None, :]
            assert max_rel_err(gw, W[idx], Ws[idx]) <= TOL[spec.dtype], (name, variant, t)
            report_plain("%s/%s full size" % (name, variant), "weights_" + spec.dtype, gw, W[idx])
            if spec.master:
                gm = layer.gather_master_rows(t, torch.from_numpy(np.ascontiguousarray(st.row[sel])).cuda())
                assert max_rel_err(gm.cpu().numpy(), M[idx], Ws[idx]) <= 1e-5, (name, variant, t)
            if spec.opt != "sgd":
                ra, rs = ref_state(spec, A, As, idx)
                assert max_rel_err(ga, ra, rs) <= 1e-5, (name, variant, t)

        # ---- untouched rows keep their initial values ----
        rb = oracle.row_base([s.rows for s in w.tables])
        for t, spec in enumerate(w.tables[:8]):
            cand = rng.integers(0, spec.rows, size=64)
            g = rb[t] + cand
            k = np.searchsorted(uniq, g)
            untouched = cand[(k >= U) | (uniq[np.minimum(k, U - 1)] != g)]
            if untouched.size == 0:
                continue
            gw, ga = gather_rows(layer, w, t, untouched)
            init = ci.stored_to_f64(ci.init_values(seed, t, untouched, spec.dim, w.w_lo, w.w_hi, spec.dtype),
                                    spec.dtype)
            assert np.array_equal(gw, init)
            if ga is not None:
                assert np.all(ga == np.float32(spec.init_acc))
    finally:
        layer.close()
