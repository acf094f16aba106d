"""The allocation-free unique entry point agrees with emb_unique.

emb_unique_noalloc exists for callers that cannot allocate device memory when
they call it (for example a framework plugin whose enqueue path must not call
cudaMalloc).  It runs emb_unique's computation on a scratch array compiled
into the library.  This file is named so that pytest collects it last; it
passes both on its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def _call(fn_name, keys_np, with_workspace):
    import torch
    from dlrm_sparse_embedding_gb300 import lib, unique_workspace_bytes
    dev = torch.device("cuda", 0)
    n = keys_np.size
    keys = torch.from_numpy(keys_np).to(dev)
    m = max(n, 1)
    uniq = torch.full((m,), -7, dtype=torch.int64, device=dev)
    inv = torch.full((m,), -7, dtype=torch.int32, device=dev)
    cnt = torch.full((m,), -7, dtype=torch.int32, device=dev)
    seg = torch.full((m + 1,), -7, dtype=torch.int32, device=dev)
    nu = torch.full((1,), -7, dtype=torch.int64, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if with_workspace:
        ws_bytes = unique_workspace_bytes(n)
        ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
        base = (ws.data_ptr() + 255) & ~255
        rc = lib.emb_unique(_vp(keys), n, _vp(uniq), _vp(inv), _vp(cnt), _vp(seg), _vp(nu),
                            ctypes.c_void_p(base), ws_bytes, stream)
    else:
        rc = lib.emb_unique_noalloc(_vp(keys), n, _vp(uniq), _vp(inv), _vp(cnt), _vp(seg), _vp(nu), stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    U = int(nu.item())
    return U, uniq[:U].cpu().numpy(), inv[:n].cpu().numpy(), cnt[:U].cpu().numpy(), seg[:U + 1].cpu().numpy()


def test_noalloc_unique_matches_emb_unique_on_two_calls_in_a_row():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    torch.cuda.set_device(0)
    from dlrm_sparse_embedding_gb300._lib import UNIQUE_NOALLOC_MAX_KEYS
    rng = np.random.default_rng(2024)
    first = rng.integers(-(1 << 40), 1 << 40, size=UNIQUE_NOALLOC_MAX_KEYS, dtype=np.int64)
    first[::3] = first[7]                                  # heavy duplicates
    second = rng.integers(0, 50, size=777, dtype=np.int64)  # smaller, different range: stale contents must not leak
    import oracle
    for keys in (first, second):
        ref = _call("emb_unique", keys, with_workspace=True)
        got = _call("emb_unique_noalloc", keys, with_workspace=False)
        # integer outputs: identical, element by element
        assert got[0] == ref[0]
        for a, b in zip(got[1:], ref[1:]):
            assert np.array_equal(a, b)
        # and the CPU oracle's sort + run-length unique, directly
        u, inv, cnt, seg = oracle.unique(keys)
        assert got[0] == u.size
        assert np.array_equal(got[1], u) and np.array_equal(got[2], inv)
        assert np.array_equal(got[3], cnt) and np.array_equal(got[4], seg)


def test_noalloc_unique_rejects_sizes_beyond_its_scratch():
    import torch
    from dlrm_sparse_embedding_gb300 import EMB_ERR_INVALID_ARG, lib
    from dlrm_sparse_embedding_gb300._lib import UNIQUE_NOALLOC_MAX_KEYS
    n = UNIQUE_NOALLOC_MAX_KEYS + 1
    keys = torch.zeros(n, dtype=torch.int64, device="cuda")
    out = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    o32 = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    rc = lib.emb_unique_noalloc(_vp(keys), n, _vp(out), _vp(o32), _vp(o32), _vp(o32), _vp(out),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == EMB_ERR_INVALID_ARG
