"""CPU checks of the C-ABI library: it loads, exports every declared symbol,
and validates host-side arguments without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def emb():
    import __graft_entry__
    __graft_entry__.build()
    import dlrm_sparse_embedding_gb300 as m
    return m


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "emb.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(emb_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(emb):
    declared = _declared_symbols()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(emb.lib, name), name
    assert sorted(emb.EXPORTS) == declared


# page titles (and the one phrase for calls with no passage) a declaration's
# comment may cite
_PASSAGE_MARKS = ("HugeCTR slides", "NVIDIA EMBark", "Merlin overview article", "No passage: library convenience",
                  "no counterpart on the pages", "Passage: as for")


def test_every_declaration_is_documented():
    # each entry point sits in a group of declarations (with any #define or
    # enum it needs) directly under a comment: no blank line in between
    with open(os.path.join(ROOT, "include", "emb.h")) as f:
        lines = f.read().splitlines()
    found = 0
    for i, line in enumerate(lines):
        m = re.match(r"(?:int|const char\*)\s+(emb_[a-z_0-9]+)\s*\(", line)
        if not m:
            continue
        found += 1
        j = i - 1
        while j >= 0 and lines[j].strip() and not lines[j].rstrip().endswith("*/"):
            j -= 1
        assert j >= 0 and lines[j].rstrip().endswith("*/"), m.group(1)
        # the comment above the group names the passage the call follows, a
        # page it points to through another call, or says it has none
        k = j
        while k >= 0 and "/*" not in lines[k]:
            k -= 1
        comment = " ".join(x.strip(" */") for x in lines[k:j + 1])
        assert any(p in comment for p in _PASSAGE_MARKS), m.group(1)
    assert found == len(_declared_symbols())


def test_status_strings(emb):
    for s in range(0, -8, -1):
        assert emb.lib.emb_status_string(s)
    assert emb.lib.emb_status_string(-4).decode() == "key outside [0, rows)"


def test_create_rejects_bad_specs_on_host(emb):
    from dlrm_sparse_embedding_gb300._lib import EmbTableSpec
    h = ctypes.c_void_p()
    good = (EmbTableSpec * 1)()
    good[0].rows, good[0].dim = 10, 16
    cases = []
    for field, val in [("dim", 6), ("dim", 0), ("dim", 132), ("rows", 0), ("dtype", 3), ("pooling", 2), ("opt", 5)]:
        a = (EmbTableSpec * 1)()
        a[0].rows, a[0].dim = 10, 16
        setattr(a[0], field, val)
        cases.append((a, 1, 8, 100))
    cases += [(good, 0, 8, 100), (good, 1, 0, 100), (good, 1, 8, -1), (good, 1, 8, 1 << 31)]
    huge = (EmbTableSpec * 2)()
    for i in range(2):
        huge[i].rows, huge[i].dim = 3_000_000_000, 4
    cases.append((huge, 2, 8, 100))
    for a, T, B, nnz in cases:
        assert emb.lib.emb_create(a, T, B, nnz, ctypes.byref(h)) == emb.EMB_ERR_INVALID_ARG


def test_calls_reject_null_layer(emb):
    L = emb.lib
    assert L.emb_forward(None, None, None, None, 0, 1, None, None) == emb.EMB_ERR_INVALID_ARG
    assert L.emb_backward_update(None, None, 0, None) == emb.EMB_ERR_INVALID_ARG
    assert L.emb_sync_status(None, None) == emb.EMB_ERR_INVALID_ARG
    assert L.emb_destroy(None) == emb.EMB_OK


def test_unique_workspace_is_host_computable(emb):
    sizes = [emb.unique_workspace_bytes(n) for n in (0, 1, 4096, 4097, 1 << 20)]
    assert all(s > 0 and s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes)
    b = ctypes.c_size_t()
    assert emb.lib.emb_unique_workspace(-1, ctypes.byref(b)) == emb.EMB_ERR_INVALID_ARG
    assert emb.lib.emb_unique(None, 10, None, None, None, None, None, None, 0, None) == emb.EMB_ERR_INVALID_ARG


def _no_cuda_device():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


# The pointers below are addresses no allocation returned.  Each case is
# rejected by the host checks before any CUDA call; the test still runs only
# where no GPU is present, so nothing could ever reach a kernel.
@pytest.mark.skipif(not _no_cuda_device(), reason="host-only check: runs where no GPU is present")
def test_unique_rejects_misaligned_arrays_on_host(emb):
    vp = ctypes.c_void_p
    ws_bytes = emb.unique_workspace_bytes(10)
    ok = dict(keys=0x10000, uniq=0x20000, inv=0x30000, cnt=0x40000, seg=0x50000, nu=0x60000)
    for name, bad in [("keys", 0x10004), ("uniq", 0x20004), ("nu", 0x60004), ("inv", 0x30002),
                      ("cnt", 0x40001), ("seg", 0x50002)]:
        a = dict(ok, **{name: bad})
        args = [vp(a["keys"]), 10, vp(a["uniq"]), vp(a["inv"]), vp(a["cnt"]), vp(a["seg"]), vp(a["nu"])]
        assert emb.lib.emb_unique(*args, vp(0x100000), ws_bytes, None) == emb.EMB_ERR_INVALID_ARG, name
        assert emb.lib.emb_unique_noalloc(*args, None) == emb.EMB_ERR_INVALID_ARG, name
    # a workspace that is not 256-byte aligned, or too small
    args = [vp(ok["keys"]), 10, vp(ok["uniq"]), vp(ok["inv"]), vp(ok["cnt"]), vp(ok["seg"]), vp(ok["nu"])]
    assert emb.lib.emb_unique(*args, vp(0x100010), ws_bytes, None) == emb.EMB_ERR_INVALID_ARG
    assert emb.lib.emb_unique(*args, vp(0x100000), ws_bytes - 1, None) == emb.EMB_ERR_INVALID_ARG


def test_product_package_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "dlrm_sparse_embedding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    text = f.read()
                assert "oracle" not in text.lower(), fn
                assert "ctr_inputs" not in text, fn
