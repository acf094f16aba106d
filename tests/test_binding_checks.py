"""Argument checks of the Python binding, on CPU.

The C ABI takes bare pointers, so the binding is the last place where a
tensor's dtype, size and device can be checked; these tests make each bad
argument fail there, with ValueError, before anything reaches the library.
The layer object is built without a device (no emb_create)."""
import pytest
import torch

import ctr_inputs as ci
from dlrm_sparse_embedding_gb300 import layer as binding


def _bare_layer(tables, last_batch=None):
    lay = object.__new__(binding.EmbeddingLayer)
    lay.tables = list(tables)
    lay.total_dim = sum(t.dim for t in tables)
    lay.last_nnz = 0
    lay.last_batch = last_batch
    lay._h = None
    return lay


TABLES = [ci.TableSpec(10, 8), ci.TableSpec(20, 4)]
B = 3


def _batch(**over):
    args = dict(keys=torch.zeros(6, dtype=torch.int64), offsets=torch.arange(0, 7, dtype=torch.int64),
                table_ids=torch.tensor([0, 0, 0, 1, 1, 1], dtype=torch.int32), batch=B,
                out=torch.empty((B, 12), dtype=torch.float32))
    args.update(over)
    return args


@pytest.mark.parametrize("method", ["forward", "forward_infer"])
@pytest.mark.parametrize("bad,match", [
    (dict(keys=torch.zeros(6, dtype=torch.int32)), "keys"),
    (dict(offsets=torch.arange(0, 7, dtype=torch.int32)), "offsets"),
    (dict(offsets=torch.arange(0, 6, dtype=torch.int64)), "offsets"),          # T*B+1 = 7 needed
    (dict(table_ids=torch.zeros(6, dtype=torch.int64)), "table_ids"),
    (dict(table_ids=torch.zeros(5, dtype=torch.int32)), "table_ids"),
    (dict(out=torch.empty((B, 11), dtype=torch.float32)), "out"),
    (dict(out=torch.empty((B, 12), dtype=torch.float64)), "out"),
    (dict(keys=torch.zeros(6, dtype=torch.int64, device="meta")), "keys"),      # not on the batch's device
    (dict(keys=[0, 1, 2]), "keys"),
])
def test_bad_batch_arguments_are_rejected(method, bad, match):
    lay = _bare_layer(TABLES)
    with pytest.raises(ValueError, match=match):
        getattr(lay, method)(**_batch(**bad))


def test_well_formed_cpu_batch_passes_the_checks_and_stops_at_the_device():
    lay = _bare_layer(TABLES)
    # every check passes; the pointer marshalling then insists on CUDA tensors
    with pytest.raises(ValueError, match="CUDA"):
        lay.forward(**_batch(offsets=torch.arange(0, 9, dtype=torch.int64)))   # longer offsets are fine


@pytest.mark.parametrize("grad,match", [
    (torch.zeros((B, 12), dtype=torch.float64), "grad_out"),
    (torch.zeros((B - 1, 12), dtype=torch.float32), "grad_out"),
    (torch.zeros((B, 13), dtype=torch.float32), "grad_out"),
    (torch.zeros(B * 12, dtype=torch.float32), "grad_out"),
])
def test_bad_gradients_are_rejected(grad, match):
    lay = _bare_layer(TABLES, last_batch=B)
    with pytest.raises(ValueError, match=match):
        lay.backward_update(grad)


def test_unknown_variant_is_rejected():
    lay = _bare_layer(TABLES, last_batch=B)
    with pytest.raises(ValueError, match="variant"):
        lay.backward_update(torch.zeros((B, 12)), "sorted")


@pytest.mark.parametrize("call", [
    lambda lay: lay.gather_rows(0, torch.zeros(2, dtype=torch.int32)),
    lambda lay: lay.gather_master_rows(0, torch.zeros(2, dtype=torch.int32)),
    lambda lay: lay.cache_build(0, torch.zeros(2, dtype=torch.float32)),
    lambda lay: lay.find_keys(0, torch.zeros(2, dtype=torch.int32)),
    lambda lay: binding.unique(torch.zeros(2, dtype=torch.int32)),
])
def test_row_and_key_arguments_must_be_int64(call):
    with pytest.raises(ValueError, match="int64"):
        call(_bare_layer(TABLES))
