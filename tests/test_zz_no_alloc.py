"""dsa_indexer_logits_topk_noalloc: the fused call for callers that cannot allocate device
memory (a process whose device memory is all reserved up front and handed out by its own
pool, or a latency-critical loop that cannot pay for cudaMalloc / cudaFree).  Its scratch
is a fixed array inside the library, so it must give exactly what the regular call with a
caller-provided workspace gives -- also on a second call, when the array still holds the
first call's contents.  (This file sorts last so a stop-at-first-failure run has already
run every other test.)"""
import gc

import numpy as np
import pytest

import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch  # noqa: E402


def _noalloc(db, k):
    idx = torch.full((db.T, k), -7, dtype=torch.int32, device="cuda")
    val = torch.full((db.T, k), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_indexer_logits_topk_noalloc(db.q, db.q_scale, db.dtype, db.weights, 64, 128, db.keys(),
                                        db.queries(), k, idx, val)
    return idx, val


def test_noalloc_matches_workspace_call_twice():
    cases = [
        # rows long enough to be split over several key chunks (the merge path)
        parity.make_case(201, [30000, 9000, 200, 0], next_n=1, block_size=64, topk=512),
        # a different shape right after: two queries per group, larger k
        parity.make_case(202, [20000, 5000, 77], next_n=2, block_size=32, topk=1024),
        # E4M3 queries and keys, four rows per group (prefill-shaped items)
        parity.make_case(203, [2500], next_n=40, paged=False, dtype="e4m3", topk=256),
    ]
    for wl in cases:
        db = DeviceBatch.from_workload(wl)
        ref_idx, ref_val = db.logits_topk()          # regular call, torch-allocated workspace
        idx, val = _noalloc(db, wl.topk)
        assert dsa.dsa_device_error() == 0
        assert torch.equal(idx, ref_idx)
        assert torch.equal(val, ref_val)
        # and against the oracle's ranking of the same scores
        lg = db.logits().cpu().numpy()
        parity.assert_topk_exact(idx.cpu().numpy(), lg, wl.topk, val.cpu().numpy())


def test_noalloc_rejects_batches_beyond_its_scratch():
    # four query rows per sequence at k = 2048: the partial top-k lists alone need ~20 MB
    lens = torch.full((256,), 1 << 20, dtype=torch.int32, device="cuda")
    qs = dsa.make_queries(256, 4, lens, 1 << 20, True)
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_LOGITS_TOPK, dsa.DSA_BF16, qs, 2048) > 16 << 20
    keys = dsa.dsa_keys(0x100000, None, 0x100000, 1 << 14, 64, 1 << 20)
    before = dsa.dsa_launch_count()
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_logits_topk_noalloc(0x100000, None, dsa.DSA_BF16, 0x100000, 64, 128, keys, qs, 2048,
                                            0x100000, None)
    assert e.value.status == dsa.DSA_ERR_WORKSPACE
    assert dsa.dsa_launch_count() == before


def test_noalloc_allocates_nothing():
    # after a first call (which looks up the array's address), further calls change
    # neither torch's allocations nor the device's free memory
    wl = parity.make_case(211, [30000, 9000, 200], next_n=1, block_size=64, topk=512)
    db = DeviceBatch.from_workload(wl)
    idx = torch.empty((db.T, wl.topk), dtype=torch.int32, device="cuda")
    val = torch.empty((db.T, wl.topk), dtype=torch.float32, device="cuda")

    def call():
        dsa.dsa_indexer_logits_topk_noalloc(db.q, db.q_scale, db.dtype, db.weights, 64, 128, db.keys(),
                                            db.queries(), wl.topk, idx, val)

    call()
    torch.cuda.synchronize()
    # garbage left by earlier tests (tensors in reference cycles) is collected now, so the
    # collector cannot free it while the calls below run and shift the baseline
    gc.collect()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert dsa.dsa_device_error() == 0
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_bad_argument_reported_before_the_size():
    # a batch too large for the array, but with an unsupported head count: the argument
    # error comes first, as for the regular call
    lens = torch.full((256,), 1 << 20, dtype=torch.int32, device="cuda")
    qs = dsa.make_queries(256, 4, lens, 1 << 20, True)
    keys = dsa.dsa_keys(0x100000, None, 0x100000, 1 << 14, 64, 1 << 20)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_logits_topk_noalloc(0x100000, None, dsa.DSA_BF16, 0x100000, 32, 128, keys, qs, 2048,
                                            0x100000, None)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
