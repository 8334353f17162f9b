"""Failure paths on the GPU, made without faulting it, and the producer's block-table
window refill.

* Every device-side wait of the library is bounded.  With the limit set to 1 ns any
  wait that does not succeed at once gives up: the kernels abandon the call's work,
  drain their own copies and MMAs, free tensor memory, flag DSA_DEVERR_TIMEOUT and
  return.  The host reads the flag, and the next call on the same context is correct.
  The same holds for the FP4-key score's converter warps and for the sparse attention
  (whose group barriers AND the waits' results, so its warps leave together).
* A paged sequence whose work items span more than the producer's 256-entry window of
  block-table entries (block size 8, items of up to 5000 keys = 625 pages) makes the
  producer refill that window in the middle of an item.
"""
import numpy as np
import pytest

import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch  # noqa: E402


def _with_wait_limit(ns, fn):
    dsa.dsa_device_error()                       # start from a clear error word
    dsa.dsa_set_wait_limit_ns(ns)
    try:
        fn()
        return dsa.dsa_device_error()
    finally:
        dsa.dsa_set_wait_limit_ns(0)             # back to the default limit


@pytest.mark.parametrize("lens,next_n,topk", [
    ([20000, 9000, 3000], 1, 512),               # decode rows split over CTAs + merge
    ([6000], 300, 256),                          # prefill-shaped: whole query groups of 4
])
def test_expired_waits_flag_timeout_and_leave_the_context_usable(lens, next_n, topk):
    wl = parity.make_case(300 + next_n, lens, next_n=next_n, block_size=64, topk=topk)
    db = DeviceBatch.from_workload(wl)
    err = _with_wait_limit(1, lambda: db.logits_topk())
    assert err >= 0 and err & dsa.DSA_DEVERR_TIMEOUT, err
    err = _with_wait_limit(1, lambda: db.logits())
    assert err >= 0 and err & dsa.DSA_DEVERR_TIMEOUT, err
    # the same context, default limit: both calls are right again
    idx, val = db.logits_topk()
    lg = db.logits()
    assert dsa.dsa_device_error() == 0
    lg = lg.cpu().numpy()
    parity.assert_topk_exact(idx.cpu().numpy(), lg, topk, val.cpu().numpy())
    rows = parity.sample_rows(wl.T, 8, 3)
    parity.assert_logits_close(lg[rows], parity.oracle_logits(wl, rows=rows))


def test_merge_is_safe_on_a_stale_workspace():
    # Lists left in the workspace by an abandoned call are read by the next merge.  Fill it
    # with one repeated nonzero word (two -inf floats, as a freed logits buffer leaves it):
    # every stale list then holds the same key, which no cut can thin, so the merge's
    # candidate count runs past its shared buffer and must be held there.  A completed call
    # rewrites every list it merges, so its result does not depend on what was there.
    wl = parity.make_case(305, [20000, 9000, 3000], next_n=1, block_size=64, topk=512)
    db = DeviceBatch.from_workload(wl)
    poison = np.array([0xFF800000FF800000], dtype=np.uint64).view(np.int64)[0]

    def stale_ws():
        ws = db.workspace(dsa.DSA_OP_LOGITS_TOPK, wl.topk)
        ws[: ws.numel() // 8 * 8].view(torch.int64).fill_(int(poison))
        return ws

    err = _with_wait_limit(1, lambda: db.logits_topk(ws=stale_ws()))
    assert err >= 0 and err & dsa.DSA_DEVERR_TIMEOUT, err
    idx, val = db.logits_topk(ws=stale_ws())
    lg = db.logits()
    assert dsa.dsa_device_error() == 0
    parity.assert_topk_exact(idx.cpu().numpy(), lg.cpu().numpy(), wl.topk, val.cpu().numpy())


def test_block_table_window_refilled_mid_item():
    # one sequence of 5000 keys in blocks of 8 (625 pages), 1216 causal queries: the
    # fused call's items cover up to 40 key tiles = 640 pages each
    wl = parity.make_case(311, [5000], next_n=1216, block_size=8, topk=256)
    db = DeviceBatch.from_workload(wl)
    idx, val = db.logits_topk()
    lg = db.logits()
    assert dsa.dsa_device_error() == 0
    lg = lg.cpu().numpy()
    parity.assert_topk_exact(idx.cpu().numpy(), lg, wl.topk, val.cpu().numpy())
    rows = parity.sample_rows(wl.T, 64, 311)
    ref = parity.oracle_logits(wl, rows=rows)
    parity.assert_logits_close(lg[rows], ref)
    parity.selection_parity(idx.cpu().numpy()[rows], ref, wl.topk)


def test_expired_waits_in_fp4_key_mode():
    # the converter warps' waits are bounded too; the next call on the context is right
    wl = parity.make_case(321, [9000, 3000], next_n=2, block_size=64, dtype="e4m3", topk=128, k_format="mxfp4")
    db = DeviceBatch.from_workload(wl)
    err = _with_wait_limit(1, lambda: db.logits_topk())
    assert err >= 0 and err & dsa.DSA_DEVERR_TIMEOUT, err
    idx, val = db.logits_topk()
    lg = db.logits()
    assert dsa.dsa_device_error() == 0
    lg = lg.cpu().numpy()
    parity.assert_topk_exact(idx.cpu().numpy(), lg, wl.topk, val.cpu().numpy())
    parity.assert_logits_close(lg, parity.oracle_logits(wl))


def test_expired_waits_in_sparse_attention():
    # every wait of the attention kernel is bounded: with a 1 ns limit its group leaves
    # together through the barrier's AND, the MMA thread drains, tensor memory is freed
    import test_gpu_attn as ta
    from deepseek_v4_sparse_dsa_gb300 import synth
    ab = synth.make_attn(331, [3000, 900], next_n=2, topk=512)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, sel, fp4, sc, tab, sink = (d(ab.q.view(np.int16)), d(ab.sel), d(ab.kv_fp4), d(ab.kv_scale), d(ab.table),
                                  d(ab.sink))
    out = torch.empty((ab.T, 64, 128), dtype=torch.float32, device="cuda")
    err = _with_wait_limit(1, lambda: dsa.dsa_sparse_attn_mxfp4(
        q, ab.T, 64, 128, sel, ab.topk, fp4, sc, fp4.shape[0], ab.block_size, tab, tab.shape[1], ab.next_n, sink,
        ab.scale, out))
    assert err >= 0 and err & dsa.DSA_DEVERR_TIMEOUT, err
    ta.check(ab)                                  # default limit: right again
