"""FP8-q x FP4-k score (dtype DSA_E4M3_MXFP4K): E4M3 queries against keys read straight
from the paged mxfp4 cache, on the GPU against the CPU oracle's score over the
dequantised keys (orc.indexer_logits(..., k_dtype="mxfp4")):

* logits within 1e-3 (1 + |ref|), -inf exactly where the oracle masks;
* the fused top-k equal, bit for bit, to the oracle's top-k of the GPU's own logits;
* the selection against the oracle's logits at mean Jaccard >= 0.999.
"""
import numpy as np
import pytest

import parity
from deepseek_v4_sparse_dsa_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch  # noqa: E402


def check(wl, rows=None, jaccard=True):
    db = DeviceBatch.from_workload(wl)
    assert db.dtype == dsa.DSA_E4M3_MXFP4K
    lg = db.logits()
    idx, val = db.logits_topk()
    assert dsa.dsa_device_error() == 0
    lg = lg.cpu().numpy()
    idx, val = idx.cpu().numpy(), val.cpu().numpy()
    rows = np.arange(wl.T) if rows is None else rows
    ref = parity.oracle_logits(wl, rows=rows)
    parity.assert_logits_close(lg[rows], ref)
    parity.assert_topk_exact(idx, lg, wl.topk, val)
    if jaccard:
        parity.selection_parity(idx[rows], ref, wl.topk)


@pytest.mark.parametrize("bs", [16, 64, 128])
def test_fp4_keys_paged_decode(bs):
    wl = parity.make_case(601 + bs, [700, 129, 1, 2050, 0], next_n=1, block_size=bs, dtype="e4m3",
                          topk=96, k_format="mxfp4")
    check(wl)


def test_fp4_keys_split_rows_and_mtp():
    # long rows split over CTAs (merged), two causal queries per group
    wl = parity.make_case(611, [30000, 9000, 200], next_n=2, block_size=64, dtype="e4m3", topk=512,
                          k_format="mxfp4")
    check(wl)


def test_fp4_keys_contiguous_many_queries():
    # one contiguous sequence, 9 causal queries (groups of two rows and a ragged tail)
    wl = parity.make_case(621, [3001], next_n=9, paged=False, dtype="e4m3", topk=128, k_format="mxfp4")
    check(wl)


def test_fp4_keys_flash_decode_full_size():
    # the Flash decode batch in its FP8-q x FP4-k form: keys from the gather's own cache
    wl = synth.make_flash_decode_fp4k()
    check(wl)


def test_fp4_keys_bad_block_id_masks_and_flags():
    wl = parity.make_case(631, [500, 300], next_n=1, block_size=64, dtype="e4m3", topk=32, k_format="mxfp4")
    wl.block_table[0, 2] = 10 ** 6        # keys 128..191 of sequence 0 point nowhere
    db = DeviceBatch.from_workload(wl)
    lg = db.logits()
    assert dsa.dsa_device_error() & dsa.DSA_DEVERR_INDEX
    lg = lg.cpu().numpy()
    assert np.isneginf(lg[0, 128:192]).all()
    assert np.isfinite(lg[0, :128]).all() and np.isfinite(lg[0, 192:500]).all()


def test_fp4_keys_subnormal_scale_bytes():
    # scale bytes 0 and 1 (subnormal bf16 keys) take the exact per-nibble decode, 0xFF the
    # table's signed zeros; the other rows of the same tiles keep the table path
    wl = parity.make_case(641, [900, 300], next_n=1, block_size=64, dtype="e4m3", topk=64, k_format="mxfp4")
    r = np.random.default_rng(641)
    sc = wl.k_scale.copy()
    rows = r.choice(sc.shape[0], sc.shape[0] // 10, replace=False)
    sc[rows, r.integers(0, 4, rows.size)] = r.choice(np.array([0, 1, 2, 255], np.uint8), rows.size)
    wl.k_scale = sc
    check(wl)
