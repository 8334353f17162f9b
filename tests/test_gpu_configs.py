"""The five workload configurations at full size, in the launch configuration the benchmark
times.  Where the oracle cannot score every row in seconds, it scores a seeded sample of
rows (always the first and the last) and the checks run on those rows."""
import numpy as np
import pytest

import parity
from deepseek_v4_sparse_dsa_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch  # noqa: E402
from oracle import dsa_oracle as orc  # noqa: E402


def pipeline(wl, rows):
    """Fused score+top-k (the benchmarked call), the unfused score for the same batch,
    and the gather of the fused selection; returns host copies of the sampled rows."""
    db = DeviceBatch.from_workload(wl)
    idx_f, val_f = db.logits_topk()
    out = None
    sel = None
    if wl.kv_fp4 is not None:
        sel_d = idx_f
        if wl.gather_pad_frac > 0:
            sel_d = torch.from_numpy(synth.pad_sel_pos(idx_f.cpu().numpy(), wl.gather_pad_frac, wl.seed)).cuda()
        out = db.gather(sel_d)
        sel = sel_d.cpu().numpy()
    lg = db.logits()
    assert dsa.dsa_device_error() == 0
    r = torch.from_numpy(rows).cuda()
    got = {
        "logits": lg.index_select(0, r).cpu().numpy(),
        "idx": idx_f.index_select(0, r).cpu().numpy(),
        "val": val_f.index_select(0, r).cpu().numpy(),
    }
    if out is not None:
        got["gather"] = out.index_select(0, r).cpu().numpy().view(np.uint16)
        got["sel"] = sel[rows]
    return got


def check(wl, rows):
    got = pipeline(wl, rows)
    ref = parity.oracle_logits(wl, rows=rows)
    parity.assert_logits_close(got["logits"], ref)
    parity.assert_topk_exact(got["idx"], got["logits"], wl.topk, got["val"])
    parity.selection_parity(got["idx"], ref, wl.topk)
    if "gather" in got:
        b = rows // wl.next_n
        want = orc.mxfp4_paged_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table[b], got["sel"],
                                      len(rows), 1, wl.block_size)
        assert np.array_equal(got["gather"], want)


def test_flash_decode_full():
    wl = synth.make_flash_decode()
    check(wl, np.arange(wl.T))


def test_pro_mtp_full():
    wl = synth.make_pro_mtp()
    check(wl, np.arange(wl.T))


def test_prefill_full_sampled():
    wl = synth.make_prefill()
    check(wl, parity.sample_rows(wl.T, 48, 4))


def test_fp8_chunked_full_sampled():
    wl = synth.make_fp8_chunked()
    check(wl, parity.sample_rows(wl.T, 24, 5))
