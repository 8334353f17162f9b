"""Indexer score, standalone top-k and fused score+top-k on the GPU against the CPU oracle."""
import numpy as np
import pytest

import parity
from deepseek_v4_sparse_dsa_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch  # noqa: E402
from oracle import dsa_oracle as orc  # noqa: E402


def run_all(wl, topk=None):
    """GPU logits (unfused), top-k of those logits, fused top-k; device error word."""
    db = DeviceBatch.from_workload(wl)
    k = topk or wl.topk
    W = max(wl.max_context_len, 1)
    logits = torch.full((wl.T, W + 3), float("nan"), device="cuda")        # sentinel incl. padding
    dsa.dsa_indexer_logits(db.q, db.q_scale, db.dtype, db.weights, 64, 128, db.keys(), db.queries(), logits,
                           logits.shape[1])
    idx_u, val_u = db.topk_of(logits, k)
    idx_f, val_f = db.logits_topk(k)
    err = dsa.dsa_device_error()
    lg = logits.cpu().numpy()
    assert np.isnan(lg[:, W:]).all(), "columns past max_context_len must stay untouched"
    return (lg[:, :W], idx_u.cpu().numpy(), val_u.cpu().numpy(), idx_f.cpu().numpy(), val_f.cpu().numpy(),
            err)


def check_case(wl, topk=None, jaccard=True):
    k = topk or wl.topk
    lg, idx_u, val_u, idx_f, val_f, err = run_all(wl, k)
    assert err == 0
    ref = parity.oracle_logits(wl)
    parity.assert_logits_close(lg, ref)
    parity.assert_topk_exact(idx_u, lg, k, val_u)       # standalone top-k on GPU logits
    parity.assert_topk_exact(idx_f, lg, k, val_f)       # fused == top-k of unfused logits
    if jaccard:
        parity.selection_parity(idx_f, ref, k)
    return lg, ref


def test_tiny_config():
    check_case(synth.make_tiny())


def test_tiny_noncausal_contiguous_ragged_groups():
    # next_n = 7: query groups of 4 with a ragged tail; K not a multiple of 128
    wl = parity.make_case(31, [1000], next_n=7, paged=False, causal=False, topk=100)
    check_case(wl)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256])
def test_paged_block_sizes(bs):
    wl = parity.make_case(40 + bs, [700, 129, 1, 2050], next_n=1, block_size=bs, topk=96)
    check_case(wl)


def test_mtp_pairs_paged():
    wl = parity.make_case(51, [3000, 77, 4097, 1500, 2], next_n=2, block_size=64, topk=256)
    check_case(wl)


def test_decode_split_rows():
    # few sequences with long rows: the key range is split over CTAs and merged
    wl = parity.make_case(61, [30000, 9000, 200, 0], next_n=1, block_size=64, topk=512)
    qs = dsa.make_queries(wl.B, wl.next_n, 0x1000, wl.max_context_len, True)
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_LOGITS_TOPK, dsa.DSA_BF16, qs, 512) > 0
    check_case(wl)


def test_decode_split_mtp_rows():
    # two queries per group, split rows, a group with no visible key
    wl = parity.make_case(62, [40000, 3, 0, 17000], next_n=2, block_size=32, topk=1024)
    check_case(wl)


def test_decode_split_fp8():
    wl = parity.make_case(63, [20000, 5000], next_n=1, block_size=64, dtype="e4m3", topk=512)
    check_case(wl)


@pytest.mark.parametrize("topk", [1, 7, 1024, 2048])
def test_topk_sizes(topk):
    wl = parity.make_case(70 + topk, [5000, 300], next_n=3, block_size=64, topk=topk)
    check_case(wl, jaccard=topk <= 1024)


def test_rows_shorter_than_k_pad_with_minus_one():
    wl = parity.make_case(81, [40], next_n=40, paged=False, topk=64)
    lg, idx_u, val_u, idx_f, val_f, err = run_all(wl)
    for t in range(40):
        assert (idx_f[t, :t + 1] >= 0).all() and (idx_f[t, t + 1:] == -1).all()
        assert np.isneginf(val_f[t, t + 1:]).all()


def test_fp8_small():
    wl = parity.make_case(91, [700], next_n=40, paged=False, dtype="e4m3", topk=128)
    check_case(wl)


def test_fp8_paged_mtp():
    wl = parity.make_case(92, [900, 2100], next_n=2, paged=True, block_size=32, dtype="e4m3", topk=200)
    check_case(wl)


@pytest.mark.parametrize("lens,next_n,topk", [
    ([700, 1500, 30000, 5000], 1, 1024),   # one row per item, two CTAs per SM
    ([3000, 2500], 4, 2048),               # four-row groups at k = 2048
])
def test_topk_where_the_plan_has_no_gather_buffer(lens, next_n, topk):
    # shared memory leaves no room for the binned top-k's gather buffer in these plans:
    # every whole-group row is cut back and sorted by the bitonic network instead
    wl = parity.make_case(81 + next_n, lens, next_n=next_n, block_size=64, topk=topk)
    check_case(wl)


def test_split_rows_with_tied_scores():
    # every cached key equal: all of a row's scores tie, so its top-k follows the index.
    # The merge of the split rows then finds all candidates in one value bin: the exact
    # fallback where they outnumber its limit, the in-bin tie rule where they do not.
    wl = parity.make_case(77, [20000, 9000, 3000, 700], next_n=1, block_size=64, topk=512)
    wl.k_data[:] = wl.k_data[0]
    check_case(wl, jaccard=False)


def test_topk_ties_and_signed_zero():
    """Standalone top-k on crafted logits: heavy ties, -0.0 vs +0.0, -inf holes, rows with
    fewer candidates than k, all -inf rows."""
    rng = np.random.default_rng(5)
    B, n, L, k = 3, 4, 3000, 300
    lens = np.array([3000, 10, 2999], np.int32)
    lg = rng.integers(-3, 4, (B * n, L)).astype(np.float32)
    lg[rng.random(lg.shape) < 0.3] = -0.0
    lg[rng.random(lg.shape) < 0.1] = 0.0
    lg[rng.random(lg.shape) < 0.2] = -np.inf
    lg[5] = -np.inf
    # the layout the logits op writes: -inf past each row's visible range
    vis = np.repeat(lens, n) - n + np.tile(np.arange(n), B) + 1
    for t in range(B * n):
        lg[t, max(vis[t], 0):] = -np.inf
    d_lg = torch.from_numpy(lg).cuda()
    d_lens = torch.from_numpy(lens).cuda()
    qs = dsa.make_queries(B, n, d_lens, L, True)
    idx = torch.empty((B * n, k), dtype=torch.int32, device="cuda")
    val = torch.empty((B * n, k), dtype=torch.float32, device="cuda")
    nws = dsa.dsa_workspace_bytes(dsa.DSA_OP_TOPK, dsa.DSA_BF16, qs, k)
    ws = torch.empty(max(nws, 8), dtype=torch.uint8, device="cuda")
    dsa.dsa_indexer_topk(d_lg, L, qs, k, idx, val, ws, ws.numel())
    assert dsa.dsa_device_error() == 0
    parity.assert_topk_exact(idx.cpu().numpy(), lg, k, val.cpu().numpy())


def test_bad_block_id_masks_key_and_flags():
    wl = parity.make_case(101, [500, 300], next_n=1, block_size=64, topk=32)
    wl.block_table[0, 2] = 10 ** 6        # keys 128..191 of sequence 0 point nowhere
    db = DeviceBatch.from_workload(wl)
    lg = db.logits()
    err = dsa.dsa_device_error()
    assert err & dsa.DSA_DEVERR_INDEX
    lg = lg.cpu().numpy()
    assert np.isneginf(lg[0, 128:192]).all()
    assert np.isfinite(lg[0, :128]).all() and np.isfinite(lg[0, 192:500]).all()
    idx, _ = db.logits_topk()
    assert dsa.dsa_device_error() & dsa.DSA_DEVERR_INDEX
    i0 = idx.cpu().numpy()[0]
    assert not ((i0 >= 128) & (i0 < 192)).any()


def test_empty_and_degenerate_batches():
    wl = parity.make_case(111, [0, 5, 0], next_n=2, block_size=8, topk=4)
    lg, idx_u, val_u, idx_f, val_f, err = run_all(wl)
    assert err == 0
    assert np.isneginf(lg[[0, 1, 4, 5]]).all()
    assert (idx_f[[0, 1, 4, 5]] == -1).all()
    parity.assert_topk_exact(idx_f, lg, 4, val_f)


@pytest.mark.parametrize("topk", [512, 2048])
def test_one_long_row_over_many_slices(topk):
    # one sequence long enough that its key tiles span every CTA's slice: the merge takes
    # more than 32 lists per row and cuts its buffer back while collecting
    wl = parity.make_case(121 + topk, [150000], next_n=1, block_size=64, topk=topk)
    check_case(wl, jaccard=topk <= 1024)


@pytest.mark.parametrize("topk", [64, 200, 2048])
def test_many_short_rows_finished_in_one_item(topk):
    # many short sequences: most query groups fit one CTA's slice and are ranked and
    # written by the fused kernel itself (register sort for k <= 1024, shared memory above)
    lens = synth.Rng(131).integers(100, 2000, 400, "lens")
    wl = parity.make_case(131 + topk, lens, next_n=1, block_size=64, topk=topk)
    check_case(wl, jaccard=topk <= 1024)
