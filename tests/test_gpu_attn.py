"""Sparse attention over the selection (dsa_sparse_attn_mxfp4) on the GPU against the CPU
oracle's fp64 sum (orc.sparse_attn), element by element.

Tolerance, from the arithmetic.  The kernel forms a weighted mean of the selected rows
x_j with weights w_j = 2^(s_j - m) rounded once to bf16 (relative error <= 2^-9) and
the same rounded weights in the denominator, so to first order
  |out - exact| <= sum_j w_j |eps_j| |x_j[e] - out[e]| / sum_j w_j <= 2 (2^-9 + |ds|) M_e
with M_e = max_j |x_j[e]| over the row's selected rows and ds the score error in
natural-log units: fp32 accumulation of 128 exact bf16 products, |ds| <= 128 * 2^-23 *
scale * sum_e |q_e x_je|.  The test allows twice that first-order bound,
  |got - ref| <= (2^-7 + 4 |ds|max) M_e + 1e-6 |ref| + 1e-30,
and checks in addition that rows with no selected position are exactly zero.
"""
import numpy as np
import pytest

from deepseek_v4_sparse_dsa_gb300 import synth
from oracle import dsa_oracle as orc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402


def gpu_attn(ab: synth.AttnBatch, rows=None):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, sel = d(ab.q.view(np.int16)), d(ab.sel)
    fp4, sc, tab, sink = d(ab.kv_fp4), d(ab.kv_scale), d(ab.table), d(ab.sink)
    out = torch.full((ab.T, 64, 128), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_sparse_attn_mxfp4(q, ab.T, 64, 128, sel, ab.topk, fp4, sc, fp4.shape[0], ab.block_size, tab,
                              tab.shape[1], ab.next_n, sink, ab.scale, out)
    err = dsa.dsa_device_error()
    got = out.cpu().numpy()
    return (got if rows is None else got[rows]), err


def cache_rows(ab: synth.AttnBatch, sel, rows):
    """Pool row of every selected slot of the given query rows (-1: padded / dropped)."""
    b = rows // ab.next_n
    page = np.where(sel >= 0, sel // ab.block_size, 0)
    ok = (sel >= 0) & (page < ab.table.shape[1])
    blk = np.where(ok, ab.table[b[:, None], np.minimum(page, ab.table.shape[1] - 1)], -1)
    ok &= (blk >= 0) & (blk < ab.kv_fp4.shape[0])
    return np.where(ok, blk.astype(np.int64) * ab.block_size + np.where(sel >= 0, sel % ab.block_size, 0), -1)


def selected_rows(ab: synth.AttnBatch, crow):
    """The dequantised cache rows (float64) of the slots crow [R, k]; zeros where -1."""
    X = np.zeros(crow.shape + (128,))
    live = crow >= 0
    if live.any():
        flat = crow[live]
        X[live] = orc.mxfp4_dequant(ab.kv_fp4.reshape(-1, 64)[flat], ab.kv_scale.reshape(-1, 4)[flat])
    return X


def reference(ab: synth.AttnBatch, rows, sel=None):
    """The oracle on the given query rows (a sub-batch with one row per sequence)."""
    sel = ab.sel[rows] if sel is None else sel
    tab = ab.table[rows // ab.next_n]
    return orc.sparse_attn(ab.q[rows], sel, ab.kv_fp4, ab.kv_scale, tab, len(rows), 1, ab.block_size,
                           ab.sink.astype(np.float64), ab.scale)


def assert_attn_close(ab, got, ref, rows, sel=None):
    sel = ab.sel[rows] if sel is None else sel
    crow = cache_rows(ab, sel, rows)
    X = selected_rows(ab, crow)                                                    # [R, k, 128]
    M = np.abs(X).max(axis=1) if X.shape[1] else np.zeros((len(rows), 128))     # [R, 128]
    qf = (ab.q[rows].astype(np.uint32) << 16).view(np.float32).astype(np.float64)   # [R, 64, 128]
    sabs = (np.abs(qf) @ np.abs(X).transpose(0, 2, 1)).max(axis=2, initial=0.0)  # [R, 64]
    ds = 128 * 2.0 ** -23 * ab.scale * sabs
    tol = (2.0 ** -7 + 4 * ds)[:, :, None] * M[:, None, :] + 1e-6 * np.abs(ref) + 1e-30
    diff = np.abs(got - ref)
    bad = np.argwhere(~(diff <= tol))
    assert bad.size == 0, (bad[:4], got[tuple(bad[0])], ref[tuple(bad[0])], tol[tuple(bad[0])])
    empty = (crow < 0).all(axis=1)
    assert not got[empty].any()


def check(ab, rows=None):
    rows = np.arange(ab.T) if rows is None else np.asarray(rows)
    got, err = gpu_attn(ab)
    assert err == 0
    assert np.isfinite(got).all()
    ref = reference(ab, rows)
    assert_attn_close(ab, got[rows], ref, rows)


def test_attn_small_ragged():
    # two tiles with a ragged second one, causal MTP rows, 5% padded slots
    ab = synth.make_attn(11, [700, 300, 1500], next_n=2, topk=200, pad_frac=0.05)
    check(ab)


@pytest.mark.parametrize("topk", [1, 127, 128, 129, 640])
def test_attn_topk_edges(topk):
    ab = synth.make_attn(20 + topk, [2000, 900, 50], next_n=1, topk=topk, block_size=16, pad_frac=0.1)
    check(ab)


def test_attn_empty_and_fully_padded_rows():
    ab = synth.make_attn(31, [600, 400], next_n=2, topk=300)
    ab.sel[1, :] = -1                     # a row with nothing selected: zeros
    ab.sel[2, 128:] = -1                  # a row whose second and third tiles are empty
    check(ab)
    ab0 = synth.make_attn(32, [600], next_n=1, topk=0)
    got, err = gpu_attn(ab0)
    assert err == 0 and not got.any()


def test_attn_no_sink_and_large_sink():
    ab = synth.make_attn(41, [3000, 800], next_n=1, topk=256)
    ab.sink[:] = -np.inf                  # plain softmax over the selection
    ab.sink[5] = 40.0                     # a sink that takes nearly all the mass
    check(ab)


def test_attn_rescaled_tiles():
    # scores spread over many units and rising from tile to tile: the running maximum moves
    # past its headroom several times (O and L rescaled in tensor memory)
    ab = synth.make_attn(51, [4096], next_n=1, topk=1024, pad_frac=0.0, scale=1.0, sink_lo=-30, sink_hi=-20)
    qf = (ab.q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    X = selected_rows(ab, cache_rows(ab, ab.sel, np.arange(ab.T)))
    s = X[0] @ qf[0, 0]                               # head 0's scores
    ab.sel[0] = ab.sel[0][np.argsort(s, kind="stable")]   # ascending: each tile raises the max
    check(ab)


def test_attn_bad_block_drops_position_and_flags():
    ab = synth.make_attn(61, [900, 700], next_n=1, topk=128, pad_frac=0.0)
    ab.table[0, 3] = 10 ** 6              # positions 192..255 of sequence 0 point nowhere
    got, err = gpu_attn(ab)
    assert err & dsa.DSA_DEVERR_INDEX
    rows = np.arange(ab.T)
    sel = ab.sel.copy()
    sel[0][(sel[0] // ab.block_size) == 3] = -1
    ref = reference(ab, rows, sel)
    assert_attn_close(ab, got, ref, rows, sel)


def test_attn_flash_decode_full_size():
    ab = synth.make_attn_config("flash_decode")
    check(ab)


def test_attn_fp8_chunked_full_size_sampled_rows():
    # 8192 rows x top-1024 in the bench's launch; 48 rows checked against the oracle
    ab = synth.make_attn_config("fp8_chunked")
    rows = np.sort(np.random.default_rng(7).choice(ab.T, 48, replace=False))
    check(ab, rows)


@pytest.mark.parametrize("bs", [1, 256])
def test_attn_block_sizes(bs):
    # one cache row per page, and pages larger than a tile; three causal rows per sequence
    ab = synth.make_attn(70 + bs, [1500, 333], next_n=3, topk=300, block_size=bs, pad_frac=0.03)
    check(ab)
