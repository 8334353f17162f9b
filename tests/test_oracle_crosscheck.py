"""The C++ oracle against an independent second implementation (dsa_oracle_np.py:
numpy float64, one library matmul per query, a library lexsort per row) on seeded
random cases of every input kind.  The two share no code; they agree to the rounding
of float64 summation order (scores) and exactly (top-k, gather)."""
import numpy as np
import pytest

import parity
from deepseek_v4_sparse_dsa_gb300 import synth
from oracle import dsa_oracle as orc
from oracle import dsa_oracle_np as orc_np


def _both(fn, *a, **kw):
    return getattr(orc, fn)(*a, **kw), getattr(orc_np, fn)(*a, **kw)


@pytest.mark.parametrize("dtype,paged,causal,next_n,lens", [
    ("bf16", True, True, 1, [700, 129, 1, 2050]),
    ("bf16", False, False, 7, [1000]),
    ("e4m3", True, True, 3, [900, 300]),
    ("e4m3", False, True, 40, [700]),
])
def test_scores_and_selection_agree(dtype, paged, causal, next_n, lens):
    wl = parity.make_case(501 + next_n, lens, next_n=next_n, paged=paged, block_size=32, dtype=dtype,
                          causal=causal, topk=64)
    args = (wl.q, wl.q_scale, wl.dtype, wl.weights, wl.k_data, wl.k_scale, wl.block_table, wl.block_size, wl.B,
            wl.next_n, wl.context_lens, wl.causal)
    a, b = _both("indexer_logits", *args)
    assert np.array_equal(a == -np.inf, b == -np.inf)
    fin = np.isfinite(b)
    assert np.all(np.abs(a[fin] - b[fin]) <= 1e-12 * (1 + np.abs(b[fin])))
    ia, va = orc.topk_select(a, 64)
    ib, vb = orc_np.topk_select(a, 64)
    assert np.array_equal(ia, ib) and np.array_equal(va, vb)


def test_mxfp4_keys_and_gather_agree():
    r = np.random.default_rng(77)
    B, n, bs, nblk, H, Dm = 2, 3, 4, 9, 4, 128
    lens = np.array([30, 11])
    pool_n = r.integers(0, 256, (nblk * bs, Dm // 2)).astype(np.uint8)
    pool_s = r.integers(118, 137, (nblk * bs, Dm // 32)).astype(np.uint8)
    pool_s[r.random(pool_s.shape) < 0.05] = 0xFF
    table = np.array([[5, 0, 3, 1, 8, 2, 7, 6], [4, 2, 6, -1, -1, -1, -1, -1]], np.int32)
    q, qs = synth.quantize_e4m3_rows(r.standard_normal((B * n, H, Dm)).astype(np.float32))
    w = r.random((B * n, H)).astype(np.float32)
    a, b = _both("indexer_logits", q, qs, "e4m3", w, pool_n, pool_s, table, bs, B, n, lens, True, k_dtype="mxfp4")
    fin = np.isfinite(b)
    assert np.array_equal(fin, np.isfinite(a))
    assert np.all(np.abs(a[fin] - b[fin]) <= 1e-12 * (1 + np.abs(b[fin])))
    sel = r.integers(-1, 11, (B * n, 9)).astype(np.int32)
    g1, g2 = _both("mxfp4_paged_gather", pool_n.reshape(nblk, bs, 64), pool_s.reshape(nblk, bs, 4), table, sel, B,
                   n, bs)
    assert np.array_equal(g1, g2)
