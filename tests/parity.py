"""Parity helpers for the GPU tests: case builders (from the shared seeded generators)
and the acceptance checks against the CPU oracle.

Acceptance (per row of queries):
* logits: -inf exactly where the oracle has -inf; elsewhere |gpu - ref| <= 1e-3 (1 + |ref|);
* top-k: bit-exact indices against the oracle's top-k of the GPU's own logits;
* selection: mean Jaccard(GPU set, oracle set on oracle logits) >= 0.999, and every
  element of a symmetric difference has an oracle logit within 1e-3 (1 + |v_k|) of the
  oracle's k-th value v_k;
* gather: bitwise equal bf16 patterns.
"""
from __future__ import annotations

import numpy as np

from deepseek_v4_sparse_dsa_gb300 import synth
from deepseek_v4_sparse_dsa_gb300.synth import D, H, Rng, Workload
from oracle import dsa_oracle as orc

LOGIT_RTOL = 1e-3


def make_case(seed: int, lens, next_n: int = 1, paged: bool = True, block_size: int = 64,
              dtype: str = "bf16", causal: bool = True, topk: int = 64, gather: bool = False,
              pad_frac: float = 0.0, k_format: str = "native") -> Workload:
    """A small batch with the configs' distributions: q, k ~ N(0,1), w ~ U(0,1)/8.
    k_format "mxfp4": E4M3 queries against keys in the paged mxfp4 cache layout (random
    nibble bytes, E8M0 scales uniform on 120..134 with 1% 0xFF, as the gather's cache)."""
    rng = Rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = lens.size
    T = B * next_n
    if paged:
        table, nblk = synth._page_pool(rng, lens, block_size, "block_table")
        rows = nblk * block_size
    else:
        assert B == 1
        table, rows = None, int(lens[0])
        if k_format == "mxfp4":
            rows = (rows + 3) // 4 * 4          # whole 16-byte rows of E8M0 bytes
        nblk = (rows + block_size - 1) // block_size
    if dtype == "bf16":
        q = synth.normal_bf16(rng, (T, H, D), "q")
        k = synth.normal_bf16(rng, (rows, D), "k")
        qs = ks = None
    else:
        qf = np.empty((T, H, D), np.float32)
        rng.normal_into(qf, "q")
        q, qs = synth.quantize_e4m3_rows(qf)
        kf = np.empty((rows, D), np.float32)
        rng.normal_into(kf, "k")
        k, ks = synth.quantize_e4m3_rows(kf)
    if k_format == "mxfp4":
        assert dtype == "e4m3"
        kn, ks8 = synth._mxfp4_pool(rng, (rows + block_size - 1) // block_size, block_size, "kcache")
        k = kn.reshape(-1, D // 2)[:rows]
        ks = ks8.reshape(-1, D // 32)[:rows]
    w = synth._weights(rng, T, "w")
    fp4 = sc = gtab = None
    if gather:
        gtab, gblk = (table, nblk) if paged else synth._page_pool(rng, lens, block_size, "gtab")
        fp4, sc = synth._mxfp4_pool(rng, gblk, block_size, "cache")
    return Workload("case", B, next_n, lens, causal, topk, dtype, q, qs, w, k, ks, table, block_size,
                    fp4, sc, gtab, pad_frac, seed, k_format)


def oracle_logits(wl: Workload, rows=None, width=None) -> np.ndarray:
    return orc.indexer_logits(wl.q, wl.q_scale, wl.dtype, wl.weights, wl.k_data, wl.k_scale,
                              wl.block_table, wl.block_size, wl.B, wl.next_n, wl.context_lens,
                              wl.causal, rows=rows, width=width,
                              k_dtype="mxfp4" if wl.k_format == "mxfp4" else None)


def assert_logits_close(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    gm, rm = got == -np.inf, ref == -np.inf
    bad = np.nonzero(gm != rm)
    assert bad[0].size == 0, f"mask differs at {list(zip(*bad))[:5]}"
    fin = ~rm
    assert np.isfinite(got[fin]).all()
    err = np.abs(got[fin] - ref[fin])
    tol = LOGIT_RTOL * (1.0 + np.abs(ref[fin]))
    worst = float((err / tol).max()) if err.size else 0.0
    assert worst <= 1.0, f"logit error {worst:.3f}x tolerance (max abs err {err.max():.3e})"
    return float(err.max()) if err.size else 0.0


def assert_topk_exact(gpu_idx: np.ndarray, logits_rows: np.ndarray, k: int, gpu_val=None) -> None:
    """GPU top-k == the oracle's top-k of the same (GPU) logits, bit-exact."""
    want_idx, want_val = orc.topk_select(logits_rows, k)
    bad = np.nonzero((gpu_idx != want_idx).any(axis=1))[0]
    assert bad.size == 0, (f"{bad.size} rows differ, first row {bad[0]}: "
                           f"gpu {gpu_idx[bad[0]][:8]} oracle {want_idx[bad[0]][:8]}")
    if gpu_val is not None:
        live = want_idx >= 0
        assert np.array_equal(np.asarray(gpu_val, np.float64)[live], want_val[live])
        assert np.all(np.asarray(gpu_val)[~live] == -np.inf)


def selection_parity(gpu_idx: np.ndarray, ref_logits: np.ndarray, k: int) -> float:
    """Mean Jaccard of the GPU selection against the oracle's selection on oracle logits;
    asserts the bar and the near-tie condition for every mismatch."""
    oidx, oval = orc.topk_select(ref_logits, k)
    jac = []
    for r in range(gpu_idx.shape[0]):
        a = set(int(x) for x in gpu_idx[r] if x >= 0)
        b = set(int(x) for x in oidx[r] if x >= 0)
        u = a | b
        jac.append(1.0 if not u else len(a & b) / len(u))
        diff = a ^ b
        if diff:
            live = oval[r][oidx[r] >= 0]
            vk = live[-1]
            for e in diff:
                v = ref_logits[r, e]
                assert abs(v - vk) <= LOGIT_RTOL * (1 + abs(vk)), (r, e, v, vk)
    m = float(np.mean(jac)) if jac else 1.0
    assert m >= 0.999, m
    return m


def sample_rows(T: int, n: int, seed: int) -> np.ndarray:
    """First, last and a seeded sample of query rows."""
    if T <= n:
        return np.arange(T)
    r = Rng(seed).permutation(T, "rows")[: max(0, n - 2)]
    return np.unique(np.concatenate([[0, T - 1], r])).astype(np.int64)
