"""CPU oracle of the DeepSeek-V4 DSA indexer hot path -- TEST INFRASTRUCTURE ONLY.

The oracle itself is plain, slow C++ (oracle/dsa_oracle.cpp: scalar float64 loops in
the order the problem states each step, std::thread over independent rows).  This
module only builds that file with the host C++ compiler (once, into oracle/_build/),
loads it with ctypes, and marshals numpy arrays in and out: it does no arithmetic of
its own.  Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it; the CUDA library never does, and shares no code with it.

Functions (same names and arguments as the float64 numpy cross-check in
dsa_oracle_np.py):

* ``indexer_logits`` -- the indexer score of xkernels issue #27 "DSA indexer +
  attention: validate/provide gfx942 forward path", comment 2 "What shipped";
* ``topk_select`` -- the per-query top-k under the canonical tie rule (README
  "DeepSeek V4 Flash on a single AMD MI300X", overlay table);
* ``mxfp4_paged_gather``, ``mxfp4_dequant``, ``e2m1_value``, ``e8m0_scale``,
  ``f64_to_bf16_bits`` -- the paged mxfp4 gather of xkernels issue #28
  "DeepSeek-V4 serving support -- tracking", comment 2 "What it does";
* ``bf16_to_f64``, ``e4m3_to_f64`` -- the storage decoders;
* ``e4m3_encode``, ``q_rope_quant`` -- the indexer-query RoPE + E4M3 producer (vllm PR #1
  "Sparse-MLA bring-up on MI300X", "Root cause story" items 1 and 3);
* ``e2m1_encode``, ``k_hadamard_mxfp4`` -- the indexer-key Hadamard + mxfp4 writer
  (ROCm/ATOM issue #707, "CSA");
* ``sparse_attn`` -- the sparse attention over the selection with sink logits
  (ROCm/ATOM issue #707, "CSA").

The worker count is ``DSA_ORACLE_THREADS`` (default: every hardware thread).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from ctypes import POINTER, c_double, c_float, c_int, c_int32, c_int64, c_uint8, c_uint16, c_void_p

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "dsa_oracle.cpp")
LIB = os.path.join(HERE, "_build", "libdsa_oracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]

_KIND = {"bf16": 0, "e4m3": 1, "mxfp4": 2}
_lock = threading.RLock()


def build(source: str = SOURCE, out: str = LIB, opt: str = "-O2", force: bool = False) -> str:
    """Compiles the oracle into a shared library (no-op when it is up to date)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cxx = os.environ.get("CXX", "g++")
    tmp = f"{out}.{os.getpid()}.tmp"
    flags = [opt if f == "-O2" else f for f in CXXFLAGS]
    r = subprocess.run([cxx, *flags, source, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, out)
    return out


def threads() -> int:
    return int(os.environ.get("DSA_ORACLE_THREADS", "0"))


def _p(a, ctype):
    return a.ctypes.data_as(POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The compiled oracle at `lib` (built from SOURCE when `lib` is None)."""

    def __init__(self, lib: str | None = None):
        if lib is None:
            with _lock:
                lib = build()
                try:
                    self.lib = ctypes.CDLL(lib)
                except OSError:                  # a stale library built for another machine
                    self.lib = ctypes.CDLL(build(force=True))
        else:
            self.lib = ctypes.CDLL(lib)
        L = self.lib
        L.orc_threads_used.restype = c_int
        L.orc_threads_used.argtypes = [c_int]
        for name, ctype in (("orc_bf16", c_uint16), ("orc_e4m3", c_uint8), ("orc_e2m1", c_uint8),
                            ("orc_e8m0", c_uint8)):
            fn = getattr(L, name)
            fn.restype = None
            fn.argtypes = [POINTER(ctype), c_int64, POINTER(c_double)]
        L.orc_bf16_round.restype = None
        L.orc_bf16_round.argtypes = [POINTER(c_double), c_int64, POINTER(c_uint16)]
        L.orc_mxfp4_dequant.restype = None
        L.orc_mxfp4_dequant.argtypes = [POINTER(c_uint8), POINTER(c_uint8), c_int64, c_int, POINTER(c_double)]
        L.orc_indexer_logits.restype = c_int
        L.orc_indexer_logits.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_void_p, c_void_p, c_int,
                                         c_int64, c_void_p, c_int64, c_int, c_int, c_int, c_void_p, c_int, c_void_p,
                                         c_int64, c_int64, POINTER(c_double), c_int]
        L.orc_topk.restype = c_int
        L.orc_topk.argtypes = [POINTER(c_double), c_int64, c_int64, c_int, POINTER(c_int32), POINTER(c_double), c_int]
        L.orc_e2m1_encode.restype = None
        L.orc_e2m1_encode.argtypes = [POINTER(c_double), c_int64, POINTER(c_uint8)]
        L.orc_e4m3_encode.restype = None
        L.orc_e4m3_encode.argtypes = [POINTER(c_float), c_int64, POINTER(c_uint8)]
        L.orc_q_rope_quant.restype = c_int
        L.orc_q_rope_quant.argtypes = [POINTER(c_uint16), POINTER(c_int32), POINTER(c_float), c_int64, c_int, c_int64,
                                       c_int, c_int, POINTER(c_uint8), POINTER(c_float), c_int]
        L.orc_k_hadamard_mxfp4.restype = c_int
        L.orc_k_hadamard_mxfp4.argtypes = [POINTER(c_uint16), POINTER(c_int64), c_int64, c_int, POINTER(c_uint8),
                                           POINTER(c_uint8), c_int64, c_int]
        L.orc_sparse_attn.restype = c_int
        L.orc_sparse_attn.argtypes = [POINTER(c_uint16), POINTER(c_int32), c_int64, c_int, c_int, c_int,
                                      POINTER(c_uint8), POINTER(c_uint8), c_int64, c_int, POINTER(c_int32), c_int64,
                                      c_int, POINTER(c_double), c_double, POINTER(c_double), c_int]
        L.orc_mxfp4_gather.restype = c_int
        L.orc_mxfp4_gather.argtypes = [POINTER(c_uint8), POINTER(c_uint8), c_int64, c_int, c_int, POINTER(c_int32),
                                       c_int64, POINTER(c_int32), c_int64, c_int, c_int, POINTER(c_uint16), c_int]

    # ------------------------------------------------------------------ decoders
    def _map(self, fn, x, dtype, ctype):
        a = _c(x, dtype)
        out = np.empty(a.shape, dtype=np.float64)
        fn(_p(a, ctype), a.size, _p(out, c_double))
        return out

    def bf16_to_f64(self, bits):
        return self._map(self.lib.orc_bf16, bits, np.uint16, c_uint16)

    def e4m3_to_f64(self, codes):
        return self._map(self.lib.orc_e4m3, codes, np.uint8, c_uint8)

    def e2m1_value(self, nibble):
        return self._map(self.lib.orc_e2m1, np.asarray(nibble).astype(np.int64) & 0xF, np.uint8, c_uint8)

    def e8m0_scale(self, b):
        return self._map(self.lib.orc_e8m0, np.asarray(b).astype(np.int64) & 0xFF, np.uint8, c_uint8)

    def f64_to_bf16_bits(self, x):
        a = _c(x, np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.orc_bf16_round(_p(a, c_double), a.size, _p(out, c_uint16))
        return out

    def mxfp4_dequant(self, fp4_rows, scale_rows):
        nib = _c(fp4_rows, np.uint8)
        sc = _c(scale_rows, np.uint8)
        N, half = nib.shape
        assert sc.shape == (N, 2 * half // 32)
        out = np.empty((N, 2 * half), dtype=np.float64)
        self.lib.orc_mxfp4_dequant(_p(nib, c_uint8), _p(sc, c_uint8), N, 2 * half, _p(out, c_double))
        return out

    # ------------------------------------------------------------------ score
    def indexer_logits(self, q, q_scale, dtype: str, weights, k_data, k_scale, block_table, block_size: int,
                       B: int, next_n: int, context_lens, causal: bool, rows=None, width=None, k_dtype=None):
        """Indexer score for the query rows ``rows`` (default: all T = B * next_n) as
        float64 [len(rows), width] (width = the longest context by default); -inf at
        masked keys.  ``dtype`` is the storage of q, and of the keys unless ``k_dtype``
        says otherwise ("mxfp4" keys: k_data = nibble rows [rows, D/2], k_scale = E8M0
        rows [rows, D/32])."""
        q = _c(q, np.uint16 if dtype == "bf16" else np.uint8)
        T, H, Dm = q.shape
        kd = k_dtype or dtype
        k = _c(k_data, np.uint16 if kd == "bf16" else np.uint8)
        ks = None
        if kd == "e4m3":
            ks = _c(k_scale, np.float64)
        elif kd == "mxfp4":
            ks = _c(k_scale, np.uint8)
        qs = _c(q_scale, np.float64) if dtype == "e4m3" else None
        w = _c(weights, np.float64)
        lens = _c(context_lens, np.int32)
        tab = None if block_table is None else _c(block_table, np.int32)
        rows = np.arange(B * next_n, dtype=np.int64) if rows is None else _c(rows, np.int64)
        width = int(lens.max()) if width is None else int(width)
        out = np.empty((rows.size, width), dtype=np.float64)
        rc = self.lib.orc_indexer_logits(
            q.ctypes.data, None if qs is None else qs.ctypes.data, _KIND[dtype], w.ctypes.data, H, Dm,
            k.ctypes.data, None if ks is None else ks.ctypes.data, _KIND[kd], k.shape[0],
            None if tab is None else tab.ctypes.data, 0 if tab is None else tab.shape[1], int(block_size), int(B),
            int(next_n), lens.ctypes.data, 1 if causal else 0, rows.ctypes.data, rows.size, width,
            _p(out, c_double), threads())
        assert rc == 0, "a visible key maps outside the key pool"
        return out

    # ------------------------------------------------------------------ top-k
    def topk_select(self, logits, k: int):
        """(idx int32 [R, k], val float64 [R, k]) per row under (value desc, index asc);
        -inf never selected; -1 / -inf past the candidates.  NaN logits are rejected."""
        x = _c(np.atleast_2d(np.asarray(logits, dtype=np.float64)), np.float64)
        R, K = x.shape
        idx = np.empty((R, k), dtype=np.int32)
        val = np.empty((R, k), dtype=np.float64)
        rc = self.lib.orc_topk(_p(x, c_double), R, K, int(k), _p(idx, c_int32), _p(val, c_double), threads())
        assert rc == 0, "NaN logits are outside the problem's domain"
        return idx, val

    # ------------------------------------------------------------------ gather
    def mxfp4_paged_gather(self, kv_fp4, kv_scale, block_table, sel_pos, B: int, next_n: int, block_size: int):
        """out[t, s, :] = bf16(dequant(cache row of sel_pos[t, s])), zeros where sel_pos < 0."""
        nib = _c(kv_fp4, np.uint8)
        sc = _c(kv_scale, np.uint8)
        tab = _c(block_table, np.int32)
        sel = _c(sel_pos, np.int32)
        T, K = sel.shape
        Dm = 2 * nib.shape[-1]
        out = np.empty((T, K, Dm), dtype=np.uint16)
        rc = self.lib.orc_mxfp4_gather(_p(nib, c_uint8), _p(sc, c_uint8), nib.shape[0], int(block_size), Dm,
                                       _p(tab, c_int32), tab.shape[1], _p(sel, c_int32), T, int(next_n), K,
                                       _p(out, c_uint16), threads())
        assert rc == 0, "a selected position maps outside the block table or the cache"
        return out

    # ------------------------------------------------------------------ producers
    def e2m1_encode(self, x):
        """Nearest E2M1 codes (nibbles) of values (ties to the even code, saturating at 6)."""
        a = _c(x, np.float64)
        out = np.empty(a.shape, dtype=np.uint8)
        self.lib.orc_e2m1_encode(_p(a, c_double), a.size, _p(out, c_uint8))
        return out

    def e4m3_encode(self, x):
        """Nearest OCP E4M3 codes of fp32 values (ties to even, saturating at +-448)."""
        a = _c(x, np.float32)
        out = np.empty(a.shape, dtype=np.uint8)
        self.lib.orc_e4m3_encode(_p(a, c_float), a.size, _p(out, c_uint8))
        return out

    def q_rope_quant(self, q, positions, cos_sin, rope_dim: int):
        """Indexer-Q producer: RoPE on the interleaved pairs of the first rope_dim dims of
        every head (cos / sin from the table row of the token's position), then per-row
        E4M3 quantisation.  q [T, H, D] bf16 bits -> (codes [T, H, D] uint8, scale [T, H])."""
        qb = _c(q, np.uint16)
        T, H, Dm = qb.shape
        pos = _c(positions, np.int32)
        cs = _c(cos_sin, np.float32)
        codes = np.empty((T, H, Dm), dtype=np.uint8)
        scale = np.empty((T, H), dtype=np.float32)
        rc = self.lib.orc_q_rope_quant(_p(qb, c_uint16), _p(pos, c_int32), _p(cs, c_float), cs.shape[0],
                                       int(rope_dim), T, H, Dm, _p(codes, c_uint8), _p(scale, c_float), threads())
        assert rc == 0, "a position lies outside the cos / sin table"
        return codes, scale

    def k_hadamard_mxfp4(self, k, slot, kv_fp4, kv_scale):
        """Indexer-key compressor write: Hadamard rotation + mxfp4 encoding of the keys
        k [N, D] (bf16 bits) into copies of the pools kv_fp4 [blocks, bs, D/2] and
        kv_scale [blocks, bs, D/32] at pool rows `slot` (< 0: skipped); returns them."""
        kb = _c(k, np.uint16)
        N, Dm = kb.shape
        sl = _c(slot, np.int64)
        fp4 = np.array(kv_fp4, dtype=np.uint8, copy=True, order="C")
        sc = np.array(kv_scale, dtype=np.uint8, copy=True, order="C")
        rows = fp4.size // (Dm // 2)
        rc = self.lib.orc_k_hadamard_mxfp4(_p(kb, c_uint16), _p(sl, c_int64), N, Dm, _p(fp4, c_uint8),
                                           _p(sc, c_uint8), rows, threads())
        assert rc == 0, "a slot lies outside the pool"
        return fp4, sc

    # ------------------------------------------------------------------ consumer
    def sparse_attn(self, q, sel_pos, kv_fp4, kv_scale, block_table, B: int, next_n: int, block_size: int,
                    sink, scale: float):
        """Sparse attention over the selected cache rows (key = value = the dequantised
        row), with a per-head sink logit in the softmax denominator.  q [T, H, D] bf16
        bits, sel_pos [T, k] -> out [T, H, D] float64 (zeros for a row with no selection)."""
        qb = _c(q, np.uint16)
        T, H, Dm = qb.shape
        sel = _c(sel_pos, np.int32)
        nib = _c(kv_fp4, np.uint8)
        sc = _c(kv_scale, np.uint8)
        tab = _c(block_table, np.int32)
        snk = _c(sink, np.float64)
        out = np.empty((T, H, Dm), dtype=np.float64)
        rc = self.lib.orc_sparse_attn(_p(qb, c_uint16), _p(sel, c_int32), T, H, Dm, sel.shape[1], _p(nib, c_uint8),
                                      _p(sc, c_uint8), nib.shape[0], int(block_size), _p(tab, c_int32), tab.shape[1],
                                      int(next_n), _p(snk, c_double), float(scale), _p(out, c_double), threads())
        assert rc == 0, "a selected position maps outside the block table or the cache"
        return out

    def threads_used(self) -> int:
        return int(self.lib.orc_threads_used(threads()))


_default = None


def _get() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
    return _default


def indexer_logits(*a, **kw):
    return _get().indexer_logits(*a, **kw)


def topk_select(*a, **kw):
    return _get().topk_select(*a, **kw)


def mxfp4_paged_gather(*a, **kw):
    return _get().mxfp4_paged_gather(*a, **kw)


def mxfp4_dequant(*a, **kw):
    return _get().mxfp4_dequant(*a, **kw)


def e2m1_value(*a, **kw):
    return _get().e2m1_value(*a, **kw)


def e8m0_scale(*a, **kw):
    return _get().e8m0_scale(*a, **kw)


def f64_to_bf16_bits(*a, **kw):
    return _get().f64_to_bf16_bits(*a, **kw)


def bf16_to_f64(*a, **kw):
    return _get().bf16_to_f64(*a, **kw)


def e4m3_to_f64(*a, **kw):
    return _get().e4m3_to_f64(*a, **kw)


def threads_used() -> int:
    return _get().threads_used()


def e4m3_encode(*a, **kw):
    return _get().e4m3_encode(*a, **kw)


def q_rope_quant(*a, **kw):
    return _get().q_rope_quant(*a, **kw)


def k_hadamard_mxfp4(*a, **kw):
    return _get().k_hadamard_mxfp4(*a, **kw)


def e2m1_encode(*a, **kw):
    return _get().e2m1_encode(*a, **kw)


def sparse_attn(*a, **kw):
    return _get().sparse_attn(*a, **kw)
