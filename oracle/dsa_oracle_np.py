"""Second, independent CPU implementation of the oracle -- TEST INFRASTRUCTURE ONLY.

The oracle the tests use is the plain C++ one (dsa_oracle.cpp through
dsa_oracle.py).  This numpy version is kept only as a cross-check of it
(tests/test_oracle_crosscheck.py): it shares no code with the C++ oracle or with
the CUDA library, and only tests import it.  It takes plain numpy arrays
(raw bf16 bits, E4M3 codes, mxfp4 bytes) and decodes them itself.

Every function is the plain definition, written out, in float64:

* ``indexer_logits`` -- the DSA indexer score of xkernels issue #27
  ("DSA indexer + attention: validate/provide gfx942 forward path", comment 2
  "What shipped"): logits[t, j] = sum_h weights[t, h] * relu(q[t, h, :] . k[j, :]),
  with q [T, H, D], one shared MQA key k [K, D], per-head weights and an
  optional per-query causal window.  The causal window is read as: query i of
  sequence b sits at absolute position p = L_b - next_n + i and sees key j iff
  j <= p (non-causal: j < L_b).  Masked keys get -inf (the same comment shows
  a -inf literal as the masked value).  One library matmul per query forms the
  [H, L] dot products; ReLU, the weighted head sum and the mask follow the
  formula term by term.
* ``topk_select`` -- the per-query top-k (top-512 Flash / top-1024 Pro, xkernels
  issue #27 "Context") under the deterministic tie rule: larger value first,
  then smaller index (the "canonical top-512 sort" / top-k tie-break overlays
  of README "DeepSeek V4 Flash on a single AMD MI300X", overlay table).  -0.0
  and +0.0 are one value; -inf is never selected; short rows pad with -1.
* ``e2m1_value`` / ``e8m0_scale`` / ``mxfp4_paged_gather`` -- the paged mxfp4
  gather of xkernels issue #28 ("DeepSeek-V4 serving support -- tracking",
  comment 2 "What it does"): E2M1 nibbles, one E8M0 scale 2^(b-127) per 32
  elements with 0xFF meaning 0, positions read through a block table,
  dequantised to bf16, padded slots (sel_pos < 0) -> zero row.  The E2M1 value
  set {0, 0.5, 1, 1.5, 2, 3, 4, 6} is the OCP Microscaling v1.0 definition; the
  oracle decodes by table (the GPU decodes arithmetically).  The low nibble of
  byte i holds element 2i.
* ``e4m3_to_f64`` -- OCP E4M3 (bias 7, no infinities, S.1111.111 = NaN,
  subnormals m * 2^-9), the byte format README "DeepSeek V4 Flash on a single
  AMD MI300X" ("FP8 format") contrasts with AMD's FNUZ variant.
* ``indexer_logits(..., k_dtype="mxfp4")`` -- the same score with the keys read
  from a paged mxfp4 cache (nibble rows + E8M0 scale rows, the gather's layout),
  as the fp8/fp4 logits kernel xkernels issue #27 names ("Unknown": the
  indexer forward uses an fp8-q x fp4-k MQA-logits kernel) computes it; per
  comment 2 ("Caveats / deferred") the packing is an encoding detail, so the
  definition is the score over the dequantised keys.

"""
from __future__ import annotations

import numpy as np

NEG_INF = float("-inf")

# ----------------------------------------------------------------------------- decoding

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32: widen the bits, reinterpret."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.

    e == 0: (-1)^s * (m / 8) * 2^-6 (subnormal); e == 15 and m == 7: NaN;
    otherwise (-1)^s * (1 + m / 8) * 2^(e - 7).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0**-6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


def dequantize(data: np.ndarray, scale, dtype: str) -> np.ndarray:
    """Storage -> float64 values.  E4M3 rows are multiplied by their fp32 row scale
    (exactly, in float64); bf16 has no scale; mxfp4 rows are [.., D/2] nibble bytes
    with [.., D/32] E8M0 scale bytes (see mxfp4_dequant)."""
    if dtype == "bf16":
        return bf16_to_f64(data)
    if dtype == "e4m3":
        v = e4m3_to_f64(data)
        return v * np.asarray(scale, dtype=np.float64)[..., None]
    if dtype == "mxfp4":
        return mxfp4_dequant(data, scale)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------- logits

def sequence_key_rows(b: int, L: int, block_table, block_size: int, num_rows: int) -> np.ndarray:
    """Physical row of each logical key j < L of sequence b.

    Paged: row = block_table[b, j // block_size] * block_size + j % block_size.
    Contiguous (no block table, one sequence): row = j.
    """
    j = np.arange(L, dtype=np.int64)
    if block_table is None:
        assert b == 0 and L <= num_rows
        return j
    blocks = np.asarray(block_table)[b, j // block_size].astype(np.int64)
    assert (blocks >= 0).all()
    rows = blocks * block_size + j % block_size
    assert (rows < num_rows).all()
    return rows


def indexer_logits(q, q_scale, dtype: str, weights, k_data, k_scale, block_table,
                   block_size: int, B: int, next_n: int, context_lens, causal: bool,
                   rows=None, width=None, k_dtype=None) -> np.ndarray:
    """Indexer score for the query rows ``rows`` (default: all T = B * next_n).

    ``dtype`` is the storage of q (and of the keys unless ``k_dtype`` says
    otherwise: "mxfp4" keys are k_data = nibble rows [rows, D/2] with k_scale =
    E8M0 rows [rows, D/32]).  Returns float64 [len(rows), width] with width = max
    context length by default; entries at masked or out-of-range keys are -inf.
    """
    context_lens = np.asarray(context_lens, dtype=np.int64)
    T = B * next_n
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    width = int(context_lens.max()) if width is None else int(width)
    w = np.asarray(weights, dtype=np.float64)
    out = np.full((rows.size, width), NEG_INF, dtype=np.float64)
    key_cache = {}
    for r, t in enumerate(rows):
        b, i = divmod(int(t), next_n)
        L = int(context_lens[b])
        if b not in key_cache:
            kr = sequence_key_rows(b, L, block_table, block_size, k_data.shape[0])
            ks = None if k_scale is None else np.asarray(k_scale)[kr]
            key_cache = {b: dequantize(np.asarray(k_data)[kr], ks, k_dtype or dtype)}  # [L, D]
        k = key_cache[b]
        qs = None if q_scale is None else np.asarray(q_scale)[t]
        qt = dequantize(np.asarray(q)[t], qs, dtype)                      # [H, D]
        visible = (L - next_n + i + 1) if causal else L
        visible = max(0, min(visible, L))
        s = qt @ k[:visible].T                                          # [H, visible]
        relu = np.maximum(s, 0.0)
        out[r, :visible] = w[t] @ relu                                  # sum over heads
    return out


# ----------------------------------------------------------------------------- top-k

def topk_select(logits: np.ndarray, k: int):
    """Top-k per row under (value descending, index ascending); -inf never selected.

    Returns (idx int32 [R, k], val float64 [R, k]); slots past the number of
    finite candidates hold -1 / -inf.  NaN logits are not part of the problem
    (ReLU and finite weights cannot produce them) and are rejected.
    """
    x = np.atleast_2d(np.asarray(logits))
    assert not np.isnan(x).any(), "NaN logits are outside the problem's domain"
    R = x.shape[0]
    idx = np.full((R, k), -1, dtype=np.int32)
    val = np.full((R, k), NEG_INF, dtype=np.float64)
    for r in range(R):
        row = x[r] + 0.0          # canonical zero: -0.0 + 0.0 == +0.0
        cand = np.nonzero(row != NEG_INF)[0]
        v = row[cand]
        order = np.lexsort((cand, -v))   # primary: value desc; secondary: index asc
        take = order[:k]
        idx[r, :take.size] = cand[take]
        val[r, :take.size] = v[take]
    return idx, val


# ----------------------------------------------------------------------------- mxfp4

_E2M1_MAGNITUDE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_value(nibble: np.ndarray) -> np.ndarray:
    """E2M1 nibble s|e1 e0|m -> value, by the OCP MX magnitude table and sign bit 3."""
    n = np.asarray(nibble, dtype=np.int64) & 0xF
    mag = np.asarray(_E2M1_MAGNITUDE, dtype=np.float64)[n & 7]
    return np.where((n & 8) != 0, -mag, mag)


def e8m0_scale(b: np.ndarray) -> np.ndarray:
    """E8M0 group scale: 2^(b-127); the byte 0xFF means a scale of 0."""
    b = np.asarray(b, dtype=np.int64)
    return np.where(b == 0xFF, 0.0, np.ldexp(1.0, (b - 127).astype(np.int32)))


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16, nearest-even, returning bit patterns.

    Goes through binary32 first; every value this oracle rounds (an E2M1 value
    times a power of two) has at most two significant bits, so that step is
    exact (or overflows to inf, as the bf16 rounding would).
    """
    with np.errstate(over="ignore"):
        f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    r[nan] = np.uint16(0x7FC0)
    return r


def mxfp4_dequant(fp4_rows: np.ndarray, scale_rows: np.ndarray) -> np.ndarray:
    """[N, D/2] nibble bytes + [N, D/32] E8M0 bytes -> float64 [N, D].

    Element e is nibble (e & 1) of byte e // 2 (low nibble first) times the
    scale of its group e // 32.
    """
    fp4_rows = np.asarray(fp4_rows, dtype=np.uint8)
    N, half = fp4_rows.shape
    Dm = 2 * half
    nib = np.empty((N, Dm), dtype=np.uint8)
    nib[:, 0::2] = fp4_rows & 0xF
    nib[:, 1::2] = fp4_rows >> 4
    vals = e2m1_value(nib)
    sc = e8m0_scale(np.asarray(scale_rows, dtype=np.uint8))       # [N, D/32]
    return vals * np.repeat(sc, 32, axis=1)


def mxfp4_paged_gather(kv_fp4, kv_scale, block_table, sel_pos, B: int, next_n: int,
                       block_size: int) -> np.ndarray:
    """out[t, s, :] = bf16(dequant(cache row of sel_pos[t, s])) or zeros when sel_pos < 0.

    Sequence of row t is b = t // next_n; the cache row of logical position pos is
    (block_table[b, pos // block_size], pos % block_size).
    """
    kv_fp4 = np.asarray(kv_fp4, dtype=np.uint8)
    kv_scale = np.asarray(kv_scale, dtype=np.uint8)
    sel = np.asarray(sel_pos, dtype=np.int64)
    T, K = sel.shape
    Dm = 2 * kv_fp4.shape[-1]
    out = np.zeros((T, K, Dm), dtype=np.uint16)
    b = np.repeat(np.arange(B), next_n)[:, None].repeat(K, axis=1)
    live = sel >= 0
    pos = sel[live]
    blk = np.asarray(block_table, dtype=np.int64)[b[live], pos // block_size]
    off = pos % block_size
    vals = mxfp4_dequant(kv_fp4[blk, off], kv_scale[blk, off])
    out[live] = f64_to_bf16_bits(vals)
    return out
