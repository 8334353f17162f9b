"""Seeded synthetic workloads for the DSA indexer hot path.

This module only *draws* inputs: random bits, normals, uniform integers,
permutations, and the rounding of the drawn reals into the storage formats
the kernels consume (bf16 bits, OCP E4M3 codes with a per-row scale, raw
mxfp4 bytes).  It holds none of the method's arithmetic (no logits, no
top-k, no mxfp4 decode), so the CPU oracle and the CUDA path can both take
their inputs from here without sharing any of the computation they check.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used in counter mode so every named draw is
an independent stream that does not shift when other draws are added:
``x_i = mix(base(seed, stream) + (i + 1) * 0x9E3779B97F4A7C15)``.
Normals come from the Box-Muller transform in float64, rounded to float32
(numpy RNE) and then to bf16 (round to nearest even).  Uniform integers use a
32x32->64 multiply-shift on the high 32 bits (bias <= range / 2**32).

Workload shapes follow the five configurations of the DeepSeek-V4 indexer
problem statement (xkernels issue #27 "Context": index_n_heads 64,
index_head_dim 128; top-512 Flash / top-1024 Pro; xkernels issue #28,
comment 2 "What it does": paged mxfp4 cache, E2M1 nibbles plus one E8M0 scale
per 32 elements, padded slots sel_pos < 0).
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np

H = 64
D = 128

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: str) -> np.uint64:
    tag = int.from_bytes(hashlib.sha256(stream.encode()).digest()[:8], "little")
    z = np.array([(seed * 0x9E3779B97F4A7C15 + tag) & (2**64 - 1)], dtype=np.uint64)
    return _mix(z)[0]


class Rng:
    """Counter-mode SplitMix64 with named, independent streams."""

    def __init__(self, seed: int):
        self.seed = int(seed)

    def u64(self, n: int, stream: str, start: int = 0) -> np.ndarray:
        base = _stream_base(self.seed, stream)
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            return _mix(base + i * _GAMMA)

    def uniform(self, n: int, stream: str, start: int = 0) -> np.ndarray:
        """Doubles in [0, 1) from the top 53 bits."""
        return (self.u64(n, stream, start) >> np.uint64(11)).astype(np.float64) * (2.0**-53)

    def integers(self, lo: int, hi: int, n: int, stream: str) -> np.ndarray:
        """Integers uniform on [lo, hi] (inclusive), multiply-shift on 32 bits."""
        span = np.uint64(hi - lo + 1)
        top = self.u64(n, stream) >> np.uint64(32)
        return (lo + ((top * span) >> np.uint64(32)).astype(np.int64)).astype(np.int64)

    def permutation(self, n: int, stream: str) -> np.ndarray:
        """Uniform shuffle: order of n random 64-bit keys (ties broken by position)."""
        return np.argsort(self.u64(n, stream), kind="stable").astype(np.int64)

    def normal_into(self, out: np.ndarray, stream: str) -> None:
        """Fill a float32 array with N(0,1) via Box-Muller in float64."""
        flat = out.reshape(-1)
        n = flat.size
        pairs = (n + 1) // 2
        for p0 in range(0, pairs, _CHUNK):
            m = min(_CHUNK, pairs - p0)
            u1 = self.uniform(m, stream + "/u1", p0)
            u2 = self.uniform(m, stream + "/u2", p0)
            r = np.sqrt(-2.0 * np.log1p(-u1))
            th = (2.0 * np.pi) * u2
            blk = np.empty(2 * m, dtype=np.float64)
            blk[0::2] = r * np.cos(th)
            blk[1::2] = r * np.sin(th)
            lo = 2 * p0
            hi = min(n, lo + 2 * m)
            flat[lo:hi] = blk[: hi - lo].astype(np.float32)

    def bytes_into(self, out: np.ndarray, stream: str) -> None:
        """Fill a uint8 array with uniform random bytes."""
        flat = out.reshape(-1)
        n = flat.size
        words = (n + 7) // 8
        for w0 in range(0, words, _CHUNK):
            m = min(_CHUNK, words - w0)
            b = self.u64(m, stream, w0).view(np.uint8)
            lo = 8 * w0
            hi = min(n, lo + 8 * m)
            flat[lo:hi] = b[: hi - lo]


# ---------------------------------------------------------------- storage formats

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def normal_bf16(rng: Rng, shape, stream: str) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    # Draw in slices so multi-GB key pools never hold a float64 copy.  Every slice has
    # its own named stream, so the slices are independent and are drawn by a few
    # threads at once (numpy releases the GIL in the transcendental functions); the
    # values do not depend on the thread count.
    step = max(1, min(flat.size, 2 * _CHUNK))
    starts = list(range(0, flat.size, step))

    def draw(s0):
        m = min(step, flat.size - s0)
        buf = np.empty(m, dtype=np.float32)
        rng.normal_into(buf, f"{stream}@{s0}")
        flat[s0:s0 + m] = f32_to_bf16_bits(buf)

    if len(starts) <= 1:
        for s0 in starts:
            draw(s0)
    else:
        import concurrent.futures as cf
        import os
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1, len(starts))) as ex:
            list(ex.map(draw, starts))
    return out


def quantize_e4m3_rows(x: np.ndarray):
    """Per-row OCP E4M3 quantisation of a float32 array [..., R].

    scale = max|x_row| / 448 (float32), code = E4M3(RNE, saturating)(x / scale);
    an all-zero row gets scale 1.  The E4M3 rounding is torch's float32 ->
    float8_e4m3fn conversion after clamping to +-448 (the format's largest
    finite magnitude), which makes it saturating.
    """
    import torch

    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    scale[amax == 0] = np.float32(1.0)
    y = np.clip(x / scale[..., None], np.float32(-448.0), np.float32(448.0)).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, scale


# ---------------------------------------------------------------- workloads

@dataclasses.dataclass
class Workload:
    """One batch of indexer + gather inputs (host arrays).

    q         [T, H, D] uint16 (bf16 bits) or uint8 (E4M3 codes); T = B * next_n
    q_scale   [T, H] float32 or None
    weights   [T, H] float32
    k_data    [rows, D] uint16 / uint8: the paged pool (nblk * block_size rows)
              when block_table is set, else the contiguous keys of one sequence
              (k_format "mxfp4": [rows, D/2] nibble bytes of the paged mxfp4 cache)
    k_scale   [rows] float32 or None (k_format "mxfp4": [rows, D/32] E8M0 bytes)
    block_table [B, max_blocks] int32 or None (unused entries are -1)
    kv_fp4    [nblk_g, block_size, D/2] uint8, low nibble = even element
    kv_scale  [nblk_g, block_size, D/32] uint8 E8M0
    gather_block_table [B, max_blocks_g] int32
    """

    name: str
    B: int
    next_n: int
    context_lens: np.ndarray
    causal: bool
    topk: int
    dtype: str
    q: np.ndarray
    q_scale: Optional[np.ndarray]
    weights: np.ndarray
    k_data: np.ndarray
    k_scale: Optional[np.ndarray]
    block_table: Optional[np.ndarray]
    block_size: int
    kv_fp4: Optional[np.ndarray] = None
    kv_scale: Optional[np.ndarray] = None
    gather_block_table: Optional[np.ndarray] = None
    gather_pad_frac: float = 0.0
    seed: int = 0
    k_format: str = "native"   # "mxfp4": k_data = nibble rows [rows, D/2], k_scale = E8M0 rows [rows, D/32]

    @property
    def T(self) -> int:
        return self.B * self.next_n

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.B else 0

    def positions(self) -> np.ndarray:
        """Absolute position p of every query row: L_b - next_n + i."""
        L = np.repeat(self.context_lens.astype(np.int64), self.next_n)
        i = np.tile(np.arange(self.next_n, dtype=np.int64), self.B)
        return L - self.next_n + i

    def visible_len(self) -> np.ndarray:
        """Number of leading keys each query row may see (causal: p + 1, else L_b)."""
        if self.causal:
            return self.positions() + 1
        return np.repeat(self.context_lens.astype(np.int64), self.next_n)


def _page_pool(rng: Rng, context_lens: np.ndarray, block_size: int, stream: str):
    """Deal a random permutation of all physical blocks to the sequences in order."""
    nblocks = [(int(L) + block_size - 1) // block_size for L in context_lens]
    total = int(sum(nblocks))
    perm = rng.permutation(total, stream).astype(np.int32)
    width = max(nblocks) if nblocks else 0
    table = np.full((len(context_lens), max(width, 1)), -1, dtype=np.int32)
    o = 0
    for b, nb in enumerate(nblocks):
        table[b, :nb] = perm[o:o + nb]
        o += nb
    return table, total


def _mxfp4_pool(rng: Rng, nblk: int, block_size: int, stream: str, ff_frac: float = 0.01, sc_lo: int = 120,
                sc_span: int = 14):
    """Random nibble bytes; E8M0 scales uniform on sc_lo .. sc_lo + sc_span - 1 (120..133
    by default) with ~1% set to 0xFF."""
    fp4 = np.empty((nblk, block_size, D // 2), dtype=np.uint8)
    rng.bytes_into(fp4, stream + "/nib")
    n_sc = nblk * block_size * (D // 32)
    sc = (sc_lo + rng.integers(0, sc_span, n_sc, stream + "/sc")).astype(np.uint8)
    ff = rng.uniform(n_sc, stream + "/ff") < ff_frac
    sc[ff] = 0xFF
    return fp4, sc.reshape(nblk, block_size, D // 32)


def _weights(rng: Rng, T: int, stream: str) -> np.ndarray:
    return (rng.uniform(T * H, stream).astype(np.float32) / np.float32(8.0)).reshape(T, H)


def make_tiny(seed: int = 1, T: int = 64, L: int = 2048, topk: int = 512) -> Workload:
    """T queries at positions L-T..L-1 over L contiguous bf16 keys, causal."""
    rng = Rng(seed)
    q = normal_bf16(rng, (T, H, D), "q")
    k = normal_bf16(rng, (L, D), "k")
    w = _weights(rng, T, "w")
    lens = np.array([L], dtype=np.int32)
    gtab, nblk = _page_pool(rng, lens, 64, "gather_table")
    fp4, sc = _mxfp4_pool(rng, nblk, 64, "cache")
    return Workload("tiny", 1, T, lens, True, topk, "bf16", q, None, w, k, None, None, 64,
                    fp4, sc, gtab, 0.05, seed)


def make_decode(seed: int, B: int, next_n: int, lmin: int, lmax: int, topk: int,
                name: str, pad_frac: float, block_size: int = 64, with_keys: bool = True) -> Workload:
    """Paged bf16 decode batch: B sequences, next_n causal query tokens each.
    with_keys=False leaves the bf16 key pool empty (for gather-only use)."""
    rng = Rng(seed)
    lens = rng.integers(lmin, lmax, B, "context_lens").astype(np.int32)
    table, nblk = _page_pool(rng, lens, block_size, "block_table")
    T = B * next_n
    q = normal_bf16(rng, (T, H, D), "q")
    k = normal_bf16(rng, (nblk * block_size if with_keys else 0, D), "k_pool")
    w = _weights(rng, T, "w")
    fp4, sc = _mxfp4_pool(rng, nblk, block_size, "cache")
    return Workload(name, B, next_n, lens, True, topk, "bf16", q, None, w, k, None, table,
                    block_size, fp4, sc, table, pad_frac, seed)


def make_flash_decode(seed: int = 2, B: int = 64, lmin: int = 4096, lmax: int = 65536,
                      with_keys: bool = True) -> Workload:
    return make_decode(seed, B, 1, lmin, lmax, 512, "flash_decode", 0.0, with_keys=with_keys)


def make_pro_mtp(seed: int = 3, B: int = 32, lmin: int = 32768, lmax: int = 131072,
                 with_keys: bool = True) -> Workload:
    return make_decode(seed, B, 2, lmin, lmax, 1024, "pro_mtp", 0.02, with_keys=with_keys)


def make_flash_decode_fp4k(seed: int = 2, B: int = 64) -> Workload:
    """The Flash decode batch scored in its FP8-q x FP4-k form: the queries quantised to
    E4M3 with a per-(token, head) scale (rowmax / 448), the keys read straight from the
    batch's paged mxfp4 cache (the cache the gather reads, through the same table)."""
    wl = make_flash_decode(seed=seed, B=B, with_keys=False)
    qf = (wl.q.astype(np.uint32) << np.uint32(16)).view(np.float32)
    wl.q, wl.q_scale = quantize_e4m3_rows(qf)
    wl.dtype = "e4m3"
    wl.k_format = "mxfp4"
    nblk = wl.kv_fp4.shape[0]
    wl.k_data = wl.kv_fp4.reshape(nblk * wl.block_size, D // 2)
    wl.k_scale = wl.kv_scale.reshape(nblk * wl.block_size, D // 32)
    wl.name = "flash_decode_fp4k"
    return wl


def make_prefill(seed: int = 4, T: int = 16384, topk: int = 512) -> Workload:
    """One sequence, T = K, full causal mask, contiguous bf16 keys, no gather."""
    rng = Rng(seed)
    q = normal_bf16(rng, (T, H, D), "q")
    k = normal_bf16(rng, (T, D), "k")
    w = _weights(rng, T, "w")
    lens = np.array([T], dtype=np.int32)
    return Workload("prefill", 1, T, lens, True, topk, "bf16", q, None, w, k, None, None, 64,
                    seed=seed)


def make_fp8_chunked(seed: int = 5, T: int = 8192, L: int = 65536, topk: int = 1024,
                     gather_blocks: Optional[int] = None) -> Workload:
    """T E4M3 queries at positions L-T..L-1 over L contiguous E4M3 keys, causal,
    per-row fp32 scales; then a gather of every selection from a paged mxfp4 pool."""
    rng = Rng(seed)
    T_rows = T
    qf = np.empty((T_rows, H, D), dtype=np.float32)
    rng.normal_into(qf, "q")
    q, q_scale = quantize_e4m3_rows(qf)
    del qf
    kf = np.empty((L, D), dtype=np.float32)
    rng.normal_into(kf, "k")
    k, k_scale = quantize_e4m3_rows(kf)
    del kf
    w = _weights(rng, T_rows, "w")
    lens = np.array([L], dtype=np.int32)
    gtab, nblk = _page_pool(rng, lens, 64, "gather_table")
    if gather_blocks is not None:
        assert gather_blocks == nblk
    fp4, sc = _mxfp4_pool(rng, nblk, 64, "cache")
    return Workload("fp8_chunked", 1, T_rows, lens, True, topk, "e4m3", q, q_scale, w, k,
                    k_scale, None, 64, fp4, sc, gtab, 0.0, seed)


def pad_sel_pos(sel_pos: np.ndarray, frac: float, seed: int, stream: str = "pad") -> np.ndarray:
    """Overwrite a seeded fraction of the selected positions with -1 (padded slots)."""
    out = np.array(sel_pos, dtype=np.int32, copy=True)
    if frac > 0:
        m = Rng(seed).uniform(out.size, stream) < frac
        out.reshape(-1)[m] = -1
    return out


def random_sel_pos(wl: Workload, seed: int, stream: str = "sel") -> np.ndarray:
    """Distinct random visible positions per query row (a stand-in selection),
    padded with -1 where a row sees fewer than topk keys."""
    rng = Rng(seed)
    vis = wl.visible_len()
    out = np.full((wl.T, wl.topk), -1, dtype=np.int32)
    for t in range(wl.T):
        n = int(vis[t])
        keys = rng.u64(n, f"{stream}/{t}")
        pick = np.argsort(keys, kind="stable")[: min(n, wl.topk)]
        out[t, : pick.size] = pick
    return out


@dataclasses.dataclass
class AttnBatch:
    """Sparse-attention inputs: query rows, their selection and the paged mxfp4 cache.

    q        [T, 64, 128] uint16 (bf16 bits); row t belongs to sequence t // next_n
    sel      [T, topk] int32 positions (-1: padded slot)
    kv_fp4   [nblk, block_size, 64] uint8, kv_scale [nblk, block_size, 4] uint8
    table    [B, max_blocks] int32
    sink     [64] float32 per-head sink logits; scale = the softmax scale
    """

    name: str
    B: int
    next_n: int
    context_lens: np.ndarray
    topk: int
    block_size: int
    q: np.ndarray
    sel: np.ndarray
    kv_fp4: np.ndarray
    kv_scale: np.ndarray
    table: np.ndarray
    sink: np.ndarray
    scale: float

    @property
    def T(self) -> int:
        return self.B * self.next_n


def make_attn(seed: int, lens, next_n: int, topk: int, block_size: int = 64, pad_frac: float = 0.02,
              distinct: bool = True, name: str = "attn", sc_lo: int = 124, sc_span: int = 5,
              sink_lo: float = -2.0, sink_hi: float = 2.0, scale: float = 128 ** -0.5) -> AttnBatch:
    """A sparse-attention batch: len(lens) sequences with next_n causal query rows each,
    topk selected positions per row (distinct when `distinct`, else drawn uniformly with
    repeats), a seeded fraction padded; a cache whose scale bytes span sc_lo ..
    sc_lo + sc_span - 1 (124..128: elements within +-12, like a Hadamard-rotated key
    quantised per 32 elements) with ~1% 0xFF groups; sinks uniform on [sink_lo, sink_hi)."""
    rng = Rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = lens.size
    table, nblk = _page_pool(rng, lens, block_size, "attn_table")
    fp4, sc = _mxfp4_pool(rng, nblk, block_size, "attn_cache", sc_lo=sc_lo, sc_span=sc_span)
    T = B * next_n
    q = normal_bf16(rng, (T, H, D), "attn_q")
    vis = np.repeat(lens.astype(np.int64), next_n) - next_n + np.tile(np.arange(next_n), B) + 1
    sel = np.full((T, topk), -1, dtype=np.int32)
    if distinct:
        for t in range(T):
            n = int(vis[t])
            pick = np.argsort(rng.u64(n, f"attn_sel/{t}"), kind="stable")[: min(n, topk)]
            sel[t, : pick.size] = pick
    else:
        u = rng.uniform(T * topk, "attn_sel").reshape(T, topk)
        sel[:] = np.minimum((u * vis[:, None]).astype(np.int64), vis[:, None] - 1)
    sel = pad_sel_pos(sel, pad_frac, seed, "attn_pad")
    sink = (sink_lo + (sink_hi - sink_lo) * rng.uniform(H, "attn_sink")).astype(np.float32)
    return AttnBatch(name, B, next_n, lens, topk, block_size, q, sel, fp4, sc, table, sink, float(scale))


def make_attn_config(name: str, seed: int = 7) -> AttnBatch:
    """The sparse-attention batch of a named shape: Flash decode (64 sequences of 4K-64K
    keys, top-512), Pro decode MTP (32 sequences of 32K-128K keys, two query rows each,
    top-1024), FP8 chunked prefill (8192 causal rows at the end of a 64K-key sequence,
    top-1024); selections drawn uniformly (with repeats), 2% padded."""
    rng = Rng(seed)
    if name == "flash_decode":
        return make_attn(seed, rng.integers(4096, 65536, 64, "lens"), 1, 512, distinct=False, name=name)
    if name == "pro_mtp":
        return make_attn(seed, rng.integers(32768, 131072, 32, "lens"), 2, 1024, distinct=False, name=name)
    if name == "fp8_chunked":
        return make_attn(seed, [65536], 8192, 1024, distinct=False, name=name)
    raise KeyError(name)


CONFIGS = {
    "tiny": make_tiny,
    "flash_decode": make_flash_decode,
    "pro_mtp": make_pro_mtp,
    "prefill": make_prefill,
    "fp8_chunked": make_fp8_chunked,
}
