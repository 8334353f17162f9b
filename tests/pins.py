"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each ``check_*`` takes an oracle module and raises AssertionError when the
oracle disagrees with a value or property that does not come from the oracle
itself: hand-worked fixtures under tests/golden/ (each cites its passage),
library routines (torch's bf16 / float8_e4m3fn conversions), closed forms,
invariants and brute force on tiny inputs.  The same checks run against
deliberately broken copies of the oracle in test_oracle_mutants.py, to show
that a plausible mistake in it would be caught.
"""
from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- fixtures

def load_mxfp4_rows():
    rows = []
    cur = None
    with open(os.path.join(GOLDEN, "mxfp4_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tag, *rest = line.split()
            if tag == "row":
                cur = {"name": rest[0], "bytes": np.zeros(64, np.uint8),
                       "scales": None, "expect": np.zeros(128, np.uint16)}
                rows.append(cur)
            elif tag == "scales":
                cur["scales"] = np.array([int(x, 16) for x in rest], dtype=np.uint8)
            elif tag == "bytes":
                for item in rest:
                    i, v = item.split(":")
                    cur["bytes"][int(i)] = int(v, 16)
            elif tag == "expect":
                for item in rest:
                    e, v = item.split(":")
                    cur["expect"][int(e)] = int(v, 16)
    return rows


def load_logits_case():
    vals = {}
    with open(os.path.join(GOLDEN, "logits_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                tag, *rest = line.split()
                vals[tag] = rest
    H, Dm, L, n = (int(vals[k][0]) for k in ("H", "D", "L", "next_n"))
    q = np.array([float(x) for x in vals["q"]]).reshape(n, H, Dm)
    w = np.array([float(x) for x in vals["w"]]).reshape(n, H)
    k = np.array([float(x) for x in vals["k"]]).reshape(L, Dm)
    expect = np.array([float(x) for x in vals["expect"]]).reshape(n, L)
    return H, Dm, L, n, q, w, k, expect


def load_topk_cases():
    cases = []
    row = None
    with open(os.path.join(GOLDEN, "topk_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tag, *rest = line.split()
            if tag == "row":
                row = np.array([float(x) for x in rest], dtype=np.float64)
            elif tag == "k":
                k = int(rest[0])
                assert rest[1] == "expect"
                cases.append((row, k, np.array([int(x) for x in rest[2:]], dtype=np.int32)))
    return cases


def f64_to_bf16_exact(x: np.ndarray) -> np.ndarray:
    """bf16 bits of values that bf16 represents exactly (fixtures are chosen so)."""
    f = np.asarray(x, dtype=np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64))
    u = f.view(np.uint32)
    assert (u & 0xFFFF == 0).all()
    return (u >> 16).astype(np.uint16)


# --------------------------------------------------------------------------- decoders

def check_bf16_decode(orc):
    import torch
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = orc.bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan].astype(np.float64))
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def check_e4m3_decode(orc):
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = orc.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2                       # S.1111.111 only
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan].astype(np.float64))
    # hand values from the OCP E4M3 definition
    hand = {0x38: 1.0, 0x7E: 448.0, 0x01: 2.0**-9, 0x08: 2.0**-6, 0xBC: -1.5, 0x00: 0.0, 0x40: 2.0}
    for c, v in hand.items():
        assert orc.e4m3_to_f64(np.array([c], np.uint8))[0] == v, hex(c)
    assert np.signbit(orc.e4m3_to_f64(np.array([0x80], np.uint8))[0])


def check_bf16_rounding(orc):
    import torch
    x = np.concatenate([
        np.random.default_rng(0).standard_normal(20000).astype(np.float32) * 1e3,
        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, 3.4e38, -3.4e38, 1e-40, -1e-40, 2.0**-128,
                  0.0, -0.0, np.inf, -np.inf], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------- mxfp4

def check_e8m0(orc):
    b = np.arange(256)
    s = orc.e8m0_scale(b)
    assert s[127] == 1.0 and s[128] == 2.0 and s[126] == 0.5
    assert s[0] == 2.0**-127 and s[254] == 2.0**127
    assert s[255] == 0.0
    assert np.all(s[1:255] == 2.0 * s[0:254])   # one binade per step


def check_e2m1(orc):
    # OCP MX E2M1 magnitudes, then the sign bit
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = orc.e2m1_value(np.arange(16))
    assert list(got[:8]) == mags
    assert list(-got[8:]) == mags
    assert np.signbit(got[8])


def check_mxfp4_hand_rows(orc):
    for row in load_mxfp4_rows():
        vals = orc.mxfp4_dequant(row["bytes"][None, :], row["scales"][None, :])[0]
        got = orc.f64_to_bf16_bits(vals)
        bad = np.nonzero(got != row["expect"])[0]
        assert bad.size == 0, (row["name"], bad[:8], got[bad[:8]], row["expect"][bad[:8]])


def check_mxfp4_gather_hand(orc):
    """Padded slot -> 256 zero bytes; a live slot reads its row through the table."""
    rows = load_mxfp4_rows()
    bs = 2
    nblk = 2
    fp4 = np.zeros((nblk, bs, 64), np.uint8)
    sc = np.full((nblk, bs, 4), 0x7F, np.uint8)
    # logical position 1 of sequence 0 -> block_table[0, 0] = 1, offset 1
    fp4[1, 1] = rows[0]["bytes"]
    sc[1, 1] = rows[0]["scales"]
    table = np.array([[1, 0]], np.int32)
    sel = np.array([[1, -1, 2]], np.int32)        # position 2 -> block 0, offset 0 (zeros)
    out = orc.mxfp4_paged_gather(fp4, sc, table, sel, 1, 1, bs)
    assert out.shape == (1, 3, 128) and out.dtype == np.uint16
    assert np.array_equal(out[0, 0], rows[0]["expect"])
    assert not out[0, 1].any()
    assert not out[0, 2].any()


def check_gather_invariant(orc, seed=7):
    """Dequantise the whole cache then index == gather (index then dequantise), bitwise.

    The indexing on the left is an explicit loop over (t, s) written here.
    """
    r = np.random.default_rng(seed)
    B, n, K, bs, nblk = 3, 2, 9, 4, 7
    fp4 = r.integers(0, 256, (nblk, bs, 64), dtype=np.uint8)
    sc = r.integers(118, 137, (nblk, bs, 4)).astype(np.uint8)
    sc[r.random(sc.shape) < 0.1] = 0xFF
    table = np.stack([r.permutation(nblk)[:3] for _ in range(B)]).astype(np.int32)
    sel = r.integers(-1, 3 * bs, (B * n, K)).astype(np.int32)
    flat_vals = orc.mxfp4_dequant(fp4.reshape(-1, 64), sc.reshape(-1, 4))
    flat_bits = orc.f64_to_bf16_bits(flat_vals)
    expect = np.zeros((B * n, K, 128), np.uint16)
    for t in range(B * n):
        for s in range(K):
            pos = int(sel[t, s])
            if pos < 0:
                continue
            blk = int(table[t // n, pos // bs])
            expect[t, s] = flat_bits[blk * bs + pos % bs]
    got = orc.mxfp4_paged_gather(fp4, sc, table, sel, B, n, bs)
    assert np.array_equal(got, expect)


# --------------------------------------------------------------------------- logits

def _logits(orc, q, w, k, B, n, lens, causal=True, table=None, bs=1, q_scale=None,
            k_scale=None, dtype="bf16"):
    return orc.indexer_logits(q, q_scale, dtype, w, k, k_scale, table, bs, B, n, lens, causal)


def _as_bf16(x):
    return f64_to_bf16_exact(np.asarray(x, dtype=np.float64))


def check_logits_hand(orc):
    H, Dm, L, n, q, w, k, expect = load_logits_case()
    lens = np.array([L])
    got = _logits(orc, _as_bf16(q), w, _as_bf16(k), 1, n, lens)
    assert np.array_equal(got, expect), got
    # the same keys through a permuted page table (block size 2)
    pool = np.concatenate([k[2:4], k[0:2]])          # physical block 0 = keys 2,3; block 1 = keys 0,1
    table = np.array([[1, 0]], np.int32)
    got_p = _logits(orc, _as_bf16(q), w, _as_bf16(pool), 1, n, lens, table=table, bs=2)
    assert np.array_equal(got_p, expect)
    # non-causal: query 0 also sees key 3: h0 = 1+2 = 3, h1 = -1+0.5 < 0 -> 2*3 = 6
    got_nc = _logits(orc, _as_bf16(q), w, _as_bf16(k), 1, n, lens, causal=False)
    assert got_nc[0, 3] == 6.0 and np.array_equal(got_nc[1], expect[1])


def check_logits_plain_matmul(orc, seed=3):
    """H = 1, w = 1 and positive q, k: the score is the plain product q k^T,
    checked against a triple loop."""
    r = np.random.default_rng(seed)
    T, L, Dm = 5, 7, 6
    qv = r.integers(1, 9, (T, 1, Dm)).astype(np.float64) / 4
    kv = r.integers(1, 9, (L, Dm)).astype(np.float64) / 8
    got = _logits(orc, _as_bf16(qv), np.ones((T, 1)), _as_bf16(kv), 1, T, np.array([L]),
                  causal=False)
    for t in range(T):
        for j in range(L):
            acc = 0.0
            for d in range(Dm):
                acc += qv[t, 0, d] * kv[j, d]
            assert got[t, j] == acc


def check_logits_special(orc, seed=4):
    r = np.random.default_rng(seed)
    H, Dm, L, T = 4, 8, 6, 3
    # one-hot q and k: q[t,h] = e_(h), k[j] = c_j * e_(j mod Dm) -> only head (j mod Dm) fires
    q = np.zeros((T, H, Dm))
    for h in range(H):
        q[:, h, h] = 1.0
    k = np.zeros((L, Dm))
    for j in range(L):
        k[j, j % Dm] = j + 1.0
    w = np.arange(1, T * H + 1, dtype=np.float64).reshape(T, H)
    got = _logits(orc, _as_bf16(q), w, _as_bf16(k), 1, T, np.array([L]), causal=False)
    for t in range(T):
        for j in range(L):
            want = w[t, j % Dm] * (j + 1.0) if j % Dm < H else 0.0
            assert got[t, j] == want
    # all dot products negative -> +0.0
    qn = -np.abs(r.integers(1, 5, (T, H, Dm))).astype(np.float64)
    kp = np.abs(r.integers(1, 5, (L, Dm))).astype(np.float64)
    z = _logits(orc, _as_bf16(qn), np.abs(r.random((T, H))) + 0.1, _as_bf16(kp), 1, T,
                np.array([L]), causal=False)
    assert np.all(z == 0.0) and not np.signbit(z).any()
    # one live head: w = e_h -> relu(q_h . k)
    qr = r.integers(-4, 5, (T, H, Dm)).astype(np.float64)
    kr = r.integers(-4, 5, (L, Dm)).astype(np.float64)
    for h in range(H):
        wh = np.zeros((T, H))
        wh[:, h] = 1.0
        g = _logits(orc, _as_bf16(qr), wh, _as_bf16(kr), 1, T, np.array([L]), causal=False)
        for t in range(T):
            for j in range(L):
                dot = float(np.dot(qr[t, h], kr[j]))
                assert g[t, j] == max(dot, 0.0)


def check_logits_invariances(orc, seed=5):
    r = np.random.default_rng(seed)
    H, Dm, L, n, B = 8, 16, 20, 3, 2
    lens = np.array([L, L - 5])
    q = _as_bf16(r.integers(-8, 9, (B * n, H, Dm)) / 8.0)
    k = _as_bf16(r.integers(-8, 9, (L, Dm)) / 8.0)
    w = r.random((B * n, H))
    # keys of both sequences from one pool through two tables (block size 5)
    pool = np.concatenate([k, k])
    table = np.array([[0, 1, 2, 3], [4, 5, 6, 7]], np.int32)
    base = _logits(orc, q, w, pool, B, n, lens, table=table, bs=5)
    # weights x2 -> logits x2 exactly
    assert np.array_equal(_logits(orc, q, 2 * w, pool, B, n, lens, table=table, bs=5),
                          2 * base)
    # jointly permuting heads in q and w, or dims in q and k, changes nothing
    ph = r.permutation(H)
    got = _logits(orc, q[:, ph], w[:, ph], pool, B, n, lens, table=table, bs=5)
    assert np.allclose(got, base, rtol=1e-12, atol=0) and np.array_equal(got == -np.inf,
                                                                         base == -np.inf)
    pd = r.permutation(Dm)
    got = _logits(orc, q[:, :, pd], w, pool[:, pd], B, n, lens, table=table, bs=5)
    assert np.allclose(got, base, rtol=1e-12, atol=0)
    # causal visibility, brute force: row t = b*n + i sees j <= L_b - n + i, and j < L_b
    for t in range(B * n):
        b, i = divmod(t, n)
        for j in range(L):
            vis = j <= lens[b] - n + i and j < lens[b]
            assert (base[t, j] != -np.inf) == vis, (t, j)
    # sequence 1 scores depend on its own keys only (pool rows 20..34 through table row 1)
    pool2 = pool.copy()
    pool2[:L] = _as_bf16(np.zeros((L, Dm)))
    got = _logits(orc, q, w, pool2, B, n, lens, table=table, bs=5)
    assert np.array_equal(got[n:], base[n:])


def check_logits_e4m3(orc, seed=6):
    """E4M3 inputs with per-row scales score like their dequantised float values."""
    r = np.random.default_rng(seed)
    H, Dm, L, T = 4, 8, 9, 3
    qc = r.integers(0, 256, (T, H, Dm)).astype(np.uint8)
    qc[(qc & 0x7F) == 0x7F] = 0x30                    # no NaN codes
    kc = r.integers(0, 256, (L, Dm)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x31
    qs = (r.random((T, H)) + 0.5).astype(np.float32)
    ks = (r.random(L) + 0.5).astype(np.float32)
    w = r.random((T, H))
    got = _logits(orc, qc, w, kc, 1, T, np.array([L]), causal=False, q_scale=qs, k_scale=ks,
                  dtype="e4m3")
    # rebuild the float inputs from the torch decode of the codes and compare scores
    import torch
    qf = torch.from_numpy(qc).view(torch.float8_e4m3fn).double().numpy() * qs[..., None]
    kf = torch.from_numpy(kc).view(torch.float8_e4m3fn).double().numpy() * ks[:, None]
    for t in range(T):
        for j in range(L):
            want = sum(w[t, h] * max(float(np.dot(qf[t, h], kf[j])), 0.0) for h in range(H))
            assert abs(got[t, j] - want) <= 1e-12 * (1 + abs(want))
    # the same keys and row scales through a reversed page table (block size 3)
    perm = np.array([2, 0, 1])
    pool = np.concatenate([kc[3 * p:3 * p + 3] for p in np.argsort(perm)])
    pool_s = np.concatenate([ks[3 * p:3 * p + 3] for p in np.argsort(perm)])
    table = perm[None, :].astype(np.int32)
    got_p = _logits(orc, qc, w, pool, 1, T, np.array([L]), causal=False, q_scale=qs,
                    k_scale=pool_s, dtype="e4m3", table=table, bs=3)
    assert np.array_equal(got_p, got)


def check_logits_mxfp4_keys(orc, seed=9):
    """Keys read from a paged mxfp4 cache (the fp8-q x fp4-k form of the score, xkernels
    issue #27): a hand-worked case, then the same score as over the bf16 patterns of the
    dequantised keys."""
    H, Dm = 2, 128
    nib = np.full((3, Dm // 2), 0x21, np.uint8)   # every byte: even element code 1 (0.5), odd code 2 (1.0)
    sc = np.array([[127] * 4, [128] * 4, [0xFF] * 4], np.uint8)   # scale 1, 2, and 0xFF -> 0
    # block size 2, table [1, 0]: keys 0, 1 are pool rows 2, 3; key 2 is pool row 0
    pool_n = np.stack([nib[2], nib[2], nib[0], nib[1]])
    pool_s = np.stack([sc[2], sc[2], sc[0], sc[1]])
    table = np.array([[1, 0]], np.int32)
    qc = np.zeros((1, H, Dm), np.uint8)
    qc[0, 0, 0::2] = 0x38                          # head 0: 1.0 on the even dims; head 1: 0
    qs = np.ones((1, H), np.float32)
    w = np.array([[1.0, 5.0]])
    got = orc.indexer_logits(qc, qs, "e4m3", w, pool_n, pool_s, table, 2, 1, 1, np.array([3]), False,
                             k_dtype="mxfp4")
    assert np.array_equal(got, [[32.0, 64.0, 0.0]]), got   # 64 x 0.5, x 2, x 0
    # random cache, scales in the normal range (so every dequantised key is exact in bf16)
    r = np.random.default_rng(seed)
    B, n, bs, nblk = 2, 3, 4, 6
    lens = np.array([13, 7])
    pool_n = r.integers(0, 256, (nblk * bs, Dm // 2)).astype(np.uint8)
    pool_s = r.integers(120, 135, (nblk * bs, Dm // 32)).astype(np.uint8)
    table = np.array([[5, 0, 3, 1], [2, 4, -1, -1]], np.int32)
    qc = r.integers(0, 256, (B * n, H, Dm)).astype(np.uint8)
    qc[(qc & 0x7F) == 0x7F] = 0x30                 # no NaN codes
    qs = (r.random((B * n, H)) + 0.5).astype(np.float32)
    w = r.random((B * n, H))
    got = orc.indexer_logits(qc, qs, "e4m3", w, pool_n, pool_s, table, bs, B, n, lens, True, k_dtype="mxfp4")
    kb = f64_to_bf16_exact(orc.mxfp4_dequant(pool_n, pool_s))
    want = orc.indexer_logits(qc, qs, "e4m3", w, kb, None, table, bs, B, n, lens, True, k_dtype="bf16")
    assert np.array_equal(got, want)
    assert np.array_equal(np.isfinite(got[0]), np.arange(13) <= 13 - 3)   # causal window, row 0


# --------------------------------------------------------------------------- top-k

def check_topk_hand(orc):
    for row, k, expect in load_topk_cases():
        idx, val = orc.topk_select(row[None, :], k)
        assert np.array_equal(idx[0], expect), (row, k, idx[0], expect)


def _brute_topk(row, k):
    """Selection by pairwise dominance: i ranks before j iff v_i > v_j or
    (v_i == v_j and i < j); rank = number of candidates ranking before."""
    cand = [j for j in range(len(row)) if row[j] != -np.inf]
    rank = {}
    for a in cand:
        rank[a] = sum(1 for b in cand if row[b] > row[a] or (row[b] == row[a] and b < a))
    out = [-1] * k
    for a, rk in rank.items():
        if rk < k:
            out[rk] = a
    return out


def check_topk_bruteforce(orc, seed=8):
    r = np.random.default_rng(seed)
    # every ordering of a small multiset with ties, -0/+0 and -inf
    base = [2.0, 2.0, -0.0, 0.0, -np.inf, 1.5]
    for perm in set(itertools.permutations(range(len(base)))):
        row = np.array([base[p] for p in perm])
        for k in (1, 3, 6, 7):
            idx, _ = orc.topk_select(row[None, :], k)
            assert list(idx[0]) == _brute_topk(row, k)
    for trial in range(200):
        K = int(r.integers(1, 65))
        k = int(r.integers(1, 17))
        row = r.integers(-3, 4, K).astype(np.float64)
        row[r.random(K) < 0.2] = -np.inf
        idx, val = orc.topk_select(row[None, :], k)
        assert list(idx[0]) == _brute_topk(row, k)
        live = idx[0] >= 0
        assert np.array_equal(val[0][live], row[idx[0][live]])


# --------------------------------------------------------------------------- producers

def check_e4m3_encode(orc):
    """Nearest-even, saturating E4M3 rounding == torch's float32 -> float8_e4m3fn after a
    clamp to +-448, on random values, binade edges, subnormals, ties and signed zeros."""
    import torch
    r = np.random.default_rng(10)
    x = np.concatenate([
        (r.standard_normal(20000) * np.exp2(r.integers(-12, 10, 20000))).astype(np.float32),
        np.float32([0.0, -0.0, 448, 449, 464, 480, -1e9, 2**-9, 2**-10, 3 * 2**-11, -3 * 2**-11, 1e-30,
                    -1e-30, 1.0625, 1.1875, 17.0, 19.0, 2**-6, 15 * 2**-10]),
    ])
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(x)
    assert np.array_equal(got, ref), (x[got != ref][:5], got[got != ref][:5], ref[got != ref][:5])
    # decode(encode(v)) == v for every finite code value
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = orc.e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(orc.e4m3_to_f64(orc.e4m3_encode(vals)), vals.astype(np.float64))


def check_e2m1_encode(orc):
    """OCP E2M1 rounding: nearest grid value, ties to the even code, saturation at 6."""
    x = np.array([0.0, 0.1, 0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.1, 7.0, 100.0, -0.3, -2.5, -6.5])
    want = [0, 0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 7, 9, 12, 15]
    assert list(orc.e2m1_encode(x)) == want


def _rope_table(max_pos, rope_dim, base=10000.0):
    """cos / sin of pos * base^(-2i / rope_dim), float64 rounded to fp32, laid out per
    position as rope_dim / 2 cosines then rope_dim / 2 sines (the standard table)."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / rope_dim)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def check_q_rope_quant(orc, seed=11):
    from deepseek_v4_sparse_dsa_gb300 import synth
    r = np.random.default_rng(seed)
    T, H, Dm, R = 5, 3, 128, 64
    qf = r.standard_normal((T, H, Dm)).astype(np.float32)
    qb = (qf.view(np.uint32) >> 16).astype(np.uint16)          # bf16 patterns (truncation)
    qv = orc.bf16_to_f64(qb).astype(np.float32)
    pos = np.array([0, 3, 1, 4, 2], np.int32)
    # identity rotation (cos 1, sin 0): the per-row quantisation of the config generator
    ident = np.concatenate([np.ones((6, R // 2)), np.zeros((6, R // 2))], axis=1).astype(np.float32)
    codes, scale = orc.q_rope_quant(qb, pos, ident, R)
    want_c, want_s = synth.quantize_e4m3_rows(qv)
    assert np.array_equal(codes, want_c) and np.array_equal(scale, want_s)
    # a quarter turn (cos 0, sin 1): (x0, x1) -> (-x1, x0) on the first R dims, exactly
    quarter = np.concatenate([np.zeros((6, R // 2)), np.ones((6, R // 2))], axis=1).astype(np.float32)
    codes, scale = orc.q_rope_quant(qb, pos, quarter, R)
    rot = qv.copy()
    rot[..., 0:R:2] = -qv[..., 1:R:2]
    rot[..., 1:R:2] = qv[..., 0:R:2]
    want_c, want_s = synth.quantize_e4m3_rows(rot)
    assert np.array_equal(codes, want_c) and np.array_equal(scale, want_s)
    # hand case: head 0 of token 0 = e_0 rotated by 90 degrees -> e_1 -> code 448 = 0x7E at dim 1
    one = np.zeros((1, 1, Dm), np.uint16)
    one[0, 0, 0] = 0x3F80                            # 1.0
    codes, scale = orc.q_rope_quant(one, np.array([2], np.int32), quarter, R)
    assert scale[0, 0] == np.float32(1.0) / np.float32(448.0)
    assert codes[0, 0, 1] == 0x7E and not np.delete(codes[0, 0], 1).any()
    # a real RoPE table: the dequantised result is the exact rotation to within E4M3
    # rounding (half a step, 2^-4 relative) of each element
    tab = _rope_table(8, R)
    codes, scale = orc.q_rope_quant(qb, pos, tab, R)
    deq = orc.e4m3_to_f64(codes) * scale[..., None]
    exact = qv.astype(np.float64).copy()
    c = tab[pos][:, None, :R // 2].astype(np.float64)
    sn = tab[pos][:, None, R // 2:].astype(np.float64)
    x0, x1 = qv[..., 0:R:2].astype(np.float64), qv[..., 1:R:2].astype(np.float64)
    exact[..., 0:R:2] = x0 * c - x1 * sn
    exact[..., 1:R:2] = x0 * sn + x1 * c
    step = np.maximum(np.abs(exact), 2.0**-6 * scale[..., None]) * 2.0**-4 + 1e-6 * np.abs(exact)
    assert np.all(np.abs(deq - exact) <= step)
    # dims past rope_dim pass through: their codes are the plain quantisation of the input
    # at the row's scale (torch's float8 conversion)
    import torch
    y = np.clip(qv[..., R:] / scale[..., None], -448, 448).astype(np.float32)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[..., R:], want)


def _hadamard(Dm):
    Hm = np.array([[1.0]])
    while Hm.shape[0] < Dm:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    return Hm


def check_k_hadamard_mxfp4(orc, seed=12):
    Dm, bs, nblk = 128, 4, 3
    pool = np.full((nblk, bs, Dm // 2), 0xAA, np.uint8)
    psc = np.full((nblk, bs, Dm // 32), 0x55, np.uint8)
    # hand case: a one-hot key e_j -> column j of H / sqrt(128): every entry +-2^-3.5;
    # amax 0.0884 -> shared exponent floor(log2) - 2 = -6 (byte 121); 0.0884 * 2^6 = 5.66
    # rounds to 6.0 (code 7); signs (-1)^popcount(i & j)
    j = 5
    k = np.zeros((1, Dm), np.uint16)
    k[0, j] = 0x3F80
    fp4, sc = orc.k_hadamard_mxfp4(k, np.array([1 * bs + 2]), pool, psc)
    assert (sc[1, 2] == 121).all()
    want = np.where(np.array([bin(i & j).count("1") % 2 for i in range(Dm)]) == 1, 0xF, 0x7)
    assert np.array_equal(fp4[1, 2] & 0xF, want[0::2]) and np.array_equal(fp4[1, 2] >> 4, want[1::2])
    # other rows untouched; a negative slot writes nothing
    mask = np.ones((nblk, bs), bool)
    mask[1, 2] = False
    assert (fp4[mask] == 0xAA).all() and (sc[mask] == 0x55).all()
    fp4b, scb = orc.k_hadamard_mxfp4(k, np.array([-1]), pool, psc)
    assert np.array_equal(fp4b, pool) and np.array_equal(scb, psc)
    # random keys: decoding the written rows gives H x / sqrt(128) to within half an
    # E2M1 step at the group's scale (the step is 0.5, 1 or 2 units of 2^exponent)
    r = np.random.default_rng(seed)
    N = 6
    k = f64_to_bf16_exact(r.integers(-64, 65, (N, Dm)) / 16.0)
    slots = r.permutation(nblk * bs)[:N]
    fp4, sc = orc.k_hadamard_mxfp4(k, slots, pool, psc)
    y = orc.bf16_to_f64(k) @ _hadamard(Dm).T / np.sqrt(Dm)
    deq = orc.mxfp4_dequant(fp4.reshape(-1, Dm // 2)[slots], sc.reshape(-1, Dm // 32)[slots])
    g = y.reshape(N, Dm // 32, 32)
    amax = np.abs(g).max(axis=2, keepdims=True)
    e = np.floor(np.log2(amax)) - 2
    assert np.array_equal(sc.reshape(-1, Dm // 32)[slots], (e[..., 0] + 127).astype(np.uint8))
    v = np.abs(g) / 2.0**e
    half_step = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0)) * 2.0**e
    err = np.abs(deq.reshape(N, Dm // 32, 32) - g)
    assert np.all(err <= half_step * (1 + 1e-6) + np.where(v > 6, np.abs(g) - 6 * 2.0**e, 0))


# --------------------------------------------------------------------------- consumer

def _attn_cache(seed, nblk=4, bs=8):
    r = np.random.default_rng(seed)
    fp4 = r.integers(0, 256, (nblk, bs, 64)).astype(np.uint8)
    sc = r.integers(124, 129, (nblk, bs, 4)).astype(np.uint8)
    table = np.array([r.permutation(nblk)], np.int32)
    return fp4, sc, table, bs


def check_sparse_attn(orc, seed=13):
    """Sparse attention with a sink: closed forms on special cases (a zero query gives the
    plain mean of the selected rows when the sink is negligible; one selected row is
    scaled by the logistic of its score against the sink; two rows mix by their softmax),
    padded slots ignored, order of the selection irrelevant, an empty selection -> 0."""
    fp4, sc, table, bs = _attn_cache(seed)
    H, Dm = 3, 128
    rows = orc.mxfp4_dequant(fp4.reshape(-1, 64), sc.reshape(-1, 4))       # pool rows, pinned above
    def x_of(pos):
        return rows[int(table[0, pos // bs]) * bs + pos % bs]
    r = np.random.default_rng(seed)
    q0 = np.zeros((1, H, Dm), np.uint16)
    sel = np.array([[3, 17, -1, 9, 30]], np.int32)
    sink_off = np.full(H, -1e300)
    got = orc.sparse_attn(q0, sel, fp4, sc, table, 1, 1, bs, sink_off, 0.125)
    want = np.mean([x_of(p) for p in (3, 17, 9, 30)], axis=0)
    assert np.allclose(got[0], want[None, :], rtol=1e-12, atol=1e-12)
    # one selected row, sink 0.5: out = x * sigmoid(s - 0.5), s = scale * q . x
    qv = r.integers(-4, 5, (1, H, Dm)).astype(np.float64) / 16
    qb = f64_to_bf16_exact(qv)
    sel1 = np.array([[-1, 12, -1]], np.int32)
    got = orc.sparse_attn(qb, sel1, fp4, sc, table, 1, 1, bs, np.full(H, 0.5), 0.0625)
    x = x_of(12)
    for h in range(H):
        sc_ = 0.0625 * float(np.dot(qv[0, h], x))
        assert np.allclose(got[0, h], x / (1.0 + np.exp(0.5 - sc_)), rtol=1e-10, atol=1e-12)
    # two rows, negligible sink: softmax of the two scores
    sel2 = np.array([[5, 22]], np.int32)
    got = orc.sparse_attn(qb, sel2, fp4, sc, table, 1, 1, bs, sink_off, 0.0625)
    x5, x22 = x_of(5), x_of(22)
    for h in range(H):
        a5, a22 = 0.0625 * float(np.dot(qv[0, h], x5)), 0.0625 * float(np.dot(qv[0, h], x22))
        w5 = 1.0 / (1.0 + np.exp(a22 - a5))
        assert np.allclose(got[0, h], w5 * x5 + (1 - w5) * x22, rtol=1e-10, atol=1e-12)
    # order of the selection and padded slots do not matter; an empty selection gives 0
    sel3 = np.array([[9, 30, 3, 17]], np.int32)
    sel4 = np.array([[-1, 17, 3, -1, 30, 9, -1]], np.int32)
    a = orc.sparse_attn(qb, sel3, fp4, sc, table, 1, 1, bs, np.full(H, 0.25), 0.0625)
    b = orc.sparse_attn(qb, sel4, fp4, sc, table, 1, 1, bs, np.full(H, 0.25), 0.0625)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    e = orc.sparse_attn(qb, np.full((1, 4), -1, np.int32), fp4, sc, table, 1, 1, bs, np.zeros(H), 0.0625)
    assert not e.any()


ALL_CHECKS = [
    check_bf16_decode, check_e4m3_decode, check_bf16_rounding, check_e8m0, check_e2m1,
    check_mxfp4_hand_rows, check_mxfp4_gather_hand, check_gather_invariant,
    check_logits_hand, check_logits_plain_matmul, check_logits_special,
    check_logits_invariances, check_logits_e4m3, check_logits_mxfp4_keys, check_topk_hand,
    check_topk_bruteforce, check_e4m3_encode, check_e2m1_encode, check_q_rope_quant, check_k_hadamard_mxfp4,
    check_sparse_attn,
]
