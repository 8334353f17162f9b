"""The two producers around the score on the GPU against the CPU oracle:

* dsa_indexer_q_rope_quant -- RoPE + per-row E4M3 quantisation of the indexer query:
  bit-exact codes and scales (the arithmetic is fixed fp32, product by product);
* dsa_indexer_k_hadamard_mxfp4 -- Hadamard rotation + mxfp4 write of keys into the
  paged cache: scale bytes and codes equal to the oracle's except where the oracle's
  rotated value lies within a few fp32 ulps of a rounding boundary (the GPU sums the
  transform by butterflies, the oracle exactly); untouched rows stay untouched.

Both also feed the path: the produced (q, q_scale) scores like the config generator's
E4M3 queries, and the written cache gathers to the oracle's dequantisation.
"""
import numpy as np
import pytest

import parity
import pins
from deepseek_v4_sparse_dsa_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from oracle import dsa_oracle as orc  # noqa: E402


def _gpu_q(qb, pos, table, R):
    T, H, Dm = qb.shape
    d_q = torch.from_numpy(qb.view(np.int16).copy()).cuda()
    d_pos = torch.from_numpy(pos.astype(np.int32)).cuda()
    d_tab = torch.from_numpy(np.ascontiguousarray(table, np.float32)).cuda()
    codes = torch.full((T, H, Dm), 0x5A, dtype=torch.uint8, device="cuda")
    scale = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_indexer_q_rope_quant(d_q, d_pos, d_tab, table.shape[0], R, T, H, Dm, codes, scale)
    err = dsa.dsa_device_error()
    return codes.cpu().numpy(), scale.cpu().numpy(), err


@pytest.mark.parametrize("T,R", [(1, 64), (37, 64), (300, 128), (9, 0)])
def test_q_rope_quant_matches_oracle(T, R):
    rng = synth.Rng(700 + T)
    qb = synth.normal_bf16(rng, (T, 64, 128), "q")
    qb[0, 0] = 0                                   # an all-zero row: scale 1, codes 0
    maxp = 70000
    pos = rng.integers(0, maxp - 1, T, "pos").astype(np.int32)
    pos[-1] = maxp - 1
    table = pins._rope_table(maxp, R) if R else np.zeros((maxp, 0), np.float32)
    codes, scale, err = _gpu_q(qb, pos, table, R)
    assert err == 0
    want_c, want_s = orc.q_rope_quant(qb, pos, table, R)
    assert np.array_equal(scale, want_s)
    assert np.array_equal(codes, want_c), np.argwhere(codes != want_c)[:5]
    # the all-zero row: scale 1 and zero codes (+0 or -0: the rotated zeros keep the sign
    # IEEE gives x * c - y * s, e.g. -0 when c < 0 < s)
    assert scale[0, 0] == 1.0 and not (codes[0, 0] & 0x7F).any()


def test_q_rope_quant_feeds_the_score():
    # the produced E4M3 queries score like the oracle's on the same codes (a small
    # decode batch over paged E4M3 keys)
    wl = parity.make_case(711, [3000, 700], next_n=2, block_size=64, dtype="e4m3", topk=64)
    rng = synth.Rng(712)
    qb = synth.normal_bf16(rng, (wl.T, 64, 128), "q")
    pos = (np.repeat(wl.context_lens, 2) - 2 + np.tile([0, 1], 2)).astype(np.int32)
    table = pins._rope_table(4096, 64)
    codes, scale, err = _gpu_q(qb, pos, table, 64)
    assert err == 0
    wl.q, wl.q_scale = codes, scale
    from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch
    db = DeviceBatch.from_workload(wl)
    lg = db.logits().cpu().numpy()
    parity.assert_logits_close(lg, parity.oracle_logits(wl))


def test_q_rope_quant_bad_position_flags():
    qb = np.full((2, 64, 128), 0x3F80, np.uint16)
    codes, scale, err = _gpu_q(qb, np.array([5, 99], np.int32), pins._rope_table(10, 64), 64)
    assert err & dsa.DSA_DEVERR_INDEX
    assert not codes[1].any() and (scale[1] == 0).all()
    assert codes[0].any()


def _gpu_k(kb, slots, fp4, sc):
    d_k = torch.from_numpy(kb.view(np.int16).copy()).cuda()
    d_s = torch.from_numpy(slots.astype(np.int64)).cuda()
    d_fp4 = torch.from_numpy(fp4.copy()).cuda()
    d_sc = torch.from_numpy(sc.copy()).cuda()
    rows = fp4.shape[0] * fp4.shape[1]
    dsa.dsa_indexer_k_hadamard_mxfp4(d_k, d_s, kb.shape[0], 128, d_fp4, d_sc, rows)
    err = dsa.dsa_device_error()
    return d_fp4.cpu().numpy(), d_sc.cpu().numpy(), err


def _near_boundary(y, scale_byte):
    """Elements whose exactly rounded rotation lies within 4 fp32 ulps of an E2M1
    rounding boundary at their group's scale (where butterfly rounding may tip a code)."""
    bounds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    v = np.abs(y) / np.exp2(np.repeat(scale_byte.astype(np.float64) - 127, 32, axis=-1))
    d = np.min(np.abs(v[..., None] - bounds), axis=-1)
    return d <= 4 * np.spacing(np.float32(np.maximum(v, 1e-30))).astype(np.float64)


@pytest.mark.parametrize("N", [1, 100, 5000])
def test_k_hadamard_mxfp4_matches_oracle(N):
    rng = synth.Rng(800 + N)
    nblk, bs = (N + 63) // 64 + 2, 64
    kb = synth.normal_bf16(rng, (N, 128), "k")
    if N > 1:
        kb[1] = 0                                  # an all-zero key: bytes 0, codes 0
    slots = rng.permutation(nblk * bs, "slots")[:N].astype(np.int64)
    if N > 2:
        slots[2] = -1                              # skipped
    fp4 = np.full((nblk, bs, 64), 0xA5, np.uint8)
    sc = np.full((nblk, bs, 4), 0x3C, np.uint8)
    g_fp4, g_sc, err = _gpu_k(kb, slots, fp4, sc)
    assert err == 0
    w_fp4, w_sc = orc.k_hadamard_mxfp4(kb, slots, fp4, sc)
    assert np.array_equal(g_sc, w_sc)
    diff = np.argwhere(g_fp4 != w_fp4)
    if diff.size:
        # every differing byte must hold an element at a rounding boundary
        Hm = pins._hadamard(128)
        for blk, off, byte in diff:
            row = blk * bs + off
            n = int(np.nonzero(slots == row)[0][0])
            y = (orc.bf16_to_f64(kb[n]) @ Hm.T / np.sqrt(128)).astype(np.float32).astype(np.float64)
            near = _near_boundary(y.reshape(4, 32), w_sc.reshape(-1, 4)[row])
            assert near.reshape(-1)[2 * byte] or near.reshape(-1)[2 * byte + 1], (n, byte)
    assert diff.shape[0] <= max(2, N // 100)


def test_k_hadamard_write_then_gather():
    # keys written by the GPU writer and read back by the GPU gather equal the oracle's
    # dequantisation of the same cache bytes
    rng = synth.Rng(901)
    nblk, bs, N = 8, 16, 100
    kb = synth.normal_bf16(rng, (N, 128), "k")
    slots = np.arange(N, dtype=np.int64)
    fp4, sc, err = _gpu_k(kb, slots, np.zeros((nblk, bs, 64), np.uint8), np.zeros((nblk, bs, 4), np.uint8))
    assert err == 0
    table = np.arange(nblk, dtype=np.int32)[None, :]
    sel = np.arange(N, dtype=np.int32)[None, :]
    out = torch.empty((1, N, 128), dtype=torch.int16, device="cuda")
    dsa.mxfp4_paged_gather(torch.from_numpy(fp4).cuda(), torch.from_numpy(sc).cuda(), nblk, bs, 128,
                           torch.from_numpy(table).cuda(), nblk, torch.from_numpy(sel).cuda(), 1, 1, N, out)
    assert dsa.dsa_device_error() == 0
    want = orc.mxfp4_paged_gather(fp4, sc, table, sel, 1, 1, bs)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), want)
    # and the decoded keys are the rotation to within half an E2M1 step of each group
    y = orc.bf16_to_f64(kb) @ pins._hadamard(128).T / np.sqrt(128)
    deq = orc.bf16_to_f64(want[0])
    e = np.repeat(sc.reshape(-1, 4)[:N].astype(np.float64) - 127, 32, axis=1)
    assert np.all(np.abs(deq - y) <= 2.0 ** e * 2.0 + 1e-6)      # half a step, or the clip at 6


def test_k_hadamard_bad_slot_flags():
    kb = np.full((2, 128), 0x3F80, np.uint16)
    fp4 = np.zeros((1, 4, 64), np.uint8)
    sc = np.zeros((1, 4, 4), np.uint8)
    g_fp4, g_sc, err = _gpu_k(kb, np.array([1, 4], np.int64), fp4, sc)
    assert err & dsa.DSA_DEVERR_INDEX
    assert g_fp4[0, 1].any() and not g_fp4[0, [0, 2, 3]].any()
