"""mxfp4_paged_gather on the GPU against the CPU oracle: bit-exact bf16 patterns."""
import numpy as np
import pytest

import parity
import pins
from deepseek_v4_sparse_dsa_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from deepseek_v4_sparse_dsa_gb300 import dsa  # noqa: E402
from oracle import dsa_oracle as orc  # noqa: E402


def gpu_gather(fp4, sc, table, sel, B, next_n, bs):
    dev = "cuda"
    fp4_d = torch.from_numpy(np.ascontiguousarray(fp4)).to(dev)
    sc_d = torch.from_numpy(np.ascontiguousarray(sc)).to(dev)
    tab_d = torch.from_numpy(np.ascontiguousarray(table, dtype=np.int32)).to(dev)
    sel_d = torch.from_numpy(np.ascontiguousarray(sel, dtype=np.int32)).to(dev)
    T, k = sel.shape
    out = torch.full((T, k, 128), 0x5A5A, dtype=torch.int16, device=dev)   # sentinel
    dsa.mxfp4_paged_gather(fp4_d, sc_d, fp4.shape[0], bs, 128, tab_d, table.shape[1], sel_d, B, next_n, k,
                           out)
    err = dsa.dsa_device_error()
    return out.cpu().numpy().view(np.uint16), err


def test_gather_hand_rows():
    rows = pins.load_mxfp4_rows()
    bs = 4
    fp4 = np.zeros((2, bs, 64), np.uint8)
    sc = np.full((2, bs, 4), 0x7F, np.uint8)
    for i, r in enumerate(rows):
        fp4[1, i] = r["bytes"]
        sc[1, i] = r["scales"]
    table = np.array([[1, 0]], np.int32)
    sel = np.array([[0, 1, -1, 2, 5, -7]], np.int32)
    got, err = gpu_gather(fp4, sc, table, sel, 1, 1, bs)
    assert err == 0
    for s, r in zip((0, 1, 3), rows):
        assert np.array_equal(got[0, s], r["expect"]), r["name"]
    assert not got[0, 2].any() and not got[0, 5].any()
    want = orc.mxfp4_paged_gather(fp4, sc, table, sel, 1, 1, bs)
    assert np.array_equal(got, want)


def test_gather_every_scale_and_byte():
    """All 256 E8M0 bytes x all 256 nibble bytes: row r, group g uses scale (4r + g) % 256
    over nibble bytes 16 per group cycling through every value."""
    nrows = 1024
    fp4 = np.empty((nrows, 64), np.uint8)
    sc = np.empty((nrows, 4), np.uint8)
    for r in range(nrows):
        for g in range(4):
            sc[r, g] = (4 * r + g) % 256
            fp4[r, 16 * g:16 * g + 16] = (np.arange(16) + 16 * ((r // 64) % 16)) % 256
    fp4 = fp4.reshape(nrows // 16, 16, 64)
    sc = sc.reshape(nrows // 16, 16, 4)
    table = np.arange(nrows // 16, dtype=np.int32)[None, :]
    sel = np.arange(nrows, dtype=np.int32)[None, :]
    got, err = gpu_gather(fp4, sc, table, sel, 1, 1, 16)
    assert err == 0
    want = orc.mxfp4_paged_gather(fp4, sc, table, sel, 1, 1, 16)
    bad = np.nonzero(got != want)
    assert bad[0].size == 0, (bad[0][:4], bad[1][:4], bad[2][:4])


def test_gather_tiny_config():
    wl = synth.make_tiny()
    sel = synth.pad_sel_pos(synth.random_sel_pos(wl, 11), 0.05, 1)
    got, err = gpu_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table, sel, wl.B, wl.next_n, 64)
    assert err == 0
    want = orc.mxfp4_paged_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table, sel, wl.B, wl.next_n, 64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("bs,topk", [(16, 37), (64, 1), (1, 33), (128, 300)])
def test_gather_ragged(bs, topk):
    wl = parity.make_case(21 + bs, [300, 1, 517], next_n=2, block_size=bs,
                          topk=topk, gather=True)
    sel = synth.pad_sel_pos(synth.random_sel_pos(wl, 5), 0.1, 2)
    got, err = gpu_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table, sel, wl.B, wl.next_n,
                          wl.block_size)
    assert err == 0
    want = orc.mxfp4_paged_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table, sel, wl.B, wl.next_n,
                                  wl.block_size)
    assert np.array_equal(got, want)


def test_gather_bad_block_ids_give_zero_rows_and_flag():
    fp4 = np.full((2, 8, 64), 0x22, np.uint8)
    sc = np.full((2, 8, 4), 127, np.uint8)
    table = np.array([[1, 7, -3]], np.int32)          # 7 and -3 are out of range
    sel = np.array([[0, 9, 17, 30, 3]], np.int32)     # 30 // 8 = 3 >= bt_stride
    got, err = gpu_gather(fp4, sc, table, sel, 1, 1, 8)
    assert err & dsa.DSA_DEVERR_INDEX
    assert (got[0, 0] == 0x3F80).all() and (got[0, 4] == 0x3F80).all()   # nibble 2 -> 1.0
    for s in (1, 2, 3):
        assert not got[0, s].any()
    assert dsa.dsa_device_error() == 0                 # reading clears the word


def test_gather_flash_decode_full_size():
    wl = synth.make_flash_decode(with_keys=False)
    rng = synth.Rng(9)
    vis = wl.visible_len()
    sel = (rng.uniform(wl.T * 512, "pos").reshape(wl.T, 512) * vis[:, None]).astype(np.int32)
    got, err = gpu_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table, sel, wl.B, wl.next_n, 64)
    assert err == 0
    want = orc.mxfp4_paged_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table, sel, wl.B, wl.next_n, 64)
    assert np.array_equal(got, want)
