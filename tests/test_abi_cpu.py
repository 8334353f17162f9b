"""The C-ABI library on a machine without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before any CUDA call."""
import os
import re

import pytest

from deepseek_v4_sparse_dsa_gb300 import dsa
from deepseek_v4_sparse_dsa_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    srcs = [os.path.join(dsa_build.CSRC, s) for s in os.listdir(dsa_build.CSRC)]
    newest = max(os.path.getmtime(p) for p in srcs + [HEADER])
    if not os.path.exists(dsa.LIB_PATH) or os.path.getmtime(dsa.LIB_PATH) < newest:
        dsa_build.build()
    return dsa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["dsa_indexer_logits", "dsa_indexer_topk", "dsa_indexer_logits_topk", "mxfp4_paged_gather",
              "dsa_workspace_bytes", "dsa_status_string", "dsa_device_error", "dsa_sparse_attn_mxfp4"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(5):
        assert dsa.status_string(s) not in ("", "unknown status")
    assert dsa.status_string(99) == "unknown status"


def _qs(B=1, n=1, L=4096, causal=True):
    return dsa.make_queries(B, n, 0x1000, L, causal)


def test_workspace_plans_are_host_only(lib):
    ws = lambda qs, k: dsa.dsa_workspace_bytes(dsa.DSA_OP_LOGITS_TOPK, dsa.DSA_BF16, qs, k)
    # the fused call's workspace: the plan (8 B per query group) plus two partial top-k
    # lists per CTA (one CTA per slice of the work, at least one per SM)
    flash = dsa.make_queries(64, 1, 0x1000, 65536, True)
    n = ws(flash, 512)
    assert n >= 148 * 2 * 512 * 8
    assert ws(dsa.make_queries(128, 1, 0x1000, 65536, True), 512) - n == 64 * 8
    # the partial lists grow with k for one epilogue group; two groups take buffers of up
    # to k + 2048 keys where shared memory allows, so theirs need not (the prefill shape's
    # at k = 512 are wider than at k = 1024)
    prefill = dsa.make_queries(1, 16384, 0x1000, 16384, True)
    assert ws(flash, 2048) > ws(flash, 1024) > ws(flash, 512) > ws(flash, 256) > 0
    for k in (256, 512, 1024, 2048):
        assert ws(prefill, k) > 4096 * 4
    assert ws(prefill, 512) > 4096 * 4
    # the standalone top-k needs no workspace at any shape
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_TOPK, dsa.DSA_BF16, prefill, 512) == 0
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_TOPK, dsa.DSA_BF16, flash, 512) == 0
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_TOPK, dsa.DSA_BF16, flash, 0) == 0
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_TOPK, dsa.DSA_BF16, flash, 4096) == 0


FAKE = 0x100000  # 1 MiB-aligned address: passes alignment checks, never dereferenced


def _status(fn, *args):
    try:
        fn(*args)
    except dsa.DsaError as e:
        return e.status
    return dsa.DSA_OK


def test_host_side_rejections_launch_nothing(lib):
    before = dsa.dsa_launch_count()
    keys = dsa.dsa_keys(FAKE, None, None, 0, 0, 4096)
    qs = _qs()
    s = 0  # stream handle, never used on a rejected call
    # unsupported head count / head dim
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_BF16, FAKE, 32, 128, keys, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_BF16, FAKE, 64, 64, keys, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    # null q, misaligned q, ld too small
    assert _status(dsa.dsa_indexer_logits, None, None, dsa.DSA_BF16, FAKE, 64, 128, keys, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_logits, FAKE + 2, None, dsa.DSA_BF16, FAKE, 64, 128, keys, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_BF16, FAKE, 64, 128, keys, qs, FAKE, 100, s) \
        == dsa.DSA_ERR_INVALID_ARG
    # E4M3 without scales
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_E4M3, FAKE, 64, 128, keys, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    # FP4 keys: E8M0 rows required and 16-byte aligned; q scales required; a contiguous key
    # array needs whole 16-byte rows of scale bytes
    f4 = dsa.dsa_keys(FAKE, None, None, 0, 0, 4096, None)
    assert _status(dsa.dsa_indexer_logits, FAKE, FAKE, dsa.DSA_E4M3_MXFP4K, FAKE, 64, 128, f4, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    f4 = dsa.dsa_keys(FAKE, None, None, 0, 0, 4096, FAKE + 4)
    assert _status(dsa.dsa_indexer_logits, FAKE, FAKE, dsa.DSA_E4M3_MXFP4K, FAKE, 64, 128, f4, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    f4 = dsa.dsa_keys(FAKE, None, None, 0, 0, 4098, FAKE)
    assert _status(dsa.dsa_indexer_logits, FAKE, FAKE, dsa.DSA_E4M3_MXFP4K, FAKE, 64, 128, f4, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    f4 = dsa.dsa_keys(FAKE, None, None, 0, 0, 4096, FAKE)
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_E4M3_MXFP4K, FAKE, 64, 128, f4, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_logits, FAKE, FAKE, 3, FAKE, 64, 128, f4, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_INVALID_ARG
    # contiguous keys with more than one sequence
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_BF16, FAKE, 64, 128, keys, _qs(B=2), FAKE,
                   4096, s) == dsa.DSA_ERR_INVALID_ARG
    # paged keys with an unsupported block size
    bad = dsa.dsa_keys(FAKE, None, FAKE, 64, 12, 4096 * 12)
    assert _status(dsa.dsa_indexer_logits, FAKE, None, dsa.DSA_BF16, FAKE, 64, 128, bad, qs, FAKE, 4096, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    # top-k bounds
    for k in (0, 2049):
        assert _status(dsa.dsa_indexer_topk, FAKE, 4096, qs, k, FAKE, None, None, 0, s) == dsa.DSA_ERR_INVALID_ARG
        assert _status(dsa.dsa_indexer_logits_topk, FAKE, None, dsa.DSA_BF16, FAKE, 64, 128, keys, qs, k, FAKE,
                       None, None, 0, s) == dsa.DSA_ERR_INVALID_ARG
    # split fused top-k without a workspace
    flash = dsa.make_queries(64, 1, FAKE, 65536, True)
    pkeys = dsa.dsa_keys(FAKE, None, FAKE, 1024, 64, 1 << 20)
    assert _status(dsa.dsa_indexer_logits_topk, FAKE, None, dsa.DSA_BF16, FAKE, 64, 128, pkeys, flash, 512, FAKE,
                   None, FAKE, 16, s) == dsa.DSA_ERR_WORKSPACE
    # gather: head dim, misaligned output, bad sizes
    assert _status(dsa.mxfp4_paged_gather, FAKE, FAKE, 8, 64, 64, FAKE, 8, FAKE, 1, 1, 4, FAKE, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    assert _status(dsa.mxfp4_paged_gather, FAKE, FAKE, 8, 64, 128, FAKE, 8, FAKE, 1, 1, 4, FAKE + 8, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.mxfp4_paged_gather, FAKE, FAKE, 8, 0, 128, FAKE, 8, FAKE, 1, 1, 4, FAKE, s) \
        == dsa.DSA_ERR_INVALID_ARG
    # a batch whose work-plan line (key tiles + per-item costs of every query group) would
    # not fit the plan's 32-bit positions is refused, not wrapped around
    huge = dsa.make_queries(1000, 1, FAKE, 2**31 - 1, True)
    assert dsa.dsa_workspace_bytes(dsa.DSA_OP_LOGITS_TOPK, dsa.DSA_BF16, huge, 512) == 0
    assert _status(dsa.dsa_indexer_logits_topk, FAKE, None, dsa.DSA_BF16, FAKE, 64, 128, pkeys, huge, 512, FAKE,
                   None, FAKE, 1 << 40, s) == dsa.DSA_ERR_UNSUPPORTED
    # producers: head dim, RoPE width, misalignment, empty batches
    assert _status(dsa.dsa_indexer_q_rope_quant, FAKE, FAKE, FAKE, 100, 64, 4, 64, 64, FAKE, FAKE, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    for rope in (-4, 66, 132):
        assert _status(dsa.dsa_indexer_q_rope_quant, FAKE, FAKE, FAKE, 100, rope, 4, 64, 128, FAKE, FAKE, s) \
            == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_q_rope_quant, FAKE + 4, FAKE, FAKE, 100, 64, 4, 64, 128, FAKE, FAKE, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_q_rope_quant, FAKE, FAKE, None, 100, 64, 4, 64, 128, FAKE, FAKE, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_q_rope_quant, None, None, None, 0, 0, 0, 64, 128, None, None, s) == dsa.DSA_OK
    assert _status(dsa.dsa_indexer_k_hadamard_mxfp4, FAKE, FAKE, 10, 64, FAKE, FAKE, 100, s) \
        == dsa.DSA_ERR_UNSUPPORTED
    assert _status(dsa.dsa_indexer_k_hadamard_mxfp4, FAKE, FAKE, 10, 128, FAKE, FAKE + 2, 100, s) \
        == dsa.DSA_ERR_INVALID_ARG
    assert _status(dsa.dsa_indexer_k_hadamard_mxfp4, None, None, 0, 128, None, None, 0, s) == dsa.DSA_OK
    # sparse attention: heads / dim, misaligned q or cache, null selection, bad scale, empty batch
    def attn(q=FAKE, T=4, H=64, D=128, sel=FAKE, topk=512, fp4=FAKE, sc=FAKE, bs=64, tab=FAKE, stride=8, nn=1,
             sink=FAKE, scale=0.088, out=FAKE):
        return _status(dsa.dsa_sparse_attn_mxfp4, q, T, H, D, sel, topk, fp4, sc, 100, bs, tab, stride, nn, sink,
                       scale, out, s)
    assert attn(H=128) == dsa.DSA_ERR_UNSUPPORTED and attn(D=64) == dsa.DSA_ERR_UNSUPPORTED
    assert attn(topk=16385) == dsa.DSA_ERR_UNSUPPORTED and attn(bs=1 << 25) == dsa.DSA_ERR_UNSUPPORTED
    assert attn(q=FAKE + 8) == dsa.DSA_ERR_INVALID_ARG and attn(fp4=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG
    assert attn(sel=None) == dsa.DSA_ERR_INVALID_ARG and attn(sink=None) == dsa.DSA_ERR_INVALID_ARG
    assert attn(scale=float("nan")) == dsa.DSA_ERR_INVALID_ARG and attn(scale=float("inf")) == dsa.DSA_ERR_INVALID_ARG
    assert attn(bs=0) == dsa.DSA_ERR_INVALID_ARG and attn(T=-1) == dsa.DSA_ERR_INVALID_ARG
    assert attn(nn=0) == dsa.DSA_ERR_INVALID_ARG and attn(topk=-1) == dsa.DSA_ERR_INVALID_ARG
    assert attn(q=None, T=0, sel=None, fp4=None, sc=None, tab=None, sink=None, out=None) == dsa.DSA_OK
    # empty problems are valid no-ops
    assert _status(dsa.mxfp4_paged_gather, None, None, 0, 64, 128, None, 0, None, 0, 1, 512, None, s) == dsa.DSA_OK
    assert dsa.dsa_launch_count() == before
