"""Python binding of the C ABI in include/dsa.h (ctypes; argument marshalling only).

The functions carry the C names and arguments.  Pointer arguments accept a torch
tensor (its data_ptr), a plain integer address, or None.  `stream` accepts a
torch.cuda.Stream, a raw cudaStream_t integer, or None for torch's current stream.
A non-OK status raises DsaError.  All computation happens in the CUDA library; this
module never computes anything itself, and importing it fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_int32, c_int64, c_size_t, c_uint64, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_gb300.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_WORKSPACE = 0, 1, 2, 3, 4
DSA_BF16, DSA_E4M3, DSA_E4M3_MXFP4K = 0, 1, 2
DSA_OP_TOPK, DSA_OP_LOGITS_TOPK = 1, 2
DSA_DEVERR_INDEX, DSA_DEVERR_TIMEOUT = 1, 2


class DsaError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {status_string(status)} (status {status})")


class dsa_keys(ctypes.Structure):
    _fields_ = [
        ("data", c_void_p),
        ("scale", c_void_p),
        ("block_table", c_void_p),
        ("bt_stride", c_int64),
        ("block_size", c_int32),
        ("num_rows", c_int64),
        ("scale_e8m0", c_void_p),
    ]


class dsa_queries(ctypes.Structure):
    _fields_ = [
        ("B", c_int32),
        ("next_n", c_int32),
        ("context_lens", c_void_p),
        ("max_context_len", c_int32),
        ("causal", c_int32),
    ]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads (once) and returns the CUDA library; raises if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -m deepseek_v4_sparse_dsa_gb300.build). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    sigs = {
        "dsa_indexer_logits": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, dsa_keys,
                                       dsa_queries, c_void_p, c_int64, c_void_p]),
        "dsa_indexer_topk": (c_int, [c_void_p, c_int64, dsa_queries, c_int, c_void_p, c_void_p, c_void_p,
                                     c_size_t, c_void_p]),
        "dsa_indexer_logits_topk": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, dsa_keys,
                                            dsa_queries, c_int, c_void_p, c_void_p, c_void_p, c_size_t,
                                            c_void_p]),
        "dsa_indexer_logits_topk_noalloc": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, dsa_keys,
                                                    dsa_queries, c_int, c_void_p, c_void_p, c_void_p]),
        "mxfp4_paged_gather": (c_int, [c_void_p, c_void_p, c_int64, c_int, c_int, c_void_p, c_int64,
                                       c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
        "dsa_indexer_q_rope_quant": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int, c_int, c_int,
                                             c_void_p, c_void_p, c_void_p]),
        "dsa_indexer_k_hadamard_mxfp4": (c_int, [c_void_p, c_void_p, c_int64, c_int, c_void_p, c_void_p, c_int64,
                                                 c_void_p]),
        "dsa_sparse_attn_mxfp4": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p, c_int, c_void_p, c_void_p,
                                          c_int64, c_int, c_void_p, c_int64, c_int, c_void_p, c_float, c_void_p,
                                          c_void_p]),
        "dsa_workspace_bytes": (c_size_t, [c_int, c_int, dsa_queries, c_int]),
        "dsa_status_string": (ctypes.c_char_p, [c_int]),
        "dsa_device_error": (c_int, [c_void_p]),
        "dsa_launch_count": (c_uint64, []),
        "dsa_set_wait_limit_ns": (c_int, [c_uint64]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, call: str) -> None:
    if status != DSA_OK:
        raise DsaError(status, call)


def status_string(status: int) -> str:
    return load().dsa_status_string(status).decode()


def make_keys(data, scale=None, block_table=None, block_size: int = 64, num_rows=None, scale_e8m0=None) -> dsa_keys:
    """dsa_keys from tensors: data [rows, 128] (mxfp4 keys: [rows, 64] nibble bytes with
    scale_e8m0 [rows, 4]); block_table [B, stride] (or None)."""
    rows = int(num_rows if num_rows is not None else data.shape[0])
    stride = int(block_table.shape[1]) if block_table is not None else 0
    return dsa_keys(_ptr(data), _ptr(scale), _ptr(block_table), stride, int(block_size), rows, _ptr(scale_e8m0))


def make_queries(B: int, next_n: int, context_lens, max_context_len: int, causal: bool) -> dsa_queries:
    return dsa_queries(int(B), int(next_n), _ptr(context_lens), int(max_context_len), 1 if causal else 0)


def dsa_indexer_logits(q, q_scale, dtype, weights, H, D, keys, qs, logits, ld_logits, stream=None):
    _check(load().dsa_indexer_logits(_ptr(q), _ptr(q_scale), int(dtype), _ptr(weights), int(H), int(D), keys, qs,
                                     _ptr(logits), int(ld_logits), _stream(stream)), "dsa_indexer_logits")


def dsa_indexer_topk(logits, ld_logits, qs, topk, out_idx, out_val, ws, ws_bytes, stream=None):
    _check(load().dsa_indexer_topk(_ptr(logits), int(ld_logits), qs, int(topk), _ptr(out_idx), _ptr(out_val),
                                   _ptr(ws), int(ws_bytes), _stream(stream)), "dsa_indexer_topk")


def dsa_indexer_logits_topk(q, q_scale, dtype, weights, H, D, keys, qs, topk, out_idx, out_val, ws, ws_bytes,
                            stream=None):
    _check(load().dsa_indexer_logits_topk(_ptr(q), _ptr(q_scale), int(dtype), _ptr(weights), int(H), int(D), keys,
                                          qs, int(topk), _ptr(out_idx), _ptr(out_val), _ptr(ws), int(ws_bytes),
                                          _stream(stream)), "dsa_indexer_logits_topk")


def dsa_indexer_logits_topk_noalloc(q, q_scale, dtype, weights, H, D, keys, qs, topk, out_idx, out_val,
                                    stream=None):
    """The fused call without a caller workspace, for callers that cannot allocate
    device memory (scratch is a fixed 16 MiB array inside the library)."""
    _check(load().dsa_indexer_logits_topk_noalloc(_ptr(q), _ptr(q_scale), int(dtype), _ptr(weights), int(H),
                                                  int(D), keys, qs, int(topk), _ptr(out_idx), _ptr(out_val),
                                                  _stream(stream)), "dsa_indexer_logits_topk_noalloc")


def mxfp4_paged_gather(kv_fp4, kv_scale, num_blocks, block_size, D, block_table, bt_stride, sel_pos, B, next_n,
                       topk, out, stream=None):
    _check(load().mxfp4_paged_gather(_ptr(kv_fp4), _ptr(kv_scale), int(num_blocks), int(block_size), int(D),
                                     _ptr(block_table), int(bt_stride), _ptr(sel_pos), int(B), int(next_n),
                                     int(topk), _ptr(out), _stream(stream)), "mxfp4_paged_gather")


def dsa_indexer_q_rope_quant(q, positions, cos_sin, max_pos, rope_dim, T, H, D, q_fp8, q_scale, stream=None):
    _check(load().dsa_indexer_q_rope_quant(_ptr(q), _ptr(positions), _ptr(cos_sin), int(max_pos), int(rope_dim),
                                           int(T), int(H), int(D), _ptr(q_fp8), _ptr(q_scale), _stream(stream)),
           "dsa_indexer_q_rope_quant")


def dsa_sparse_attn_mxfp4(q, T, H, D, sel_pos, topk, kv_fp4, kv_scale, num_blocks, block_size, block_table,
                          bt_stride, next_n, sink, softmax_scale, out, stream=None):
    _check(load().dsa_sparse_attn_mxfp4(_ptr(q), int(T), int(H), int(D), _ptr(sel_pos), int(topk), _ptr(kv_fp4),
                                        _ptr(kv_scale), int(num_blocks), int(block_size), _ptr(block_table),
                                        int(bt_stride), int(next_n), _ptr(sink), float(softmax_scale), _ptr(out),
                                        _stream(stream)),
           "dsa_sparse_attn_mxfp4")


def dsa_indexer_k_hadamard_mxfp4(k, slot_mapping, N, D, kv_fp4, kv_scale, num_rows, stream=None):
    _check(load().dsa_indexer_k_hadamard_mxfp4(_ptr(k), _ptr(slot_mapping), int(N), int(D), _ptr(kv_fp4),
                                               _ptr(kv_scale), int(num_rows), _stream(stream)),
           "dsa_indexer_k_hadamard_mxfp4")


def dsa_workspace_bytes(op, dtype, qs, topk) -> int:
    return int(load().dsa_workspace_bytes(int(op), int(dtype), qs, int(topk)))


def dsa_device_error(stream=None) -> int:
    return int(load().dsa_device_error(_stream(stream)))


def dsa_launch_count() -> int:
    return int(load().dsa_launch_count())


def dsa_set_wait_limit_ns(ns: int) -> None:
    _check(load().dsa_set_wait_limit_ns(int(ns)), "dsa_set_wait_limit_ns")
