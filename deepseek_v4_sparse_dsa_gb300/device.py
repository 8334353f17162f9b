"""Device-resident batches and the four calls of the C ABI over them.

PyTorch only owns the device memory and the stream here; every step of the indexer
path runs in the CUDA library through the binding in ``dsa``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import dsa

H = 64
D = 128


def _dev(a: Optional[np.ndarray], device) -> Optional[torch.Tensor]:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


@dataclasses.dataclass
class DeviceBatch:
    """A synthetic Workload uploaded to one GPU (see synth.Workload for layouts)."""

    B: int
    next_n: int
    causal: bool
    topk: int
    dtype: int
    max_context_len: int
    context_lens: torch.Tensor
    q: torch.Tensor
    q_scale: Optional[torch.Tensor]
    weights: torch.Tensor
    k_data: torch.Tensor
    k_scale: Optional[torch.Tensor]
    block_table: Optional[torch.Tensor]
    block_size: int
    kv_fp4: Optional[torch.Tensor]
    kv_scale: Optional[torch.Tensor]
    gather_block_table: Optional[torch.Tensor]

    @property
    def T(self) -> int:
        return self.B * self.next_n

    @classmethod
    def from_workload(cls, wl, device="cuda") -> "DeviceBatch":
        dt = dsa.DSA_E4M3 if wl.dtype == "e4m3" else dsa.DSA_BF16
        if getattr(wl, "k_format", "native") == "mxfp4":
            dt = dsa.DSA_E4M3_MXFP4K
        return cls(wl.B, wl.next_n, wl.causal, wl.topk, dt, wl.max_context_len,
                   _dev(wl.context_lens.astype(np.int32), device),
                   _dev(wl.q, device), _dev(wl.q_scale, device), _dev(wl.weights, device),
                   _dev(wl.k_data, device), _dev(wl.k_scale, device), _dev(wl.block_table, device),
                   wl.block_size, _dev(wl.kv_fp4, device), _dev(wl.kv_scale, device),
                   _dev(wl.gather_block_table, device))

    def keys(self) -> dsa.dsa_keys:
        if self.dtype == dsa.DSA_E4M3_MXFP4K:     # mxfp4 cache rows: nibbles + E8M0 bytes
            return dsa.make_keys(self.k_data, None, self.block_table, self.block_size, scale_e8m0=self.k_scale)
        return dsa.make_keys(self.k_data, self.k_scale, self.block_table, self.block_size)

    def queries(self) -> dsa.dsa_queries:
        return dsa.make_queries(self.B, self.next_n, self.context_lens, self.max_context_len, self.causal)

    # ------------------------------------------------------------------ calls
    def logits(self, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((self.T, max(self.max_context_len, 1)), dtype=torch.float32,
                              device=self.q.device)
        dsa.dsa_indexer_logits(self.q, self.q_scale, self.dtype, self.weights, H, D, self.keys(),
                               self.queries(), out, out.shape[1], stream)
        return out

    def workspace(self, op: int, topk: Optional[int] = None) -> torch.Tensor:
        n = dsa.dsa_workspace_bytes(op, self.dtype, self.queries(), topk or self.topk)
        return torch.empty(max(n, 8), dtype=torch.uint8, device=self.q.device)

    def topk_of(self, logits: torch.Tensor, topk: Optional[int] = None, ws=None, stream=None,
                with_values: bool = True):
        k = topk or self.topk
        idx = torch.empty((self.T, k), dtype=torch.int32, device=self.q.device)
        val = torch.empty((self.T, k), dtype=torch.float32, device=self.q.device) if with_values else None
        if ws is None:
            ws = self.workspace(dsa.DSA_OP_TOPK, k)
        dsa.dsa_indexer_topk(logits, logits.shape[1], self.queries(), k, idx, val, ws, ws.numel(), stream)
        return idx, val

    def logits_topk(self, topk: Optional[int] = None, ws=None, out_idx=None, out_val=None, stream=None,
                    with_values: bool = True):
        k = topk or self.topk
        idx = out_idx if out_idx is not None else torch.empty((self.T, k), dtype=torch.int32,
                                                              device=self.q.device)
        val = out_val
        if val is None and with_values:
            val = torch.empty((self.T, k), dtype=torch.float32, device=self.q.device)
        if ws is None:
            ws = self.workspace(dsa.DSA_OP_LOGITS_TOPK, k)
        dsa.dsa_indexer_logits_topk(self.q, self.q_scale, self.dtype, self.weights, H, D, self.keys(),
                                    self.queries(), k, idx, val, ws, ws.numel(), stream)
        return idx, val

    def gather(self, sel_pos: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        k = sel_pos.shape[1]
        if out is None:
            out = torch.empty((self.T, k, D), dtype=torch.int16, device=self.q.device)
        nblk = self.kv_fp4.shape[0]
        dsa.mxfp4_paged_gather(self.kv_fp4, self.kv_scale, nblk, self.kv_fp4.shape[1], D,
                               self.gather_block_table, self.gather_block_table.shape[1], sel_pos,
                               self.B, self.next_n, k, out, stream)
        return out
