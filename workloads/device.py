"""Moves a seeded workload to the GPU and runs the library on it (harness code).

Used by the GPU tests, __graft_entry__.smoke() and bench.py.  It only uploads
inputs, calls the public API of block_sparse_flashattention_gb300 and copies
results back; it holds none of the method's arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch

import block_sparse_flashattention_gb300 as bsa


def bf16_to_device(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def i32(a, device):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


class DeviceWorkload:
    """Device copies of a workload's inputs plus the sizes the API needs."""

    def __init__(self, wl, device="cuda", qkv=None):
        """qkv: host (q, k, v) bf16 bits, None to generate them, False to skip them
        (enough for the metadata kernel, which never reads q/k/v)."""
        self.wl = wl
        self.device = device
        if qkv is False:
            self.q = self.k = self.v = None
        else:
            q, k, v = qkv if qkv is not None else wl.qkv()
            self.q = bf16_to_device(q, device)
            self.k = bf16_to_device(k, device)
            self.v = bf16_to_device(v, device)
        self.block_map = torch.from_numpy(np.ascontiguousarray(wl.block_map, np.uint8)).to(device)
        self.cu_q = i32(wl.cu_seqlens_q, device) if wl.varlen else None
        self.cu_k = i32(wl.cu_seqlens_k, device) if wl.varlen else None
        self.vl = i32(wl.kv_valid_len, device)
        self.doc_q = i32(wl.doc_id_q, device)
        self.doc_k = i32(wl.doc_id_k, device)
        self.mask_params = bsa.MaskParams(window_left=wl.window_left, sink_tokens=wl.sink_tokens,
                                          prefix_len=wl.prefix_len, doc_id_q=self.doc_q,
                                          doc_id_k=self.doc_k)

    def seqlens(self):
        wl = self.wl
        if wl.varlen:
            return wl.rows_q, wl.rows_k
        return int(wl.seqlens_q[0]), int(wl.seqlens_k[0])

    def alloc_meta(self):
        wl = self.wl
        sq, sk = self.seqlens()
        if wl.varlen:
            return bsa.alloc_meta(wl.B, wl.H, varlen=True, total_m_blocks=wl.total_m_blocks,
                                  total_n_blocks=wl.total_n_blocks, max_num_n=wl.num_n,
                                  device=self.device)
        return bsa.alloc_meta(wl.B, wl.H, seqlen_q=sq, seqlen_k=sk, tile_m=wl.tile_m,
                              tile_n=wl.tile_n, device=self.device)

    def build_meta(self, meta=None, err_flag=None, stream=None):
        meta = meta or self.alloc_meta()
        sq, sk = self.seqlens()
        return bsa.build_meta(self.block_map, meta, cu_seqlens_q=self.cu_q, cu_seqlens_k=self.cu_k,
                              seqlen_q=sq, seqlen_k=sk, kv_valid_len=self.vl, kind=self.wl.kind,
                              mask_params=self.mask_params, err_flag=err_flag, stream=stream)

    def forward(self, meta, out=None, lse=None, err_flag=None, stream=None, out_dtype=None,
                workspace="auto"):
        return bsa.forward(self.q, self.k, self.v, meta, cu_seqlens_q=self.cu_q,
                           cu_seqlens_k=self.cu_k, kv_valid_len=self.vl, kind=self.wl.kind,
                           mask_params=self.mask_params, softmax_scale=self.wl.scale, out=out,
                           out_dtype=out_dtype, lse=lse, workspace=workspace, err_flag=err_flag,
                           stream=stream)


def meta_to_numpy(meta) -> dict:
    out = {k: getattr(meta, k).cpu().numpy() for k in ("full_cnt", "full_idx", "mask_cnt",
                                                        "mask_idx")}
    if meta.varlen:
        out["cu_total_m_blocks"] = meta.cu_total_m_blocks.cpu().numpy()
        out["cu_block_idx_offsets"] = meta.cu_block_idx_offsets.cpu().numpy()
        out["total_m_blocks"] = meta.total_m_blocks
        out["total_n_blocks"] = meta.total_n_blocks
    return out


def meta_from_numpy(wl, arrays: dict, device="cuda"):
    """A device Meta holding the given (oracle-made or hand-edited) lists."""
    m = bsa.Meta(full_cnt=i32(arrays["full_cnt"], device), full_idx=i32(arrays["full_idx"], device),
                 mask_cnt=i32(arrays["mask_cnt"], device), mask_idx=i32(arrays["mask_idx"], device),
                 varlen=int(wl.varlen), B=wl.B, H=wl.H, num_m=0 if wl.varlen else wl.num_m,
                 num_n=wl.num_n)
    if wl.varlen:
        m.total_m_blocks = int(arrays["total_m_blocks"])
        m.total_n_blocks = int(arrays["total_n_blocks"])
        m.cu_total_m_blocks = i32(arrays["cu_total_m_blocks"], device)
        m.cu_block_idx_offsets = i32(arrays["cu_block_idx_offsets"], device)
    return m


def out_to_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def computed_blocks(meta_np: dict) -> int:
    """Number of (head, Q tile, KV tile) blocks the forward computes."""
    return int(meta_np["full_cnt"].sum() + meta_np["mask_cnt"].sum())
