"""Block-sparse attention forward for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library libbsattn.so (include/bsattn.h): a metadata
kernel that turns a boolean block map into full / mask block lists, and a
persistent TMA + tcgen05 attention kernel that walks those lists.  This package
is the Python face of that C ABI: ``bsattn_build_meta``, ``bsattn_fwd``,
``bsattn_bwd`` and the rest carry the C names and only marshal arguments;
``alloc_meta``, ``build_meta``, ``forward`` and ``backward`` add torch
allocation of the outputs around them.  PyTorch provides
device memory and streams only.
"""
from __future__ import annotations

import math
from typing import Optional

from ._binding import (BSATTN_ERR_CAPACITY, BSATTN_ERR_CUDA, BSATTN_ERR_INVALID_ARG,
                       BSATTN_ERR_UNSUPPORTED, BSATTN_OK, BSATTN_STATIC_SCRATCH_UNITS, FLAG_BAD_COUNT, FLAG_BAD_INDEX, FLAG_BAD_SEQLENS, FLAG_TIMEOUT,
                       MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX, MASK_SLIDING_WINDOW,
                       OUT_BF16, OUT_F32,
                       BsattnError, MaskParams, Meta, bsattn_abi_version, bsattn_build_meta,
                       bsattn_build_meta_bitmask, bsattn_build_meta_blocks, bsattn_build_meta_bsr,
                       bsattn_fwd_proxy, bsattn_kv_summaries, bsattn_bwd, bsattn_bwd_workspace_size,
                       bsattn_fwd, bsattn_fwd_static_scratch, bsattn_fwd_workspace_size,
                       bsattn_testing_set_wait_limit, library, status_string)

TILE = 128

__all__ = ["bsattn_bwd", "bsattn_bwd_workspace_size", "backward", "bsattn_fwd_proxy", "bsattn_kv_summaries", "bsattn_build_meta", "bsattn_build_meta_bitmask", "bsattn_build_meta_blocks", "bsattn_build_meta_bsr", "bsattn_fwd", "bsattn_fwd_static_scratch", "bsattn_fwd_workspace_size", "bsattn_abi_version", "bsattn_testing_set_wait_limit",
           "alloc_meta", "alloc_workspace", "build_meta",
           "forward", "block_sparse_attention", "Meta", "MaskParams", "BsattnError", "status_string", "library", "TILE",
           "OUT_BF16", "OUT_F32", "MASK_NONE", "MASK_CAUSAL", "MASK_SLIDING_WINDOW", "MASK_DOCUMENT", "MASK_PREFIX",
           "BSATTN_OK", "BSATTN_ERR_INVALID_ARG", "BSATTN_ERR_UNSUPPORTED", "BSATTN_ERR_CUDA", "BSATTN_ERR_CAPACITY", "BSATTN_STATIC_SCRATCH_UNITS",
           "FLAG_BAD_COUNT", "FLAG_BAD_INDEX", "FLAG_TIMEOUT", "FLAG_BAD_SEQLENS"]


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def alloc_meta(B: int, H: int, *, varlen: bool = False, seqlen_q: int = 0, seqlen_k: int = 0,
               total_m_blocks: int = 0, total_n_blocks: int = 0, max_num_n: int = 0,
               tile_m: int = TILE, tile_n: int = TILE, device="cuda") -> Meta:
    """Allocates the metadata tensors.

    Batched: pass seqlen_q / seqlen_k (per sequence); tile_m / tile_n give the
    listed block size (128 x 128 tiles, or sparse blocks of 256 x 128 or
    256 x 256 tokens, whose lists the forward walks directly).  Varlen: pass
    total_m_blocks, total_n_blocks (sum of num_m(b) and of num_m(b) * num_n(b))
    and max_num_n (row stride of kv_valid_len, at least the largest num_n(b))."""
    import torch
    i32 = dict(dtype=torch.int32, device=device)
    if varlen:
        return Meta(full_cnt=torch.empty((H, total_m_blocks), **i32),
                    full_idx=torch.empty((H, total_n_blocks), **i32),
                    mask_cnt=torch.empty((H, total_m_blocks), **i32),
                    mask_idx=torch.empty((H, total_n_blocks), **i32), varlen=1, B=B, H=H,
                    num_m=0, num_n=max_num_n, total_m_blocks=total_m_blocks,
                    total_n_blocks=total_n_blocks,
                    cu_total_m_blocks=torch.empty(B + 1, **i32),
                    cu_block_idx_offsets=torch.empty(B + 1, **i32))
    nm, nn = _cdiv(seqlen_q, tile_m), _cdiv(seqlen_k, tile_n)
    return Meta(full_cnt=torch.empty((B, H, nm), **i32),
                full_idx=torch.empty((B, H, nm, nn), **i32),
                mask_cnt=torch.empty((B, H, nm), **i32),
                mask_idx=torch.empty((B, H, nm, nn), **i32), varlen=0, B=B, H=H, num_m=nm,
                num_n=nn, tile_m=tile_m, tile_n=tile_n)


def alloc_workspace(meta: Meta, device="cuda"):
    """Scheduling workspace for bsattn_fwd (None when the problem needs none)."""
    import torch
    n = bsattn_fwd_workspace_size(meta)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


def _check(status: int, where: str) -> None:
    if status != BSATTN_OK:
        raise BsattnError(status, where)


def build_meta(block_map, meta: Meta, *, cu_seqlens_q=None, cu_seqlens_k=None, seqlen_q: int = 0,
               seqlen_k: int = 0, kv_valid_len=None, kind: int = MASK_NONE,
               mask_params: Optional[MaskParams] = None, err_flag=None, stream=None) -> Meta:
    """Runs the metadata kernel into `meta` (see alloc_meta); raises on a bad status."""
    _check(bsattn_build_meta(block_map, cu_seqlens_q, cu_seqlens_k, seqlen_q, seqlen_k,
                             kv_valid_len, kind, mask_params, meta, err_flag, stream),
           "bsattn_build_meta")
    return meta


def forward(q, k, v, meta: Meta, *, cu_seqlens_q=None, cu_seqlens_k=None, kv_valid_len=None,
            kind: int = MASK_NONE, mask_params: Optional[MaskParams] = None,
            softmax_scale: Optional[float] = None, out=None, out_dtype=None, lse=None,
            workspace="auto", err_flag=None, stream=None):
    """Block-sparse attention forward.  q/k/v: bf16 [B, S, H, D] or packed [total, H, D].

    Returns (out, lse): out shaped like q (bf16 by default, or torch.float32),
    lse fp32 [B, H, S_q] (batched) or [H, total_q].  workspace: "auto" allocates
    the scheduling workspace for this call, None uses the fixed-stride schedule,
    a tensor is used as given (see alloc_workspace)."""
    import torch
    varlen = bool(meta.varlen)
    if varlen:
        rows_q, H, D = q.shape
        seqlen_q, seqlen_k = rows_q, k.shape[0]
        lse_shape = (H, rows_q)
    else:
        _, seqlen_q, H, D = q.shape
        seqlen_k = k.shape[1]
        lse_shape = (meta.B, H, seqlen_q)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    elif out.dtype != out_dtype:
        raise ValueError("out.dtype and out_dtype disagree")
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    if isinstance(workspace, str):
        workspace = alloc_workspace(meta, q.device)
    _check(bsattn_fwd(q, k, v, meta.B, seqlen_q, seqlen_k, H, D, cu_seqlens_q, cu_seqlens_k, meta,
                      kv_valid_len, kind, mask_params, softmax_scale, out,
                      OUT_F32 if out_dtype == torch.float32 else OUT_BF16, lse, workspace=workspace,
                      err_flag=err_flag, stream=stream),
           "bsattn_fwd")
    return out, lse


def backward(q, k, v, out, lse, dout, meta: Meta, *, cu_seqlens_q=None, cu_seqlens_k=None,
             kv_valid_len=None, kind: int = MASK_NONE, mask_params: Optional[MaskParams] = None,
             softmax_scale: Optional[float] = None, grad_dtype=None, workspace=None,
             err_flag=None, stream=None):
    """Gradients (dq, dk, dv) of ``forward`` for upstream gradient dout.

    q/k/v/dout: bf16 [B, S, H, D] or packed [total, H, D] (varlen, with
    cu_seqlens_q / cu_seqlens_k); out, lse: the forward's results for the same
    arguments.  Gradients are bf16 by default, or torch.float32.  workspace: a
    uint8 tensor of at least bsattn_bwd_workspace_size(meta) bytes, or None to
    allocate one for this call."""
    import torch
    if meta.varlen:
        rows_q, H, D = q.shape
        seqlen_q, seqlen_k = rows_q, k.shape[0]
    else:
        _, seqlen_q, H, D = q.shape
        seqlen_k = k.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if grad_dtype is None:
        grad_dtype = torch.bfloat16
    if grad_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("grad_dtype must be torch.bfloat16 or torch.float32")
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=q.device)
    if workspace is None:
        workspace = torch.empty(bsattn_bwd_workspace_size(meta), dtype=torch.uint8, device=q.device)
    gd = OUT_F32 if grad_dtype == torch.float32 else OUT_BF16
    od = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(bsattn_bwd(q, k, v, out, od, lse, dout, meta.B, seqlen_q, seqlen_k, H, D, cu_seqlens_q,
                      cu_seqlens_k, meta, kv_valid_len, kind, mask_params, softmax_scale, dq, dk, dv,
                      gd, workspace, err_flag=err_flag, stream=stream),
           "bsattn_bwd")
    return dq, dk, dv


_attention_fn = None


def _attention_function():
    """The autograd Function behind ``block_sparse_attention`` (built on first use,
    so that importing the package does not import torch)."""
    global _attention_fn
    if _attention_fn is None:
        import torch

        class BlockSparseAttention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, meta, opts):
                out, lse = forward(q, k, v, meta, **opts)
                ctx.save_for_backward(q, k, v, out, lse)
                ctx.meta, ctx.opts = meta, opts
                return out

            @staticmethod
            def backward(ctx, dout):
                q, k, v, out, lse = ctx.saved_tensors
                dq, dk, dv = backward(q, k, v, out, lse, dout.to(q.dtype).contiguous(), ctx.meta,
                                      grad_dtype=q.dtype, **ctx.opts)
                return dq, dk, dv, None, None

        _attention_fn = BlockSparseAttention
    return _attention_fn


def block_sparse_attention(q, k, v, meta: Meta, *, cu_seqlens_q=None, cu_seqlens_k=None,
                           kv_valid_len=None, kind: int = MASK_NONE,
                           mask_params: Optional[MaskParams] = None,
                           softmax_scale: Optional[float] = None, err_flag=None, stream=None):
    """Differentiable block-sparse attention: ``forward`` with the bf16 output,
    and on the way back ``backward`` for the incoming gradient of the output
    (dq, dk, dv in bf16, like q/k/v).  Arguments as for ``forward``; the
    metadata, sequence offsets, valid lengths and mask parameters are taken as
    constants (no gradient)."""
    opts = dict(cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, kv_valid_len=kv_valid_len,
                kind=kind, mask_params=mask_params, softmax_scale=softmax_scale,
                err_flag=err_flag, stream=stream)
    return _attention_function().apply(q, k, v, meta, opts)
