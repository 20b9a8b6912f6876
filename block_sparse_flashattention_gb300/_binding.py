"""ctypes binding of the C ABI declared in include/bsattn.h (argument marshalling only).

Every function here forwards to libbsattn.so; all arithmetic runs in the CUDA
kernels.  Loading fails loudly when the library has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

from ._build import LIB

BSATTN_OK, BSATTN_ERR_INVALID_ARG, BSATTN_ERR_UNSUPPORTED, BSATTN_ERR_CUDA = 0, 1, 2, 3
BSATTN_ERR_CAPACITY = 4
BSATTN_STATIC_SCRATCH_UNITS = 65536
MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT, MASK_PREFIX = 0, 1, 2, 3, 4
OUT_BF16, OUT_F32 = 0, 1
FLAG_BAD_COUNT, FLAG_BAD_INDEX, FLAG_TIMEOUT, FLAG_BAD_SEQLENS = 0x1, 0x2, 0x4, 0x8

_I32P = ctypes.POINTER(ctypes.c_int32)


class bsattn_mask_params(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int32), ("sink_tokens", ctypes.c_int32),
                ("prefix_len", ctypes.c_int32), ("doc_id_q", ctypes.c_void_p),
                ("doc_id_k", ctypes.c_void_p)]


class bsattn_meta(ctypes.Structure):
    _fields_ = [("full_cnt", ctypes.c_void_p), ("full_idx", ctypes.c_void_p),
                ("mask_cnt", ctypes.c_void_p), ("mask_idx", ctypes.c_void_p),
                ("cu_total_m_blocks", ctypes.c_void_p), ("cu_block_idx_offsets", ctypes.c_void_p),
                ("varlen", ctypes.c_int32), ("B", ctypes.c_int32), ("H", ctypes.c_int32),
                ("num_m", ctypes.c_int32), ("num_n", ctypes.c_int32),
                ("total_m_blocks", ctypes.c_int32), ("total_n_blocks", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32)]


class BsattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libbsattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: build it with __graft_entry__.build() or "
                               "block_sparse_flashattention_gb300._build.build()")
        lib = ctypes.CDLL(LIB)
        lib.bsattn_build_meta.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(bsattn_mask_params),
            ctypes.POINTER(bsattn_meta), ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_build_meta.restype = ctypes.c_int
        lib.bsattn_kv_summaries.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_kv_summaries.restype = ctypes.c_int
        lib.bsattn_build_meta_blocks.argtypes = [
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(bsattn_mask_params),
            ctypes.POINTER(bsattn_meta), ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_build_meta_blocks.restype = ctypes.c_int
        lib.bsattn_build_meta_bitmask.argtypes = [ctypes.c_void_p, ctypes.c_int32] + \
            lib.bsattn_build_meta.argtypes[1:]
        lib.bsattn_build_meta_bitmask.restype = ctypes.c_int
        lib.bsattn_build_meta_bsr.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + \
            lib.bsattn_build_meta.argtypes[1:]
        lib.bsattn_build_meta_bsr.restype = ctypes.c_int
        lib.bsattn_fwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.POINTER(bsattn_meta), ctypes.c_void_p, ctypes.c_int,
            ctypes.POINTER(bsattn_mask_params), ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_fwd.restype = ctypes.c_int
        lib.bsattn_fwd_proxy.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(bsattn_meta),
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
            ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_fwd_proxy.restype = ctypes.c_int
        lib.bsattn_fwd_static_scratch.argtypes = lib.bsattn_fwd.argtypes[:18] + [
            ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_fwd_static_scratch.restype = ctypes.c_int
        lib.bsattn_fwd_workspace_size.argtypes = [ctypes.POINTER(bsattn_meta),
                                                  ctypes.POINTER(ctypes.c_size_t)]
        lib.bsattn_fwd_workspace_size.restype = ctypes.c_int
        lib.bsattn_bwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.POINTER(bsattn_meta), ctypes.c_void_p,
            ctypes.c_int, ctypes.POINTER(bsattn_mask_params), ctypes.c_float, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
            ctypes.c_void_p, ctypes.c_void_p]
        lib.bsattn_bwd.restype = ctypes.c_int
        lib.bsattn_bwd_workspace_size.argtypes = [ctypes.POINTER(bsattn_meta),
                                                  ctypes.POINTER(ctypes.c_size_t)]
        lib.bsattn_bwd_workspace_size.restype = ctypes.c_int
        lib.bsattn_status_string.argtypes = [ctypes.c_int]
        lib.bsattn_status_string.restype = ctypes.c_char_p
        lib.bsattn_abi_version.argtypes = []
        lib.bsattn_abi_version.restype = ctypes.c_int32
        lib.bsattn_testing_set_wait_limit.argtypes = [ctypes.c_longlong]
        lib.bsattn_testing_set_wait_limit.restype = ctypes.c_int
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().bsattn_status_string(int(status)).decode()


def _ptr(x) -> Optional[int]:
    """Device (or host) address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class MaskParams:
    window_left: int = 0
    sink_tokens: int = 0
    prefix_len: int = 0
    doc_id_q: object = None   # device int32 tensor (or address), one id per packed q row
    doc_id_k: object = None

    def to_c(self) -> bsattn_mask_params:
        return bsattn_mask_params(self.window_left, self.sink_tokens, self.prefix_len,
                                  _ptr(self.doc_id_q), _ptr(self.doc_id_k))


@dataclass
class Meta:
    """Block-sparse metadata tensors (device int32) with their sizes."""
    full_cnt: object
    full_idx: object
    mask_cnt: object
    mask_idx: object
    varlen: int
    B: int
    H: int
    num_m: int
    num_n: int
    total_m_blocks: int = 0
    total_n_blocks: int = 0
    cu_total_m_blocks: object = None
    cu_block_idx_offsets: object = None
    tile_m: int = 128
    tile_n: int = 128

    def to_c(self) -> bsattn_meta:
        return bsattn_meta(_ptr(self.full_cnt), _ptr(self.full_idx), _ptr(self.mask_cnt),
                           _ptr(self.mask_idx), _ptr(self.cu_total_m_blocks),
                           _ptr(self.cu_block_idx_offsets), int(self.varlen), int(self.B),
                           int(self.H), int(self.num_m), int(self.num_n), int(self.total_m_blocks),
                           int(self.total_n_blocks), int(self.tile_m), int(self.tile_n))


def bsattn_build_meta(block_map, cu_seqlens_q, cu_seqlens_k, seqlen_q: int, seqlen_k: int,
                      kv_valid_len, kind: int, mask_params: Optional[MaskParams], meta: Meta,
                      err_flag=None, stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    return library().bsattn_build_meta(
        _ptr(block_map), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(seqlen_q), int(seqlen_k),
        _ptr(kv_valid_len), int(kind), ctypes.byref(mp) if mp is not None else None,
        ctypes.byref(mt), _ptr(err_flag), _stream(stream))


def bsattn_kv_summaries(k, v, B: int, seqlen_k: int, H: int, D: int, k_sum, v_sum,
                        stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    return library().bsattn_kv_summaries(_ptr(k), _ptr(v), int(B), int(seqlen_k), int(H), int(D),
                                         _ptr(k_sum), _ptr(v_sum), _stream(stream))


def bsattn_build_meta_blocks(block_map, q_block_tiles: int, kv_block_tiles: int, seqlen_q: int,
                             seqlen_k: int, kv_valid_len_blocks, kv_valid_len_tiles, kind: int,
                             mask_params: Optional[MaskParams], meta: Meta, err_flag=None,
                             stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    return library().bsattn_build_meta_blocks(
        _ptr(block_map), int(q_block_tiles), int(kv_block_tiles), int(seqlen_q), int(seqlen_k),
        _ptr(kv_valid_len_blocks), _ptr(kv_valid_len_tiles), int(kind),
        ctypes.byref(mp) if mp is not None else None, ctypes.byref(mt), _ptr(err_flag),
        _stream(stream))


def bsattn_build_meta_bitmask(words, words_per_row: int, cu_seqlens_q, cu_seqlens_k,
                              seqlen_q: int, seqlen_k: int, kv_valid_len, kind: int,
                              mask_params: Optional[MaskParams], meta: Meta, err_flag=None,
                              stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    return library().bsattn_build_meta_bitmask(
        _ptr(words), int(words_per_row), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(seqlen_q),
        int(seqlen_k), _ptr(kv_valid_len), int(kind), ctypes.byref(mp) if mp is not None else None,
        ctypes.byref(mt), _ptr(err_flag), _stream(stream))


def bsattn_build_meta_bsr(block_indptr, block_indices, cu_seqlens_q, cu_seqlens_k, seqlen_q: int,
                          seqlen_k: int, kv_valid_len, kind: int,
                          mask_params: Optional[MaskParams], meta: Meta, err_flag=None,
                          stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    return library().bsattn_build_meta_bsr(
        _ptr(block_indptr), _ptr(block_indices), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        int(seqlen_q), int(seqlen_k), _ptr(kv_valid_len), int(kind),
        ctypes.byref(mp) if mp is not None else None, ctypes.byref(mt), _ptr(err_flag),
        _stream(stream))


def bsattn_fwd(q, k, v, B: int, seqlen_q: int, seqlen_k: int, H: int, D: int, cu_seqlens_q,
               cu_seqlens_k, meta: Meta, kv_valid_len, kind: int,
               mask_params: Optional[MaskParams], softmax_scale: float, out, out_dtype: int, lse,
               workspace=None, workspace_bytes: int = 0, err_flag=None, stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    if workspace is not None and not isinstance(workspace, int) and workspace_bytes == 0:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return library().bsattn_fwd(
        _ptr(q), _ptr(k), _ptr(v), int(B), int(seqlen_q), int(seqlen_k), int(H), int(D),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), ctypes.byref(mt), _ptr(kv_valid_len), int(kind),
        ctypes.byref(mp) if mp is not None else None, float(softmax_scale), _ptr(out),
        int(out_dtype), _ptr(lse), _ptr(workspace), int(workspace_bytes), _ptr(err_flag),
        _stream(stream))


def bsattn_fwd_proxy(q, k, v, B: int, seqlen_q: int, seqlen_k: int, H: int, D: int, meta: Meta,
                     sel_words, words_per_row: int, k_sum, v_sum, softmax_scale: float, out,
                     out_dtype: int, lse, workspace=None, workspace_bytes: int = 0, err_flag=None,
                     stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mt = meta.to_c()
    if workspace is not None and not isinstance(workspace, int) and workspace_bytes == 0:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return library().bsattn_fwd_proxy(
        _ptr(q), _ptr(k), _ptr(v), int(B), int(seqlen_q), int(seqlen_k), int(H), int(D),
        ctypes.byref(mt), _ptr(sel_words), int(words_per_row), _ptr(k_sum), _ptr(v_sum),
        float(softmax_scale), _ptr(out), int(out_dtype), _ptr(lse), _ptr(workspace),
        int(workspace_bytes), _ptr(err_flag), _stream(stream))


def bsattn_fwd_static_scratch(q, k, v, B: int, seqlen_q: int, seqlen_k: int, H: int, D: int,
                              cu_seqlens_q, cu_seqlens_k, meta: Meta, kv_valid_len, kind: int,
                              mask_params: Optional[MaskParams], softmax_scale: float, out,
                              out_dtype: int, lse, err_flag=None, stream=None) -> int:
    """Forwards to the C function of the same name (bsattn_fwd with the library's
    fixed scheduling scratch; allocates nothing); returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    return library().bsattn_fwd_static_scratch(
        _ptr(q), _ptr(k), _ptr(v), int(B), int(seqlen_q), int(seqlen_k), int(H), int(D),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), ctypes.byref(mt), _ptr(kv_valid_len), int(kind),
        ctypes.byref(mp) if mp is not None else None, float(softmax_scale), _ptr(out),
        int(out_dtype), _ptr(lse), _ptr(err_flag), _stream(stream))


def bsattn_fwd_workspace_size(meta: Meta) -> int:
    """Bytes of scheduling workspace bsattn_fwd can use for `meta` (0: none)."""
    mt = meta.to_c()
    n = ctypes.c_size_t(0)
    st = library().bsattn_fwd_workspace_size(ctypes.byref(mt), ctypes.byref(n))
    if st != BSATTN_OK:
        raise BsattnError(st, "bsattn_fwd_workspace_size")
    return int(n.value)


def bsattn_bwd(q, k, v, out, out_dtype: int, lse, dout, B: int, seqlen_q: int, seqlen_k: int,
               H: int, D: int, cu_seqlens_q, cu_seqlens_k, meta: Meta, kv_valid_len, kind: int,
               mask_params: Optional[MaskParams], softmax_scale: float, dq, dk, dv,
               grad_dtype: int, workspace, workspace_bytes: int = 0, err_flag=None,
               stream=None) -> int:
    """Forwards to the C function of the same name; returns its status code."""
    mp = mask_params.to_c() if mask_params is not None else None
    mt = meta.to_c()
    if workspace is not None and not isinstance(workspace, int) and workspace_bytes == 0:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return library().bsattn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), int(out_dtype), _ptr(lse), _ptr(dout), int(B),
        int(seqlen_q), int(seqlen_k), int(H), int(D), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        ctypes.byref(mt), _ptr(kv_valid_len),
        int(kind), ctypes.byref(mp) if mp is not None else None, float(softmax_scale), _ptr(dq),
        _ptr(dk), _ptr(dv), int(grad_dtype), _ptr(workspace), int(workspace_bytes),
        _ptr(err_flag), _stream(stream))


def bsattn_bwd_workspace_size(meta: Meta) -> int:
    """Bytes of workspace bsattn_bwd needs for `meta`."""
    mt = meta.to_c()
    n = ctypes.c_size_t(0)
    st = library().bsattn_bwd_workspace_size(ctypes.byref(mt), ctypes.byref(n))
    if st != BSATTN_OK:
        raise BsattnError(st, "bsattn_bwd_workspace_size")
    return int(n.value)


def bsattn_abi_version() -> int:
    return int(library().bsattn_abi_version())


def bsattn_testing_set_wait_limit(cycles: int) -> None:
    """Testing hook: pipeline wait limit (SM cycles) of later forward launches;
    cycles <= 0 restores the default."""
    st = library().bsattn_testing_set_wait_limit(int(cycles))
    if st != BSATTN_OK:
        raise BsattnError(st, "bsattn_testing_set_wait_limit")
