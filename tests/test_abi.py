"""The C-ABI library loads, exports what include/bsattn.h declares, and rejects
bad arguments on the host (no GPU needed: every case here fails validation
before any CUDA call)."""
import ctypes
import os
import re

import pytest

import block_sparse_flashattention_gb300 as bsa
from block_sparse_flashattention_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bsattn.h")
FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced here


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(bsattn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"bsattn_build_meta", "bsattn_fwd", "bsattn_status_string",
            "bsattn_abi_version"} <= set(names)


def test_library_exports_every_declared_function():
    lib = ctypes.CDLL(_build.LIB)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared but not exported"


def test_abi_version_and_status_strings():
    text = open(HEADER).read()
    ver = int(re.search(r"#define BSATTN_ABI_VERSION (\d+)", text).group(1))
    assert bsa.bsattn_abi_version() == ver
    assert bsa.status_string(bsa.BSATTN_OK) == "BSATTN_OK"
    assert bsa.status_string(bsa.BSATTN_ERR_INVALID_ARG) == "BSATTN_ERR_INVALID_ARG"
    assert bsa.status_string(bsa.BSATTN_ERR_UNSUPPORTED) == "BSATTN_ERR_UNSUPPORTED"
    assert bsa.status_string(bsa.BSATTN_ERR_CUDA) == "BSATTN_ERR_CUDA"
    assert bsa.status_string(bsa.BSATTN_ERR_CAPACITY) == "BSATTN_ERR_CAPACITY"
    assert bsa.status_string(99) == "BSATTN_ERR_UNKNOWN"


def _meta(**kw):
    base = dict(full_cnt=FAKE, full_idx=FAKE, mask_cnt=FAKE, mask_idx=FAKE, varlen=0, B=1, H=2,
                num_m=2, num_n=2)
    base.update(kw)
    return bsa.Meta(**base)


def _fwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, seqlen_q=256, seqlen_k=256, H=2, D=128,
             cu_seqlens_q=None, cu_seqlens_k=None, meta=_meta(), kv_valid_len=None,
             kind=bsa.MASK_CAUSAL, mask_params=None, softmax_scale=0.125, out=FAKE,
             out_dtype=bsa.OUT_BF16, lse=FAKE, workspace=None, workspace_bytes=0,
             err_flag=None, stream=0)
    a.update(kw)
    return bsa.bsattn_fwd(**a)


def _bm(**kw):
    a = dict(block_map=FAKE, cu_seqlens_q=None, cu_seqlens_k=None, seqlen_q=256, seqlen_k=256,
             kv_valid_len=None, kind=bsa.MASK_CAUSAL, mask_params=None, meta=_meta(),
             err_flag=None, stream=0)
    a.update(kw)
    return bsa.bsattn_build_meta(**a)


INV, UNS = bsa.BSATTN_ERR_INVALID_ARG, bsa.BSATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,expect", [
    (dict(D=96), UNS),
    (dict(D=256), UNS),
    (dict(q=FAKE + 2), INV),                       # not 16-byte aligned
    (dict(out=None), INV),
    (dict(out_dtype=7), INV),
    (dict(workspace=FAKE + 8, workspace_bytes=1 << 20), INV),   # misaligned workspace
    (dict(workspace=FAKE, workspace_bytes=16), INV),             # too small
    (dict(lse=None), INV),
    (dict(softmax_scale=0.0), INV),
    (dict(softmax_scale=-1.0), INV),
    (dict(softmax_scale=float("inf")), INV),
    (dict(seqlen_q=300), INV),                     # num_m would be 3, meta says 2
    (dict(B=2), INV),                              # meta.B disagrees
    (dict(H=3), INV),
    (dict(cu_seqlens_q=FAKE, cu_seqlens_k=FAKE), INV),   # batched meta with cu_seqlens
    (dict(meta=_meta(tile_m=64)), UNS),
    (dict(meta=_meta(full_idx=None)), INV),
    (dict(meta=_meta(varlen=1)), INV),             # varlen meta without offset tensors
    (dict(kind=7), INV),
    (dict(kind=bsa.MASK_SLIDING_WINDOW), INV),     # needs mask params
    (dict(kind=bsa.MASK_DOCUMENT, mask_params=bsa.MaskParams()), INV),
    (dict(kind=bsa.MASK_PREFIX, mask_params=bsa.MaskParams(prefix_len=-1)), INV),
])
def test_fwd_rejects_bad_arguments(kw, expect):
    assert _fwd(**kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(block_map=None), INV),
    (dict(seqlen_k=600), INV),
    (dict(seqlen_q=-1), INV),
    (dict(cu_seqlens_q=FAKE), INV),
    (dict(meta=_meta(tile_n=256)), UNS),
    (dict(meta=_meta(varlen=1, cu_total_m_blocks=FAKE, cu_block_idx_offsets=FAKE)), INV),
    (dict(kind=bsa.MASK_SLIDING_WINDOW, mask_params=bsa.MaskParams(window_left=-5)), INV),
])
def test_build_meta_rejects_bad_arguments(kw, expect):
    assert _bm(**kw) == expect


def test_workspace_size():
    # 2 heads x ceil(2 tiles / 2) = 2 units -> 256-byte header + 2 int32
    assert bsa.bsattn_fwd_workspace_size(_meta()) == 256 + 4 * 2
    assert bsa.bsattn_fwd_workspace_size(_meta(B=3, num_m=5)) == 256 + 4 * 2 * 8
    huge = _meta(H=1000, num_m=1000)
    assert bsa.bsattn_fwd_workspace_size(huge) == 0          # beyond the scheduling pass
    with pytest.raises(bsa.BsattnError):
        bsa.bsattn_fwd_workspace_size(_meta(tile_m=64))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from block_sparse_flashattention_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _binding.library()


def test_static_scratch_capacity_and_validation():
    """The fixed-scratch forward rejects problems beyond its capacity (and bad
    metadata) before any CUDA call."""
    text = open(HEADER).read()
    cap = int(re.search(r"#define BSATTN_STATIC_SCRATCH_UNITS (\d+)", text).group(1))
    assert cap == bsa.BSATTN_STATIC_SCRATCH_UNITS

    def call(meta):
        return bsa.bsattn_fwd_static_scratch(
            q=FAKE, k=FAKE, v=FAKE, B=1, seqlen_q=meta.num_m * 128, seqlen_k=256, H=meta.H, D=128,
            cu_seqlens_q=None, cu_seqlens_k=None, meta=meta, kv_valid_len=None,
            kind=bsa.MASK_CAUSAL, mask_params=None, softmax_scale=0.125, out=FAKE,
            out_dtype=bsa.OUT_BF16, lse=FAKE, err_flag=None, stream=0)

    # H * ceil(num_m / 2) units: 2 * 65538 / 2 = cap + 2 > cap
    assert call(_meta(H=2, num_m=cap + 2)) == bsa.BSATTN_ERR_CAPACITY
    assert call(_meta(full_idx=None)) == INV
    assert call(_meta(tile_m=64)) == UNS


def _bmf(fmt, **kw):
    a = dict(cu_seqlens_q=None, cu_seqlens_k=None, seqlen_q=256, seqlen_k=256, kv_valid_len=None,
             kind=bsa.MASK_CAUSAL, mask_params=None, meta=_meta(), err_flag=None, stream=0)
    if fmt == "bitmask":
        a.update(words=FAKE, words_per_row=1)
        a.update(kw)
        return bsa.bsattn_build_meta_bitmask(**a)
    a.update(block_indptr=FAKE, block_indices=FAKE)
    a.update(kw)
    return bsa.bsattn_build_meta_bsr(**a)


@pytest.mark.parametrize("fmt,kw,expect", [
    ("bitmask", dict(words=None), INV),
    ("bitmask", dict(words_per_row=0), INV),
    ("bitmask", dict(meta=_meta(num_n=40), seqlen_k=5000), INV),   # 1 word cannot hold 40 tiles
    ("bitmask", dict(seqlen_k=600), INV),                          # same checks as the byte map
    ("bitmask", dict(meta=_meta(tile_n=256)), UNS),
    ("bsr", dict(block_indptr=None), INV),
    ("bsr", dict(block_indices=None), INV),
    ("bsr", dict(seqlen_k=0), INV),
    ("bsr", dict(seqlen_k=600), INV),
    ("bsr", dict(kind=bsa.MASK_SLIDING_WINDOW), INV),
])
def test_format_entry_points_reject_bad_arguments(fmt, kw, expect):
    assert _bmf(fmt, **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(block_map=None), INV),
    (dict(q_block_tiles=0), INV),
    (dict(kv_block_tiles=2000), INV),
    (dict(kv_valid_len_blocks=FAKE, kv_valid_len_tiles=None), INV),   # lengths need an output
    (dict(meta=_meta(varlen=1, cu_total_m_blocks=FAKE, cu_block_idx_offsets=FAKE)), UNS),
    (dict(seqlen_k=600), INV),
    (dict(meta=_meta(tile_m=64)), UNS),
])
def test_block_map_entry_point_rejects_bad_arguments(kw, expect):
    a = dict(block_map=FAKE, q_block_tiles=2, kv_block_tiles=2, seqlen_q=256, seqlen_k=256,
             kv_valid_len_blocks=None, kv_valid_len_tiles=None, kind=bsa.MASK_CAUSAL,
             mask_params=None, meta=_meta(), err_flag=None, stream=0)
    a.update(kw)
    assert bsa.bsattn_build_meta_blocks(**a) == expect


def _prox(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, seqlen_q=256, seqlen_k=256, H=2, D=128, meta=_meta(),
             sel_words=FAKE, words_per_row=1, k_sum=FAKE, v_sum=FAKE, softmax_scale=0.125,
             out=FAKE, out_dtype=bsa.OUT_F32, lse=FAKE, workspace=None, workspace_bytes=0,
             err_flag=None, stream=0)
    a.update(kw)
    return bsa.bsattn_fwd_proxy(**a)


@pytest.mark.parametrize("kw,expect", [
    (dict(sel_words=None), INV),
    (dict(k_sum=None), INV),
    (dict(v_sum=FAKE + 4), INV),                                  # not 16-byte aligned
    (dict(words_per_row=0), INV),
    (dict(meta=_meta(num_n=40), seqlen_k=5000), INV),             # 1 word < 40 tiles
    (dict(meta=_meta(varlen=1, cu_total_m_blocks=FAKE, cu_block_idx_offsets=FAKE)), UNS),
    (dict(D=96), UNS),
    (dict(softmax_scale=0.0), INV),
])
def test_proxy_forward_rejects_bad_arguments(kw, expect):
    assert _prox(**kw) == expect


@pytest.mark.parametrize("kw", [dict(k=None), dict(B=0), dict(D=7), dict(seqlen_k=0),
                                dict(k_sum=FAKE + 2)])
def test_kv_summaries_rejects_bad_arguments(kw):
    a = dict(k=FAKE, v=FAKE, B=1, seqlen_k=256, H=2, D=128, k_sum=FAKE, v_sum=FAKE, stream=0)
    a.update(kw)
    assert bsa.bsattn_kv_summaries(**a) == INV


def _bwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, out_dtype=bsa.OUT_F32, lse=FAKE, dout=FAKE, B=1,
             seqlen_q=256, seqlen_k=256, H=2, D=128, cu_seqlens_q=None, cu_seqlens_k=None,
             meta=_meta(), kv_valid_len=None,
             kind=bsa.MASK_CAUSAL, mask_params=None, softmax_scale=0.125, dq=FAKE, dk=FAKE,
             dv=FAKE, grad_dtype=bsa.OUT_F32, workspace=FAKE, workspace_bytes=1 << 20,
             err_flag=None, stream=0)
    a.update(kw)
    return bsa.bsattn_bwd(**a)


@pytest.mark.parametrize("kw,expect", [
    (dict(D=96), UNS),
    (dict(meta=_meta(varlen=1, cu_total_m_blocks=FAKE, cu_block_idx_offsets=FAKE)), INV),  # no cu_seqlens
    (dict(cu_seqlens_q=FAKE, cu_seqlens_k=FAKE), INV),            # batched meta with cu_seqlens
    (dict(dout=None), INV),
    (dict(lse=None), INV),
    (dict(dq=FAKE + 2), INV),                                  # not 16-byte aligned
    (dict(dv=None), INV),
    (dict(workspace=None), INV),
    (dict(workspace=FAKE + 16), INV),                          # not 256-byte aligned
    (dict(workspace_bytes=16), INV),                           # too small
    (dict(grad_dtype=5), INV),
    (dict(out_dtype=9), INV),
    (dict(seqlen_k=300), INV),                                 # num_n would be 3
    (dict(B=2), INV),
    (dict(kind=bsa.MASK_SLIDING_WINDOW), INV),
    (dict(softmax_scale=0.0), INV),
    (dict(meta=_meta(tile_n=64)), UNS),
])
def test_bwd_rejects_bad_arguments(kw, expect):
    assert _bwd(**kw) == expect


def test_bwd_workspace_size():
    # counts 2 x and order 1 x [B*H*num_n] int32; KV-major lists 2 x int32 and codes
    # 1 x byte per forward index entry ([B*H*num_m*num_n] batched, [H*total_n]
    # varlen); prefix [B+1] int32; rows 2 x 128 fp32 per Q tile and head; each
    # region rounded up to 256 bytes
    up = lambda x: -(-x // 256) * 256  # noqa: E731
    assert bsa.bsattn_bwd_workspace_size(_meta()) == 3 * 256 + 2 * 256 + 256 + 256 + 2 * 2048
    m = _meta(B=3, H=5, num_m=17, num_n=9)
    assert bsa.bsattn_bwd_workspace_size(m) == (3 * up(4 * 135) + 2 * up(4 * 135 * 17)
                                                + up(135 * 17) + up(4 * 4)
                                                + 2 * up(4 * 255 * 128))
    v = _meta(varlen=1, B=4, H=3, num_m=0, num_n=6, total_m_blocks=11, total_n_blocks=40,
              cu_total_m_blocks=FAKE, cu_block_idx_offsets=FAKE)
    assert bsa.bsattn_bwd_workspace_size(v) == (3 * up(4 * 72) + 2 * up(4 * 120) + up(120)
                                                + up(4 * 5) + 2 * up(4 * 33 * 128))
    with pytest.raises(bsa.BsattnError):
        bsa.bsattn_bwd_workspace_size(_meta(varlen=1, num_n=0, cu_total_m_blocks=FAKE,
                                            cu_block_idx_offsets=FAKE))


def test_sparse_block_metadata_rules():
    """Metadata per sparse block (tile_m 256, tile_n 256 or 128) is batched only;
    the forward needs an even number of 128-row Q tiles per sequence (each unit
    one whole block); the backward, the proxy forward and the block-map
    expansion take per-tile metadata only."""
    UNS = bsa.BSATTN_ERR_UNSUPPORTED
    blk = dict(tile_m=256, tile_n=256, num_m=2, num_n=2)
    # accepted sizes reach the device launch, which FAKE pointers cannot pass:
    # they must not fail the host checks (any status but INVALID_ARG/UNSUPPORTED)
    assert bsa.bsattn_fwd_workspace_size(_meta(**blk)) == 256 + 4 * 2 * 2
    assert _fwd(meta=_meta(tile_m=256, tile_n=128, num_m=2, num_n=4), seqlen_q=512,
                seqlen_k=512) not in (bsa.BSATTN_ERR_INVALID_ARG, UNS)
    # an odd number of Q tiles (384 rows = 3 tiles): a unit would hold half a block
    assert _fwd(meta=_meta(tile_m=256, tile_n=256, num_m=2, num_n=2), seqlen_q=384,
                seqlen_k=512) == UNS
    # sizes must follow the block size
    assert _fwd(meta=_meta(**blk), seqlen_q=256, seqlen_k=512) == bsa.BSATTN_ERR_INVALID_ARG
    # unsupported block shapes and layouts
    assert _fwd(meta=_meta(tile_m=128, tile_n=256, num_m=4, num_n=2), seqlen_q=512,
                seqlen_k=512) == UNS
    assert _fwd(meta=_meta(tile_m=512, tile_n=512, num_m=1, num_n=1), seqlen_q=512,
                seqlen_k=512) == UNS
    assert _fwd(meta=_meta(varlen=1, cu_total_m_blocks=FAKE, cu_block_idx_offsets=FAKE, **blk),
                cu_seqlens_q=FAKE, cu_seqlens_k=FAKE) == UNS
    with pytest.raises(bsa.BsattnError):
        bsa.bsattn_bwd_workspace_size(_meta(**blk))
    assert bsa.bsattn_build_meta_blocks(FAKE, 2, 2, 512, 512, None, None, bsa.MASK_NONE, None,
                                        _meta(**blk), stream=0) == UNS
