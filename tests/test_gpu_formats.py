"""Metadata from packed bitmask words and from BSR rows (FlashInfer #4872,
bitmask format) against the byte-map path and the oracle: the lists must be
bit-identical.  Also the error flags of malformed rows."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.formats import to_bitmask, to_bsr  # noqa: E402
from workloads.device import DeviceWorkload, meta_to_numpy  # noqa: E402
from workloads import make_workload  # noqa: E402
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE,  # noqa: E402
                               MASK_SLIDING_WINDOW, random_workload)

pytestmark = pytest.mark.gpu

KEYS = ("full_cnt", "full_idx", "mask_cnt", "mask_idx")


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a).astype(dtype)).to("cuda")


def _run(dw, fmt, data, err):
    wl = dw.wl
    meta = dw.alloc_meta()
    sq, sk = dw.seqlens()
    args = dict(cu_seqlens_q=dw.cu_q, cu_seqlens_k=dw.cu_k, seqlen_q=sq, seqlen_k=sk,
                kv_valid_len=dw.vl, kind=wl.kind, mask_params=dw.mask_params, meta=meta,
                err_flag=err, stream=torch.cuda.current_stream().cuda_stream)
    if fmt == "bitmask":
        words, W = data
        st = bsa.bsattn_build_meta_bitmask(_dev(words.view(np.int32), np.int32), W, **args)
    else:
        indptr, indices = data
        st = bsa.bsattn_build_meta_bsr(_dev(indptr, np.int32), _dev(indices, np.int32), **args)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    torch.cuda.synchronize()
    return meta_to_numpy(meta)


def _cases():
    return [
        ("cfg1", make_workload(1)), ("cfg2", make_workload(2)), ("cfg3", make_workload(3)),
        ("rand_varlen", random_workload(41, B=4, H=2, D=64, seqlens_q=[130, 257, 40, 1],
                                        varlen=True, kind=MASK_CAUSAL, valid_len=True)),
        ("rand_window", random_workload(42, B=2, H=2, D=64, seqlens_q=[200, 450],
                                        seqlens_k=[333, 129], varlen=True,
                                        kind=MASK_SLIDING_WINDOW, window_left=150,
                                        sink_tokens=70, valid_len=True)),
        ("rand_doc", random_workload(43, B=2, H=1, D=64, seqlens_q=[300, 77], varlen=True,
                                     kind=MASK_DOCUMENT, n_docs=4)),
        ("rand_wide", random_workload(44, B=1, H=2, D=64, seqlens_q=[600], seqlens_k=[9000],
                                      kind=MASK_NONE, density=0.3)),   # 71 KV tiles: 3 words
    ]


@pytest.mark.parametrize("idx", range(7))
def test_formats_match_byte_map_and_oracle(idx):
    name, wl = _cases()[idx]
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_dev = meta_to_numpy(dw.build_meta(err_flag=err))
    torch.cuda.synchronize()
    ref = oracle.build_meta(wl)
    datas = {"bitmask": to_bitmask(wl, wl.block_map, pad_seed=idx),
             "bsr": to_bsr(wl, wl.block_map, shuffle_seed=idx, dup_every=3)}
    for fmt, data in datas.items():
        got = _run(dw, fmt, data, err)
        assert int(err.item()) == 0, (name, fmt)
        for key in KEYS:
            assert np.array_equal(got[key], ref_dev[key]), (name, fmt, key)
            assert np.array_equal(got[key], ref[key]), (name, fmt, key)


@pytest.mark.parametrize("cfg", [4, 5])
def test_formats_full_size(cfg):
    wl = make_workload(cfg)
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_dev = meta_to_numpy(dw.build_meta(err_flag=err))
    for fmt, data in (("bitmask", to_bitmask(wl, wl.block_map, pad_seed=cfg)),
                      ("bsr", to_bsr(wl, wl.block_map, shuffle_seed=cfg))):
        got = _run(dw, fmt, data, err)
        assert int(err.item()) == 0
        for key in KEYS:
            assert np.array_equal(got[key], ref_dev[key]), (cfg, fmt, key)


def test_bsr_bad_rows_are_flagged_and_skipped():
    wl = random_workload(45, B=1, H=1, D=64, seqlens_q=[384], kind=MASK_CAUSAL, density=0.6)
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    indptr, indices = to_bsr(wl, wl.block_map)
    # an out-of-range id appended to row 1 must be skipped and flagged
    bad_indptr = indptr.copy()
    bad_indptr[2:] += 1
    bad_indices = np.insert(indices, indptr[2], 99)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(dw, "bsr", (bad_indptr, bad_indices), err)
    assert int(err.item()) & bsa.FLAG_BAD_INDEX
    ref = oracle.build_meta(wl)
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key
    # a row whose end lies below its start selects nothing and is flagged
    dec = indptr.copy()
    dec[2] = dec[1] - 1   # row 1 ends below its start (row 0 holds its forced diagonal tile)
    err.zero_()
    got = _run(dw, "bsr", (dec, indices), err)
    assert int(err.item()) & bsa.FLAG_BAD_COUNT
    expect = oracle.build_meta(wl, block_map=oracle.map_from_bsr(wl, dec, indices))
    for key in KEYS:
        assert np.array_equal(got[key], expect[key]), key


def test_bitmask_varlen_rows_wider_than_words_are_flagged():
    wl = random_workload(46, B=2, H=1, D=64, seqlens_q=[200, 300], seqlens_k=[200, 5000],
                         varlen=True, kind=MASK_NONE, density=0.5)
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    words, W = to_bitmask(wl, wl.block_map, words_per_row=1)   # sequence 1 has 40 KV tiles
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(dw, "bitmask", (words, 1), err)
    assert int(err.item()) & bsa.FLAG_BAD_COUNT
    expect = oracle.build_meta(wl, block_map=oracle.map_from_bitmask(wl, words, 1))
    for key in KEYS:
        assert np.array_equal(got[key], expect[key]), key
