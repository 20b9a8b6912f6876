"""Metadata kernel vs the oracle: bit-exact on every config and on randomised
cases covering every mask kind, varlen packing, ragged tails and valid lengths."""
import numpy as np
import pytest
import torch

import oracle
from workloads.device import DeviceWorkload, meta_to_numpy
from workloads import make_workload
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,
                               MASK_SLIDING_WINDOW, random_workload)

pytestmark = pytest.mark.gpu

KEYS = ("full_cnt", "full_idx", "mask_cnt", "mask_idx")


def _check(wl):
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    torch.cuda.synchronize()
    got = meta_to_numpy(meta)
    ref = oracle.build_meta(wl)
    assert int(err.item()) == 0
    for key in KEYS:
        assert got[key].shape == ref[key].shape
        assert np.array_equal(got[key], ref[key]), f"{key} differs"
    if wl.varlen:
        assert np.array_equal(got["cu_total_m_blocks"], ref["cu_total_m_blocks"])
        assert np.array_equal(got["cu_block_idx_offsets"], ref["cu_block_idx_offsets"])


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_meta_configs_small(cfg):
    _check(make_workload(cfg))


@pytest.mark.parametrize("cfg", [4, 5])
def test_meta_configs_full_size(cfg):
    _check(make_workload(cfg))


CASES = [
    dict(seed=101, B=2, H=3, D=64, seqlens_q=[384, 384], kind=MASK_CAUSAL),
    dict(seed=102, B=1, H=2, D=64, seqlens_q=[300], seqlens_k=[520], kind=MASK_NONE, valid_len=True),
    dict(seed=103, B=4, H=2, D=64, seqlens_q=[130, 257, 40, 1], varlen=True, kind=MASK_CAUSAL,
         valid_len=True),
    dict(seed=104, B=2, H=2, D=64, seqlens_q=[200, 450], seqlens_k=[333, 129], varlen=True,
         kind=MASK_SLIDING_WINDOW, window_left=150, sink_tokens=70, valid_len=True),
    dict(seed=105, B=1, H=2, D=64, seqlens_q=[1000], kind=MASK_SLIDING_WINDOW, window_left=256,
         sink_tokens=200, density=0.8),
    dict(seed=106, B=1, H=2, D=64, seqlens_q=[512], kind=MASK_PREFIX, prefix_len=200),
    dict(seed=107, B=2, H=1, D=64, seqlens_q=[300, 77], varlen=True, kind=MASK_DOCUMENT, n_docs=4),
    dict(seed=108, B=1, H=2, D=64, seqlens_q=[640], seqlens_k=[1300], kind=MASK_PREFIX,
         prefix_len=700, valid_len=True),
    dict(seed=109, B=3, H=2, D=64, seqlens_q=[4096, 100, 2000], varlen=True, kind=MASK_CAUSAL,
         density=0.3),
    dict(seed=110, B=1, H=2, D=64, seqlens_q=[256], kind=MASK_CAUSAL, density=0.0,
         force_diag=False),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_meta_random_cases(case):
    _check(random_workload(**CASES[case]))


def test_meta_error_flag_on_inconsistent_varlen_totals():
    """The caller's packed sizes disagree with cu_seqlens: flagged on the device,
    nothing written past the caller's arrays, no fault."""
    wl = random_workload(120, B=2, H=2, D=64, seqlens_q=[300, 200], varlen=True, kind=MASK_CAUSAL)
    dev = torch.device("cuda")
    import block_sparse_flashattention_gb300 as bsa
    from workloads.device import i32
    small_m, small_n = wl.total_m_blocks - 1, wl.total_n_blocks - 3
    meta = bsa.alloc_meta(wl.B, wl.H, varlen=True, total_m_blocks=small_m, total_n_blocks=small_n,
                          max_num_n=wl.num_n, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bm = torch.from_numpy(np.ascontiguousarray(wl.block_map[:, :small_n])).to(dev)
    bsa.build_meta(bm, meta, cu_seqlens_q=i32(wl.cu_seqlens_q, dev),
                   cu_seqlens_k=i32(wl.cu_seqlens_k, dev), kind=wl.kind, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & bsa.FLAG_BAD_SEQLENS
