"""Metadata from a block map given per sparse block of several tiles
(bsattn_build_meta_blocks) against the per-tile path and the oracle: identical
lists, and per-tile valid lengths equal to the oracle's split of the block
lengths; a forward fed those lengths equals the forward fed the host's."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.device import DeviceWorkload, meta_to_numpy  # noqa: E402
from workloads import make_workload  # noqa: E402
from workloads.configs import (MASK_CAUSAL, MASK_NONE, MASK_PREFIX,  # noqa: E402
                               MASK_SLIDING_WINDOW, Workload)

pytestmark = pytest.mark.gpu

KEYS = ("full_cnt", "full_idx", "mask_cnt", "mask_idx")


def _blocks_meta(dw, coarse, qf, kf, vl_blocks, err):
    wl = dw.wl
    meta = dw.alloc_meta()
    sq, sk = dw.seqlens()
    d_map = torch.from_numpy(np.ascontiguousarray(coarse)).to("cuda")
    d_vlb = torch.from_numpy(np.ascontiguousarray(vl_blocks)).to("cuda") if vl_blocks is not None else None
    d_vlt = torch.full((wl.B, wl.num_n), -7, dtype=torch.int32, device="cuda")
    st = bsa.bsattn_build_meta_blocks(d_map, qf, kf, sq, sk, d_vlb, d_vlt, wl.kind, dw.mask_params,
                                      meta, err_flag=err,
                                      stream=torch.cuda.current_stream().cuda_stream)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    torch.cuda.synchronize()
    return meta, d_vlt


def test_vsa_native_256_token_blocks():
    wl = make_workload(4)
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = meta_to_numpy(dw.build_meta(err_flag=err))
    meta, vlt = _blocks_meta(dw, wl.extra["logical_map"][None], 2, 2,
                             wl.extra["logical_block_valid_len"][None].astype(np.int32), err)
    assert int(err.item()) == 0
    got = meta_to_numpy(meta)
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key
    assert np.array_equal(vlt.cpu().numpy(), wl.kv_valid_len)


def _case(seed, B, H, sq, sk, qf, kf, kind, valid, **mask):
    rng = np.random.default_rng(seed)
    nm, nn = math.ceil(sq / 128), math.ceil(sk / 128)
    bm_, bn_ = math.ceil(nm / qf), math.ceil(nn / kf)
    coarse = (rng.random((B, H, bm_, bn_)) < 0.5).astype(np.uint8)
    for i in range(min(bm_, bn_)):
        coarse[:, :, i, i] = 1
    vlb = rng.integers(0, kf * 128 + 1, (B, bn_)).astype(np.int32) if valid else None
    tiles = oracle.expand_blocks(coarse, qf, kf, nm, nn)
    vlt = oracle.split_valid_len(vlb, kf, nn) if valid else None
    wl = Workload(name=f"blocks_{seed}", B=B, H=H, D=64, varlen=False,
                  seqlens_q=np.full(B, sq, np.int32), seqlens_k=np.full(B, sk, np.int32),
                  block_map=np.ascontiguousarray(tiles), kind=kind, scale=0.125, data_seed=seed,
                  kv_valid_len=vlt, **mask)
    return wl, coarse, vlb


CASES = [
    dict(seed=61, B=2, H=2, sq=700, sk=900, qf=2, kf=2, kind=MASK_CAUSAL, valid=True),
    dict(seed=62, B=1, H=3, sq=1000, sk=1000, qf=2, kf=1, kind=MASK_NONE, valid=True),
    dict(seed=63, B=1, H=2, sq=600, sk=1500, qf=1, kf=3, kind=MASK_PREFIX, valid=False,
         prefix_len=300),
    dict(seed=64, B=2, H=1, sq=1300, sk=1300, qf=3, kf=2, kind=MASK_SLIDING_WINDOW, valid=True,
         window_left=400, sink_tokens=100),
    dict(seed=65, B=1, H=2, sq=2048, sk=2048, qf=4, kf=4, kind=MASK_CAUSAL, valid=False),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_block_maps_match_oracle(idx):
    c = dict(CASES[idx])
    mask = {k: c.pop(k) for k in ("prefix_len", "window_left", "sink_tokens") if k in c}
    wl, coarse, vlb = _case(**c, **mask)
    dw = DeviceWorkload(wl, "cuda", qkv=False)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta, vlt = _blocks_meta(dw, coarse, c["qf"], c["kf"], vlb, err)
    assert int(err.item()) == 0
    got = meta_to_numpy(meta)
    ref = oracle.build_meta(wl)
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key
    expect_vl = wl.kv_valid_len if vlb is not None else np.full((wl.B, wl.num_n), 128, np.int32)
    assert np.array_equal(vlt.cpu().numpy(), expect_vl)


def test_forward_with_block_valid_lengths_equals_tile_lengths():
    wl, coarse, vlb = _case(seed=66, B=1, H=2, sq=640, sk=768, qf=2, kf=2, kind=MASK_CAUSAL,
                            valid=True)
    wl.D = 128
    dw = DeviceWorkload(wl, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta, vlt = _blocks_meta(dw, coarse, 2, 2, vlb, err)
    out_host, lse_host = dw.forward(meta, err_flag=err, out_dtype=torch.float32)
    dw.vl = vlt
    out_dev, lse_dev = dw.forward(meta, err_flag=err, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_host, out_dev) and torch.equal(lse_host, lse_dev)
