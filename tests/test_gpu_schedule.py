"""The forward's scheduling pass (heaviest-first claiming order of the work
units, written into the caller's workspace) against the order defined on the
host from the metadata counts:

- unit u = (head h, pair p of Q tiles 2p, 2p+1); its work is the number of KV
  tiles both tiles' lists hold (per sparse-block list: entries x KV tiles per
  entry, counted once per block), clamped to 1023;
- units in order of decreasing work, units of equal work in increasing unit
  index (a stable sort).

The order is unique, so it is compared exactly, on workloads whose unit counts
are below, at and far above one warp's 32 lanes and one run per warp."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
from workloads import make_workload  # noqa: E402
from workloads.configs import MASK_CAUSAL, MASK_NONE, as_sparse_blocks, random_workload  # noqa: E402
from workloads.device import DeviceWorkload  # noqa: E402

pytestmark = pytest.mark.gpu

HEADER = 256  # workspace bytes before the order array


def _expected_order(meta, wl, list_q_tiles=1, list_kv_tiles=1):
    full = meta.full_cnt.cpu().numpy().astype(np.int64)
    mask = meta.mask_cnt.cpu().numpy().astype(np.int64)
    cnt = np.maximum(full, 0) + np.maximum(mask, 0)
    if wl.varlen:
        total_m = int(meta.total_m_blocks)
        per_tile = cnt.reshape(wl.H, total_m)
    else:
        num_m = -(-int(wl.seqlens_q[0]) // 128)  # Q tiles of 128 rows per sequence
        total_m = wl.B * num_m
        per_tile = np.zeros((wl.H, total_m), np.int64)
        for b in range(wl.B):
            for m in range(0, num_m, list_q_tiles):
                if b * num_m + m < total_m:
                    per_tile[:, b * num_m + m] = cnt[b, :, m // list_q_tiles]
    per_tile = np.minimum(per_tile * list_kv_tiles, 32767)
    pairs = (total_m + 1) // 2
    padded = np.zeros((wl.H, 2 * pairs), np.int64)
    padded[:, :total_m] = per_tile
    work = np.minimum(padded[:, 0::2] + padded[:, 1::2], 1023).reshape(-1)
    return np.argsort(-work, kind="stable").astype(np.int32)


def _order_after_forward(wl):
    dw = DeviceWorkload(wl, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    ws = bsa.alloc_workspace(meta)
    assert ws is not None
    ws.fill_(0xFF)
    dw.forward(meta, err_flag=err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n = (ws.numel() - HEADER) // 4
    order = ws[HEADER:HEADER + 4 * n].view(torch.int32).cpu().numpy()
    return meta, order


CASES = {
    "batched_3_units": dict(seed=401, B=1, H=3, D=64, seqlens_q=[200], kind=MASK_CAUSAL,
                            density=0.6),
    "batched_odd_tiles": dict(seed=402, B=2, H=5, D=128, seqlens_q=[1300, 1300],
                              kind=MASK_NONE, density=0.4),
    "varlen_mixed": dict(seed=403, B=4, H=7, D=128, seqlens_q=[100, 2000, 777, 3000],
                         varlen=True, kind=MASK_CAUSAL, density=0.5),
}


@pytest.mark.parametrize("name", list(CASES))
def test_order_on_random_workloads(name):
    wl = random_workload(**CASES[name])
    meta, order = _order_after_forward(wl)
    assert np.array_equal(order, _expected_order(meta, wl))


@pytest.mark.parametrize("cfg", [3, 4])
def test_order_on_the_target_workloads(cfg):
    wl = make_workload(cfg)
    meta, order = _order_after_forward(wl)
    exp = _expected_order(meta, wl)
    assert np.array_equal(np.sort(order), np.arange(order.size, dtype=np.int32))
    assert np.array_equal(order, exp)


def test_order_with_lists_per_sparse_block():
    wl = as_sparse_blocks(make_workload(4))
    meta, order = _order_after_forward(wl)
    assert np.array_equal(order, _expected_order(meta, wl, list_q_tiles=2,
                                                 list_kv_tiles=wl.tile_n // 128))
