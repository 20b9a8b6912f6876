"""The oracle's readers of the bitmask and BSR selection formats, pinned to a
hand-worked example (tests/golden/bitmask_bsr_example.json), and the three
formats giving the same lists through the oracle."""
import json
import os

import numpy as np

import oracle
from workloads.formats import to_bitmask, to_bsr
from workloads import make_workload
from workloads.configs import MASK_CAUSAL, MASK_NONE, Workload, random_workload

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "bitmask_bsr_example.json")))


def _batched_wl():
    g = GOLD["batched"]
    nm, nn = -(-g["seqlen_q"] // 128), -(-g["seqlen_k"] // 128)
    return Workload(name="gold", B=g["B"], H=g["H"], D=64, varlen=False,
                    seqlens_q=np.array([g["seqlen_q"]], np.int32),
                    seqlens_k=np.array([g["seqlen_k"]], np.int32),
                    block_map=np.zeros((g["B"], g["H"], nm, nn), np.uint8), kind=MASK_NONE,
                    scale=0.125, data_seed=0)


def _selected(bm):
    return [list(np.nonzero(bm[0, h, m])[0]) for h in range(bm.shape[1]) for m in range(bm.shape[2])]


def test_bitmask_worked_example():
    g = GOLD["batched"]
    wl = _batched_wl()
    bm = oracle.map_from_bitmask(wl, np.array(g["words"], np.uint32), g["words_per_row"])
    assert _selected(bm) == g["selected"]


def test_bsr_worked_example():
    g = GOLD["batched"]
    wl = _batched_wl()
    bm = oracle.map_from_bsr(wl, np.array(g["bsr_indptr"]), np.array(g["bsr_indices"]))
    assert _selected(bm) == g["selected"]


def test_varlen_row_order_worked_example():
    g = GOLD["varlen"]
    wl = Workload(name="gold_varlen", B=2, H=g["H"], D=64, varlen=True,
                  seqlens_q=np.array(g["seqlens_q"], np.int32),
                  seqlens_k=np.array(g["seqlens_k"], np.int32),
                  block_map=np.zeros((g["H"], 8), np.uint8), kind=MASK_NONE, scale=0.125,
                  data_seed=0)
    bm = oracle.map_from_bitmask(wl, np.array(g["words"], np.uint32), g["words_per_row"])
    assert bm.tolist() == g["map"]


def test_bsr_decreasing_row_selects_nothing():
    wl = _batched_wl()
    indptr = np.array([0, 2, 1, 1, 1])   # row 1 ends below its start
    indices = np.array([5, 6])
    bm = oracle.map_from_bsr(wl, indptr, indices)
    assert _selected(bm) == [[5, 6], [], [], []]


def test_formats_give_identical_lists():
    for wl in (make_workload(1), make_workload(2), make_workload(3),
               random_workload(31, B=3, H=2, D=64, seqlens_q=[130, 700, 40], varlen=True,
                               kind=MASK_CAUSAL, density=0.4)):
        words, W = to_bitmask(wl, wl.block_map, pad_seed=1)
        indptr, indices = to_bsr(wl, wl.block_map, shuffle_seed=2, dup_every=2)
        ref = oracle.build_meta(wl)
        for bm in (oracle.map_from_bitmask(wl, words, W), oracle.map_from_bsr(wl, indptr, indices)):
            got = oracle.build_meta(wl, block_map=bm)
            for key in ("full_cnt", "full_idx", "mask_cnt", "mask_idx"):
                assert np.array_equal(got[key], ref[key]), (wl.name, key)


# ---- sparse blocks larger than the tile -----------------------------------

def test_expand_blocks_worked_example():
    # 2 x 2 tiles per block; 3 Q tiles (the last block row holds one tile), 4 KV tiles
    coarse = np.array([[[[1, 0], [0, 1]]]], np.uint8)
    tiles = oracle.expand_blocks(coarse, 2, 2, 3, 4)
    assert tiles[0, 0].tolist() == [[1, 1, 0, 0], [1, 1, 0, 0], [0, 0, 1, 1]]
    # 1 x 3: a block of three KV tiles, ragged at the end (5 tiles)
    coarse = np.array([[[[0, 1]]]], np.uint8)
    assert oracle.expand_blocks(coarse, 1, 3, 1, 5)[0, 0].tolist() == [[0, 0, 0, 1, 1]]


def test_split_valid_len_worked_example():
    # the 256-token split: min(v, 128) and v - min(v, 128)
    got = oracle.split_valid_len(np.array([[200, 100, 256, 0]]), 2, 8)
    assert got.tolist() == [[128, 72, 100, 0, 128, 128, 0, 0]]
    # three tiles per block
    assert oracle.split_valid_len(np.array([[300]]), 3, 3).tolist() == [[128, 128, 44]]


def test_vsa_native_blocks_reproduce_the_tile_inputs():
    wl = make_workload(4)
    logical = wl.extra["logical_map"][None]             # [1, H, 240, 240]
    v = wl.extra["logical_block_valid_len"][None]       # [1, 240]
    assert np.array_equal(oracle.expand_blocks(logical, 2, 2, wl.num_m, wl.num_n), wl.block_map)
    assert np.array_equal(oracle.split_valid_len(v, 2, wl.num_n), wl.kv_valid_len)
