"""The oracle's proxy-compensated forward and KV summaries ("feat(prims-ts):
support proxy-compensated block-sparse attention", FlashInfer #4872), pinned to
closed forms: a tile whose keys are all equal is represented exactly by its
summaries, so proxies over such tiles reproduce exact attention (computed by the
C oracle); with every tile selected the proxy form is exact attention; and a
hand-worked mean / sum over a partial tile.  The per-row form (for full-size
checks) equals the dense one on every row."""
import numpy as np
import pytest

import oracle
from workloads.configs import MASK_NONE, random_workload


def _bits(x):
    """float values exactly representable in bf16 -> bf16 bits."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _wl(seed, sq, sk, D=64, H=2, density=0.5):
    return random_workload(seed, B=1, H=H, D=D, seqlens_q=[sq], seqlens_k=[sk], kind=MASK_NONE,
                           density=density, force_diag=False)


def test_summaries_worked_example():
    wl = _wl(80, 128, 130)
    q, k, v = wl.qkv()
    kf = np.zeros(k.shape, np.float32)
    vf = np.zeros(v.shape, np.float32)
    kf[0, :, 0, 0] = np.arange(130)             # integers, exact in bf16
    vf[0, :, 1, 3] = np.arange(130)
    km, vs = oracle.kv_summaries(wl, _bits(kf), _bits(vf))
    assert km[0, 0, 0, 0] == 63.5 and km[0, 1, 0, 0] == 128.5      # (0+...+127)/128, (128+129)/2
    assert vs[0, 0, 1, 3] == 8128.0 and vs[0, 1, 1, 3] == 257.0
    assert np.count_nonzero(km) == 2 and np.count_nonzero(vs) == 2


def _constant_key_tiles(wl):
    """k with every 128-key tile made of one repeated key row (per head)."""
    q, k, v = wl.qkv()
    k = k.copy()
    S = k.shape[1]
    for n0 in range(0, S, 128):
        k[:, n0:min(n0 + 128, S)] = k[:, n0:n0 + 1]
    return q, k, v


def test_proxy_over_constant_key_tiles_is_exact_attention():
    for sk in (384, 300):                       # 300: a 44-key last tile
        wl = _wl(81, 256, sk)
        q, k, v = _constant_key_tiles(wl)
        km, vs = oracle.kv_summaries(wl, k, v)  # exact: the mean of equal keys is that key
        none = np.zeros_like(wl.block_map)
        o_p, l_p = oracle.fwd_proxy(wl, q, k, v, km, vs, none)
        wl.block_map = np.ones_like(wl.block_map)
        o_e, l_e = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
        assert np.max(np.abs(o_p - o_e)) < 1e-12 and np.max(np.abs(l_p - l_e)) < 1e-12


def test_proxy_with_every_tile_selected_is_exact_attention():
    wl = _wl(82, 384, 700, density=1.0)
    q, k, v = wl.qkv()
    km, vs = oracle.kv_summaries(wl, k, v)
    o_p, l_p = oracle.fwd_proxy(wl, q, k, v, km, vs, np.ones_like(wl.block_map))
    o_e, l_e = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    assert np.max(np.abs(o_p - o_e)) < 1e-12 and np.max(np.abs(l_p - l_e)) < 1e-12


def test_mixed_selection_splits_between_exact_and_proxy():
    # constant-key tiles again, now half selected: still exact attention overall
    wl = _wl(83, 384, 900)
    q, k, v = _constant_key_tiles(wl)
    km, vs = oracle.kv_summaries(wl, k, v)
    o_p, l_p = oracle.fwd_proxy(wl, q, k, v, km, vs, wl.block_map)
    wl.block_map = np.ones_like(wl.block_map)
    o_e, l_e = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    assert np.max(np.abs(o_p - o_e)) < 1e-12 and np.max(np.abs(l_p - l_e)) < 1e-12


@pytest.mark.parametrize("seed,density,sk", [(701, 0.5, 300), (702, 0.0, 640), (703, 0.3, 1000)])
def test_proxy_rows_equal_the_dense_proxy(seed, density, sk):
    # the per-row form (grouped by Q tile, for full-size checks) against fwd_proxy on every row
    wl = random_workload(seed, B=2, H=2, D=16, seqlens_q=[384, 384], seqlens_k=[sk, sk],
                         kind=MASK_NONE, density=density, force_diag=density > 0)
    q, k, v = wl.qkv()
    km, vsum = oracle.kv_summaries(wl, k, v)
    o_ref, l_ref = oracle.fwd_proxy(wl, q, k, v, km, vsum, wl.block_map)
    S, H = 384, 2
    b, t, h = np.meshgrid(np.arange(2), np.arange(S), np.arange(H), indexing="ij")
    o, l = oracle.fwd_proxy_rows(wl, q, k, v, km, vsum, wl.block_map, t.ravel(), h.ravel(), b.ravel())
    assert np.max(np.abs(o - o_ref[b.ravel(), t.ravel(), h.ravel()])) < 1e-12
    assert np.max(np.abs(l - l_ref[b.ravel(), h.ravel(), t.ravel()])) < 1e-12
