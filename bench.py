#!/usr/bin/env python
"""Benchmark of the block-sparse attention forward on GB300.

One step = the whole hot path over one batch of synthetic input: the metadata
kernel (boolean block map -> full / mask lists) and the attention kernel.
Default workload: video sparse attention, B=1 H=24 S=61440 d=128, top-32 of 240
logical 256-token KV blocks per logical Q block, valid length U[192,256] per
logical block, run as 128-token tiles (737,280 computed tiles, 6.185 TFLOP).

Metric: effective TFLOP/s = sum over computed tiles of 4 * 128 * 128 * d,
divided by the time.  Also reported: the attention kernel's own roofline
(CUDA events around its launches), an end-to-end number through the public
API with pinned host buffers (host->device inputs and device->host outputs
inside the timed region), and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
Under torchrun each rank runs its own replica on its own GPU (no data-path
collective); rank 0 prints one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective TFLOP/s over computed blocks, bf16 fwd; % of GB300 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_CONFIG = 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG,
                    help="workload number (1-5); the benchmark line uses 4")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-meta-formats", action="store_true",
                    help="skip the side measurements (metadata formats, proxy A/B)")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward timing")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the forward timing of configs 3 and 5")
    ap.add_argument("--no-oracle-timing", action="store_true",
                    help="skip the oracle timing over configs 1-5")
    ap.add_argument("--heads", type=int, default=0,
                    help="keep only the first N heads (a smaller case for profiling)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(pg, ms: float, device) -> float:
    """The largest of the ranks' timings (ms); `pg` is torch.distributed with an
    initialised process group, or None for one rank."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flop_per_rank_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank processes flop_per_rank_step per step
    (replicas, weak scaling) and the job takes the slowest rank's time."""
    return world * flop_per_rank_step * steps / (ms * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def flop_per_tile(d: int) -> int:
    return 4 * 128 * 128 * d


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if gpu_index is not None:
            cmd += ["-i", str(gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                for name, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_index_for_smi(torch, dev):
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", None)
        devid = getattr(props, "pci_device_id", None)
        if bus is not None and dom is not None and devid is not None:
            return f"{dom:08x}:{bus:02x}:{devid:02x}.0"
    except Exception:
        pass
    return None


def one_head(wl, q, k, v):
    """Head 0 of a workload as a workload of its own (heads are independent)."""
    import numpy as np
    from dataclasses import replace
    bm = wl.block_map[:1] if wl.varlen else wl.block_map[:, :1]
    w1 = replace(wl, H=1, block_map=np.ascontiguousarray(bm))
    cut = (lambda x: np.ascontiguousarray(x[:, :1])) if wl.varlen else (
        lambda x: np.ascontiguousarray(x[:, :, :1]))
    return w1, cut(q), cut(k), cut(v)


def cpu_baseline(wl, q, k, v, seconds, threads=None):
    """The oracle on whole Q tiles of head 0, drawn at random, until about
    `seconds` of oracle time; returns (TFLOP/s over the sample's computed tiles,
    threads used, description of the sample)."""
    import numpy as np
    import oracle
    threads = threads or oracle.default_threads()
    w1, q1, k1, v1 = one_head(wl, q, k, v)
    meta = oracle.build_meta(w1, threads=threads)
    cnt = (meta["full_cnt"] + meta["mask_cnt"]).reshape(-1)     # per packed Q tile
    starts = (np.concatenate([[0], np.cumsum(np.ceil(w1.seqlens_q / 128).astype(int))])
              if w1.varlen else None)
    rng = np.random.default_rng(0)
    done_flop, done_tiles, elapsed = 0, 0, 0.0
    while elapsed < seconds and done_tiles < 4096:
        t = int(rng.integers(0, cnt.size))
        if w1.varlen:
            b = int(np.searchsorted(starts, t, side="right") - 1)
            r0 = int(w1.cu_seqlens_q[b]) + (t - int(starts[b])) * 128
            r1 = min(r0 + 128, int(w1.cu_seqlens_q[b + 1]))
        else:
            S = int(w1.seqlens_q[0])
            b, m = divmod(t, S // 128 if S % 128 == 0 else -(-S // 128))
            r0 = b * S + m * 128
            r1 = min(r0 + 128, (b + 1) * S)
        tok = np.arange(r0, r1, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.fwd_rows(w1, q1, k1, v1, meta, tok, np.zeros_like(tok), threads=threads)
        elapsed += time.perf_counter() - t0
        done_flop += int(cnt[t]) * flop_per_tile(wl.D)
        done_tiles += 1
    value = done_flop / elapsed / 1e12
    desc = (f"oracle (fp64, plain C, {threads} threads) on {done_tiles} whole Q tiles of head 0 "
            f"drawn at random from the workload: {done_flop / 1e9:.1f} GFLOP of computed tiles "
            f"in {elapsed:.1f} s")
    return value, threads, desc


def time_meta_formats(wl, dw, meta, err, stream, iters=20):
    """The metadata kernel fed by each selection format (byte map, packed bitmask
    words, BSR rows, and, where the workload has one, its native map per 256-token
    block with per-block valid lengths) on the benchmark workload, outside the timed region: mean ms
    over `iters` launches and achieved GB/s over the bytes each must move (its
    input and the two -1-padded lists and counts it writes; the valid lengths,
    read once per selected mask tile, are left out)."""
    import numpy as np
    import torch
    import block_sparse_flashattention_gb300 as bsa
    from workloads.formats import to_bitmask, to_bsr
    words, W = to_bitmask(wl, wl.block_map)
    indptr, indices = to_bsr(wl, wl.block_map)
    dev = dw.q.device
    d_words = torch.from_numpy(words.view(np.int32)).to(dev)
    d_indptr = torch.from_numpy(indptr).to(dev)
    d_indices = torch.from_numpy(indices).to(dev)
    sq, sk = dw.seqlens()
    rows = words.shape[0]
    out_bytes = 2 * int(wl.block_map.size) * 4 + 2 * rows * 4   # both lists (num_n per row) + counts
    in_bytes = {"byte_map": int(wl.block_map.size), "bitmask": int(words.nbytes),
                "bsr": int(indptr.nbytes + indices.nbytes)}
    common = dict(cu_seqlens_q=dw.cu_q, cu_seqlens_k=dw.cu_k, seqlen_q=sq, seqlen_k=sk,
                  kv_valid_len=dw.vl, kind=wl.kind, mask_params=dw.mask_params, meta=meta,
                  err_flag=err, stream=stream.cuda_stream)

    native = wl.extra.get("logical_map") if not wl.varlen else None
    if native is not None:   # the map also exists per 256-token block (2 x 2 tiles)
        d_blocks = torch.from_numpy(np.ascontiguousarray(native[None] if native.ndim == 3
                                                         else native)).to(dev)
        vlb = wl.extra.get("logical_block_valid_len")
        d_vlb = torch.from_numpy(np.ascontiguousarray(vlb).reshape(wl.B, -1).astype(np.int32)).to(dev) \
            if vlb is not None else None
        d_vlt = torch.empty((wl.B, wl.num_n), dtype=torch.int32, device=dev)
        in_bytes["blocks_2x2"] = int(native.size) + (int(vlb.size) * 4 if vlb is not None else 0)

    def call(fmt):
        if fmt == "byte_map":
            dw.build_meta(meta, err_flag=err)
            return
        if fmt == "blocks_2x2":
            st = bsa.bsattn_build_meta_blocks(d_blocks, 2, 2, sq, sk, d_vlb, d_vlt, wl.kind,
                                              dw.mask_params, meta, err_flag=err,
                                              stream=stream.cuda_stream)
            if st != bsa.BSATTN_OK:
                raise RuntimeError(f"{fmt}: {bsa.status_string(st)}")
            return
        if fmt == "bitmask":
            st = bsa.bsattn_build_meta_bitmask(d_words, W, **common)
        else:
            st = bsa.bsattn_build_meta_bsr(d_indptr, d_indices, **common)
        if st != bsa.BSATTN_OK:
            raise RuntimeError(f"{fmt}: {bsa.status_string(st)}")

    out = {}
    for fmt in ("byte_map", "bitmask", "bsr") + (("blocks_2x2",) if native is not None else ()):
        for _ in range(3):
            call(fmt)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            call(fmt)
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / iters
        nbytes = in_bytes[fmt] + out_bytes + (wl.B * wl.num_n * 4 if fmt == "blocks_2x2" else 0)
        out[fmt] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9}
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())} after the metadata formats")
    return out


def time_proxy(wl, dw, err, stream, iters=10):
    """Proxy-compensation A/B on the benchmark map with identical inputs: the exact
    forward against the proxy forward (summaries of every omitted KV tile), both
    on metadata built with mask kind none and no valid lengths (the proxy mode
    needs a dense mask), plus the time of the KV summaries kernel."""
    import math
    import numpy as np
    import torch
    import block_sparse_flashattention_gb300 as bsa
    from workloads.formats import to_bitmask
    if wl.varlen or wl.kind != bsa.MASK_NONE:
        return None
    dev = dw.q.device
    sq, sk = dw.seqlens()
    meta = dw.alloc_meta()
    st = bsa.bsattn_build_meta(dw.block_map, None, None, sq, sk, None, bsa.MASK_NONE, None, meta,
                               err, stream.cuda_stream)
    if st != bsa.BSATTN_OK:
        raise RuntimeError(bsa.status_string(st))
    nn = math.ceil(sk / 128)
    ks = torch.empty((wl.B, nn, wl.H, wl.D), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    words, W = to_bitmask(wl, wl.block_map)
    d_words = torch.from_numpy(words.view(np.int32)).to(dev)
    out = torch.empty(dw.q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.B, wl.H, sq), dtype=torch.float32, device=dev)
    ws = bsa.alloc_workspace(meta, dev)

    def summaries():
        st = bsa.bsattn_kv_summaries(dw.k, dw.v, wl.B, sk, wl.H, wl.D, ks, vs, stream.cuda_stream)
        if st != bsa.BSATTN_OK:
            raise RuntimeError(bsa.status_string(st))

    def exact():
        st = bsa.bsattn_fwd(dw.q, dw.k, dw.v, wl.B, sq, sk, wl.H, wl.D, None, None, meta, None,
                            bsa.MASK_NONE, None, wl.scale, out, bsa.OUT_BF16, lse, workspace=ws,
                            err_flag=err, stream=stream.cuda_stream)
        if st != bsa.BSATTN_OK:
            raise RuntimeError(bsa.status_string(st))

    def proxy():
        st = bsa.bsattn_fwd_proxy(dw.q, dw.k, dw.v, wl.B, sq, sk, wl.H, wl.D, meta, d_words, W, ks,
                                  vs, wl.scale, out, bsa.OUT_BF16, lse, workspace=ws, err_flag=err,
                                  stream=stream.cuda_stream)
        if st != bsa.BSATTN_OK:
            raise RuntimeError(bsa.status_string(st))

    res = {}
    for name, fn in (("summaries", summaries), ("exact", exact), ("proxy", proxy)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        res[name + "_ms"] = a.elapsed_time(b) / iters
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())} in the proxy A/B")
    res["overhead"] = res["proxy_ms"] / res["exact_ms"] - 1.0
    res["note"] = "benchmark map, mask kind none, no valid lengths; summaries outside both arms"
    return res


def time_bwd(wl, dw, meta, out, lse, err, stream, flop_fwd, iters=5):
    """Backward (bsattn_bwd: list transpose, row pass, dK/dV kernel, dQ kernel) on
    the benchmark's metadata and forward results, with a seeded upstream gradient.
    Effective TFLOP/s counts 2.5x the forward's FLOPs per computed block (the five
    128x128xD products S, dP, dV, dK, dQ), the usual attention-backward
    convention; the kernels recompute S and dP once more (seven products)."""
    import torch
    import block_sparse_flashattention_gb300 as bsa
    dev = dw.q.device
    sq, sk = dw.seqlens()
    hdo = torch.empty(wl.q_shape(), dtype=torch.int16, pin_memory=True)
    wl.fill("do", hdo.data_ptr())
    dout = hdo.to(dev).view(torch.bfloat16)
    dq = torch.empty_like(dw.q)
    dk = torch.empty_like(dw.k)
    dv = torch.empty_like(dw.v)
    wsb = torch.empty(bsa.bsattn_bwd_workspace_size(meta), dtype=torch.uint8, device=dev)

    def bwd():
        st = bsa.bsattn_bwd(dw.q, dw.k, dw.v, out, bsa.OUT_BF16, lse, dout, wl.B, sq, sk, wl.H,
                            wl.D, dw.cu_q, dw.cu_k, meta, dw.vl, wl.kind, dw.mask_params, wl.scale,
                            dq, dk, dv,
                            bsa.OUT_BF16, wsb, err_flag=err, stream=stream.cuda_stream)
        if st != bsa.BSATTN_OK:
            raise RuntimeError(bsa.status_string(st))

    for _ in range(3):
        bwd()
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bwd()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms.append(a.elapsed_time(b))
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())} in the backward")
    mean = statistics.mean(ms)
    flop = 2.5 * flop_fwd
    return {"ms": mean, "tflops": flop / (mean * 1e-3) / 1e12, "flop": flop,
            "launches_per_call": 6 + (1 if wl.varlen else 0), "grad_dtype": "bf16",
            "note": "flop = 2.5 x forward flop over computed blocks; events around each call"}


def time_forward(dw, meta, err, stream, ws, warmup=5, iters=20):
    """Median of `iters` CUDA-event-timed forward calls (scheduling pass +
    attention kernel) after `warmup` untimed ones, and the same for the metadata
    kernel (K-META), on the launching stream."""
    import torch
    out = torch.empty_like(dw.q)
    lse = None
    for _ in range(warmup):
        dw.build_meta(meta, err_flag=err, stream=stream)
        out, lse = dw.forward(meta, out=out, lse=lse, err_flag=err, workspace=ws, stream=stream)
    torch.cuda.synchronize(dw.q.device)
    f_ms, m_ms = [], []
    for _ in range(iters):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        dw.build_meta(meta, err_flag=err, stream=stream)
        e[1].record(stream)
        dw.forward(meta, out=out, lse=lse, err_flag=err, workspace=ws, stream=stream)
        e[2].record(stream)
        torch.cuda.synchronize(dw.q.device)
        m_ms.append(e[0].elapsed_time(e[1]))
        f_ms.append(e[1].elapsed_time(e[2]))
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())}")
    return statistics.median(f_ms), statistics.median(m_ms)


def per_config(cfgs, dev, peak, stream):
    """Forward and K-META of further workloads, each on its full seeded inputs
    (median of 20 CUDA-event-timed runs after 5 warm-ups)."""
    import torch
    import block_sparse_flashattention_gb300 as bsa
    from workloads import make_workload
    from workloads.device import DeviceWorkload, computed_blocks, meta_to_numpy
    res = {}
    for cfg in cfgs:
        wl = make_workload(cfg)
        dw = DeviceWorkload(wl, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        meta = dw.build_meta(err_flag=err, stream=stream)
        ws = bsa.alloc_workspace(meta, dev)
        torch.cuda.synchronize(dev)
        blocks = computed_blocks(meta_to_numpy(meta))
        flop = blocks * flop_per_tile(wl.D)
        f_ms, m_ms = time_forward(dw, meta, err, stream, ws)
        tf = flop / (f_ms * 1e-3) / 1e12
        res[str(cfg)] = {"workload": wl.name, "computed_tiles": blocks, "flop": flop,
                         "fwd_ms": f_ms, "tflops": tf, "frac": tf / peak, "meta_ms": m_ms,
                         "timing": "median of 20 CUDA-event-timed calls after 5 warm-ups"}
        del dw, meta, ws
        torch.cuda.empty_cache()
    return res


def time_sparse_blocks(wl, dw, meta, dev, stream, peak):
    """A/B on a workload with a native sparse-block map (config 4: 256-token
    blocks): the metadata kernel and the forward fed lists per 256 x 256 block
    against the same fed per-tile lists, on the same device inputs (median of 20
    CUDA-event-timed calls after 5 warm-ups each)."""
    import copy
    import torch
    import block_sparse_flashattention_gb300 as bsa
    from workloads.configs import as_sparse_blocks
    from workloads.device import computed_blocks, meta_to_numpy
    w2 = as_sparse_blocks(wl)
    dw2 = copy.copy(dw)
    dw2.wl = w2
    dw2.block_map = torch.from_numpy(w2.block_map).to(dev)
    dw2.vl = torch.from_numpy(w2.kv_valid_len).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    meta2 = dw2.build_meta(err_flag=err, stream=stream)
    ws1, ws2 = bsa.alloc_workspace(meta, dev), bsa.alloc_workspace(meta2, dev)
    torch.cuda.synchronize(dev)
    flop = computed_blocks(meta_to_numpy(meta)) * flop_per_tile(wl.D)
    f1, m1 = time_forward(dw, meta, err, stream, ws1)
    f2, m2 = time_forward(dw2, meta2, err, stream, ws2)
    return {"per_tile": {"fwd_ms": f1, "meta_ms": m1, "tflops": flop / (f1 * 1e-3) / 1e12,
                         "list_entries": int(meta.full_idx.numel())},
            "blocks_256x256": {"fwd_ms": f2, "meta_ms": m2, "tflops": flop / (f2 * 1e-3) / 1e12,
                               "frac": flop / (f2 * 1e-3) / 1e12 / peak,
                               "list_entries": int(meta2.full_idx.numel())},
            "note": "same inputs and outputs; FLOP of the 128 x 128 tiles computed"}


def oracle_timing(cpu_seconds):
    """The oracle (fp64, plain C) as it stands, on the host cores: the metadata
    oracle against nothing but the clock on every config; the forward oracle over
    whole configs 1-3 (measured) and configs 4-5 (extrapolated from a sample of
    whole Q tiles of head 0 at the sampled rate), with all threads and with one."""
    import numpy as np
    import oracle
    from workloads import make_workload
    threads = oracle.default_threads()
    res = {"threads": threads, "configs": {}}
    sample_s = max(2.0, cpu_seconds / 4)
    for cfg in (1, 2, 3, 4, 5):
        wl = make_workload(cfg)
        q, k, v = wl.qkv()
        t0 = time.perf_counter()
        meta = oracle.build_meta(wl, threads=threads)
        meta_s = time.perf_counter() - t0
        cnt = int(meta["full_cnt"].sum() + meta["mask_cnt"].sum())
        flop = cnt * flop_per_tile(wl.D)
        e = {"meta_oracle_s": meta_s, "computed_tiles": cnt, "flop": flop}
        if cfg <= 3:
            t0 = time.perf_counter()
            oracle.fwd(wl, q, k, v, meta, threads=threads)
            fwd_s = time.perf_counter() - t0
            e.update(fwd_oracle_s=fwd_s, fwd_oracle_tflops=flop / fwd_s / 1e12,
                     fwd_oracle_kind="measured, whole config")
        else:
            rate, _, desc = cpu_baseline(wl, q, k, v, sample_s, threads=threads)
            e.update(fwd_oracle_s=flop / (rate * 1e12), fwd_oracle_tflops=rate,
                     fwd_oracle_kind="extrapolated from a sample: " + desc)
        if cfg <= 2:
            t0 = time.perf_counter()
            oracle.fwd(wl, q, k, v, meta, threads=1)
            one_s = time.perf_counter() - t0
            e.update(fwd_oracle_1thread_s=one_s, fwd_oracle_1thread_tflops=flop / one_s / 1e12,
                     fwd_oracle_1thread_kind="measured, whole config")
        else:
            rate1, _, desc1 = cpu_baseline(wl, q, k, v, sample_s / 2, threads=1)
            e.update(fwd_oracle_1thread_s=flop / (rate1 * 1e12), fwd_oracle_1thread_tflops=rate1,
                     fwd_oracle_1thread_kind="extrapolated from a sample: " + desc1)
        res["configs"][str(cfg)] = e
        del q, k, v, meta
    return res


def workload_config(wl, blocks, ws):
    """The `config` object of both arms: the workload, its computed tiles and FLOP."""
    import numpy as np
    q_bytes = 2 * int(np.prod(wl.q_shape()))
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "S": int(wl.seqlens_q[0]), "D": wl.D,
            "tile": "128x128", "computed_tiles": int(blocks),
            "flop_per_step": int(blocks) * flop_per_tile(wl.D),
            "step": "metadata kernel + attention kernel",
            "l2": "inputs larger than L2 (Q/K/V %.2f GB vs 129 MB)" % (3 * q_bytes / 1e9),
            "parallelism": f"replicas x{ws}"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from workloads import make_workload
    wl = make_workload(args.config)
    q, k, v = wl.qkv()
    ref_meta = oracle.build_meta(wl)
    blocks = int(ref_meta["full_cnt"].sum() + ref_meta["mask_cnt"].sum())
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(wl, q, k, v, per_step)
    vals = []
    t0 = time.perf_counter()
    threads = oracle.default_threads()
    desc = ""
    for _ in range(args.steps):
        val, threads, desc = cpu_baseline(wl, q, k, v, per_step)
        vals.append(val)
    wall = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall * 1e3 / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, blocks, ws),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_native(args):
    import numpy as np
    import torch

    import block_sparse_flashattention_gb300 as bsa
    from workloads.device import DeviceWorkload, meta_to_numpy, computed_blocks
    from workloads import make_workload

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    wl = make_workload(args.config)
    if args.heads:
        from workloads.configs import with_heads
        wl = with_heads(wl, args.heads)
    # inputs in pinned host memory (the e2e leg copies them every step)
    pin = dict(pin_memory=True)
    hq = torch.empty(wl.q_shape(), dtype=torch.int16, **pin)
    hk = torch.empty(wl.k_shape(), dtype=torch.int16, **pin)
    hv = torch.empty(wl.k_shape(), dtype=torch.int16, **pin)
    wl.fill("q", hq.data_ptr())
    wl.fill("k", hk.data_ptr())
    wl.fill("v", hv.data_ptr())
    hmap = torch.from_numpy(np.ascontiguousarray(wl.block_map)).pin_memory()
    hvl = (torch.from_numpy(np.ascontiguousarray(wl.kv_valid_len)).pin_memory()
           if wl.kv_valid_len is not None else None)

    dw = DeviceWorkload(wl, dev, qkv=False)
    dw.q = hq.to(dev).view(torch.bfloat16)
    dw.k = hk.to(dev).view(torch.bfloat16)
    dw.v = hv.to(dev).view(torch.bfloat16)
    meta = dw.alloc_meta()
    out = torch.empty_like(dw.q)
    sq, sk = dw.seqlens()
    lse = torch.empty((wl.H, wl.rows_q) if wl.varlen else (wl.B, wl.H, sq), dtype=torch.float32,
                      device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sched_ws = bsa.alloc_workspace(meta, dev)   # scheduling workspace, allocated once

    def step():
        dw.build_meta(meta, err_flag=err)
        dw.forward(meta, out=out, lse=lse, err_flag=err, workspace=sched_ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())}")
    blocks = computed_blocks(meta_to_numpy(meta))
    flop_step = blocks * flop_per_tile(wl.D)

    # ---------------------------------------------------------- timed region
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_index_for_smi(torch, dev))
    time.sleep(0.5)   # the sampler is running before the timed region starts
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        dw.build_meta(meta, err_flag=err)
        ev[i][1].record(stream)
        dw.forward(meta, out=out, lse=lse, err_flag=err, workspace=sched_ws)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if pg:
        pg.barrier()
    total_ms = t_start.elapsed_time(t_end)
    meta_ms = [a.elapsed_time(b) for a, b, _ in ev]
    fwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(pg, total_ms, dev)
    value = whole_job_tflops(ws, flop_step, K, total_ms)

    # ------------------------------------------------------- end-to-end leg
    # Every step copies its inputs in from pinned host memory and its O / LSE back
    # out, through the public API on explicit streams, pipelined the way a
    # serving loop would run it: two device buffer sets, host->device copies on
    # one stream, compute on another, device->host copies on a third, so step
    # i's compute overlaps step i+1's copy in and step i-1's copy out.  (Spreading
    # the copy-in over three streams measured no faster: the host link, not one
    # copy engine, bounds it: ~212 GB/s host-to-device alone, ~157 GB/s each way
    # with both directions busy, as measured.)
    import copy as _copy
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    slots = [dw, _copy.copy(dw)]
    slots[1].q = torch.empty_like(dw.q)
    slots[1].k = torch.empty_like(dw.k)
    slots[1].v = torch.empty_like(dw.v)
    slots[1].block_map = torch.empty_like(dw.block_map)
    slots[1].vl = torch.empty_like(dw.vl) if dw.vl is not None else None
    outs, lses = [out, torch.empty_like(out)], [lse, torch.empty_like(lse)]
    h_outs = [torch.empty(out.shape, dtype=torch.int16, pin_memory=True) for _ in range(2)]
    h_lses = [torch.empty(lse.shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        j = i & 1
        d = slots[j]
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev_cmp[j])      # step i-2 has finished reading slot j
            d.q.view(torch.int16).copy_(hq, non_blocking=True)
            d.k.view(torch.int16).copy_(hk, non_blocking=True)
            d.v.view(torch.int16).copy_(hv, non_blocking=True)
            d.block_map.copy_(hmap, non_blocking=True)
            if d.vl is not None:
                d.vl.copy_(hvl, non_blocking=True)
            ev_in[j].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[j])
            if used[j]:
                s_cmp.wait_event(ev_out[j])     # step i-2's O / LSE have been copied out
            d.build_meta(meta, err_flag=err, stream=s_cmp)
            d.forward(meta, out=outs[j], lse=lses[j], err_flag=err, workspace=sched_ws, stream=s_cmp)
            ev_cmp[j].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[j])
            h_outs[j].copy_(outs[j].view(torch.int16), non_blocking=True)
            h_lses[j].copy_(lses[j], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_stream(s_in)
    s_out.wait_stream(s_in)
    for i in range(K):
        e2e_step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1), dev)
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2 + hmap.numel() + (
        hvl.numel() * 4 if hvl is not None else 0)
    d2h = out.numel() * 2 + lse.numel() * 4
    e2e_value = whole_job_tflops(ws, flop_step, K, e2e_ms)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())}")
    meta_formats = time_meta_formats(wl, dw, meta, err, stream) if not args.no_meta_formats else None
    proxy_ab = time_proxy(wl, dw, err, stream) if not args.no_meta_formats else None
    bwd = time_bwd(wl, dw, meta, out, lse, err, stream, flop_step) if not args.no_bwd else None
    peaks, peak_src = measured_peaks()
    others = [c for c in (3, 5) if c != args.config]
    cfg_lines = (per_config(others, dev, float(peaks["bf16_tflops"]), stream)
                 if not args.no_per_config and not args.heads else None)
    blocks_ab = (time_sparse_blocks(wl, dw, meta, dev, stream, float(peaks["bf16_tflops"]))
                 if "logical_map" in wl.extra and not args.heads and not args.no_per_config else None)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    fwd_mean = statistics.mean(fwd_ms)
    achieved = flop_step / (fwd_mean * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = None
    prof = os.path.join(ROOT, "profiles", "bsattn_fwd_traffic.json")
    if os.path.exists(prof):
        # the DRAM counters count only while the kernel source is the one profiled
        import hashlib
        src = os.path.join(ROOT, "block_sparse_flashattention_gb300", "csrc", "bsattn_fwd.cu")
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        try:
            with open(prof) as f:
                tr = json.load(f)
            if tr.get("workload") == wl.name and tr.get("kernel_sha256_prefix") == sha:
                traffic = tr.get("bytes_per_launch")
        except (OSError, ValueError):
            traffic = None
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        q_np = hq.numpy().view(np.uint16)
        k_np = hk.numpy().view(np.uint16)
        v_np = hv.numpy().view(np.uint16)
        cval, cores, desc = cpu_baseline(wl, q_np, k_np, v_np, args.cpu_seconds)
        cval1, _, desc1 = cpu_baseline(wl, q_np, k_np, v_np, args.cpu_seconds / 3, threads=1)
        cpu = {"value": cval, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "cores_1": {"value": cval1, "unit": UNIT, "cores": 1, "sample": desc1}}
        if not args.no_oracle_timing:
            cpu["oracle_timing"] = oracle_timing(args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, blocks, ws),
        "fwd_ms": fwd_mean, "meta_ms": statistics.mean(meta_ms),
        "fwd_tflops": achieved, "frac_of_peak_step": value / ws / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 dense burst (MEASURED_PEAKS.json)",
                     "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained",
                                                                      peak))},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / K,
                "pipeline": "copy-in, compute and copy-out on three streams, two buffer sets"},
        "meta_formats": meta_formats,
        "proxy_ab": proxy_ab,
        "bwd": bwd if bwd is None or "ms" not in bwd else dict(
            bwd, frac=bwd["tflops"] / peak,
            frac_of_sustained=bwd["tflops"] / float(peaks.get("bf16_tflops_sustained", peak))),
        "per_config": cfg_lines,
        "sparse_blocks": blocks_ab,
        "gpu_launches": K * (2 + (1 if wl.varlen else 0) + (1 if sched_ws is not None else 0)),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
