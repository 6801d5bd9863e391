#!/usr/bin/env python3
"""Throughput of LUT-driven block-sparse attention forward on GB300.

One step = the whole hot path over one batch of the headline workload
(b=2, h=32, s=16384, d=128, fp16, non-causal, BLKQ=BLKK=64, simthreshd1=0.001):
sparge_block_map (pool + similarity + pooled-score top-k -> LUT) followed by
sparse_fmha_fwd over the selected tiles.  Inputs (Q, K, V: 805 MB) are larger
than the 129 MB L2, so no flush is needed between steps.

Metric: effective TFLOP/s = (selected tiles x 4 * 64 * 64 * d) / step time,
plus the speedup over this library's own dense FMHA (no LUT, the 128-row
tile kernel: the fastest dense attention this library has) at the same shape.  `--topk` picks the step's topk
(default 0.4); the sweep over {0.1, 0.2, 0.4, 0.6, 1.0} is reported alongside,
with the q-block pair path (lut_pair_union + sparse_fmha_fwd_pairs) next to
the 64-row kernel the step uses.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own batch on its own GPU (no
collective on the data path); value = all ranks' work / the slowest rank.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective TFLOP/s & speedup vs own dense FMHA, b2 h32 s16k d128 per topk"
FLOP_PER_TILE = 4 * 64 * 64 * 128  # QK^T and PV of one selected 64x64 tile at d = 128
TOPKS = (0.1, 0.2, 0.4, 0.6, 1.0)

# DRAM bytes (read + written) per launch of the sparse FMHA kernel at the
# headline workload, from one ncu capture, keyed by the sha256 prefix of the
# kernel source the capture ran; a kernel edited since reports traffic = null.
NCU_TRAFFIC = {
    "e3db23bf8f9d04b6": 1070720512,  # 814.50 MB read + 256.22 MB written
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--topk", type=float, default=0.4)
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the causal-GQA prefill and sparse-decode measurements")
    p.add_argument("--decode-only", action="store_true",
                   help="only the sparse-decode measurement (a small command for profiling it)")
    p.add_argument("--causal-gqa-only", action="store_true",
                   help="only the causal GQA measurement (a small command for profiling it)")
    p.add_argument("--small", action="store_true",
                   help="b1 h16 s16384 d128 (Q, K, V 201 MB: still larger than L2) with every "
                        "leg but the step, the dense runs and the pair path off: a small case "
                        "of the same kernels for profiler captures, not a bench number")
    args = p.parse_args()
    if args.small:
        args.no_sweep = args.no_e2e = args.no_cpu = args.no_extra = True
    return args


def headline_config(cfg, topk, small=False):
    """The `config` object of the JSON line (the same for both arms)."""
    in_mb = cfg.b * (cfg.hq + 2 * cfg.hk) * cfg.s * cfg.d * 2 / 1e6
    return {"workload": f"b{cfg.b} h{cfg.hq} s{cfg.s} d{cfg.d} fp16 non-causal, BLKQ=BLKK=64, "
                        f"topk={topk}, simthreshd1=0.001"
                        + (" (small profiling case)" if small else ""),
            "b": cfg.b, "h": cfg.hq, "s": cfg.s, "d": cfg.d, "topk": topk,
            "l2": f"inputs ({in_mb:.0f} MB) larger than L2; no flush"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_config(cfg, rank: int):
    """Each rank runs its own independent batch: the same workload shape with
    a per-rank seed (rank 0 keeps the base seed)."""
    return cfg.replace(seed=cfg.seed + 7919 * rank)


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The slowest rank's time (the job finishes when the last rank does)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash():
    path = os.path.join(ROOT, "fmha_block_map_gb300", "csrc", "fmha_tc.cu")
    try:
        return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    except OSError:
        return None


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------


def run_ours(args):
    import numpy as np
    import torch

    import fmha_block_map_gb300 as fbm
    import synth
    from fmha_block_map_gb300 import build as fbuild

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    fbuild.build()
    fbm.lib()
    cfg = rank_config(synth.C3.replace(topk=args.topk), rank)
    if args.small:
        cfg = cfg.replace(b=1, hq=16, hk=16)
    x = synth.prefill(cfg)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.float16).cuda()
    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    stream = torch.cuda.current_stream()
    ws = torch.empty(fbm.block_map_workspace_bytes(cfg.b, cfg.hq, cfg.hk, cfg.s, cfg.d),
                     dtype=torch.uint8, device="cuda")
    nq = cfg.nq
    lut = torch.empty((cfg.b, cfg.hq, nq, nq), dtype=torch.int32, device="cuda")
    cnt = torch.empty((cfg.b, cfg.hq, nq), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()

    def block_map(topk, smooth_k=False):
        fbm.sparge_block_map(q, k, topk=topk, simthreshd1=cfg.simthreshd1, scale=cfg.scale,
                             lut=lut, lut_count=cnt, workspace=ws, smooth_k=smooth_k)

    def attn(dense=False):
        fbm.sparse_fmha_fwd(q, k, v, None if dense else lut, None if dense else cnt,
                            scale=cfg.scale, out=out)

    # 128-row tiles over q-block pairs: the dense attention of this library at
    # full tensor-core rate (the speedup denominator), and the sparse pair path
    npq = (nq + 1) // 2
    plut = torch.empty((cfg.b, cfg.hq, npq, nq), dtype=torch.int32, device="cuda")
    pcnt = torch.empty((cfg.b, cfg.hq, npq), dtype=torch.int32, device="cuda")

    def attn_pairs(dense=False):
        fbm.sparse_fmha_fwd_pairs(q, k, v, None if dense else plut, None if dense else pcnt,
                                  scale=cfg.scale, out=out)

    def overlap_pair_gain():
        """(|A| + |B|) / |A u B| summed over q-block pairs chosen by LUT
        overlap within each head: each q block in order takes its unmatched
        partner of largest overlap (greedy; a statistic, not a kernel path)."""
        m = torch.zeros((cfg.b * cfg.hq, nq, nq + 1), dtype=torch.float32, device="cuda")
        ar = torch.arange(nq, device="cuda")
        idx = torch.where(ar[None, None, :] < cnt.view(-1, nq, 1), lut.view(-1, nq, nq).long(),
                          torch.full_like(lut.view(-1, nq, nq).long(), nq))
        m.scatter_(2, idx, 1.0)
        m = m[:, :, :nq]
        ov = torch.bmm(m, m.transpose(1, 2)).cpu().numpy()
        sizes = cnt.view(-1, nq).cpu().numpy().astype(np.int64)
        tot = uni = 0
        for hh in range(ov.shape[0]):
            o = ov[hh]
            free = np.ones(nq, dtype=bool)
            for i in range(nq):
                if not free[i]:
                    continue
                free[i] = False
                cand = np.where(free, o[i], -1.0)
                j = int(cand.argmax())
                if cand[j] < 0:  # i is left alone (odd count)
                    tot += sizes[hh, i]
                    uni += sizes[hh, i]
                    continue
                free[j] = False
                tot += sizes[hh, i] + sizes[hh, j]
                uni += sizes[hh, i] + sizes[hh, j] - int(o[i, j])
        return round(tot / uni, 3) if uni else None

    def timed(fn, steps, warm):
        for _ in range(warm):
            fn()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / steps

    def timed_local(fn, steps, warm):
        # for the rank-0-only measurements: no collective (the other ranks are
        # not there to meet it)
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    # ---- the timed step: block map + sparse attention, per-kernel events
    for _ in range(args.warmup):
        block_map(args.topk)
        attn()
    barrier()
    sampler = ClockSampler(local)
    sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    t0.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        block_map(args.topk)
        ev[s][1].record(stream)
        attn()
        ev[s][2].record(stream)
    t1.record(stream)
    barrier()
    clocks = sampler.stop()
    step_ms = t0.elapsed_time(t1) / args.steps
    bm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    at_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    tiles = int(cnt.sum().item())
    assert fbm.get_error() == 0
    flops = tiles * FLOP_PER_TILE
    step_ms = max_over_ranks(step_ms, world, device="cuda")
    value = flops * world / (step_ms * 1e-3) / 1e12

    # ---- the block map with K smoothing (one more K read), dense FMHA, topk sweep
    smooth_ms = timed(lambda: block_map(args.topk, smooth_k=True), 5, 1)
    # the same call replayed from a CUDA graph (20 calls per replay): no host
    # launch gaps between its three kernels or between calls
    bm_graph_ms = _graph_ms(lambda: block_map(args.topk), reps=20, warm=3)
    block_map(args.topk)
    dense64_ms = timed(lambda: attn(dense=True), max(2, args.steps // 10), 1)
    dense_ms = timed(lambda: attn_pairs(dense=True), max(2, args.steps // 10), 1)
    if args.small:
        # one sparse launch of the pair path at the step's topk, for profiler captures
        fbm.lut_pair_union(lut, cnt, nq, pair_lut=plut, pair_count=pcnt)
        attn_pairs()
    sweep = []
    if not args.no_sweep:
        for tk in TOPKS:
            block_map(tk)
            fbm.lut_pair_union(lut, cnt, nq, pair_lut=plut, pair_count=pcnt)
            torch.cuda.synchronize()
            tl = int(cnt.sum().item())
            ul = int(pcnt.sum().item())
            bm = timed(lambda: block_map(tk), 5, 1)
            a = timed(lambda: attn(), max(2, args.steps // 10), 1)
            un = timed(lambda: fbm.lut_pair_union(lut, cnt, nq, pair_lut=plut, pair_count=pcnt),
                       5, 1)
            ap = timed(lambda: attn_pairs(), max(2, args.steps // 10), 1)
            sweep.append({"topk": tk, "selected_tiles": tl, "block_map_ms": round(bm, 4),
                          "attn_ms": round(a, 4),
                          "eff_tflops_attn": round(tl * FLOP_PER_TILE / (a * 1e-3) / 1e12, 1),
                          "eff_tflops_step": round(tl * FLOP_PER_TILE / ((a + bm) * 1e-3) / 1e12, 1),
                          "speedup_vs_dense_attn": round(dense_ms / a, 3),
                          "speedup_vs_dense_step": round(dense_ms / (a + bm), 3),
                          # q-block pairs: (|A| + |B|) / |A u B| over adjacent q blocks,
                          # and over pairs chosen by LUT overlap within the head
                          "pair_union_gain": round(tl / ul, 3) if ul else None,
                          "pair_union_gain_by_overlap": overlap_pair_gain(),
                          "pairs_attn_ms": round(ap, 4), "pair_union_ms": round(un, 4),
                          "pairs_eff_tflops_attn": round(tl * FLOP_PER_TILE / (ap * 1e-3) / 1e12, 1)})
        block_map(args.topk)

    # ---- context parallelism over kv-block ranges, two ranks emulated one after
    # the other on this GPU: each rank's LUT shard + fp32 partial, then the combine
    cp_res = None
    if rank == 0 and not args.no_extra:
        from fmha_block_map_gb300 import cp

        bounds = cp.kv_shard_bounds(cfg.nq, 2)
        shards = []
        for lo, hi in bounds:
            r0, r1 = cp.shard_rows(cfg.s, lo, hi)
            shards.append((k[:, :, r0:r1].contiguous(), v[:, :, r0:r1].contiguous(), lo, hi))
        o_all = torch.empty((2,) + tuple(out.shape), dtype=torch.float32, device="cuda")
        l_all = torch.empty((2,) + tuple(out.shape[:-1]), dtype=torch.float32, device="cuda")

        def cp_step():
            for r, (ks, vs, lo, hi) in enumerate(shards):
                cp.rank_partial(q, ks, vs, lut, cnt, lo, hi, scale=cfg.scale, o_slot=o_all[r],
                                lse_slot=l_all[r])
            fbm.attn_combine(o_all, l_all, out_dtype=q.dtype, out=out)

        cp_ms = timed_local(cp_step, 5, 1)
        comb_ms = timed_local(lambda: fbm.attn_combine(o_all, l_all, out_dtype=q.dtype, out=out),
                              5, 1)
        cp_res = {"ranks": 2, "emulated": "both ranks on one GPU, one after the other",
                  "ms": round(cp_ms, 4), "combine_ms": round(comb_ms, 4),
                  "eff_tflops": round(flops / (cp_ms * 1e-3) / 1e12, 1),
                  "partial_kernel": "tcgen05 (fp32 partial output)"}
        del shards, o_all, l_all

    # ---- per-Q-tile PV skip: the same step's attention with pv_threshold set
    pv_res = None
    if rank == 0 and not args.no_extra:
        pv_res = []
        for tau in (2.0, 6.0):
            ms = timed_local(lambda: fbm.sparse_fmha_fwd(q, k, v, lut, cnt, scale=cfg.scale,
                                                         out=out, pv_threshold=tau), 5, 1)
            pv_res.append({"pv_threshold": tau, "attn_ms": round(ms, 4),
                           "vs_no_skip": round(at_ms / ms, 3),
                           "eff_tflops_attn": round(flops / (ms * 1e-3) / 1e12, 1)})

    # ---- end to end through the public API with host buffers: every step copies
    # its Q, K, V from pinned host memory and reads its O back.  Double buffers;
    # the uploads and the read-backs run on two copy streams (the host link is
    # full duplex): the upload of step i + 1 and the read-back of step i - 1
    # overlap the compute of step i.
    e2e = None
    if not args.no_e2e:
        attn()  # the device-resident sparse result the end-to-end output must equal
        torch.cuda.synchronize()
        host_in = [[t.cpu().pin_memory() for t in (q, k, v)] for _ in range(2)]
        host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        dev_in = [[torch.empty_like(t) for t in (q, k, v)] for _ in range(2)]
        dev_out = [torch.empty_like(out) for _ in range(2)]
        luts = [torch.empty_like(lut) for _ in range(2)]
        cnts = [torch.empty_like(cnt) for _ in range(2)]
        wss = [torch.empty_like(ws) for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        comp_s = torch.cuda.current_stream()
        ev = lambda: torch.cuda.Event()
        loaded = [ev(), ev()]
        computed = [ev(), ev()]
        drained = [ev(), ev()]

        def upload(i):
            b = i % 2
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(computed[b])  # the compute of step i - 2 has read these inputs
                for d, h in zip(dev_in[b], host_in[b]):
                    d.copy_(h, non_blocking=True)
                loaded[b].record(h2d_s)

        def run_steps(n):
            upload(0)
            for i in range(n):
                b = i % 2
                if i + 1 < n:
                    upload(i + 1)
                comp_s.wait_event(loaded[b])
                comp_s.wait_event(drained[b])  # the read-back of step i - 2 has read dev_out[b]
                dq, dk, dv_ = dev_in[b]
                fbm.sparge_block_map(dq, dk, topk=args.topk, simthreshd1=cfg.simthreshd1,
                                     scale=cfg.scale, lut=luts[b], lut_count=cnts[b],
                                     workspace=wss[b], stream=comp_s)
                fbm.sparse_fmha_fwd(dq, dk, dv_, luts[b], cnts[b], scale=cfg.scale,
                                    out=dev_out[b], stream=comp_s)
                computed[b].record(comp_s)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(computed[b])
                    host_out[b].copy_(dev_out[b], non_blocking=True)
                    drained[b].record(d2h_s)
            torch.cuda.synchronize()

        run_steps(2)  # warm-up
        n_e2e = max(4, args.steps // 2)  # the pipeline fill (first upload) is paid once
        barrier()
        w0 = time.perf_counter()
        run_steps(n_e2e)
        barrier()
        e2e_ms = (time.perf_counter() - w0) * 1e3 / n_e2e
        assert torch.equal(host_out[(n_e2e - 1) % 2], out.cpu())
        h2d = 3 * q.numel() * q.element_size()
        d2h = out.numel() * out.element_size()
        e2e = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "timing": "host wall clock around synchronised steps; the H2D of step i+1 and "
                         "the D2H of step i-1 (two copy streams) overlap the compute of step i"}

    peaks, peak_kind = load_peaks()
    # the FMHA is timed on its own (tens of ms of launches, not a seconds-long
    # loop): the burst peak is its denominator; the sustained one is reported too
    peak = peaks.get("bf16_tflops", 1900.0)
    peak_sus = peaks.get("bf16_tflops_sustained", 1700.0)
    achieved = flops / (at_ms * 1e-3) / 1e12
    kind = fbm.fmha_kernel_kind(torch.float16, 128, 128, 1, cfg.s, cfg.s)
    src_hash = kernel_source_hash()
    # the stored figure is for the headline workload's launch
    traffic = None if args.small else NCU_TRAFFIC.get(src_hash)
    # block map algorithmic bytes: Q and K read once, pooled means + sims written
    # and read back once, the -1-padded LUT rows and the counts written
    pooled = (cfg.b * cfg.hq * nq + cfg.b * cfg.hk * nq) * (cfg.d + 1) * 4
    bm_bytes = (q.numel() + k.numel()) * 2 + 2 * pooled + lut.numel() * 4 + cnt.numel() * 4

    # ---- fp8 (e4m3) Q / K: block quantisation of Q and K, then the attention
    # over the quantised scores (same LUT; V, P and O 16-bit)
    fp8_res = None
    if rank == 0 and not args.no_extra:
        q8, qsc = fbm.quantize_e4m3_blocks(q)
        k8, ksc = fbm.quantize_e4m3_blocks(k)
        quant_ms = timed_local(lambda: (fbm.quantize_e4m3_blocks(q, codes=q8, scales=qsc),
                                        fbm.quantize_e4m3_blocks(k, codes=k8, scales=ksc)), 5, 1)
        a8_ms = timed_local(lambda: fbm.sparse_fmha_fwd_fp8(q8, qsc, k8, ksc, v, lut, cnt,
                                                            scale=cfg.scale, out=out), 5, 1)
        qbytes = (q.numel() + k.numel()) * (2 + 1) + (qsc.numel() + ksc.numel()) * 4
        # the quantisation fused into the block map's pooling pass: the fp8
        # step is sparge_block_map_e4m3 + the fp8 attention
        fused_ms = timed_local(lambda: fbm.sparge_block_map_e4m3(
            q, k, topk=args.topk, simthreshd1=cfg.simthreshd1, scale=cfg.scale, lut=lut,
            lut_count=cnt, workspace=ws, q8=q8, q_scale=qsc, k8=k8, k_scale=ksc), 5, 1)
        fp8_res = {"fused_block_map_ms": round(fused_ms, 4),
                   "fused_quant_cost_ms": round(fused_ms - bm_ms, 4),
                   "eff_tflops_fused_step": round(flops / ((a8_ms + fused_ms) * 1e-3) / 1e12, 1),
                   "quant_ms": round(quant_ms, 4),
                   "quant_GB_s": round(qbytes / (quant_ms * 1e-3) / 1e9, 1),
                   "attn_ms": round(a8_ms, 4), "vs_16bit_attn": round(at_ms / a8_ms, 3),
                   "eff_tflops_attn": round(flops / (a8_ms * 1e-3) / 1e12, 1),
                   "eff_tflops_quant_plus_attn": round(flops / ((a8_ms + quant_ms) * 1e-3) / 1e12,
                                                       1)}
        del q8, k8, qsc, ksc

    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded centroid-plus-noise blocks, 25% diffuse)",
        "config": headline_config(cfg, args.topk, args.small),
        "speedup_vs_dense": {"dense_attn_ms": round(dense_ms, 4),
                             "dense_kernel": "sparse_fmha_fwd_pairs, no LUT (128-row tiles)",
                             "dense_eff_tflops": round(4 * cfg.b * cfg.hq * cfg.s * cfg.s * cfg.d
                                                       / (dense_ms * 1e-3) / 1e12, 1),
                             "dense_64row_attn_ms": round(dense64_ms, 4),
                             "vs_attn": round(dense_ms / at_ms, 3),
                             "vs_step": round(dense_ms / step_ms, 3)},
        "block_map": {"ms": round(bm_ms, 4), "algorithmic_bytes": bm_bytes,
                      "GB_s": round(bm_bytes / (bm_ms * 1e-3) / 1e9, 1),
                      "frac_hbm": round(bm_bytes / (bm_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                      "share_of_step": round(bm_ms / step_ms, 3),
                      "smooth_k_ms": round(smooth_ms, 4),
                      "graph_ms": round(bm_graph_ms, 4),
                      "graph_frac_hbm": round(bm_bytes / (bm_graph_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)},
        "roofline": {"kernel": "sparse_fmha_fwd (k_fmha_tc, tcgen05)", "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} bf16 burst (fp16 tensor rate = bf16)",
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_sustained": peak_sus,
                     "frac_of_sustained": round(achieved / peak_sus, 4),
                     "traffic": traffic, "selected_tiles": tiles,
                     "flop_per_tile": FLOP_PER_TILE, "attn_ms": round(at_ms, 4)},
        "sweep": sweep,
        "context_parallel": cp_res,
        "pv_skip": pv_res,
        "fp8_qk": fp8_res,
        "e2e": e2e,
        "clocks": clocks,
        # per step: k_pool_sim, k_pooled_scores, k_select and k_fmha_tc
        "gpu_launches": 4 * args.steps,
    }
    if rank == 0 and not args.no_extra:
        res["causal_gqa"] = measure_causal_gqa(peaks["hbm_gbs"], peak)
        res["decode"] = measure_decode(peaks["hbm_gbs"])
    if rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(cfg, x, args.topk)
        res["cpu_baselines"] = cpu_baselines()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return res if rank == 0 else None


# ----------------------------------------------------------------------------
# the other rows of the path, measured on their own workloads (not the step)
# ----------------------------------------------------------------------------


def _graph_ms(fn, reps=20, warm=3):
    """Device time of a short, launch-bound call: `reps` calls captured in one
    CUDA graph, the graph replayed (after `warm` eager calls) and timed with
    CUDA events, per call."""
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _events_ms(fn, steps, warm):
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def measure_causal_gqa(hbm_gbs, peak):
    """b=1, 32 query heads on 8 KV heads, s=32768, d=128, bf16, causal, sink,
    topk=0.2 of the causal-eligible blocks, LSE on."""
    import numpy as np
    import torch

    import fmha_block_map_gb300 as fbm
    import synth

    cfg = synth.C4
    x = synth.prefill(cfg)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    nq = cfg.nq
    ws = torch.empty(fbm.block_map_workspace_bytes(1, 32, 8, cfg.s, 128), dtype=torch.uint8,
                     device="cuda")
    lut = torch.empty((1, 32, nq, nq), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 32, nq), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((1, 32, cfg.s), dtype=torch.float32, device="cuda")
    bm = lambda: fbm.sparge_block_map(q, k, topk=cfg.topk, simthreshd1=cfg.simthreshd1,
                                      scale=cfg.scale, causal=True, attention_sink=True,
                                      lut=lut, lut_count=cnt, workspace=ws)
    at = lambda: fbm.sparse_fmha_fwd(q, k, v, lut, cnt, scale=cfg.scale, causal=True, out=out,
                                     lse=lse, return_lse=True)
    bm()
    torch.cuda.synchronize()
    tiles = int(cnt.sum().item())
    # 30 back-to-back calls: the host's start-up before the first launch is
    # then a small share of the timed span
    bm_ms = _events_ms(bm, 30, 3)
    bm_graph_ms = _graph_ms(bm, reps=20, warm=3)
    at_ms = _events_ms(at, 10, 3)
    bm_bytes = (q.numel() + k.numel()) * 2 + 2 * (32 * nq + 8 * nq) * 129 * 4 + lut.numel() * 4
    assert fbm.get_error() == 0
    return {"workload": "b1 hq32 hk8 s32768 d128 bf16 causal + sink, topk=0.2, LSE on",
            "selected_tiles": tiles, "block_map_ms": round(bm_ms, 4),
            "block_map_GB_s": round(bm_bytes / (bm_ms * 1e-3) / 1e9, 1),
            "block_map_frac_hbm": round(bm_bytes / (bm_ms * 1e-3) / 1e9 / hbm_gbs, 3),
            "block_map_graph_ms": round(bm_graph_ms, 4),
            "block_map_graph_frac_hbm": round(bm_bytes / (bm_graph_ms * 1e-3) / 1e9 / hbm_gbs, 3),
            "attn_ms": round(at_ms, 4),
            "attn_eff_tflops": round(tiles * FLOP_PER_TILE / (at_ms * 1e-3) / 1e12, 1),
            "attn_frac_peak": round(tiles * FLOP_PER_TILE / (at_ms * 1e-3) / 1e12 / peak, 4)}


def measure_decode(hbm_gbs, small=False):
    """64 queries x 16 heads on one 576-wide KV head, 2048 listed tokens each,
    65536-page cache (4.8 GB bf16): split-KV decode + LSE combine.  small:
    the same queries and list lengths over 128 pages per query (a 0.6 GB
    cache, still larger than L2), for profiler captures."""
    import numpy as np
    import torch

    import fmha_block_map_gb300 as fbm
    import synth

    cfg = synth.C5.replace(pages_per_query=128) if small else synth.C5
    inp = synth.decode(cfg)
    n_rows = cfg.n_pages * cfg.page
    cache = torch.empty((n_rows, cfg.d), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, n_rows, 1 << 18):
        r1 = min(n_rows, r0 + (1 << 18))
        cache[r0:r1] = synth.cache_rows_torch(cfg, r0, r1, "cuda")
    cache = cache.view(cfg.n_pages, cfg.page, cfg.d)
    q = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16).cuda()
    pt = torch.from_numpy(inp["page_table"]).cuda()
    ix = torch.from_numpy(inp["idx"]).cuda()
    res = []
    for S in (2, 4, 8):
        op = torch.empty((S, cfg.n_queries, cfg.hq, cfg.dv), dtype=torch.float32, device="cuda")
        lp = torch.empty((S, cfg.n_queries, cfg.hq), dtype=torch.float32, device="cuda")
        o = torch.empty((cfg.n_queries, cfg.hq, cfg.dv), dtype=torch.bfloat16, device="cuda")
        dec = lambda: fbm.sparse_decode_fwd(q, cache, pt, ix, dv=cfg.dv, scale=cfg.sm_scale,
                                            num_splits=S, o_partial=op, lse_partial=lp)
        comb = lambda: fbm.attn_combine(op, lp, out=o, return_lse=False)
        d_ms = _events_ms(dec, 20, 3)
        # a few µs of device work: timed inside a CUDA graph, or the host's
        # launch overhead would be measured instead
        c_ms = _graph_ms(comb, 20, 3)

        def dec_comb():
            dec()
            comb()

        # the pair as a decode step runs it (the combine a chained launch)
        p_ms = _events_ms(dec_comb, 20, 3)
        rows_bytes = cfg.n_queries * cfg.topk * cfg.d * 2
        part_bytes = S * cfg.n_queries * cfg.hq * (cfg.dv + 1) * 4
        d_bytes = rows_bytes + q.numel() * 2 + ix.numel() * 4 + part_bytes \
            + cfg.n_queries * cfg.topk * 4  # page-table entries looked up
        c_bytes = part_bytes + o.numel() * 2
        res.append({"splits": S, "decode_ms": round(d_ms, 4),
                    "decode_GB_s": round(d_bytes / (d_ms * 1e-3) / 1e9, 1),
                    "decode_frac_hbm": round(d_bytes / (d_ms * 1e-3) / 1e9 / hbm_gbs, 3),
                    "combine_ms": round(c_ms, 4),
                    "combine_GB_s": round(c_bytes / (c_ms * 1e-3) / 1e9, 1),
                    "decode_plus_combine_ms": round(p_ms, 4)})
    # the same calls replayed from CUDA graphs (20 per replay): no host launch
    # gaps.  After the eager legs, so that their launch order is unchanged.
    for r in res:
        S = r["splits"]
        op = torch.empty((S, cfg.n_queries, cfg.hq, cfg.dv), dtype=torch.float32, device="cuda")
        lp = torch.empty((S, cfg.n_queries, cfg.hq), dtype=torch.float32, device="cuda")
        o = torch.empty((cfg.n_queries, cfg.hq, cfg.dv), dtype=torch.bfloat16, device="cuda")

        def dec_g(S=S, op=op, lp=lp):
            fbm.sparse_decode_fwd(q, cache, pt, ix, dv=cfg.dv, scale=cfg.sm_scale, num_splits=S,
                                  o_partial=op, lse_partial=lp)

        def dec_comb_g(op=op, lp=lp, o=o):
            dec_g()
            fbm.attn_combine(op, lp, out=o, return_lse=False)

        dg_ms = _graph_ms(dec_g, 20, 3)
        pg_ms = _graph_ms(dec_comb_g, 20, 3)
        d_bytes = (cfg.n_queries * cfg.topk * cfg.d * 2 + q.numel() * 2 + ix.numel() * 4
                   + S * cfg.n_queries * cfg.hq * (cfg.dv + 1) * 4 + cfg.n_queries * cfg.topk * 4)
        r["decode_graph_ms"] = round(dg_ms, 4)
        r["decode_graph_frac_hbm"] = round(d_bytes / (dg_ms * 1e-3) / 1e9 / hbm_gbs, 3)
        r["decode_plus_combine_graph_ms"] = round(pg_ms, 4)
    assert fbm.get_error() == 0
    del cache
    torch.cuda.empty_cache()
    return {"workload": f"{cfg.n_queries} queries x {cfg.hq} heads, d={cfg.d} (V = first "
                        f"{cfg.dv}), {cfg.topk} tokens each, {cfg.n_pages} pages of {cfg.page} "
                        "rows, bf16" + (" (small profiling case)" if small else ""),
            "by_splits": res}


# ----------------------------------------------------------------------------
# the fp64 oracle on the host cores (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------


def cpu_baseline(cfg, x, topk, qblocks=None, heads=10):
    """The oracle as it stands on a bounded sample of the same workload: the
    block map of `heads` (batch, head) pairs, then sparse attention of
    `qblocks` q blocks of each (all of them by default: about 10 s of work
    for 10 heads on 16 Arm cores); effective TFLOP/s over the selected tiles of the
    sample, charging the block map in proportion to the q blocks done."""
    import numpy as np

    import oracle
    import synth

    units = [(0, h) for h in range(heads)]
    t0 = time.perf_counter()
    r = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, topk), None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, False, False,
                                dtype=cfg.dtype, heads=units)
    t_bm = time.perf_counter() - t0
    nqb = cfg.nq if qblocks is None else qblocks
    rng = np.random.default_rng(0)
    todo = [(b, h, int(i)) for b, h in units for i in rng.choice(cfg.nq, nqb, replace=False)]
    t0 = time.perf_counter()
    oracle.sparse_fmha(x["q"], x["k"], x["v"], r["lut"], r["count"], cfg.scale, False,
                       units=todo, dtype=cfg.dtype)
    t_at = time.perf_counter() - t0
    tiles = sum(int(r["count"][b, h, i]) for b, h, i in todo)
    t = t_at + t_bm * nqb / cfg.nq
    return {"value": round(tiles * FLOP_PER_TILE / t / 1e12, 6), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"block map of {heads} (batch, head), attention of {len(todo)} q blocks "
                      f"({tiles} selected tiles) at topk={topk}; {t_bm + t_at:.1f} s of CPU work"}


def _oracle_config_time(name, heads=None, qblocks=None):
    """Seconds the oracle takes on config `name` (C1, C2, C4: block map then
    attention; a (batch, head) / q-block sample when given) and the selected
    tiles it covered; C5: the decode of every query over its listed tokens."""
    import numpy as np

    import oracle
    import synth

    if name == "C5":
        cfg = synth.C5
        inp = synth.decode(cfg)
        t0 = time.perf_counter()
        rows = oracle.decode_rows(inp["page_table"], inp["idx"], cfg.page)
        qf = synth.bits_to_f64(inp["q"], "bf16")
        for c in range(cfg.n_queries):
            kv = synth.bits_to_f64(synth.cache_rows(cfg, rows[c]), "bf16")
            oracle.decode_attention(qf[c], kv, cfg.dv, cfg.sm_scale)
        return time.perf_counter() - t0, cfg.n_queries * cfg.topk
    cfg = synth.PREFILL_CONFIGS[name]
    x = synth.prefill(cfg)
    mode = "topk" if cfg.topk is not None else "cdf"
    ph = synth.per_head(cfg, cfg.topk if mode == "topk" else cfg.cdfthreshd)
    todo = heads or [(b, h) for b in range(cfg.b) for h in range(cfg.hq)]
    t0 = time.perf_counter()
    r = oracle.sparge_block_map(x["q"], x["k"], ph if mode == "topk" else None,
                                ph if mode == "cdf" else None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, cfg.causal,
                                cfg.attention_sink, dtype=cfg.dtype, heads=todo)
    rng = np.random.default_rng(0)
    units = [(b, h, int(i)) for b, h in todo
             for i in (range(cfg.nq) if qblocks is None
                       else rng.choice(cfg.nq, qblocks, replace=False))]
    oracle.sparse_fmha(x["q"], x["k"], x["v"], r["lut"], r["count"], cfg.scale, cfg.causal,
                       units=units, dtype=cfg.dtype)
    tiles = sum(int(r["count"][b, h, i]) for b, h, i in units)
    return time.perf_counter() - t0, tiles


def _oracle_c4_tiles():
    """Selected tiles of the whole C4 map (b1 hq32 s32768, topk 0.2 + sink),
    from the oracle's block map of every head (not timed)."""
    import oracle
    import synth

    cfg = synth.C4
    x = synth.prefill(cfg)
    r = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, cfg.topk), None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, cfg.causal,
                                cfg.attention_sink, dtype=cfg.dtype)
    return int(r["count"].sum())


def cpu_baselines():
    """The oracle's own costs beside the headline sample: full C1, C2 and C5
    runs on all host cores, C4 on a sample (2 heads, 16 q blocks each) with
    its full-config time extrapolated by selected tiles, and the headline
    sample again on one core (a child process with one BLAS / OpenMP
    thread)."""
    out = {"cores": os.cpu_count()}
    for name in ("C1", "C2", "C5"):
        t, units = _oracle_config_time(name)
        out[name] = {"seconds": round(t, 2), "full": True,
                     ("listed_tokens" if name == "C5" else "selected_tiles"): units}
    import synth

    t, tiles = _oracle_config_time("C4", heads=[(0, 0), (0, 17)], qblocks=16)
    full_tiles = _oracle_c4_tiles()
    out["C4"] = {"seconds": round(t, 2), "sample": "2 heads x 16 q blocks",
                 "sample_tiles": tiles,
                 "full_config_seconds_extrapolated": round(t * full_tiles / max(tiles, 1), 1)}
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench, synth; cfg = synth.C3; x = synth.prefill(cfg.replace(b=1, hq=2, hk=2)); "
            "print(json.dumps(bench.cpu_baseline(cfg, x, 0.4, qblocks=64, heads=2)))")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=600)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        one["cores"] = 1
        out["C3_one_core"] = one
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        out["C3_one_core"] = {"error": str(e)[:200]}
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import synth

    cfg = synth.C3.replace(topk=args.topk)
    x = synth.prefill(cfg.replace(b=1, hq=1, hk=1))
    for _ in range(args.warmup):
        cpu_baseline(cfg, x, args.topk, qblocks=4, heads=1)
    vals, t_all = [], time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(cfg, x, args.topk, qblocks=8, heads=1))
    t_all = time.perf_counter() - t_all
    v = round(statistics.mean(r["value"] for r in vals), 6)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_all / args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded centroid-plus-noise blocks, 25% diffuse)",
            "config": headline_config(synth.C3, args.topk),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": vals[0]["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.decode_only:
        import torch

        torch.cuda.set_device(0)
        print(json.dumps({"decode": measure_decode(load_peaks()[0]["hbm_gbs"], small=args.small)}))
        return
    if args.causal_gqa_only:
        import torch

        from fmha_block_map_gb300 import build as fbuild

        torch.cuda.set_device(0)
        fbuild.build()
        peaks = load_peaks()[0]
        print(json.dumps({"causal_gqa": measure_causal_gqa(peaks["hbm_gbs"],
                                                           peaks.get("bf16_tflops", 1900.0))}))
        return
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
