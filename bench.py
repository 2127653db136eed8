#!/usr/bin/env python3
"""Benchmark: paged KV store + GQA paged attention on GB300.

One step = one pass of the whole hot path over one batch: the metadata plan,
then for each of the 28 layers store_kv of the step's new K/V and the paged
attention (one fused kernel per layer, msg_paged_attention_store) over the
64-request decode batch (context U[512, 4096], page_size 1,
16 query / 8 KV heads, head_dim 128, bf16, 28 independent 300k-slot layer
pools, one shared page table).  The headline metric is decode KV-read GB/s
(algorithmic bytes: every needed K/V row once, q, out and page-table entries,
plus the store_kv rows) over the device time of the step.

Also printed, in the same JSON line:
  roofline      -- the decode kernel's achieved GB/s against the measured HBM peak,
                   timed with CUDA events around each launch in the timed region;
  e2e           -- the same metric through the C ABI with the step's inputs in
                   pinned host memory (H2D copies and the D2H of the outputs timed);
  extend        -- extend attention TFLOP/s on the 8-request extend batch;
  small_batch_graph -- an 8-request x 28-layer decode step, eager vs CUDA-graph replay;
  large_decode  -- 256 decode requests, page_size 16, pools at 90% of free HBM;
  long_mixed    -- 32 long decodes + 2 extends (page_size 64): each part alone and
                   the mixed call against the max() and sum() of the two bounds;
  chunked_prefill -- one 128-token tile over a 32,768-token prefix (8 work items):
                   the extend key split over every SM vs items taken whole;
  prologue      -- fused q/k RMSNorm + RoPE + store_kv over the extend batch's tokens;
  cpu_baseline  -- the fp64 oracle on the host cores, on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) each rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_gqa_store_gb300 import workload as wl  # noqa: E402

METRIC = "paged GQA attn: decode KV-read GB/s (% HBM peak); extend TFLOP/s"
KV_ROW = wl.HKV * wl.HEAD_DIM * 2            # bytes of one token's K (or V) row, one layer
QO_ROW = wl.HQ * wl.HEAD_DIM * 2             # bytes of one token's q (or out) row


def decode_attn_bytes(spec) -> int:
    """Algorithmic bytes of one layer's attention: K and V of every key once,
    q and out rows, one page-table entry per page read."""
    dev = spec.device_len
    pages = (dev + spec.page_size - 1) // spec.page_size
    return int(dev.sum() * 2 * KV_ROW + spec.total_q * 2 * QO_ROW + pages.sum() * 4)


def store_bytes(spec) -> int:
    return int(spec.total_q * 2 * KV_ROW * 2)   # read k,v rows + write them


def extend_flops(spec) -> float:
    """4 * D * Hq per unmasked (query, key) pair: 2 for Q.K^T, 2 for P.V."""
    c = spec.cached_len.astype(np.float64)
    e = spec.extend_len.astype(np.float64)
    pairs = (e * c + e * (e + 1) / 2).sum()
    return 4.0 * wl.HEAD_DIM * wl.HQ * pairs


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, only if the kernel
    source is unchanged since the counters were taken."""
    try:
        d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kernel]
        if d["source_hash"] != source_hash(d["sources"]):
            return None
        return d
    except Exception:
        return None


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Max of a per-rank value over all ranks (the slowest rank sets the step time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves its own batch's bytes in the (max) step time."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ our implementation
def run_ours(args, rank, world, dist):
    import torch
    import paged_kv_gqa_store_gb300 as msg

    msg.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()

    spec = wl.config_decode_28_layers()
    L = args.layers
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    pt, cached, ext, rows = (i32(spec.page_table), i32(spec.cached_len), i32(spec.extend_len),
                             i32(spec.req_rows))
    T, R = spec.total_q, spec.num_reqs
    qo = torch.zeros(R + 1, dtype=torch.int32, device=dev)
    loc = torch.zeros(T, dtype=torch.int64, device=dev)
    ws = torch.zeros(msg.msg_workspace_size(R, T), dtype=torch.uint8, device=dev)
    layers = [wl.device_tensors(spec, layer, device=dev) for layer in range(L)]
    outs = [torch.empty_like(t["q"]) for t in layers]
    flags = msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY
    attn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(L * args.steps)]

    def step(ev=None):
        msg.msg_plan(pt, cached, ext, T, spec.num_slots, ws, req_rows=rows, qo_indptr_out=qo,
                     out_loc_out=loc)
        for i, t in enumerate(layers):
            # store_kv of the step's new rows and the decode attention, in one kernel
            if ev is not None:
                ev[i][0].record(stream)
            msg.msg_paged_attention_store(t["q"], t["k_new"], t["v_new"], t["k_pool"],
                                          t["v_pool"], pt, cached, ext, qo, outs[i], ws,
                                          page_size=spec.page_size, req_rows=rows,
                                          max_kv_len=spec.max_kv_len, flags=flags)
            if ev is not None:
                ev[i][1].record(stream)

    launches_per_step = 2 + L                     # plan + token meta, store + decode per layer

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st, info = msg.msg_read_device_status(ws)
    if st != msg.MSG_OK:
        raise RuntimeError(f"device status after warm-up: {info}")

    clocks = ClockSampler(dev.index)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    # The step's kernels start their set-up while the previous kernel finishes
    # (programmatic dependent launch); an event between two launches would
    # serialise them, so the headline region has events only at its ends ...
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    # ... and the decode kernel's own launch time (roofline) comes from a second
    # timed pass with CUDA events around each of its launches.
    for k in range(args.steps):
        step(attn_ev[k * L:(k + 1) * L])
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), dist, dev) / args.steps

    bytes_layer = decode_attn_bytes(spec)
    bytes_step = L * (bytes_layer + store_bytes(spec))
    value = weak_scaling_gbs(bytes_step, world, ms)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in attn_ev)
    # the fused launch also writes the step's new K / V rows to the pool
    achieved = (bytes_layer + spec.total_q * 2 * KV_ROW) / (attn_ms * 1e-3) / 1e9
    traffic = ncu_traffic("decode_kernel")

    # ---- end to end through the C ABI from pinned host buffers
    if args.no_e2e:
        return finish_line(args, rank, world, spec, peaks, value, ms, achieved, attn_ms,
                           bytes_layer, bytes_step, traffic, launches_per_step, clk, None, dev, msg)
    # Each layer's q | k_new | v_new sit contiguously in one pinned host buffer
    # and one device buffer (the layer's tensors become views of it), the three
    # metadata arrays likewise, and the 28 outputs in one device buffer.  A copy
    # stream moves the inputs layer by layer ahead of the compute and reads each
    # group of 7 layers' outputs back as soon as they are computed; the timed
    # region runs from an event before the first copy to the compute stream's
    # wait on the last read-back.
    def stage(parts):
        nb = sum(x.numel() * x.element_size() for x in parts)
        dbuf = torch.empty(nb, dtype=torch.uint8, device=dev)
        views, off = [], 0
        for x in parts:
            n = x.numel() * x.element_size()
            v = dbuf[off:off + n].view(x.dtype).view(x.shape)
            v.copy_(x)
            views.append(v)
            off += n
        return dbuf, dbuf.cpu().pin_memory(), views
    dev_in, host_in = [], []
    for t in layers:
        dbuf, hbuf, (t["q"], t["k_new"], t["v_new"]) = stage([t["q"], t["k_new"], t["v_new"]])
        dev_in.append(dbuf)
        host_in.append(hbuf)
    meta_dev, meta_host, (cached, ext, rows) = stage([cached, ext, rows])
    out_dev = torch.empty((L,) + tuple(outs[0].shape), dtype=outs[0].dtype, device=dev)
    outs[:] = [out_dev[i] for i in range(L)]
    out_host = torch.empty_like(out_dev, device="cpu").pin_memory()
    h2d = meta_host.numel() + sum(h.numel() for h in host_in)
    d2h = out_host.numel() * out_host.element_size()
    group = 7
    cs = torch.cuda.Stream(device=dev)
    ev_start = torch.cuda.Event()
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_out = {i: torch.cuda.Event() for i in range(L) if (i + 1) % group == 0 or i == L - 1}
    ev_done = torch.cuda.Event()
    first_wait = min(3, L - 1)

    def e2e_step():
        ev_start.record(stream)
        cs.wait_event(ev_start)
        with torch.cuda.stream(cs):
            meta_dev.copy_(meta_host, non_blocking=True)
            for i in range(L):
                dev_in[i].copy_(host_in[i], non_blocking=True)
                ev_in[i].record(cs)
        stream.wait_event(ev_in[first_wait])
        msg.msg_plan(pt, cached, ext, T, spec.num_slots, ws, req_rows=rows, qo_indptr_out=qo,
                     out_loc_out=loc)
        for i, t in enumerate(layers):
            if i == first_wait + 1:
                stream.wait_event(ev_in[L - 1])
            msg.msg_paged_attention_store(t["q"], t["k_new"], t["v_new"], t["k_pool"],
                                          t["v_pool"], pt, cached, ext, qo, outs[i], ws,
                                          page_size=spec.page_size, req_rows=rows,
                                          max_kv_len=spec.max_kv_len, flags=flags)
            if i in ev_out:
                ev_out[i].record(stream)
        with torch.cuda.stream(cs):
            g0 = 0
            for i in sorted(ev_out):
                cs.wait_event(ev_out[i])
                out_host[g0:i + 1].copy_(out_dev[g0:i + 1], non_blocking=True)
                g0 = i + 1
            ev_done.record(cs)
        stream.wait_event(ev_done)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev) / args.steps
    if not torch.equal(out_host, out_dev.cpu()):
        raise RuntimeError("end-to-end leg: the outputs read back differ from the device's")
    e2e_value = weak_scaling_gbs(bytes_step, world, e2e_ms)
    e2e = {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)}
    del layers, outs, dev_in, host_in, out_dev, out_host
    return finish_line(args, rank, world, spec, peaks, value, ms, achieved, attn_ms, bytes_layer,
                       bytes_step, traffic, launches_per_step, clk, e2e, dev, msg)


def finish_line(args, rank, world, spec, peaks, value, ms, achieved, attn_ms, bytes_layer,
                bytes_step, traffic, launches_per_step, clk, e2e, dev, msg):
    import torch
    torch.cuda.empty_cache()
    R, L = spec.num_reqs, args.layers
    want_cpu = rank == 0 and world == 1 and not args.no_cpu
    args.cpu_samples = {} if want_cpu else None
    tiny = run_tiny_mixed(args, dev, msg) if rank == 0 and not args.no_extend else None
    ladder = run_graph_ladder(args, dev, msg) if rank == 0 and not args.no_extend else None
    extend = run_extend(args, dev, msg, peaks) if rank == 0 and not args.no_extend else None
    small = run_graph_decode(args, dev, msg) if rank == 0 and not args.no_extend else None
    large = run_large_decode(args, dev, msg, peaks) if rank == 0 and not args.no_extend else None
    mixed = run_long_mixed(args, dev, msg, peaks) if rank == 0 and not args.no_extend else None
    chunk = run_chunked_prefill(args, dev, msg, peaks) if rank == 0 and not args.no_extend else None
    prologue = run_prologue(args, dev, msg, peaks) if rank == 0 and not args.no_extend else None
    sampler = run_sampler(args, dev, msg, peaks) if rank == 0 and not args.no_extend else None
    cpu = cpu_baseline(spec) if want_cpu else None
    cpu_configs = None
    if want_cpu:
        import oracle
        cpu_configs = cpu_oracle_configs()
        cpu_configs.update(args.cpu_samples)
        cpu_configs = {"cpu_model": cpu_model(), "cores": oracle.num_threads(),
                       "kind": "oracle", **dict(sorted(cpu_configs.items()))}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, seeded page permutation)",
        "config": {
            "workload": f"decode_64req_ctx512-4096_{L}layers_page1",
            "requests": R, "layers": L, "page_size": spec.page_size, "pool_slots_per_layer":
            spec.num_slots, "q_heads": wl.HQ, "kv_heads": wl.HKV, "head_dim": wl.HEAD_DIM,
            "kv_tokens": int(spec.device_len.sum()), "bytes_per_step": bytes_step,
            "l2": "inputs larger than L2: 28 distinct layer pools, ~604 MB read per layer",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {
            "kernel": "decode_kernel", "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_source": peaks["source"], "bytes_per_launch": bytes_layer + spec.total_q * 2 * KV_ROW,
            "launch_ms": round(attn_ms, 5),
            "timing": "CUDA events around each decode launch in a second timed pass of the "
                      "same steps (events between launches disable the early start)",
            "traffic": None if traffic is None else traffic["bytes_per_launch"]},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if tiny is not None:
        line["tiny_mixed"] = tiny
    if ladder is not None:
        line["graph_ladder"] = ladder
    if extend is not None:
        line["extend"] = extend
    if small is not None:
        line["small_batch_graph"] = small
    if large is not None:
        line["large_decode"] = large
    if mixed is not None:
        line["long_mixed"] = mixed
    if chunk is not None:
        line["chunked_prefill"] = chunk
    if prologue is not None:
        line["prologue"] = prologue
    if sampler is not None:
        line["sampler"] = sampler
    if cpu is not None:
        line["cpu_baseline"] = {**cpu, "cpu_model": cpu_model()}
    if cpu_configs is not None:
        line["cpu_baseline_per_config"] = cpu_configs
    return line


def run_tiny_mixed(args, dev, msg):
    """The tiny mixed batch (1 extend of 4 over 2 cached + decodes at 5, 17 and
    64 keys): one whole step -- plan, store_kv, attention -- in microseconds,
    L2 flushed before every timed step (a latency config: no roofline)."""
    import torch
    spec = wl.config_tiny_mixed()
    host = wl.host_tensors(spec)
    b = _planned_batch(spec, dev, msg)
    q = wl.bits_to_torch(host["q"], dev)
    kn, vn = wl.bits_to_torch(host["k_new"], dev), wl.bits_to_torch(host["v_new"], dev)
    kp, vp = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    out = torch.empty_like(q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        msg.msg_plan(b["pt"], b["cached"], b["ext"], b["T"], spec.num_slots, b["ws"],
                     req_rows=b["rows"], qo_indptr_out=b["qo"], out_loc_out=b["loc"])
        msg.msg_store_kv(kn, vn, kp, vp, b["loc"], dev_status=b["ws"])
        msg.msg_paged_attention(q, kp, vp, b["pt"], b["cached"], b["ext"], b["qo"], out, b["ws"],
                                page_size=1, req_rows=b["rows"], max_kv_len=spec.max_kv_len,
                                flags=msg.MSG_ATTN_REUSE_PLAN)

    ms = _median_launch_ms(step, max(args.steps, 50), flush)
    _check_status(msg, b, "tiny mixed")
    # the same step captured once and replayed (what a graph runner pays per step)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gms = _median_launch_ms(g.replay, max(args.steps, 50), flush)
    _check_status(msg, b, "tiny mixed, graph")
    del flush, g
    return {"workload": "tiny_mixed_1ext4_cached2_3dec_ctx5-17-64_page1", "us": round(ms * 1e3, 2),
            "graph_us": round(gms * 1e3, 2),
            "launches": 5, "l2": "flushed (256 MB write) before every timed step",
            "what": "plan + token metadata + store_kv + decode + extend kernels, one step "
                    "(us: launched one by one; graph_us: one captured graph replayed)"}


def run_graph_ladder(args, dev, msg):
    """Launch-bound decode steps: 1, 2, 4 and 8 requests at contexts U[128, 512]
    over 28 layers, eager launches against CUDA-graph replay of the captured
    ladder sizes (the graph runner pads nothing here: each is a ladder size)."""
    import torch
    from paged_kv_gqa_store_gb300 import graph as mgraph
    rng = np.random.default_rng(2010)
    max_bs, L = 8, 28
    ctx = rng.integers(128, 512 + 1, size=max_bs)
    n = max(args.steps, 20)
    steps = 8 * (n + 3) + 8                          # tokens a request gains over the leg
    spec = wl.make_batch("ladder", 2011, cached_len=ctx - 1 + steps,
                         extend_len=np.ones(max_bs, np.int32), page_size=1,
                         num_pages=int((ctx + steps).sum()) + 64, num_layers=L)
    pt = np.zeros((max_bs + 1, spec.page_table.shape[1]), np.int32)
    pt[:max_bs] = spec.page_table
    pt[max_bs] = spec.num_slots                      # the dummy row -> the dummy slot
    slots = spec.num_slots + 1
    g = torch.Generator(device=dev).manual_seed(2012)
    pools = [(torch.randn(slots, wl.HKV, wl.HEAD_DIM, generator=g, device=dev).to(torch.bfloat16),
              torch.randn(slots, wl.HKV, wl.HEAD_DIM, generator=g, device=dev).to(torch.bfloat16))
             for _ in range(L)]
    runner = mgraph.DecodeGraphRunner(pools, torch.from_numpy(pt).to(dev), max_bs, max_bs)
    for i in range(L):
        for x in (runner.q[i], runner.k_new[i], runner.v_new[i]):
            x.copy_(torch.randn(x.shape, generator=g, device=dev).to(torch.bfloat16))
    runner.capture()
    res = {"workload": "decode_bs1-8_ctx128-512_28layers_page1",
           "what": "plan + 28 fused store+decode launches per step; ms per step, back to back",
           "sizes": runner.sizes}
    cached = (ctx - 1).astype(np.int64)
    for bs in (1, 2, 4, 8):
        live = np.arange(bs)
        row = {}
        for mode, fn in (("eager", runner.eager), ("graph", runner.replay)):
            for _ in range(3):
                fn(cached[live], live)
                cached[live] += 1
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(n):
                fn(cached[live], live)
                cached[live] += 1
            b.record()
            torch.cuda.synchronize()
            row[f"{mode}_ms"] = round(a.elapsed_time(b) / n, 4)
        row["speedup"] = round(row["eager_ms"] / row["graph_ms"], 3)
        res[f"bs{bs}"] = row
    st, info = msg.msg_read_device_status(runner.ws)
    if st != msg.MSG_OK:
        raise RuntimeError(f"graph ladder: device status {info}")
    del runner, pools
    torch.cuda.empty_cache()
    return res


def run_graph_decode(args, dev, msg):
    """Small-batch decode step (8 requests x 28 layers), eager vs CUDA-graph replay:
    at this size the step is launch-bound, which is what graph replay removes."""
    import torch
    rng = np.random.default_rng(2002)
    ctx = rng.integers(512, 4096 + 1, size=8)
    spec = wl.make_batch("decode_8x28", 2003, cached_len=ctx - 1, extend_len=np.ones(8, np.int32),
                         page_size=1, num_pages=int(ctx.sum()) + 1024, num_layers=28)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    pt, cached, ext, rows = (i32(spec.page_table), i32(spec.cached_len), i32(spec.extend_len),
                             i32(spec.req_rows))
    T, R = spec.total_q, spec.num_reqs
    qo = torch.zeros(R + 1, dtype=torch.int32, device=dev)
    loc = torch.zeros(T, dtype=torch.int64, device=dev)
    ws = torch.zeros(msg.msg_workspace_size(R, T), dtype=torch.uint8, device=dev)
    layers = [wl.device_tensors(spec, layer, device=dev) for layer in range(spec.num_layers)]
    outs = [torch.empty_like(t["q"]) for t in layers]
    flags = msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY

    def step():
        msg.msg_plan(pt, cached, ext, T, spec.num_slots, ws, req_rows=rows, qo_indptr_out=qo,
                     out_loc_out=loc)
        for i, t in enumerate(layers):
            msg.msg_paged_attention_store(t["q"], t["k_new"], t["v_new"], t["k_pool"], t["v_pool"],
                                          pt, cached, ext, qo, outs[i], ws, page_size=1,
                                          req_rows=rows, max_kv_len=int(spec.max_kv_len),
                                          flags=flags)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(True), torch.cuda.Event(True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    n = max(args.steps, 20)
    eager_ms = timed(step, n)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    graph_ms = timed(g.replay, n)
    del layers, outs, g
    torch.cuda.empty_cache()
    by = spec.num_layers * (decode_attn_bytes(spec) + store_bytes(spec))
    return {"workload": "decode_8req_ctx512-4096_28layers_page1", "eager_ms": round(eager_ms, 4),
            "graph_ms": round(graph_ms, 4), "eager_gbs": round(by / (eager_ms * 1e-3) / 1e9, 1),
            "graph_gbs": round(by / (graph_ms * 1e-3) / 1e9, 1), "launches_per_step": 2 + 28}


def run_extend(args, dev, msg, peaks):
    """Extend attention TFLOP/s on the 8-request extend batch (store first)."""
    import torch
    spec = wl.config_extend()
    t = wl.device_tensors(spec, device=dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    pt, cached, ext, rows = (i32(spec.page_table), i32(spec.cached_len), i32(spec.extend_len),
                             i32(spec.req_rows))
    T, R = spec.total_q, spec.num_reqs
    qo = torch.zeros(R + 1, dtype=torch.int32, device=dev)
    loc = torch.zeros(T, dtype=torch.int64, device=dev)
    ws = torch.zeros(msg.msg_workspace_size(R, T), dtype=torch.uint8, device=dev)
    out = torch.empty_like(t["q"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (129 MB)
    msg.msg_plan(pt, cached, ext, T, spec.num_slots, ws, req_rows=rows, qo_indptr_out=qo,
                 out_loc_out=loc)
    flags = msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_EXTEND_ONLY

    def attn():
        msg.msg_paged_attention(t["q"], t["k_pool"], t["v_pool"], pt, cached, ext, qo, out, ws,
                                page_size=1, req_rows=rows, max_kv_len=spec.max_kv_len,
                                flags=flags)

    def store():
        msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], loc)

    for _ in range(3):
        store()
        attn()
    n = max(args.steps, 5)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    s = torch.cuda.current_stream()
    for k in range(n):
        flush.zero_()
        ev[k][0].record(s)
        store()
        ev[k][1].record(s)
        flush.zero_()
        ev[k][2].record(s)
        attn()
        ev[k][3].record(s)
    torch.cuda.synchronize()
    st_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    at_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev)
    fl = extend_flops(spec)
    tf = fl / (at_ms * 1e-3) / 1e12
    sb = store_bytes(spec)
    traffic = ncu_traffic("extend_kernel")
    return {"workload": "extend_8req_cached0-2048_ext512-4096_page1", "tflops": round(tf, 1),
            "bound": "tensor", "kernel": "extend_kernel",
            "traffic": None if traffic is None else traffic["bytes_per_launch"],
            "tensor_pipe_pct_of_active": None if traffic is None
            else traffic.get("tensor_pipe_pct_of_active"),
            "peak_tflops": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4),
            "peak_source": peaks["source"], "attn_ms": round(at_ms, 4), "flops": fl,
            "store_kv_gbs": round(sb / (st_ms * 1e-3) / 1e9, 1), "store_kv_ms": round(st_ms, 4),
            "l2": "flushed (256 MB write) before every timed launch"}



def _planned_batch(spec, dev, msg, sel=None):
    """Device copies of a batch's metadata, planned once (qo_indptr, out_loc).
    sel (a contiguous range of request indices) makes a sub-batch of the same
    page table: its requests' tokens are rows tok[0]:tok[1] of the full q."""
    import torch
    sel = np.arange(spec.num_reqs) if sel is None else np.asarray(sel)
    qo_full = np.concatenate([[0], np.cumsum(spec.extend_len)])
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    ext = spec.extend_len[sel]
    T = int(ext.sum())
    b = {"pt": i32(spec.page_table), "cached": i32(spec.cached_len[sel]), "ext": i32(ext),
         "rows": i32(spec.req_rows[sel]), "T": T, "R": len(sel), "sel": sel,
         "tok": (int(qo_full[sel[0]]), int(qo_full[sel[0]]) + T),
         "qo": torch.zeros(len(sel) + 1, dtype=torch.int32, device=dev),
         "loc": torch.zeros(T, dtype=torch.int64, device=dev),
         "ws": torch.zeros(msg.msg_workspace_size(len(sel), T), dtype=torch.uint8, device=dev)}
    msg.msg_plan(b["pt"], b["cached"], b["ext"], T, spec.num_slots, b["ws"],
                 req_rows=b["rows"], qo_indptr_out=b["qo"], out_loc_out=b["loc"])
    return b


def _median_launch_ms(fn, n, flush=None):
    """Median CUDA-event time of fn over n launches after 3 warm-ups; the L2
    flush (if any) is written before each timed launch, outside the events."""
    import torch
    s = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        if flush is not None:
            flush.zero_()
        a.record(s)
        fn()
        b.record(s)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def _median_rotating_ms(calls, n):
    """Median CUDA-event time of one launch when the launches cycle through
    len(calls) independent copies of the inputs whose footprint together is
    larger than L2: each launch finds its own inputs evicted by the others'
    reads.  (Written-then-read flush buffers leave L2 full of dirty lines, and
    their write-back then runs inside the timed launch; evictions of clean
    lines cost nothing.)"""
    import torch
    s = torch.cuda.current_stream()
    for _ in range(3):
        for c in calls:
            c()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i, (a, b) in enumerate(ev):
        a.record(s)
        calls[i % len(calls)]()
        b.record(s)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def _attn_call(msg, spec, t, b, out, flags):
    t0, t1 = b["tok"]
    q, o = t["q"][t0:t1], out[t0:t1]

    def call():
        msg.msg_paged_attention(q, t["k_pool"], t["v_pool"], b["pt"], b["cached"], b["ext"],
                                b["qo"], o, b["ws"], page_size=spec.page_size,
                                req_rows=b["rows"], max_kv_len=spec.max_kv_len, flags=flags)
    return call


def _page_table_call(msg, spec, t, b, out, flags):
    """The same (sub)batch read through the FlashAttention / TRT-LLM dense
    page-id table ("Mini-SGLang 完整剖析" 4.6.4) instead of the token table:
    the index is built on the device, planned with it (the plan's index rows
    depend on the layout), and attention reads it."""
    import torch
    dev = b["pt"].device
    kv_len = (spec.cached_len.astype(np.int64) + spec.extend_len)[b["sel"]]
    width = int(((kv_len + spec.page_size - 1) // spec.page_size).max())
    table = torch.empty(b["R"], width, dtype=torch.int32, device=dev)
    msg.msg_build_kv_index(msg.MSG_KV_PAGE_TABLE, spec.page_size, b["pt"], b["cached"], b["ext"],
                           table, req_rows=b["rows"], dev_status=b["ws"])
    kv = msg.KvIndex(msg.MSG_KV_PAGE_TABLE, table, spec.page_size)
    ws = torch.zeros_like(b["ws"])
    msg.msg_plan_ex(kv, b["cached"], b["ext"], b["T"], spec.num_slots, ws)
    t0, t1 = b["tok"]
    q, o = t["q"][t0:t1], out[t0:t1]

    def call():
        msg.msg_paged_attention_ex(q, t["k_pool"], t["v_pool"], kv, b["cached"], b["ext"],
                                   b["qo"], o, ws, max_kv_len=spec.max_kv_len, flags=flags)
    return call, {"ws": ws, "table": table}


def _check_status(msg, b, what):
    st, info = msg.msg_read_device_status(b["ws"])
    if st != msg.MSG_OK:
        raise RuntimeError(f"{what}: device status {info}")


def run_large_decode(args, dev, msg, peaks):
    """256 decode requests, context U[1024, 8192], page_size 16, pools sized to
    90% of free HBM with the pages drawn at random from the whole pool."""
    import torch
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    pages = int(0.9 * free) // (2 * 16 * KV_ROW)
    spec = wl.config_large_decode(pages)
    t = wl.device_tensors(spec, device=dev, canary=False)
    b = _planned_batch(spec, dev, msg)
    msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], b["loc"])
    out = torch.empty_like(t["q"])
    attn = _attn_call(msg, spec, t, b, out,
                      msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY)
    ms = _median_launch_ms(attn, max(args.steps, 20))
    _check_status(msg, b, "large decode")
    by = decode_attn_bytes(spec)
    gbs = by / (ms * 1e-3) / 1e9
    # the dense page-id table layout on the same batch (one entry per page
    # either way at page_size 16: the token table is read at page starts)
    pcall, pb = _page_table_call(msg, spec, t, b, out,
                                 msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY)
    pms = _median_launch_ms(pcall, max(args.steps, 20))
    _check_status(msg, pb, "large decode, page-id table")
    cpu = None
    if getattr(args, "cpu_samples", None) is not None:
        # the CPU oracle on a sample of requests, their referenced pages
        # fetched from the device pools (never the whole pool)
        cpu = cpu_oracle_config3(spec, t)
    del t, b, out, pb
    torch.cuda.empty_cache()
    if cpu is not None:
        args.cpu_samples["3_large_decode"] = cpu
    return {"workload": "decode_256req_ctx1024-8192_page16_pool90pct", "gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4), "attn_ms": round(ms, 4),
            "page_table_layout": {"attn_ms": round(pms, 4),
                                  "gbs": round(by / (pms * 1e-3) / 1e9, 1),
                                  "frac": round(by / (pms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                  "vs_token_table": round(ms / pms, 4)},
            "bytes_per_launch": by, "pool_pages": pages,
            "pool_gb_k_plus_v": round(2 * spec.num_slots * KV_ROW / 1e9, 1),
            "kv_tokens": int(spec.device_len.sum()),
            "l2": "inputs larger than L2 (~4.8 GB of K/V per launch)"}


def prologue_bytes(T: int, max_pos_row_bytes: int = wl.HEAD_DIM * 4) -> int:
    """Algorithmic bytes of the fused prologue: the qkv rows read, q / K / V
    written, one cos/sin row, one position and one out_loc per token."""
    units = wl.HQ + 2 * wl.HKV
    return int(T * (units * wl.HEAD_DIM * 2 * 2 + max_pos_row_bytes + 4 + 8))


def run_prologue(args, dev, msg, peaks):
    """Fused q/k RMSNorm + RoPE + store_kv over the extend batch's new tokens."""
    import torch
    torch.cuda.empty_cache()
    spec = wl.config_extend()
    T = spec.total_q
    b = _planned_batch(spec, dev, msg)
    positions = torch.zeros(T, dtype=torch.int32, device=dev)
    msg.msg_plan(b["pt"], b["cached"], b["ext"], T, spec.num_slots, b["ws"], req_rows=b["rows"],
                 out_loc_out=b["loc"], positions_out=positions)
    g = torch.Generator(device=dev).manual_seed(4242)
    qkv = torch.randn(T, wl.HQ + 2 * wl.HKV, wl.HEAD_DIM, generator=g, device=dev).to(
        torch.bfloat16)
    qw = (1 + 0.1 * torch.randn(wl.HEAD_DIM, generator=g, device=dev)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(wl.HEAD_DIM, generator=g, device=dev)).to(torch.bfloat16)
    cs = msg.msg_rope_cos_sin_cache(1e6, wl.HEAD_DIM, int(spec.max_kv_len) + 1)
    q_out = torch.empty(T, wl.HQ, wl.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    kp = torch.empty(spec.num_slots, wl.HKV, wl.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        msg.msg_qk_norm_rope_store(qkv, positions, qw, kw, 1e-6, cs, q_out, kp, vp, b["loc"],
                                   wl.HQ, wl.HKV, dev_status=b["ws"])

    # a launch touches 353 MB (> L2): back to back, each finds its first inputs
    # evicted by the previous one's later ones
    ms = _median_rotating_ms([call], max(args.steps, 20))
    ms_flushed = _median_launch_ms(call, max(args.steps, 20), flush)
    _check_status(msg, b, "prologue")
    by = prologue_bytes(T)
    gbs = by / (ms * 1e-3) / 1e9
    del qkv, q_out, kp, vp, flush, b
    torch.cuda.empty_cache()
    return {"workload": f"qk_norm_rope_store_{T}tok_16q8kv_d128", "gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4), "us": round(ms * 1e3, 2),
            "us_flushed": round(ms_flushed * 1e3, 2), "bytes_per_launch": by,
            "l2": "inputs larger than L2 (353 MB a launch), launches back to back; us_flushed: "
                  "a 256 MB flush written before each launch (its dirty lines are written back "
                  "during the launch)"}


def sampler_bytes(batch: int, vocab: int, esz: int) -> int:
    """Algorithmic bytes of one sampler launch: every logit read once, the
    four per-row arguments read and one token written per row."""
    return int(batch * vocab * esz + batch * (4 * 4 + 4))


def run_sampler(args, dev, msg, peaks):
    """Batched sampler over 256 rows of Qwen3's 151,936-token vocabulary:
    bf16 and fp32 logits with the mixed parameter set (greedy, temperature,
    top-k, top-p, both), and an all-greedy batch (argmax)."""
    import torch
    torch.cuda.empty_cache()
    B, V = 256, wl.QWEN3_VOCAB
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    n = max(args.steps, 20)
    res = {"workload": f"sample_{B}rows_vocab{V}", "batch": B, "vocab": V,
           "l2": "inputs larger than L2: 3 copies of the batch's logits in rotation (233 MB "
                 "bf16, 467 MB fp32); us_flushed: one copy with a 256 MB flush written before "
                 "each launch (its dirty lines are written back during the launch)"}
    for name, bf16, greedy in (("bf16_mixed", True, False), ("f32_mixed", False, False),
                               ("bf16_greedy", True, True)):
        spec = wl.sampler_batch(name, 8100 + bf16, B, V, bf16=bf16, greedy_only=greedy)
        logits = (wl.bits_to_torch(spec.logits, dev) if bf16
                  else torch.from_numpy(spec.logits).to(dev))
        copies = [logits] + [logits.clone() for _ in range(2)]
        t, k, p = msg.sampling_args(spec.temperature, spec.top_k, spec.top_p, V, device=dev)
        u = torch.from_numpy(spec.uniforms).to(dev)
        out = torch.empty(B, dtype=torch.int32, device=dev)
        ws = torch.empty(msg.msg_sample_workspace_size(B, V), dtype=torch.uint8, device=dev)

        def call(x=logits):
            msg.msg_sample(x, t, k, p, u, tokens_out=out, workspace=ws, dev_status=status)

        ms = _median_rotating_ms([lambda x=x: call(x) for x in copies], n)
        ms_flushed = _median_launch_ms(call, n, flush)
        st, info = msg.msg_read_device_status(status)
        if st != msg.MSG_OK:
            raise RuntimeError(f"sampler {name}: device status {info}")
        by = sampler_bytes(B, V, 2 if bf16 else 4)
        gbs = by / (ms * 1e-3) / 1e9
        res[name] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "us_flushed": round(ms_flushed * 1e3, 2),
                     "bytes_per_launch": by}
        del logits, copies, out, ws
    del flush
    torch.cuda.empty_cache()
    return res


def run_long_mixed(args, dev, msg, peaks):
    """32 decode requests at context 32768 + 2 extend requests of 2048 over 16384
    cached, page_size 64: decode-only, extend-only and the mixed call, the mixed
    call against the max() and sum() of the two roofline bounds."""
    import torch
    torch.cuda.empty_cache()
    spec = wl.config_long_mixed()
    t = wl.device_tensors(spec, device=dev, canary=False)
    dec = spec.extend_len == 1
    b = _planned_batch(spec, dev, msg)
    # the same requests as a decode-only and an extend-only batch (decodes come first)
    bd = _planned_batch(spec, dev, msg, np.flatnonzero(dec))
    be = _planned_batch(spec, dev, msg, np.flatnonzero(~dec))
    msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], b["loc"])
    out = torch.empty_like(t["q"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    n = max(args.steps, 20)
    reuse = msg.MSG_ATTN_REUSE_PLAN
    dec_ms = _median_launch_ms(_attn_call(msg, spec, t, bd, out, reuse | msg.MSG_ATTN_DECODE_ONLY),
                               n, flush)
    ext_ms = _median_launch_ms(_attn_call(msg, spec, t, be, out, reuse | msg.MSG_ATTN_EXTEND_ONLY),
                               n, flush)
    mix_ms = _median_launch_ms(_attn_call(msg, spec, t, b, out, reuse), n, flush)
    pcall, pb = _page_table_call(msg, spec, t, bd, out, reuse | msg.MSG_ATTN_DECODE_ONLY)
    dec_pt_ms = _median_launch_ms(pcall, n, flush)
    for x, what in ((b, "long mixed"), (bd, "long mixed, decode part"),
                    (be, "long mixed, extend part"), (pb, "long mixed, page-id table")):
        _check_status(msg, x, what)
    pages = (spec.device_len + spec.page_size - 1) // spec.page_size
    dec_bytes = int((spec.device_len[dec].sum() * 2 * KV_ROW + dec.sum() * 2 * QO_ROW
                     + pages[dec].sum() * 4))
    fl = extend_flops(spec)
    hbm_ms = dec_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    tc_ms = fl / (peaks["bf16_tflops"] * 1e12) * 1e3
    del t, b, bd, be, out, flush, pb
    torch.cuda.empty_cache()
    return {"workload": "mixed_32dec_ctx32768_2ext2048_cached16384_page64",
            "decode_only_ms": round(dec_ms, 4),
            "decode_gbs": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
            "decode_frac": round(hbm_ms / dec_ms, 4),
            "decode_page_table_layout": {
                "attn_ms": round(dec_pt_ms, 4),
                "gbs": round(dec_bytes / (dec_pt_ms * 1e-3) / 1e9, 1),
                "frac": round(hbm_ms / dec_pt_ms, 4),
                "vs_token_table": round(dec_ms / dec_pt_ms, 4)},
            "extend_only_ms": round(ext_ms, 4),
            "extend_tflops": round(fl / (ext_ms * 1e-3) / 1e12, 1),
            "extend_frac": round(tc_ms / ext_ms, 4),
            "mixed_ms": round(mix_ms, 4), "bound_max_ms": round(max(hbm_ms, tc_ms), 4),
            "bound_sum_ms": round(hbm_ms + tc_ms, 4),
            "mixed_frac_of_max_bound": round(max(hbm_ms, tc_ms) / mix_ms, 4),
            "mixed_frac_of_sum_bound": round((hbm_ms + tc_ms) / mix_ms, 4),
            "decode_bytes": dec_bytes, "extend_flops": fl,
            "l2": "flushed (256 MB write) before every timed launch"}

def run_chunked_prefill(args, dev, msg, peaks):
    """A chunked-prefill step: one request's next 128 tokens over a 32,768-token
    cached prefix (page_size 1): 8 work items (one query tile x 8 KV heads) of
    257 key tiles each.  Timed with the workspace the library asks for (the key
    split spreads the items' key tiles over every SM) and with one too small
    for the split's partial slots (the 8 items taken whole, by 8 CTAs)."""
    import torch
    torch.cuda.empty_cache()
    cached, ext = np.array([32768]), np.array([128])
    spec = wl.make_batch("chunked_prefill", 1009, cached, ext, 1,
                         num_pages=int(cached[0] + ext[0]) + 9)
    t = wl.device_tensors(spec, device=dev, canary=False)
    b = _planned_batch(spec, dev, msg)
    msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], b["loc"])
    out = torch.empty_like(t["q"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    n = max(args.steps, 20)
    flags = msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_EXTEND_ONLY
    split_ms = _median_launch_ms(_attn_call(msg, spec, t, b, out, flags), n, flush)
    whole = dict(b, ws=b["ws"][:16 << 20])     # the plan, without the split's slots
    whole_ms = _median_launch_ms(_attn_call(msg, spec, t, whole, out, flags), n, flush)
    _check_status(msg, b, "chunked prefill")
    fl = extend_flops(spec)
    del t, b, whole, out, flush
    torch.cuda.empty_cache()
    return {"workload": "chunked_prefill_1x128_cached32768_page1",
            "split_ms": round(split_ms, 4), "whole_items_ms": round(whole_ms, 4),
            "split_tflops": round(fl / (split_ms * 1e-3) / 1e12, 1),
            "whole_items_tflops": round(fl / (whole_ms * 1e-3) / 1e12, 1),
            "split_frac": round(fl / (split_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "speedup": round(whole_ms / split_ms, 2), "flops": fl,
            "l2": "flushed (256 MB write) before every timed launch"}


# ------------------------------------------------------------ CPU oracle baseline
def oracle_layer_inputs(spec, layer):
    """Host copies of one layer's inputs for the oracle (all requests, compacted)."""
    rng = np.random.default_rng([spec.seed, layer])
    sub, src = wl.compact_requests(spec, np.arange(spec.num_reqs))
    n = src.shape[0]
    kp = wl.random_bf16(rng, (n, wl.HKV, wl.HEAD_DIM))
    vp = wl.random_bf16(rng, (n, wl.HKV, wl.HEAD_DIM))
    T = spec.total_q
    return sub, {"q": wl.random_bf16(rng, (T, wl.HQ, wl.HEAD_DIM)),
                 "k_new": wl.random_bf16(rng, (T, wl.HKV, wl.HEAD_DIM)),
                 "v_new": wl.random_bf16(rng, (T, wl.HKV, wl.HEAD_DIM)), "k_pool": kp, "v_pool": vp}


def oracle_step_time(spec, sub, data):
    import oracle
    t0 = time.perf_counter()
    meta = oracle.metadata(sub.page_table, sub.cached_len, sub.extend_len, sub.req_rows)
    oracle.store_kv(data["k_new"], data["v_new"], meta["out_loc"], data["k_pool"], data["v_pool"])
    oracle.paged_attention(data["q"], data["k_pool"], data["v_pool"], sub.page_table,
                           sub.cached_len, meta["qo_indptr"], wl.HQ, wl.HKV, wl.HEAD_DIM,
                           req_rows=sub.req_rows)
    return time.perf_counter() - t0


def cpu_baseline(spec, budget_s: float = 12.0):
    """The fp64 oracle, as it stands, on whole layers of the same workload (all 64
    requests), repeated until about budget_s of wall time; GB/s in the same unit."""
    import oracle
    sub, data = oracle_layer_inputs(spec, 0)
    per_layer = decode_attn_bytes(spec) + store_bytes(spec)
    done, elapsed = 0, 0.0
    while elapsed < budget_s:
        elapsed += oracle_step_time(spec, sub, data)
        done += 1
    return {"value": round(per_layer * done / elapsed / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} layer passes (each: all 64 requests, store + attention), fp64 C "
                      f"oracle with OpenMP, {elapsed:.1f} s"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def _oracle_sample_inputs(spec, reqs, rows_per_req=None, pools=None, seed=77):
    """Host inputs for the oracle on a sample of a config: the chosen requests
    relabelled into a compact pool (values from the device pools when given,
    fetching only the referenced pages, else seeded N(0,1) bf16), new q/k/v
    rows, and optionally a sample of query rows per request."""
    import torch
    sub, src = wl.compact_requests(spec, reqs)
    rng = np.random.default_rng([spec.seed, seed])
    n = src.shape[0]
    shape = (n, spec.num_kv_heads, spec.head_dim)
    if pools is None:
        kp, vp = wl.random_bf16(rng, shape), wl.random_bf16(rng, shape)
    else:
        idx = torch.from_numpy(src).to(pools[0].device)
        kp = wl.torch_to_bits(pools[0].index_select(0, idx))
        vp = wl.torch_to_bits(pools[1].index_select(0, idx))
    T = sub.total_q
    data = {"q": wl.random_bf16(rng, (T, spec.num_qo_heads, spec.head_dim)),
            "k_new": wl.random_bf16(rng, (T, spec.num_kv_heads, spec.head_dim)),
            "v_new": wl.random_bf16(rng, (T, spec.num_kv_heads, spec.head_dim)),
            "k_pool": kp, "v_pool": vp}
    rows = None
    if rows_per_req is not None:
        qo = np.concatenate([[0], np.cumsum(sub.extend_len)]).astype(np.int64)
        rows = np.concatenate([np.sort(rng.choice(np.arange(qo[r], qo[r + 1]),
                                                  min(rows_per_req, qo[r + 1] - qo[r]),
                                                  replace=False))
                               for r in range(sub.num_reqs)]).astype(np.int64)
    return sub, data, rows


def _oracle_pass_s(sub, data, rows, threads, budget_s):
    """Mean wall time of one oracle pass (metadata, store_kv, attention of the
    sampled rows) with `threads` OpenMP threads, over passes filling budget_s
    (at least one)."""
    import oracle
    oracle.set_num_threads(threads)
    done, elapsed = 0, 0.0
    while done == 0 or elapsed < budget_s:
        t0 = time.perf_counter()
        meta = oracle.metadata(sub.page_table, sub.cached_len, sub.extend_len, sub.req_rows)
        oracle.store_kv(data["k_new"], data["v_new"], meta["out_loc"], data["k_pool"],
                        data["v_pool"])
        oracle.paged_attention(data["q"], data["k_pool"], data["v_pool"], sub.page_table,
                               sub.cached_len, meta["qo_indptr"], sub.num_qo_heads,
                               sub.num_kv_heads, sub.head_dim, req_rows=sub.req_rows, rows=rows)
        elapsed += time.perf_counter() - t0
        done += 1
    return elapsed / done, done


def _rows_flops(sub, rows):
    """4 D Hq per visible (query, key) pair of the sampled query rows."""
    qo = np.concatenate([[0], np.cumsum(sub.extend_len)]).astype(np.int64)
    r = np.searchsorted(qo, rows, side="right") - 1
    keys = sub.cached_len[r].astype(np.int64) + (rows - qo[r]) + 1
    return 4.0 * sub.head_dim * sub.num_qo_heads * float(keys.sum())


def _cpu_entry(sub, data, rows, unit, work, all_threads, budget_s, sample):
    """The oracle on all cores and on one core; value = work / time in unit
    (GB/s, TFLOP/s) or the time of one pass (us)."""
    out = {"sample": sample}
    for name, th in (("all_cores", all_threads), ("one_core", 1)):
        s, n = _oracle_pass_s(sub, data, rows, th, budget_s)
        if unit == "us":
            v = s * 1e6
        elif unit == "GB/s":
            v = work / s / 1e9
        else:
            v = work / s / 1e12
        out[name] = {"value": round(v, 6 if unit == "TFLOP/s" else 4), "unit": unit,
                     "threads": th, "passes": n}
    return out


def cpu_oracle_configs(budget_s: float = 1.5):
    """The fp64 oracle, as it stands, on bounded samples of configs 1, 2, 4 and
    5 (config 3 is timed in its GPU leg, on pages fetched from the device)."""
    import oracle
    all_threads = oracle.num_threads()
    res = {}
    spec = wl.config_tiny_mixed()
    sub, data, rows = _oracle_sample_inputs(spec, np.arange(spec.num_reqs))
    res["1_tiny_mixed"] = _cpu_entry(sub, data, None, "us", 0, all_threads, budget_s,
                                     "the whole batch (4 requests, 7 new tokens)")
    spec = wl.config_decode_28_layers()
    reqs = np.arange(0, 64, 8)
    sub, data, _ = _oracle_sample_inputs(spec, reqs)
    res["2_decode_64x28"] = _cpu_entry(sub, data, None, "GB/s",
                                       decode_attn_bytes(sub) + store_bytes(sub), all_threads,
                                       budget_s, "8 of the 64 requests, one layer")
    spec = wl.config_extend()
    sub, data, rows = _oracle_sample_inputs(spec, [0, 5], rows_per_req=24)
    res["4_extend"] = _cpu_entry(sub, data, rows, "TFLOP/s", _rows_flops(sub, rows),
                                 all_threads, budget_s,
                                 "2 of the 8 requests, 24 query rows each")
    spec = wl.config_long_mixed()
    sub, data, _ = _oracle_sample_inputs(spec, [0, 1])
    res["5_long_mixed_decode"] = _cpu_entry(sub, data, None, "GB/s",
                                            decode_attn_bytes(sub) + store_bytes(sub),
                                            all_threads, budget_s,
                                            "2 of the 32 decode requests (32768 keys each)")
    sub, data, rows = _oracle_sample_inputs(spec, [32], rows_per_req=8)
    res["5_long_mixed_extend"] = _cpu_entry(sub, data, rows, "TFLOP/s", _rows_flops(sub, rows),
                                            all_threads, budget_s,
                                            "1 of the 2 extend requests, 8 query rows")
    oracle.set_num_threads(all_threads)
    return res


def cpu_oracle_config3(spec, t, budget_s: float = 1.5):
    import oracle
    all_threads = oracle.num_threads()
    reqs = np.arange(0, spec.num_reqs, 32)
    sub, data, _ = _oracle_sample_inputs(spec, reqs, pools=(t["k_pool"], t["v_pool"]))
    r = _cpu_entry(sub, data, None, "GB/s", decode_attn_bytes(sub) + store_bytes(sub),
                   all_threads, budget_s,
                   f"{len(reqs)} of the 256 requests, their pages fetched from the device pools")
    oracle.set_num_threads(all_threads)
    return r


def run_reference(args):
    """The oracle as the reference arm: each step is one layer of the same workload."""
    import oracle
    spec = wl.config_decode_28_layers()
    sub, data = oracle_layer_inputs(spec, 0)
    for _ in range(args.warmup):
        oracle_step_time(spec, sub, data)
    t = [oracle_step_time(spec, sub, data) for _ in range(args.steps)]
    per = decode_attn_bytes(spec) + store_bytes(spec)
    value = per * len(t) / sum(t) / 1e9
    ms = 1e3 * sum(t) / len(t)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, seeded page permutation)",
            "config": {"workload": "decode_64req_ctx512-4096_28layers_page1",
                       "step": "one layer of the 28 (all 64 requests): store + attention"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                             "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "one of the 28 layers per step, all 64 requests"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-extend", action="store_true",
                    help="skip the sub-benchmarks (extend, graph, large decode, mixed)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer leg")
    ap.add_argument("--extend-only", action="store_true",
                    help="run only the extend sub-benchmark and print its JSON (profiling)")
    ap.add_argument("--only", choices=["extend", "graph", "ladder", "tiny", "large", "mixed", "chunk",
                                       "prologue", "sampler", "cpu"],
                    default=None,
                    help="run only one sub-benchmark and print its JSON (profiling)")
    ap.add_argument("--layers", type=int, default=28,
                    help="layers per step (28 for the benchmark; fewer only for profiling)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            import oracle
            oracle.build()
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.extend_only:
        args.only = "extend"
    if args.only:
        import torch
        import paged_kv_gqa_store_gb300 as msg
        msg.load_library()
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
        torch.cuda.set_device(dev)
        peaks = measured_peaks()
        legs = {"extend": lambda: run_extend(args, dev, msg, peaks),
                "graph": lambda: run_graph_decode(args, dev, msg),
                "ladder": lambda: run_graph_ladder(args, dev, msg),
                "tiny": lambda: run_tiny_mixed(args, dev, msg),
                "cpu": lambda: cpu_oracle_configs(),
                "large": lambda: run_large_decode(args, dev, msg, peaks),
                "mixed": lambda: run_long_mixed(args, dev, msg, peaks),
                "chunk": lambda: run_chunked_prefill(args, dev, msg, peaks),
                "prologue": lambda: run_prologue(args, dev, msg, peaks),
                "sampler": lambda: run_sampler(args, dev, msg, peaks)}
        print(json.dumps(legs[args.only]()), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        line = run_ours(args, rank, world, dist)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
