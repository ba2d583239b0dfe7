#!/usr/bin/env python3
"""Benchmark: MLA paged decode, microseconds per layer-step, on GB300.

A layer-step is one pass of the whole hot path over one batch: every emulated DCP
shard's partial decode (out + LSE per shard; all shards in one ``mla_decode_shards``
launch, as the ranks of a DCP group run at the same time) and ``lse_merge`` of the
partials.  ``per_config[...]["decode_call_us"]`` is that launch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config spec] [--extra-configs tiny,cp2,plain,long] [--slot-only]

The headline workload is ``spec``, the largest single-GPU workload: 32 requests, 128
heads, q_len 4, contexts U[8192, 131072], block_size 64, 8 shards, natural-log LSE.
Its KV (2.6 GB) is far larger than L2; L2 is flushed (a 512 MB write) before every timed
step anyway, and only the step itself is inside the CUDA-event bracket.  The other
workloads are timed the same way and reported under ``per_config``; every workload with
several shards is also timed with one ``mla_decode`` call per shard
(``<name>_per_shard``), the form a real DCP rank uses, and ``cp_local_slot`` is timed on
the long workload's 1,048,576 positions (``cp_local_slot_1M``).  ``--impl reference``
times the float64 CPU oracle on the host cores.

One JSON line is printed by rank 0.  With torchrun (N > 1) every rank runs an
independent replica on its own GPU (weak scaling; the step has no cross-GPU exchange).
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
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

CONTEXTS = {"tiny": "37, 130", "cp2": "U[1024,8192]", "plain": "32768 each",
            "spec": "U[8192,131072]", "long": "U[262144,524288], 1% of KV rows x20"}
METRIC = "MLA paged decode µs/layer-step, KV GB/s & TFLOP/s vs GB300 roofline"
UNIT = "us/layer-step"
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------
# algorithmic work (per the decode definition; masked / padded work excluded)
# ---------------------------------------------------------------------------
def _row_prefixes(G, q_len):
    G = np.asarray(G, dtype=np.int64)
    return np.maximum(G[:, None] - np.arange(q_len - 1, -1, -1)[None, :], 0)


def _local(Gr, cp, rank):
    return Gr // cp + (Gr % cp > rank)


def work(w):
    """Algorithmic bytes and flops of one layer-step and of each shard's decode call."""
    G = w.G.numpy()
    Gr = _row_prefixes(G, w.q_len)
    q_bytes = w.B * w.q_len * w.H * 576 * 2
    per_shard = []
    for r in range(w.cp):
        L = np.minimum(_local(Gr, w.cp, r), _local(G, w.cp, r)[:, None])
        Lfull = _local(G, w.cp, r)
        per_shard.append(dict(flops=float((w.H * 2 * 1088 * L).sum()),
                              bytes=float(Lfull.sum() * 1152 + q_bytes)))
    return dict(kv_bytes=float(G.sum() * 1152), q_bytes=float(w.cp * q_bytes),
                flops=float(sum(s["flops"] for s in per_shard)), per_shard=per_shard)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def build_step(name, device, batch=None):
    from step_builder import step_from_workload

    w = synth.make_workload(name, device=device, B=batch)
    step = step_from_workload(w, device)
    del w.kv_global
    return w, step


def time_step(step, steps, warmup, flush, batched):
    """CUDA-event times of ``steps`` layer steps (after ``warmup`` untimed ones): the whole
    step, and each decode call in it (one call over all shards when ``batched``, else one
    per shard)."""
    import mla_paged_decode_03_gb300 as m

    step.batched = batched and step.cp > 1
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    assert m.device_status() == 0
    ncalls = 1 if (step.cp == 1 or step.batched) else step.cp
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ncalls + 2)]
          for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        flush.zero_()
        e = ev[k]
        e[0].record(stream)
        if step.cp == 1:
            step.run()
            e[1].record(stream)
        elif step.batched:
            m.mla_decode_shards(step.q, step.pool_all, step.block_table_all, step.seq_lens_all,
                                step.gseq, step.q_len, step.cp, step.scale, out=step.partials,
                                lse=step.lses, lse_base_e=step.lse_base_e,
                                workspace=step.workspace)
            e[1].record(stream)
            m.lse_merge(step.partials, step.lses, out=step.out, out_lse=step.out_lse,
                        lse_base_e=step.lse_base_e)
            e[2].record(stream)
        else:
            for r in range(step.cp):
                m.mla_decode(step.q, step.pools[r], step.block_table, step.seq_lens[r],
                             step.gseq, step.q_len, step.cp, r, step.scale,
                             out=step.partials[r], lse=step.lses[r], lse_base_e=step.lse_base_e,
                             workspace=step.workspace)
                e[r + 1].record(stream)
            m.lse_merge(step.partials, step.lses, out=step.out, out_lse=step.out_lse,
                        lse_base_e=step.lse_base_e)
            e[ncalls + 1].record(stream)
    torch.cuda.synchronize()
    step_ms, call_ms, merge_ms = [], [], []
    for k in range(steps):
        e = ev[k]
        last = e[1] if step.cp == 1 else e[ncalls + 1]
        step_ms.append(e[0].elapsed_time(last))
        for r in range(ncalls):
            call_ms.append(e[r].elapsed_time(e[r + 1]))
        if step.cp > 1:
            merge_ms.append(e[ncalls].elapsed_time(e[ncalls + 1]))
    assert m.device_status() == 0
    return dict(step_ms=step_ms, call_ms=call_ms, merge_ms=merge_ms,
                launches=step.kernel_launches_per_step(),
                call_shards=step.cp if (step.cp > 1 and step.batched) else 1)


def time_config(name, steps, warmup, device, flush, with_e2e=False, batch=None,
                per_shard=False):
    w, step = build_step(name, device, batch)
    res = time_step(step, steps, warmup, flush, batched=True)
    res.update(work=work(w), w=w, step=step)
    if per_shard and step.cp > 1:
        res["per_shard"] = time_step(step, steps, warmup, flush, batched=False)
        step.batched = True
    if with_e2e:
        res["e2e"] = time_e2e(step, steps, warmup, flush)
    return res


def time_slot(steps, warmup, device, flush):
    """cp_local_slot over the long workload's 1,048,576 positions (cp_size 8), one call
    per rank; HBM-bound at 16 B per position (8 in, 8 out)."""
    import mla_paged_decode_03_gb300 as m

    case = synth.make_workload("long", draw_values=False).slot_cases[0]
    w_pos = case.positions.to(device)
    bt = case.block_table.to(device)
    slots = torch.empty_like(w_pos)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        m.cp_local_slot(w_pos, bt, case.block_size, case.cp_size, 0, case.interleave, slots=slots)
    torch.cuda.synchronize()
    times = []
    for k in range(steps):
        for rank in range(case.cp_size):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            m.cp_local_slot(w_pos, bt, case.block_size, case.cp_size, rank, case.interleave,
                            slots=slots)
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
    assert m.device_status() == 0
    n = w_pos.numel()
    us = statistics.mean(times) * 1e3
    return dict(us_per_call=us, positions=n, cp_size=case.cp_size,
                gbs=16.0 * n / (us * 1e-6) / 1e9, bytes_per_position=16,
                calls=len(times))


def time_scatter(steps, warmup, device, flush):
    """cp_local_slot_scatter over the same 1,048,576 positions (cp_size 8), one call per
    rank, each writing the 576-dim bf16 rows of the positions it owns into its pool.
    HBM-bound: 8 B of position per position, plus 2 x 1152 B (row read and written) per
    owned position."""
    import mla_paged_decode_03_gb300 as m

    case = synth.make_workload("long", draw_values=False).slot_cases[0]
    pos = case.positions.to(device)
    bt = case.block_table.to(device)
    B, N = pos.shape
    g = torch.Generator(device=device).manual_seed(7)
    kv_new = torch.randn(B, N, 576, generator=g, device=device).to(torch.bfloat16)
    num_blocks = int(bt.max()) + 1
    pool = torch.empty(num_blocks, case.block_size, 576, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        m.cp_local_slot_scatter(pos, kv_new, bt, pool, case.cp_size, 0, case.interleave)
    torch.cuda.synchronize()
    times, owned = [], []
    for k in range(steps):
        for rank in range(case.cp_size):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            m.cp_local_slot_scatter(pos, kv_new, bt, pool, case.cp_size, rank, case.interleave)
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
            if k == 0:
                owned.append(int((((pos >= 0) & ((pos // case.interleave) % case.cp_size == rank))
                                  .sum()).item()))
    assert m.device_status() == 0
    n = pos.numel()
    us = statistics.mean(times) * 1e3
    nbytes = 8.0 * n + 2304.0 * statistics.mean(owned)
    return dict(us_per_call=us, positions=n, cp_size=case.cp_size,
                owned_per_call=statistics.mean(owned), bytes_per_call=nbytes,
                gbs=nbytes / (us * 1e-6) / 1e9, calls=len(times))


def time_e2e(step, steps, warmup, flush):
    """Same step through the public API with host buffers: every step copies the
    per-step inputs (q, block table, lengths) from pinned host memory and reads the
    result (out, lse) back."""
    dev = step.q.device
    h_q = step.q.cpu().pin_memory()
    d_in = step.input_tensors()
    h_in = [t.cpu().pin_memory() for t in d_in]
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h_lse = torch.empty(step.out_lse.shape, dtype=step.out_lse.dtype).pin_memory()
    d_q = torch.empty_like(step.q)
    stream = torch.cuda.current_stream()

    def one():
        d_q.copy_(h_q, non_blocking=True)
        for t, ht in zip(d_in, h_in):
            t.copy_(ht, non_blocking=True)
        out, lse = step.run(q=d_q)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    h2d = h_q.numel() * 2 + sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    return dict(ms=statistics.mean(times), h2d=h2d, d2h=d2h)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum under ncu) of one decode call
# of a workload, summed over the two kernels the call launches (decode + split combine),
# keyed by the SHA-256 of the tcgen05 kernel source they were taken on: a changed kernel
# reports null until it is captured again.
TRAFFIC = {
    # spec, all 8 shards in one mla_decode_shards call: decode reads 3,023.6 MB and writes
    # 131.8 MB, the split combine reads 19.0 MB (mean of 12 calls, one-pass capture of the
    # full workload)
    ("spec", "fb4df4fe4dd00e46227fbd0fe766198c749aeeababc2759acef84367040f4fc5"): 3174349632,
}


def measured_traffic(config, batch):
    if batch is not None:
        return None
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                       "mla_paged_decode_03_gb300", "csrc", "mla_decode_tc.cu")
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return TRAFFIC.get((config, digest))


def summarize(res, pk):
    wk = res["work"]
    ms = statistics.mean(res["step_ms"])
    t = ms * 1e-3
    t_hbm = (wk["kv_bytes"] + wk["q_bytes"]) / (pk["hbm"] * 1e9)
    t_tc = wk["flops"] / (pk["bf16"] * 1e12)
    roof = max(t_hbm, t_tc)
    call = statistics.mean(res["call_ms"]) * 1e-3
    # one timed call covers call_shards shards (all of them when they run in one launch)
    shard_flops = statistics.mean(s["flops"] for s in wk["per_shard"]) * res["call_shards"]
    shard_bytes = statistics.mean(s["bytes"] for s in wk["per_shard"]) * res["call_shards"]
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    return dict(us_per_step=ms * 1e3, kv_gbs=wk["kv_bytes"] / t / 1e9,
                tflops=wk["flops"] / t / 1e12, roofline_us=roof * 1e6,
                roofline_frac=roof / t, bound=bound,
                decode_call_us=call * 1e6,
                decode_call_tflops=shard_flops / call / 1e12,
                decode_call_gbs=shard_bytes / call / 1e9,
                decode_calls_per_step=len(res["call_ms"]) // max(1, len(res["step_ms"])),
                merge_us=(statistics.mean(res["merge_ms"]) * 1e3 if res.get("merge_ms") else 0.0),
                kv_gb=wk["kv_bytes"] / 1e9, gflop=wk["flops"] / 1e9,
                launches_per_step=res["launches"])


def baseline_workload(name):
    """The workload the CPU baseline samples: the same seeded draws as the GPU arm (drawn
    on the GPU when there is one, which is quicker for the large workloads)."""
    return synth.make_workload(name, device="cuda" if torch.cuda.is_available() else "cpu")


def cpu_baseline_sample(name, budget_s=12.0, w=None, first=0):
    """Times the float64 oracle on the host cores on a bounded sample of the workload:
    whole requests from ``first`` on (all shards + merge) until ~budget_s of CPU work,
    scaled to one layer-step by the share of the step's flops the sample covered."""
    import oracle.mla_ref as R

    if w is None:
        w = synth.make_workload(name)
    wk = work(w)
    q = w.q.to("cpu", torch.float64).numpy()
    G = w.G.numpy()
    order = [(first + k) % w.B for k in range(w.B)]
    done_flops, elapsed, used = 0.0, 0.0, []
    Gr = _row_prefixes(G, w.q_len)
    for b in order:
        rows_b = w.rows_of(b).to("cpu", torch.float64).numpy()
        t0 = time.perf_counter()
        outs, lses = [], []
        for r in range(w.cp):
            o, l = R.ref_mla_decode_global(q[b:b + 1], [rows_b], G[b:b + 1], w.q_len, w.cp, r,
                                           w.scale, w.base_e)
            outs.append(o)
            lses.append(l)
        if w.cp > 1:
            R.ref_lse_merge(np.stack(outs), np.stack(lses), w.base_e)
        elapsed += time.perf_counter() - t0
        done_flops += float((w.H * 2 * 1088 * Gr[b]).sum())
        used.append(b)
        if elapsed >= budget_s:
            break
    frac = done_flops / wk["flops"]
    us = elapsed / frac * 1e6
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return dict(value=us, unit=UNIT, cores=threads, kind="oracle",
                sample=f"{len(used)} of {w.B} requests of '{name}' (all {w.cp} shards + merge,"
                       f" {frac * 100:.1f}% of the step's flops, {elapsed:.1f} s), scaled to one step")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    ws, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import mla_paged_decode_03_gb300 as m
    m._lib.load()
    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    if args.decode_kernel == "mma":
        m.set_decode_kernel(m.KERNEL_MMA)
    if args.slot_only:
        r = time_slot(max(1, args.steps), args.warmup, device, flush)
        r2 = time_scatter(max(1, args.steps), args.warmup, device, flush)
        if rank == 0:
            print(json.dumps({"cp_local_slot_1M": r, "cp_local_slot_scatter_1M": r2}))
        return

    per_config = {}
    extra = [c for c in args.extra_configs.split(",") if c and c != args.config]
    for name in extra:
        r = time_config(name, max(3, args.steps), max(3, args.warmup), device, flush,
                        per_shard=True)
        per_config[name] = summarize(r, pk)
        if "per_shard" in r:
            per_config[name + "_per_shard"] = summarize(dict(r["per_shard"], work=r["work"]), pk)
        del r
        torch.cuda.empty_cache()
    if args.extra_configs:
        per_config["cp_local_slot_1M"] = time_slot(max(3, args.steps) // 3 + 1, 3, device, flush)
        per_config["cp_local_slot_scatter_1M"] = time_scatter(max(3, args.steps) // 3 + 1, 3,
                                                              device, flush)
        torch.cuda.empty_cache()

    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    wall0 = time.perf_counter()
    res = time_config(args.config, args.steps, args.warmup, device, flush, with_e2e=True,
                      batch=args.batch, per_shard=args.batch is None)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    s = summarize(res, pk)
    per_config[args.config] = s
    if "per_shard" in res:
        per_config[args.config + "_per_shard"] = summarize(dict(res["per_shard"], work=res["work"]),
                                                           pk)
    ms = reduce_max(s["us_per_step"] / 1e3, ws, device)
    e2e_ms = reduce_max(res["e2e"]["ms"], ws, device)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        return
    peak_tc = pk["bf16"]
    if s["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": s["decode_call_tflops"], "peak": peak_tc,
                "unit": "TFLOP/s", "frac": s["decode_call_tflops"] / peak_tc}
    else:
        roof = {"bound": "hbm", "achieved": s["decode_call_gbs"], "peak": pk["hbm"],
                "unit": "GB/s", "frac": s["decode_call_gbs"] / pk["hbm"]}
    roof.update({"traffic": measured_traffic(args.config, args.batch),
                 "kernel": ("mla_decode_shards call (every shard's split-KV decode + split "
                            "combine in one launch)" if res["call_shards"] > 1 else
                            "mla_decode call (split-KV decode + split combine)"),
                 "peak_source": pk["source"] + " (burst)"})
    cpu = None
    if ws == 1 and not args.no_cpu_baseline and args.batch is None:
        del res["step"]
        torch.cuda.empty_cache()
        cpu = cpu_baseline_sample(args.config, w=baseline_workload(args.config))
    line = {
        "metric": METRIC, "value": ms * 1e3, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.config, "B": res["w"].B, "H": res["w"].H,
                   "q_len": res["w"].q_len, "block_size": res["w"].bs, "shards": res["w"].cp,
                   "contexts": CONTEXTS.get(args.config, "see synth"),
                   "l2": "flushed (512 MB write) before every timed step",
                   "parallelism": (f"replicas{ws}" if ws > 1 else
                                   "single GPU, emulated DCP shards (all shards in one launch)"
                                   if res["call_shards"] > 1 else
                                   "single GPU, emulated DCP shards")},
        "kv_gbs": s["kv_gbs"], "tflops": s["tflops"], "roofline_frac": s["roofline_frac"],
        "roofline_us": s["roofline_us"],
        "roofline": roof,
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": res["e2e"]["h2d"],
                "d2h_bytes_per_step": res["e2e"]["d2h"]},
        "gpu_launches": res["launches"] * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "peaks": pk,
        "wall_s": wall,
    }
    print(json.dumps(line))


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.config
    budget = float(os.environ.get("REF_SAMPLE_SECONDS", min(8.0, 120.0 / max(1, args.steps))))
    w = baseline_workload(name)
    vals = []
    for k in range(args.warmup):
        cpu_baseline_sample(name, budget_s=0.5, w=w, first=k)
    last = None
    t0 = time.perf_counter()
    for k in range(args.steps):
        last = cpu_baseline_sample(name, budget_s=budget, w=w, first=k)
        vals.append(last["value"])
    wall = time.perf_counter() - t0
    v = statistics.mean(vals)
    last["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": name, "parallelism": "host cores (float64 CPU oracle)"},
            "cpu_baseline": last,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="spec", choices=synth.ORDER)
    ap.add_argument("--extra-configs", default="tiny,cp2,plain,long")
    ap.add_argument("--slot-only", action="store_true",
                    help="time only cp_local_slot and cp_local_slot_scatter on the "
                         "1,048,576-position case")
    ap.add_argument("--decode-kernel", default="auto", choices=["auto", "mma"],
                    help="profiling only: run the warp-level cross-check decode kernel")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the headline workload's batch (profiling runs only)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
