"""Benchmark: QSA block scoring + exact top-k at 262,144 cells x 256 queries.

One step = one pass of the whole selection path on resident inputs:
qsa_block_scores_gmax (256 queries x 4 heads x D=128 against 65,536 active
summary keys of a 65,538-block capacity; the scores plus each 32-block
group's maximum) then qsa_block_topk_gmax (k=512), which gives the same ids
as qsa_block_topk. ``--path plain`` times qsa_block_scores + qsa_block_topk
instead; the other path is timed beside the headline (``other_path``). The
inputs are the seeded synthetic full-capacity workload: q and keys
Student-t(3) at unit variance.

Prints ONE JSON line (rank 0). ``value`` is query-blocks per second over all
ranks; ``ms_per_step`` the mean device time of the K timed steps (one CUDA
event pair around both calls of each step on the launching stream, L2
flushed before every step and the flush untimed; p10/p50/p90 in
``step_us``); each kernel's own duration (``kernels_us``, the roofline's)
comes from a separate pass right after, with an event between the calls;
``roofline`` describes the dominant kernel; ``e2e`` repeats the measurement
through the public API with host buffers (pinned H2D of q and the active
keys, D2H of the ids, all inside the timed region; consecutive steps are
pipelined over two input buffers, the copy of one step overlapping the
kernels of the previous one); ``cpu_baseline`` times the CPU oracle on this
machine's cores.

Side measurements nested in the same line (rank 0): ``k_sweep`` (the
headline workload at k = 64, 256, 1024), ``decode`` (nq = 1 and 4 decode
steps: the one-launch qsa_block_select_small and the two-call forms),
``attention`` (qsa_sparse_attn at decode shapes and at 256 queries x
k = 512) and ``summary`` (qsa_block_summary over a 262,144-cell pool and a
one-block append). ``--decode-launches``, ``--attn-launches`` and
``--summary-launches`` only launch that call a few times and exit (short
runs for a profiler).

``--impl reference`` times the CPU oracle itself as the reference arm.
Under torchrun each rank runs an independent replica (no collective on the
data path); timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "score+top-k ms/call and query·blocks/s at 256 queries, 262K cells; % of roofline"
UNIT = "query·blocks/s"
WORKLOAD = ("full_262k: 262,144 cells = 65,536 active blocks (capacity 65,538), nq=256 queries x 4 heads "
            "x D=128 fp32, q and keys Student-t(3) at unit variance, top k=512")
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "sparse_attention_kv_qsa_gb300", "csrc")

# Algorithmic traffic and work at this workload (the selection path's
# definition, counted once): q 256*4*128*4 B, keys 65,536*128*4 B, scores
# 256*65,536*4 B written then read, ids 256*512*4 B written.
NQ, ACTIVE, MAX_BLOCKS, K = 256, 65536, 65538, 512


def algorithmic(nq: int, active: int, k: int) -> dict:
    q_b = nq * 4 * 128 * 4
    key_b = active * 128 * 4
    s_b = nq * active * 4
    id_b = nq * k * 4
    return {
        "score_bytes": q_b + key_b + s_b,
        "topk_bytes": s_b + id_b,
        "step_bytes": q_b + key_b + 2 * s_b + id_b,
        "flops_per_head_form": 1024 * nq * active,
        "flops_head_summed": 256 * nq * active,
    }


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def source_sha(fname: str) -> str:
    with open(os.path.join(CSRC, fname), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def decode_side_measurement(dev, stream, cells_list=(2048, 16384, 65536, 262144)):
    """Decode-shaped calls (int8 keys, k=128, nq = 1 and 4, the decode sweep's
    contexts of 2,048 to 262,144 cells = 512 to 65,536 blocks): launch- and
    latency-bound, so reported in microseconds per score + top-k step, once
    with a CUDA-event pair per step (L2 flushed first) and once per step of a
    CUDA graph of 20 back-to-back steps; for the one-launch call (fused:
    qsa_block_select_small), the group-maximum calls (gmax) and the plain
    ones. Rows of at most 8,192 blocks take the register-resident top-k.
    `layer`: the whole decode layer of the pages' breakdown (append, scores,
    top-k, attention) as one CUDA graph per step."""
    import torch
    import sparse_attention_kv_qsa_gb300 as qsa
    from sparse_attention_kv_qsa_gb300 import workloads as w
    out = {"workload": "decode: int8 keys + binary16 scales, k=128; keys nq{1,4}_c<cells>", "unit": "us"}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    for nq, cells in [(nq, c) for c in cells_list for nq in (1, 4)]:
        W = w.decode(nq, cells)
        q = torch.from_numpy(W.q).to(dev)
        kq = torch.from_numpy(W.kq8).to(dev)
        ks = torch.from_numpy(W.kscale.view(np.int16)).to(dev)
        s = torch.empty((nq, W.active), dtype=torch.float32, device=dev)
        gm = torch.empty((nq, qsa.groups(W.active)), dtype=torch.int32, device=dev)
        ids = torch.empty((nq, W.k), dtype=torch.int32, device=dev)

        def step_gmax():
            qsa.block_scores_q8_gmax(q, kq, ks, W.active, out=s, gmax_out=gm)
            qsa.block_topk_gmax(s, gm, W.k, out=ids)

        def step_plain():
            qsa.block_scores_q8(q, kq, ks, W.active, out=s)
            qsa.block_topk(s, W.k, out=ids)

        def step_fused():
            qsa.block_select_small(q, W.active, W.k, kblk_q8=kq, kscale_f16=ks, scores_out=s, ids_out=ids)

        res = {}
        for name, step in (("fused", step_fused), ("gmax", step_gmax), ("plain", step_plain)):
            for _ in range(5):
                step()
            torch.cuda.synchronize()
            ts = []
            for i in range(50):
                flush.fill_(float(i))
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step()
                e1.record(stream)
                e1.synchronize()
                ts.append(1e3 * e0.elapsed_time(e1))
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                step()
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=side):
                    for _ in range(20):
                        step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            res[name] = {"step_p50": pct(ts, 50), "step_p10": pct(ts, 10), "step_p90": pct(ts, 90),
                         "graph_step": 1e3 * e0.elapsed_time(e1) / 20}
        out[f"nq{nq}_c{cells}"] = res
    out["layer"] = decode_layer_measurement(dev, stream)
    return out


def decode_layer_measurement(dev, stream, cells=262144, k=128, nqs=(1, 4), graph=True, launches=0):
    """One decode layer per step, as the pages break it down (append +
    scores + top-k + attention), on one int8 KV pool: the summary keys of the
    block the new cell fell into are refreshed (qsa_block_summary, one
    block), the queries are scored against the int8 summary keys and the top
    k selected (the two group-maximum calls), and the 4 heads attend the
    selected blocks' cells (qsa_sparse_attn). Microseconds per step of a CUDA
    graph of 20 steps; the four calls run as programmatic dependents."""
    import torch
    import sparse_attention_kv_qsa_gb300 as qsa
    from sparse_attention_kv_qsa_gb300 import workloads as w
    nblocks = cells // 4
    out = {"workload": f"decode layer: {cells:,} int8 KV cells, k={k}, append of one block's keys + "
                       "scores + top-k + attention", "unit": "us"}
    for nq in nqs:
        A = w.attn_case(nq, cells, k)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        q, kc, vc = t(A.q), t(A.kc), t(A.vc)
        ks, vs = t(A.ks.view(np.int16)), t(A.vs.view(np.int16))
        kq = torch.empty((nblocks + 2, 128), dtype=torch.int8, device=dev)
        ksc = torch.empty((nblocks + 2,), dtype=torch.int16, device=dev)
        qsa.block_summary(kc, ks, 0, nblocks, kblk_q8=kq, kblk_scale_f16=ksc)
        s = torch.empty((nq, nblocks), dtype=torch.float32, device=dev)
        gm = torch.empty((nq, qsa.groups(nblocks)), dtype=torch.int32, device=dev)
        ids = torch.empty((nq, k), dtype=torch.int32, device=dev)
        o = torch.empty((nq, 4, 128), dtype=torch.float32, device=dev)

        def layer():
            qsa.block_summary(kc, ks, nblocks - 1, nblocks, kblk_q8=kq, kblk_scale_f16=ksc)
            qsa.block_scores_q8_gmax(q, kq, ksc, nblocks, out=s, gmax_out=gm)
            qsa.block_topk_gmax(s, gm, k, out=ids)
            qsa.sparse_attn(q, kc, ks, vc, vs, ids, out=o)

        for _ in range(5 if graph else launches):
            layer()
        torch.cuda.synchronize()
        if not graph:
            continue
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            layer()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                for _ in range(20):
                    layer()
        torch.cuda.synchronize()
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            v = 1e3 * e0.elapsed_time(e1) / 20
            best = v if best is None else min(best, v)
        out[f"nq{nq}"] = {"graph_step": best}
    return out


def pct(xs, p):
    """p-th percentile (nearest rank) of a list of floats."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(p / 100 * (len(ys) - 1)))))]


def recorded_traffic(kernel: str, fname: str):
    """DRAM bytes per launch of `kernel` from profiles/dram_traffic.txt, or
    None when absent or taken on a different source of the kernel."""
    p = os.path.join(PROFILES, "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = source_sha(fname)
    with open(p) as f:
        for line in f:
            m = dict(re.findall(r"(\w+)=(\S+)", line))
            if m.get("kernel") == kernel and m.get("source_sha") == sha and "dram_bytes_per_launch" in m:
                return float(m["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
            return
        # nvidia-smi's start-up (driver and NVML initialisation) must be over
        # before the timed steps begin: wait for its first sample (bounded).
        t0 = time.monotonic()
        while not self.lines and time.monotonic() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        time.sleep(0.2)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarise(self.lines)

    @staticmethod
    def summarise(lines: list[str]) -> dict | None:
        """Median SM clock, maximum SM clock and the throttle reasons seen
        Active in nvidia-smi's csv,noheader,nounits rows of FIELDS; rows that
        do not start with a GPU index and fields that are not numbers (such
        as [N/A]) are skipped."""
        rows = [l.split(", ") for l in lines if l and l[0].isdigit()]
        if not rows:
            return None
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in rows if len(r) > 1 and num(r[1])]
        smaxs = [float(r[2]) for r in rows if len(r) > 2 and num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if len(r) > 5 + j and r[5 + j] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smaxs) if smaxs else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_oracle_baseline(W, budget_s: float = 20.0, nq_sample: int | None = None) -> dict:
    import oracle
    o = oracle.get()
    cores = o.default_threads()
    nq_s = W.nq if nq_sample is None else nq_sample
    t0 = time.perf_counter()
    S = o.scores(W.q[:nq_s], W.kblk, W.active, nthreads=cores)
    o.topk_f64(S, W.k, nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": nq_s * W.active / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{nq_s} queries x {W.active} blocks, k={W.k}: FP64 scoring + full-sort top-k, "
                      f"{cores} threads, one pass, {dt:.2f} s"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_step: int, step_ms: float) -> float:
    """Units per second over the whole job: every rank processes
    `units_per_step` per step (weak scaling), and the step time is the max
    over ranks."""
    return world * units_per_step / (step_ms * 1e-3)


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return None
    from sparse_attention_kv_qsa_gb300 import workloads
    import oracle
    W = workloads.full(k=args.k)
    o = oracle.get()
    cores = o.default_threads()
    # each step: a bounded sample sized so warm-up + steps take ~<= 2 minutes
    per_step = max(0.02, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    t0 = time.perf_counter()
    S = o.scores(W.q[:cores], W.kblk, W.active, nthreads=cores)
    o.topk_f64(S, W.k, nthreads=cores)
    t_rows = (time.perf_counter() - t0)
    # sample cores queries x `blocks` blocks per step
    blocks = int(max(2 * W.k, min(W.active, W.active * per_step / max(t_rows, 1e-9))))
    nq_s = cores

    def step():
        S = o.scores(W.q[:nq_s], W.kblk, blocks, nthreads=cores)
        o.topk_f64(S, W.k, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * nq_s * blocks / dt
    sample = (f"{nq_s} queries x {blocks} blocks per step (k={W.k}), FP64 scoring + full-sort top-k on "
              f"{cores} host threads")
    return {"metric": METRIC, "impl": "reference", "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "nq": NQ, "active_blocks": ACTIVE,
                                            "max_blocks": MAX_BLOCKS, "k": args.k},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def attention_side_measurement(dev, stream, sm_mhz: float):
    """qsa_sparse_attn over the selected blocks' int8 KV cells (262,144 cells,
    binary16 scales): decode shapes (nq = 1 and 4, k = 128: the CUDA-core
    kernel) per call of a CUDA graph of 20 calls, and a prompt-like shape
    (256 queries, k = 512, L2 flushed before each call: the tensor-core
    kernel) with its HBM fraction and its rate in FP32-equivalent FLOPs
    against the CUDA cores' FP32 peak (the device's SM count x 128 lanes x 2
    FLOP x `sm_mhz`, the SM clock sampled during the timed steps)."""
    import torch
    import sparse_attention_kv_qsa_gb300 as qsa
    from sparse_attention_kv_qsa_gb300 import workloads as w
    out = {"workload": "attention over the selected blocks: int8 K/V cells + binary16 scales, 262,144 cells",
           "unit": "us"}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    for nq, k, name in ((1, 128, "decode_nq1_k128"), (4, 128, "decode_nq4_k128"), (256, 512, "nq256_k512")):
        W = w.attn_case(nq, 262144, k)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        q, kc, vc, ids = t(W.q), t(W.kc), t(W.vc), t(W.ids)
        ks = torch.from_numpy(W.ks.view(np.int16)).to(dev)
        vs = torch.from_numpy(W.vs.view(np.int16)).to(dev)
        o = torch.empty((nq, 4, 128), dtype=torch.float32, device=dev)
        call = lambda: qsa.sparse_attn(q, kc, ks, vc, vs, ids, out=o)
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        if nq <= 4:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                call()
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=side):
                    for _ in range(20):
                        call()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            out[name] = {"graph_call_us": 1e3 * e0.elapsed_time(e1) / 20, "kernel": "attn_kernel (CUDA cores)"}
            continue
        ts = []
        for i in range(30):
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            ts.append(1e3 * e0.elapsed_time(e1))
        us = statistics.median(ts)
        cells = nq * k * 4
        bytes_ = cells * 2 * (128 + 2) + nq * 4 * 128 * 4 * 2 + nq * k * 4
        flops = cells * 4 * 128 * 2 * 2
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak_fp32 = sms * 128 * 2 * sm_mhz * 1e6
        out[name] = {"call_us_p50": us, "algorithmic_bytes": bytes_, "hbm_gbs": bytes_ / us / 1e3,
                     "fp32_tflops": flops / us / 1e6, "fp32_frac": flops / (us * 1e-6) / peak_fp32,
                     "fp32_peak_note": f"{sms} SMs x 128 lanes x 2 FLOP x {sm_mhz:.0f} MHz (sampled)",
                     "kernel": attn_kernel_label(nq, sms)}
    return out


def attn_kernel_label(nq: int, sms: int) -> str:
    """Which attention kernel and CTA form qsa_sparse_attn launches for nq
    queries on a device with `sms` SMs (the launchers' rule): CUDA cores
    with clusters of 4 or 2 CTAs per query up to half the SM count; beyond
    it the tensor cores, 16-warp CTAs up to the SM count, then 8-warp CTAs
    two per SM up to twice it, then 4-warp CTAs four per SM."""
    if 2 * nq <= sms:
        return f"attn_kernel (CUDA cores, clusters of {4 if 4 * nq <= sms else 2} CTAs per query)"
    warps = 16 if nq <= sms else 8 if nq <= 2 * sms else 4
    return f"attn_tc_kernel (tensor cores, mma.sync; {warps}-warp CTAs, {16 // warps} per SM)"


def summary_side_measurement(dev, stream):
    """qsa_block_summary: every summary key (fp32 and int8 forms) of a
    262,144-cell pool rebuilt (65,536 blocks, L2 flushed before each call),
    and the one-block refresh after a decode append (per call of a CUDA graph
    of 20 calls)."""
    import torch
    import sparse_attention_kv_qsa_gb300 as qsa
    from sparse_attention_kv_qsa_gb300 import workloads as w
    A = w.attn_case(1, 262144, 1)
    kc = torch.from_numpy(np.ascontiguousarray(A.kc)).to(dev)
    ks = torch.from_numpy(A.ks.view(np.int16)).to(dev)
    nb = 65536
    key = torch.empty((nb, 128), dtype=torch.float32, device=dev)
    q8 = torch.empty((nb, 128), dtype=torch.int8, device=dev)
    sc = torch.empty((nb,), dtype=torch.int16, device=dev)
    full = lambda: qsa.block_summary(kc, ks, 0, nb, kblk=key, kblk_q8=q8, kblk_scale_f16=sc)
    one = lambda: qsa.block_summary(kc, ks, nb - 1, nb, kblk=key, kblk_q8=q8, kblk_scale_f16=sc)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    for _ in range(5):
        full()
    torch.cuda.synchronize()
    ts = []
    for i in range(30):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        full()
        e1.record(stream)
        e1.synchronize()
        ts.append(1e3 * e0.elapsed_time(e1))
    us = statistics.median(ts)
    bytes_ = 262144 * (128 + 2) + nb * (128 * 4 + 128 + 2)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        one()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            for _ in range(20):
                one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return {"workload": "block summary keys (fp32 + int8 forms) of a 262,144-cell int8 pool", "unit": "us",
            "rebuild_65536_blocks_us_p50": us, "algorithmic_bytes": bytes_, "hbm_gbs": bytes_ / us / 1e3,
            "append_one_block_graph_us": 1e3 * e0.elapsed_time(e1) / 20}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--k", type=int, default=K)
    ap.add_argument("--scorer", default="default", choices=["default", "ffma"])
    ap.add_argument("--path", default="gmax", choices=["gmax", "plain"],
                    help="gmax: qsa_block_scores_gmax + qsa_block_topk_gmax (the group maxima let the "
                         "top-k read only the groups that can hold its k); plain: qsa_block_scores + "
                         "qsa_block_topk. Both give the same ids.")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-flush", action="store_true", help="warm L2 (back-to-back steps)")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-shaped side measurement")
    ap.add_argument("--no-ksweep", action="store_true", help="skip the k sweep (64, 256, 1024) side measurement")
    ap.add_argument("--no-attn", action="store_true", help="skip the attention side measurement")
    ap.add_argument("--no-summary", action="store_true", help="skip the summary-key side measurement")
    ap.add_argument("--decode-launches", type=int, default=0,
                    help="only launch qsa_block_select_small this many times on the decode workload (4 queries, "
                         "int8 keys, 262,144 cells, k=128; a short run for a profiler to capture), then exit")
    ap.add_argument("--summary-launches", type=int, default=0,
                    help="only launch qsa_block_summary this many times over a 262,144-cell pool (65,536 "
                         "blocks, both key forms; a short run for a profiler to capture), then exit")
    ap.add_argument("--attn-launches", type=int, default=0,
                    help="only launch qsa_sparse_attn this many times on --attn-nq queries x k=512 over "
                         "262,144 cells (a short run for a profiler to capture), then exit")
    ap.add_argument("--layer-launches", type=int, default=0,
                    help="only run the decode layer (append + scores + top-k + attention, nq = 4, 262,144 cells, "
                         "k=128) this many times (a short run for a profiler to capture), then exit")
    ap.add_argument("--attn-nq", type=int, default=256,
                    help="queries of the --attn-launches run (at most half the SM count: the CUDA-core kernel)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    import sparse_attention_kv_qsa_gb300 as qsa
    from sparse_attention_kv_qsa_gb300 import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.decode_launches > 0:
        Wd = workloads.decode(4, 262144)
        qd = torch.from_numpy(Wd.q).to(dev)
        kqd = torch.from_numpy(Wd.kq8).to(dev)
        ksd = torch.from_numpy(Wd.kscale.view(np.int16)).to(dev)
        sd = torch.empty((4, Wd.active), dtype=torch.float32, device=dev)
        idd = torch.empty((4, Wd.k), dtype=torch.int32, device=dev)
        for _ in range(args.decode_launches):
            qsa.block_select_small(qd, Wd.active, Wd.k, kblk_q8=kqd, kscale_f16=ksd, scores_out=sd, ids_out=idd)
        torch.cuda.synchronize()
        print(json.dumps({"decode_launches": args.decode_launches, "workload": Wd.name}), flush=True)
        return
    if args.summary_launches > 0:
        A = workloads.attn_case(1, 262144, 1)
        kc = torch.from_numpy(np.ascontiguousarray(A.kc)).to(dev)
        ks = torch.from_numpy(A.ks.view(np.int16)).to(dev)
        key = torch.empty((65536, 128), dtype=torch.float32, device=dev)
        q8 = torch.empty((65536, 128), dtype=torch.int8, device=dev)
        sc = torch.empty((65536,), dtype=torch.int16, device=dev)
        for _ in range(args.summary_launches):
            qsa.block_summary(kc, ks, 0, 65536, kblk=key, kblk_q8=q8, kblk_scale_f16=sc)
        torch.cuda.synchronize()
        print(json.dumps({"summary_launches": args.summary_launches, "workload": "262,144 cells"}), flush=True)
        return
    if args.layer_launches > 0:
        decode_layer_measurement(dev, torch.cuda.current_stream(dev), nqs=(4,), graph=False,
                                 launches=args.layer_launches)
        torch.cuda.synchronize()
        print(json.dumps({"layer_launches": args.layer_launches, "workload": "decode layer, nq=4, 262,144 cells"}),
              flush=True)
        return
    if args.attn_launches > 0:
        A = workloads.attn_case(args.attn_nq, 262144, 512)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        ks, vs = t(A.ks.view(np.int16)), t(A.vs.view(np.int16))
        q, kc, vc, ids = t(A.q), t(A.kc), t(A.vc), t(A.ids)
        out = torch.empty((A.nq, 4, 128), dtype=torch.float32, device=dev)
        for _ in range(args.attn_launches):
            qsa.sparse_attn(q, kc, ks, vc, vs, ids, out=out)
        torch.cuda.synchronize()
        print(json.dumps({"attn_launches": args.attn_launches, "workload": A.name}), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    W = workloads.full(k=args.k)
    q = torch.from_numpy(W.q).to(dev)
    kblk = torch.from_numpy(W.kblk).to(dev)
    scores = torch.empty((W.nq, W.active), dtype=torch.float32, device=dev)
    gmax = torch.empty((W.nq, qsa.groups(W.active)), dtype=torch.int32, device=dev)
    ids = torch.empty((W.nq, W.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)

    path = "plain" if args.scorer == "ffma" else args.path
    calls = {}
    if args.scorer == "ffma":
        calls["plain"] = (lambda: qsa.block_scores_ffma(q, W.active, kblk=kblk, out=scores),
                          lambda: qsa.block_topk(scores, W.k, out=ids))
    else:
        calls["plain"] = (lambda: qsa.block_scores(q, kblk, W.active, out=scores),
                          lambda: qsa.block_topk(scores, W.k, out=ids))
        calls["gmax"] = (lambda: qsa.block_scores_gmax(q, kblk, W.active, out=scores, gmax_out=gmax),
                         lambda: qsa.block_topk_gmax(scores, gmax, W.k, out=ids))

    def queue_ahead():
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(2_000_000)   # ~1 ms

    def timed_steps(score, topk, n):
        """n flushed steps, each timed whole: one event pair on the launching
        stream around both calls (the top-k may launch under the scorer's
        tail, as it does in use). A short device-side sleep before the first
        event lets the host queue the first steps while the GPU is still busy,
        so no step's events also time a host launch gap; it is outside every
        timed event pair."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        queue_ahead()
        for i in range(n):
            if not args.no_flush:
                flush.fill_(float(i))
            ev[i][0].record(stream)
            score()
            topk()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]

    def split_steps(score, topk, n):
        """n flushed steps with an extra event between the calls: each
        kernel's own duration. The middle event keeps the top-k from
        launching under the scorer's tail, so these steps are not step times."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        queue_ahead()
        for i in range(n):
            if not args.no_flush:
                flush.fill_(float(i))
            ev[i][0].record(stream)
            score()
            ev[i][1].record(stream)
            topk()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        return [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)], [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]

    score, topk = calls[path]
    K_ = args.steps
    # No garbage-collection pause may land inside a timed event pair: a host
    # stall between a step's launches leaves the GPU idle inside that step.
    gc.collect()
    gc.disable()
    # The clock sampler runs from before the warm-up to after the timed steps.
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    if sampler:
        sampler.start()
    for i in range(args.warmup):
        if not args.no_flush:
            flush.fill_(float(i))
        score()
        topk()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_step = timed_steps(score, topk, K_)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    ids_headline = ids.clone()
    # Each kernel's own duration (the roofline's), in a pass of its own right
    # after the timed steps: same calls, same flushes.
    n_split = max(K_, 200)
    t_score, t_topk = split_steps(score, topk, n_split)
    other = None
    if len(calls) > 1:
        # The other path, for comparison (same ids), outside the timed region.
        o_score, o_topk = calls["plain" if path == "gmax" else "gmax"]
        for i in range(args.warmup):
            o_score()
            o_topk()
        n_o = min(max(K_, 200), 400)
        ostep = timed_steps(o_score, o_topk, n_o)
        os_, ot_ = split_steps(o_score, o_topk, n_o)
        assert torch.equal(ids, ids_headline), "the two paths disagree"
        other = {"path": "plain" if path == "gmax" else "gmax", "steps": n_o,
                 "step_us": 1e3 * statistics.mean(ostep), "step_p50_us": 1e3 * pct(ostep, 50),
                 "scores_us": 1e3 * statistics.mean(os_), "topk_us": 1e3 * statistics.mean(ot_)}
    # The fused call (qsa_block_select: the same ids without storing the
    # scores), same workload, flushes and step timing; its ids must equal the
    # headline's.
    select = None
    peaks = load_peaks()
    units_per_step = W.nq * W.active
    if args.scorer == "default":
        ids_f = torch.empty_like(ids)
        scratch = torch.empty((qsa.select_scratch_bytes(W.nq),), dtype=torch.uint8, device=dev)
        sel = lambda: qsa.block_select(q, kblk, W.active, W.k, ids_out=ids_f, scores_buf=scores, scratch=scratch)
        for i in range(args.warmup):
            sel()
        n_f = min(max(K_, 200), 1000)
        t_sel = timed_steps(sel, lambda: None, n_f)
        torch.cuda.synchronize()
        assert torch.equal(ids_f, ids_headline), "qsa_block_select disagrees with the two calls"
        f_us = 1e3 * statistics.mean(t_sel)
        f_alg = 1e6 * (W.nq * 128 * 4 * 4 + W.active * 128 * 4 + W.nq * W.k * 4) / (peaks["hbm_gbs"] * 1e9)
        f_tc = 1e6 * 1024.0 * W.nq * W.active / (peaks["bf16_tflops"] * 1e12)
        select = {"call": "qsa_block_select (five launches; scores not stored)", "steps": n_f,
                  "step_us": f_us, "step_p50_us": 1e3 * pct(t_sel, 50), "value": units_per_step / (f_us * 1e-6),
                  "roofline": {"hbm_floor_us": f_alg, "tensor_floor_us": f_tc, "floor_us": max(f_alg, f_tc),
                               "frac": max(f_alg, f_tc) / f_us,
                               "note": "q + keys + ids at the HBM copy peak; 1,024 FLOP per query-block (the 4-head "
                                       "definition) at the bf16 tensor peak; the slower of the two"}}
    step_ms_local = statistics.mean(t_step)
    step_ms = max_over_ranks(step_ms_local, world, dev)
    if qsa.device_error(dev) != 0:
        raise SystemExit("a QSA kernel reported a timed-out wait; results invalid")

    alg = algorithmic(W.nq, W.active, W.k)
    peaks = load_peaks()
    units_per_step = W.nq * W.active
    value = whole_job_rate(world, units_per_step, step_ms)
    score_us = 1e3 * statistics.mean(t_score)
    topk_us = 1e3 * statistics.mean(t_topk)

    # Dominant kernel and its roofline.
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak_tflops = sm_count * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
    scorer_kernel, scorer_src = (("scores_ffma_kernel", "scores_ffma.cu") if args.scorer == "ffma"
                                 else qsa.default_scorer_kernel())
    if score_us >= topk_us:
        if scorer_kernel == "scores_ffma_kernel":
            achieved = alg["flops_head_summed"] / (score_us * 1e-6) / 1e12
            roof = {"kernel": scorer_kernel, "bound": "alu", "achieved": achieved, "peak": fp32_peak_tflops,
                    "unit": "TFLOP/s", "frac": achieved / fp32_peak_tflops,
                    "peak_note": f"FP32 FMA: {sm_count} SMs x 128 lanes x 2 FLOP x {peaks['sm_max_mhz']:.0f} MHz"}
        else:
            achieved = alg["score_bytes"] / (score_us * 1e-6) / 1e9
            roof = {"kernel": scorer_kernel, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_note": f"{peaks['source']} HBM copy bandwidth"}
        roof["traffic"] = recorded_traffic(scorer_kernel, scorer_src)
    else:
        achieved = alg["topk_bytes"] / (topk_us * 1e-6) / 1e9
        roof = {"kernel": "topk_row_kernel", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_note": f"{peaks['source']} HBM copy bandwidth",
                "traffic": recorded_traffic("topk_row_kernel", "topk.cu")}
    floor_us = 1e6 * alg["step_bytes"] / (peaks["hbm_gbs"] * 1e9)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K_, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "nq": W.nq, "active_blocks": W.active, "max_blocks": W.max_blocks,
                   "k": W.k, "scorer": scorer_kernel,
                   "path": ("qsa_block_scores_gmax + qsa_block_topk_gmax" if path == "gmax"
                            else "qsa_block_scores + qsa_block_topk"),
                   "l2": "warm (no flush)" if args.no_flush else
                         f"flushed before every step by a {2 * l2 >> 20} MiB write, flush untimed",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kernels_us": {"scores": score_us, "topk": topk_us,
                       "scores_p50": 1e3 * statistics.median(t_score), "topk_p50": 1e3 * statistics.median(t_topk),
                       "steps": n_split,
                       "pass": "a split pass after the timed steps (an event between the two calls)"},
        "step_us": {"mean": 1e3 * step_ms_local, "p10": 1e3 * pct(t_step, 10), "p50": 1e3 * pct(t_step, 50),
                    "p90": 1e3 * pct(t_step, 90), "min": 1e3 * min(t_step), "max": 1e3 * max(t_step),
                    "argmax": int(np.argmax(t_step)), "first3": [1e3 * x for x in t_step[:3]],
                    "steps": len(t_step)},
        "roofline": roof,
        "step_roofline": {"floor_us": floor_us, "frac": floor_us / (step_ms * 1e3),
                          "note": "algorithmic step bytes at the measured HBM copy peak (the step's binding "
                                  "roof when scoring runs on tensor cores)",
                          "floor_us_nominal_8tbs": alg["step_bytes"] / 8e12 * 1e6,
                          "frac_nominal_8tbs": alg["step_bytes"] / 8e12 * 1e6 / (step_ms * 1e3)},
        "gpu_launches": 2 * K_,
        "other_path": other,
        "select": select,
        "clocks": clocks,
        "pages_context": {"r9700_score_plus_topk_ms": 2.8, "r9700_qblocks_per_s": 6.0e9,
                          "note": "AMD R9700 (gfx1201) numbers from the pages; context only"},
    }

    # End to end through the public API with host buffers.
    if not args.no_e2e:
        # End to end through the public API with host buffers: every step
        # copies its q and active keys from pinned host memory, runs both calls
        # and reads the ids back. Steps are pipelined the way a server would
        # run them: two device input buffers, the copy of step i+1 (copy
        # stream) overlapping the kernels of step i (compute stream).
        q_h = torch.from_numpy(W.q).pin_memory()
        k_h = torch.from_numpy(np.ascontiguousarray(W.kblk[:W.active])).pin_memory()
        ids_h = [torch.empty((W.nq, W.k), dtype=torch.int32).pin_memory() for _ in range(2)]
        q_d = [torch.empty_like(q_h, device=dev) for _ in range(2)]
        k_d = [torch.empty((W.max_blocks, 128), dtype=torch.float32, device=dev) for _ in range(2)]
        ids_d = [torch.empty((W.nq, W.k), dtype=torch.int32, device=dev) for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        n_e = min(args.e2e_steps, K_)

        def run_pipeline(n, copy_keys=True):
            copied = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            for i in range(n):
                b = i & 1
                with torch.cuda.stream(copy_stream):
                    if i >= 2:
                        copy_stream.wait_event(done[i - 2])      # buffer b is free again
                    q_d[b].copy_(q_h, non_blocking=True)
                    if copy_keys:
                        k_d[b][:W.active].copy_(k_h, non_blocking=True)
                    copied[i].record(copy_stream)
                stream.wait_event(copied[i])
                if path == "gmax":
                    qsa.block_scores_gmax(q_d[b], k_d[b], W.active, out=scores, gmax_out=gmax)
                    qsa.block_topk_gmax(scores, gmax, W.k, out=ids_d[b])
                elif args.scorer == "ffma":
                    qsa.block_scores_ffma(q_d[b], W.active, kblk=k_d[b], out=scores)
                    qsa.block_topk(scores, W.k, out=ids_d[b])
                else:
                    qsa.block_scores(q_d[b], k_d[b], W.active, out=scores)
                    qsa.block_topk(scores, W.k, out=ids_d[b])
                ids_h[b].copy_(ids_d[b], non_blocking=True)
                done[i].record(stream)

        run_pipeline(4)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        run_pipeline(n_e)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e, world, dev)
        assert np.array_equal(ids_h[(n_e - 1) & 1].numpy(), ids_headline.cpu().numpy())
        line["e2e"] = {"value": whole_job_rate(world, units_per_step, e_ms), "unit": UNIT, "ms_per_step": e_ms,
                       "steps": n_e, "h2d_bytes_per_step": q_h.numel() * 4 + k_h.numel() * 4,
                       "d2h_bytes_per_step": ids_h[0].numel() * 4,
                       "pipeline": "two input buffers; the H2D copy of step i+1 overlaps the kernels of step i"}
        # The same with the keys resident in device memory (copied once, as a
        # server keeps the KV cache's summary keys): per step only q goes in
        # and the ids come back. Reported beside e2e, which copies the keys too.
        for b in range(2):
            k_d[b][:W.active].copy_(k_h)
        torch.cuda.synchronize()
        run_pipeline(4, copy_keys=False)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        run_pipeline(n_e, copy_keys=False)
        e1.record(stream)
        torch.cuda.synchronize()
        r_ms = max_over_ranks(e0.elapsed_time(e1) / n_e, world, dev)
        assert np.array_equal(ids_h[(n_e - 1) & 1].numpy(), ids_headline.cpu().numpy())
        line["e2e_keys_resident"] = {"value": whole_job_rate(world, units_per_step, r_ms), "unit": UNIT,
                                     "ms_per_step": r_ms, "steps": n_e, "h2d_bytes_per_step": q_h.numel() * 4,
                                     "d2h_bytes_per_step": ids_h[0].numel() * 4,
                                     "note": "keys copied to the device once before the timed steps; no L2 "
                                             "flush between steps (the keys and scores may stay in L2)"}

    if rank == 0 and not args.no_decode:
        line["decode"] = decode_side_measurement(dev, stream)
    if rank == 0 and not args.no_attn:
        sm_mhz = (clocks or {}).get("sm_mhz") or peaks["sm_max_mhz"]
        line["attention"] = attention_side_measurement(dev, stream, sm_mhz)
    if rank == 0 and not args.no_summary:
        line["summary"] = summary_side_measurement(dev, stream)

    if rank == 0 and not args.no_ksweep and path == "gmax":
        # The headline workload's k sweep, same calls and flushes, 200 steps
        # each; ids checked against the plain path once per k.
        sweep = {}
        for ks in (64, 256, 1024):
            ids_k = torch.empty((W.nq, ks), dtype=torch.int32, device=dev)
            ids_p = torch.empty((W.nq, ks), dtype=torch.int32, device=dev)
            sc = lambda: qsa.block_scores_gmax(q, kblk, W.active, out=scores, gmax_out=gmax)
            tk = lambda: qsa.block_topk_gmax(scores, gmax, ks, out=ids_k)
            for _ in range(args.warmup):
                sc()
                tk()
            t_st = timed_steps(sc, tk, 200)
            t_s, t_k = split_steps(sc, tk, 200)
            qsa.block_topk(scores, ks, out=ids_p)
            torch.cuda.synchronize()
            assert torch.equal(ids_k, ids_p), f"k={ks}: the two top-k paths disagree"
            sweep[f"k{ks}"] = {"step_us": 1e3 * statistics.mean(t_st), "topk_us": 1e3 * statistics.mean(t_k)}
        line["k_sweep"] = sweep

    gc.enable()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_baseline(W)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
