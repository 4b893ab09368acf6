#!/usr/bin/env python
"""Benchmark of the block-batched MXFP4 MoE layer on GB300.

Workload (one GPU): the Kimi K3.1-shaped MoE layer in decode, one row per step:
d=7168, f=1536, all 896 MXFP4 experts resident in HBM (15.7 GB), top-16 softmax
routing through the bf16 router GEMV, plus the 2 Q8_0 shared experts; 100
seeded N(0,1) rows, timed one at a time.  A step is one whole layer
(moe_route -> moe_expert_block -> moe_combine) on one row.

Metric: HBM GB/s on the unique MXFP4 expert bytes the layer reads (16 experts x
17,547,264 B per row), i.e. unique expert bytes / layer time.  Inputs are
resident in HBM; L2 is flushed (256 MB write + 256 MB read) before every timed step, outside
the timed events.  Extra keys report 8- and 16-row verification blocks and the
roofline of the expert kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (under torchrun) every rank runs the same single-GPU layer on
its own GPU (replicas: the layer has no cross-GPU step); rank 0 prints.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

if "reference" in sys.argv[sys.argv.index("--impl") + 1:sys.argv.index("--impl") + 2] if "--impl" in sys.argv else False:
    # the reference arm (the CPU oracle) runs on one core: single-threaded BLAS, set
    # before numpy loads it
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as syn  # noqa: E402

SEED = 0
N_ROWS_SEEDED = 100
SLAB = 17547264
Q8_SLAB = 35094528
ROUTER_BYTES = 896 * 7168 * 2
METRIC = "MoE-layer HBM GB/s on unique MXFP4 expert bytes; layer µs at 1/8/16 rows"
UNIT = "GB/s"
WORKLOAD = ("Kimi K3.1 MoE layer decode, 1 row/step: d=7168 f=1536 E=896 top-16 + 2 Q8_0 shared, "
            "all experts resident, rows drawn in turn from 100 seeded rows")
DTYPE = ("mxfp4 weights x 5-term E2M1 (MX) activations on tcgen05 (routed experts), int8 x f16 activations "
         "on mma.sync (shared experts), fp32 accumulate, bf16 out")
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Cold-L2 reset between timed steps: write a 256 MB buffer (larger than the
    129 MB L2), then read a second 256 MB buffer so the L2 ends up holding clean
    lines and the timed step does not pay for the flush's own write-backs."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def zero_(self):
        self.w.zero_()
        self.sink.copy_(self.r.sum())


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; read-only queries)
# ---------------------------------------------------------------------------

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
            0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    def __init__(self, pci_bus_id: str | None):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thr = None
        self.ok = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if pci_bus_id is None or nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                    return
            m = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.nv, self.h = nv, h
            self.ok = True
        except OSError:
            pass

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            a = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
            b = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs))
            if a == 0:
                self.samples.append((clk.value, rs.value if b == 0 else 0))
            time.sleep(0.002)

    def start(self):
        if self.ok:
            self._thr = threading.Thread(target=self._run, daemon=True)
            self._thr.start()

    def stop(self):
        if self._thr:
            self._stop.set()
            self._thr.join()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        reasons = set()
        for _, r in busy:
            for bit, name in _REASONS.items():
                if r & bit and bit != 0x1:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in busy), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(busy)}


# ---------------------------------------------------------------------------
# CPU oracle sample (the baseline): whole layer rows through the oracle, in
# spawned worker processes with single-threaded BLAS
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name (lscpu or /proc/cpuinfo), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _oracle_row_worker(row, barrier, queue):
    """One seeded row of the 1-row Kimi decode workload through the whole oracle layer
    (router GEMV, top-16, 16 MXFP4 experts, 2 Q8_0 shared experts, combine).  Input
    creation (the row's expert slabs) happens before the barrier and is not timed."""
    from oracle import moe_oracle as orc
    sh = syn.KIMI
    router = syn.router_weight(SEED, sh)
    x = syn.x_rows(SEED, [row], sh.d_model)
    lo = orc.router_logits(x, router)
    sel = orc.select_topk(lo.astype(np.float32).astype(np.float64), sh.top_k)[0]
    slabs = {int(e): syn.mxfp4_expert_slab(SEED, int(e), sh) for e in sel}
    shared = [syn.q8_0_shared_slab(SEED, s, sh) for s in range(2)]
    barrier.wait()
    t0 = time.perf_counter()
    orc.moe_layer(x, x, sh, lambda e: slabs[e], router_w_bits=router, shared_slabs=shared)
    queue.put((row, time.perf_counter() - t0))


def oracle_layer_rows(rows):
    """Times the oracle on the given rows, one spawned process per row, all started
    together after their inputs exist.  Returns (unique expert bytes / s, wall s)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(rows))
    queue = ctx.Queue()
    procs = [ctx.Process(target=_oracle_row_worker, args=(r, barrier, queue)) for r in rows]
    for pr in procs:
        pr.start()
    times = [queue.get(timeout=900)[1] for _ in rows]
    for pr in procs:
        pr.join()
    wall = max(times)
    return len(rows) * syn.KIMI.top_k * SLAB / wall / 1e9, wall


def oracle_pairs(n_pairs: int, start: int = 0):
    """(row, expert) pairs of the workload in order: the experts each seeded row's
    oracle routing selects."""
    from oracle import moe_oracle as orc
    router = syn.router_weight(SEED, syn.KIMI)
    pairs = []
    r = 0
    while len(pairs) < start + n_pairs:
        x = syn.x_rows(SEED, [r % N_ROWS_SEEDED], syn.KIMI.d_model)
        lo = orc.router_logits(x, router)
        for e in orc.select_topk(lo.astype(np.float32).astype(np.float64), syn.KIMI.top_k)[0]:
            pairs.append((r % N_ROWS_SEEDED, int(e)))
        r += 1
    return pairs[start:start + n_pairs]


def oracle_step_seconds(pairs):
    """Times the oracle's expert MLP (slab decode + SwiGLU MLP in float64) on each
    (row, expert) pair; slab generation is input creation and is not timed."""
    from oracle import moe_oracle as orc
    times = []
    for r, e in pairs:
        x = orc.bf16_bits_to_float(syn.x_rows(SEED, [r], syn.KIMI.d_model))
        slab = syn.mxfp4_expert_slab(SEED, e, syn.KIMI)
        t0 = time.perf_counter()
        wg, wu, wd = orc.mxfp4_expert_mats(slab, syn.KIMI.d_model, syn.KIMI.d_ff)
        orc.swiglu_expert(x, wg, wu, wd)
        times.append(time.perf_counter() - t0)
    return times


def cpu_baseline(all_cores: int):
    """The oracle on this host's cores: 1 core (two rows one after the other) and all
    cores (one row per core, concurrently), single-threaded BLAS in every process."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    res = {}
    for cores, rows in ((1, "0"), (all_cores, ",".join(str(r) for r in range(all_cores)))):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--_oracle-rows", rows],
                           capture_output=True, text=True, env=env, timeout=1800)
        if r.returncode != 0:
            res[cores] = {"error": r.stderr[-300:]}
            continue
        res[cores] = json.loads(r.stdout.strip().splitlines()[-1])
    one = res.get(1, {})
    allc = res.get(all_cores, {})
    return {"value": allc.get("gbs"), "unit": UNIT, "cores": all_cores, "kind": "oracle",
            "cpu": cpu_model(),
            "one_core": {"value": one.get("gbs"), "cores": 1, "seconds": one.get("seconds")},
            "sample": f"whole 1-row layers of the Kimi decode workload (router GEMV, top-16, 16 MXFP4 experts, "
                      f"2 Q8_0 shared experts, combine) in float64: {all_cores} rows at once on {all_cores} cores "
                      f"({allc.get('seconds')} s), and 1 row on 1 core; value = unique expert bytes "
                      f"(16 x 17,547,264 per row) / time"}


# ---------------------------------------------------------------------------
# GPU layer
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the slowest rank's time); the value itself on one
    rank.  device: where the collective's tensor lives (the GPU for NCCL, CPU for gloo)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, steps: int, bytes_per_step: float, max_total_ms: float) -> float:
    """Whole-job throughput: every rank processed steps x bytes_per_step, timed by the
    slowest rank (replicas: the units of all ranks over the max time)."""
    return world * steps * bytes_per_step / (max_total_ms * 1e-3) / 1e9


def build_layer(torch, dev):
    from mxfp4_mixture_experts_router_gb300.layer import MoeLayer
    sh = syn.KIMI
    lay = MoeLayer(sh.d_model, sh.d_ff, sh.n_experts, sh.top_k, n_rows_max=16, n_shared=2, device=dev)
    router = syn.router_weight(SEED, sh)
    lay.set_router(torch.from_numpy(router.view(np.int16)).view(torch.uint16))
    lay.alloc_pool(sh.n_experts)
    threads = max(2, min(16, os.cpu_count() or 2))
    for e, slab in syn.mxfp4_slabs_parallel(SEED, range(sh.n_experts), sh, threads=threads):
        lay.put_slab(e, slab)
    lay.set_expert_slots(np.arange(sh.n_experts, dtype=np.int32))
    lay.set_shared([syn.q8_0_shared_slab(SEED, s, sh) for s in range(2)])
    return lay


class Timeline:
    """The layer's kernel timeline in its workspace (first CTA start and last CTA end of
    the routing, shared-expert and routed-expert kernels, written by the kernels
    themselves): zeroed before a step, read after it."""

    def __init__(self, torch, lay):
        self.words = lay.ws[lay.offsets.timeline: lay.offsets.timeline + 64]

    def zero_(self):
        self.words.zero_()

    def spans_us(self):
        w = self.words.cpu().numpy().view(np.uint64)
        out = {}
        for k, name in enumerate(("route", "shared_experts", "routed_experts")):
            start_inv, end = int(w[2 * k]), int(w[2 * k + 1])
            if start_inv and end:
                start = (~start_inv) & ((1 << 64) - 1)
                out[name] = ((start, end), (end - start) / 1e3)
        return out


def run_ours(args, rank, world):
    import torch

    from mxfp4_mixture_experts_router_gb300 import build as build_mod

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_mod.build()
    lay = build_layer(torch, dev)
    xs = syn.x_rows(SEED, range(N_ROWS_SEEDED), syn.KIMI.d_model)
    X = torch.from_numpy(xs.view(np.int16)).to(dev).view(torch.uint16)
    flush = L2Flush(torch, dev)
    tl = Timeline(torch, lay)
    K, W = args.steps, args.warmup

    # one captured graph per step: route -> shared experts -> routed experts -> combine
    Xs = torch.empty((1, syn.KIMI.d_model), dtype=torch.uint16, device=dev)
    Xs.copy_(X[:1])
    graph, _ = lay.capture(Xs, Xs)
    for i in range(W):
        flush.zero_()
        Xs.copy_(X[i % N_ROWS_SEEDED: i % N_ROWS_SEEDED + 1])
        graph.replay()
    torch.cuda.synchronize()
    assert lay.error_bits() == 0

    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    sampler = ClockSampler(bus if isinstance(bus, str) else None)
    layer_ms, spans = [], []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall = time.perf_counter()
    for i in range(K):
        r = (W + i) % N_ROWS_SEEDED
        flush.zero_()
        tl.zero_()
        Xs.copy_(X[r: r + 1])
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
        torch.cuda.synchronize()
        layer_ms.append(ev[i][0].elapsed_time(ev[i][1]))
        spans.append(tl.spans_us())
    wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    assert lay.error_bits() == 0
    total_ms = max_over_ranks(sum(layer_ms), world, dev)
    U = syn.KIMI.top_k  # a single row selects 16 distinct experts
    unique_bytes = U * SLAB
    value = job_gbs(world, K, unique_bytes, total_ms)
    all_bytes = unique_bytes + 2 * Q8_SLAB + ROUTER_BYTES + 3 * syn.KIMI.d_model * 2
    # routed-expert kernel, algorithmic bytes of one launch: the unique experts' slabs,
    # the row's MX_TERMS packed E2M1 activation terms with their scales, the fp32 y_part rows
    d_ = syn.KIMI.d_model
    kern_bytes = unique_bytes + 5 * (d_ // 2 + d_ // 32) + U * d_ * 4
    kern_us = [sp["routed_experts"][1] for sp in spans if "routed_experts" in sp]
    kern_avg_s = statistics.mean(kern_us) * 1e-6
    peak, peak_kind = load_peaks()
    achieved = kern_bytes / kern_avg_s / 1e9

    def seg(name):
        v = [sp[name][1] for sp in spans if name in sp]
        return round(statistics.median(v), 2) if v else None

    t0s = [min(v[0][0] for v in sp.values()) for sp in spans if sp]
    offsets = {}
    for name in ("route", "shared_experts", "routed_experts"):
        st = [sp[name][0][0] - t for sp, t in zip(spans, t0s) if name in sp]
        en = [sp[name][0][1] - t for sp, t in zip(spans, t0s) if name in sp]
        if st:
            offsets[name] = [round(statistics.median(st) / 1e3, 2), round(statistics.median(en) / 1e3, 2)]

    # end to end through the public API: one graph replay per step whose kernels read the
    # step's row from pinned host memory and write the output row to pinned host memory
    # in place (MoeLayer.capture with pinned x / residual / out: no copy launches); the
    # host puts the step's row into the pinned input buffer before the step, outside the
    # events, and the output is checked against the device-resident layer
    xh = torch.from_numpy(xs.view(np.int16)).view(torch.uint16).pin_memory()
    hin = torch.empty((1, syn.KIMI.d_model), dtype=torch.uint16).pin_memory()
    oh = torch.empty((1, syn.KIMI.d_model), dtype=torch.uint16).pin_memory()
    hin.copy_(xh[:1])
    graph_e2e, _ = lay.capture(hin, hin, out=oh)
    e2e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K + W):
        r = i % N_ROWS_SEEDED
        flush.zero_()
        hin.copy_(xh[r: r + 1])
        if i >= W:
            e2e[i - W][0].record()
        graph_e2e.replay()
        if i >= W:
            e2e[i - W][1].record()
        torch.cuda.synchronize()
        if i == W:
            Xs.copy_(hin)
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(oh, lay.out[:1].cpu()), "the host-to-host step differs from the device-resident layer"
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e), world, dev)
    e2e_value = job_gbs(world, K, unique_bytes, e2e_ms)

    # warm L2 (no flush between steps), labelled as such
    warm = []
    for i in range(max(K, 10)):
        r = i % N_ROWS_SEEDED
        Xs.copy_(X[r: r + 1])
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record()
        graph.replay()
        b_.record()
        torch.cuda.synchronize()
        warm.append(a_.elapsed_time(b_))

    med = statistics.median(layer_ms)
    blocks = {"1": {"us_median": med * 1e3, "unique_experts": U, "gbs_unique": unique_bytes / med / 1e6,
                    "frac_unique": round(unique_bytes / med / 1e6 / peak, 4),
                    "gbs_all_bytes": all_bytes / med / 1e6, "routing": "router GEMV"}}
    if not args.no_blocks:
        for sigma in (0.1, 0.5, 2.0):
            for n in (2, 4, 8, 16):
                blocks[f"{n}@{sigma}"] = time_blocks(torch, lay, X, flush, n, sigma, reps=args.block_reps, peak=peak)

    spine = time_spine(torch, flush, peak) if not args.no_blocks else None
    stacked = None
    if not args.no_stacked:
        stacked = run_stacked_legs(torch, args)
    prefill = None
    if not args.no_prefill:
        del flush  # the prefill leg makes its own flush buffer
        pf = run_prefill_bench(args, pool=(lay.pool, lay.slot_bytes, lay.n_slots))
        prefill = {"blocks": pf["blocks"], "workload": pf["config"]["workload"], "steps": args.prefill_steps}
    traffic, traffic_note = measured_traffic()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows_timed": K,
                   "rows_per_step": 1,
                   "l2": "flushed before every step (256 MB write, then 256 MB read), outside the events",
                   "parallelism": f"replicas x{world}"},
        "layer_us_p10_p50_p90": [float(np.percentile(layer_ms, q)) * 1e3 for q in (10, 50, 90)],
        "layer_us_warm_l2_median": round(statistics.median(warm) * 1e3, 2),
        "all_bytes_gbs": world * K * all_bytes / (total_ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "moe::tc::tc_expert_kernel", "peak_kind": peak_kind,
                     "bytes_per_launch": kern_bytes, "avg_launch_us": round(kern_avg_s * 1e6, 2),
                     "timing": "the kernel's own timeline: first CTA start to last CTA end (%globaltimer), "
                               "in the layer", "traffic_source": traffic_note},
        "kernel_spans_us_median": {"route": seg("route"), "shared_experts": seg("shared_experts"),
                                   "routed_experts": seg("routed_experts")},
        "kernel_start_end_us_median": offsets,
        "blocks": blocks,
        "spine_q8_0_matmul": spine,
        "prefill": prefill,
        "stacked": stacked,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": syn.KIMI.d_model * 2,
                "d2h_bytes_per_step": syn.KIMI.d_model * 2,
                "transfer": "the step's row in pinned host memory, read in place by the kernels; the output "
                            "row written in place to pinned host memory (one graph replay per step)"},
        "gpu_launches": K * 4,
        "timing": "one CUDA graph per step (route, shared experts, routed experts, combine chained on one "
                  "stream), CUDA events around the replay; kernel spans from the kernels' own timeline",
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    return line


SPINE_SHAPES = [(7168, 1536), (1536, 12288), (8192, 7168)]


def time_spine(torch, flush, peak, reps=10):
    """Q8_0 spine matmuls (q8_0_block_matmul) at attention-projection shapes for blocks
    of 1, 8 and 16 rows: weight bytes (int8 codes + fp16 scales, each read once per
    block) / kernel time, L2 flushed before each call, CUDA events around the call."""
    from mxfp4_mixture_experts_router_gb300 import binding as B
    out = {}
    for k_in, n_out in SPINE_SHAPES:
        key = int(syn.stream_key(SEED, 77, k_in, n_out))
        q = torch.from_numpy((syn.u64(key, 0, n_out * k_in // 8).view(np.int8))).cuda()
        dq = torch.from_numpy(((1e-3 + 9e-3 * syn.uniform01(key + 1, 0, n_out * k_in // 32)).astype(np.float16))
                              .view(np.int16)).cuda()
        wbytes = n_out * k_in + 2 * n_out * (k_in // 32)
        for n in (1, 8, 16):
            x = torch.from_numpy(syn.x_rows(SEED, range(n), k_in).view(np.int16)).cuda().view(torch.uint16)
            ws = torch.zeros(B.q8_0_workspace_size(n, k_in, n_out), dtype=torch.uint8, device="cuda")
            y = torch.empty((n, n_out), dtype=torch.float32, device="cuda")
            ts = []
            for r in range(reps + 3):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                B.q8_0_block_matmul(n, k_in, n_out, x, B.MOE_DTYPE_BF16, q, dq, None, None, B.MOE_EPI_NONE, y, ws)
                b.record()
                torch.cuda.synchronize()
                if r >= 3:
                    ts.append(a.elapsed_time(b))
            t = statistics.median(ts)
            out[f"{k_in}x{n_out}@{n}"] = {"us_median": round(t * 1e3, 2), "gbs": round(wbytes / t / 1e6, 1),
                                          "frac": round(wbytes / t / 1e6 / peak, 4)}
    return out


def measured_traffic():
    """DRAM bytes (read + write) of one routed-expert launch on this workload from an ncu
    capture, if one was recorded for the kernel source as it is now: profiles/ holds the
    capture's figure with the SHA-256 of csrc/experts_tc.cu it was taken on."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "routed_kernel_traffic.json")) as fh:
            rec = json.load(fh)
        with open(os.path.join(ROOT, "mxfp4_mixture_experts_router_gb300", "csrc", "experts_tc.cu"), "rb") as fh:
            sha = hashlib.sha256(fh.read()).hexdigest()
    except (OSError, ValueError):
        return None, "no ncu capture recorded"
    if rec.get("source_sha256") != sha:
        return None, "the recorded ncu capture is of an earlier version of the kernel"
    return int(rec["dram_bytes_per_launch"]), rec.get("command", "ncu")


def time_blocks(torch, lay, X, flush, n, sigma, reps, peak):
    """Verification blocks of n rows: shared N(0,1) base logits + N(0, sigma) per-row
    noise (caller logits), one captured graph replayed per block, L2 flushed before each."""
    dev = X.device
    Xs = torch.empty((n, syn.KIMI.d_model), dtype=torch.uint16, device=dev)
    Ls = torch.empty((n, syn.KIMI.n_experts), dtype=torch.float32, device=dev)
    lgs = [torch.from_numpy(syn.block_logits(SEED, n, syn.KIMI.n_experts, sigma, block=b)).to(dev)
           for b in range(reps + 3)]
    Xs.copy_(X[:n])
    Ls.copy_(lgs[0])
    graph, _ = lay.capture(Xs, Xs, logits_in=Ls)
    graph.replay()
    torch.cuda.synchronize()
    ts, us = [], []
    for b in range(reps + 3):
        x0 = (b * n) % (N_ROWS_SEEDED - n)
        flush.zero_()
        Xs.copy_(X[x0: x0 + n])
        Ls.copy_(lgs[b])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if b >= 3:
            ts.append(e0.elapsed_time(e1))
            us.append(int(lay.ws_view(lay.offsets.n_unique, 1, torch.int32).item()))
    t = statistics.median(ts)
    u = statistics.mean(us)
    allb = u * SLAB + 2 * Q8_SLAB + 3 * n * syn.KIMI.d_model * 2
    return {"us_median": round(t * 1e3, 2), "unique_experts": u, "gbs_unique": round(u * SLAB / t / 1e6, 1),
            "frac_unique": round(u * SLAB / t / 1e6 / peak, 4), "gbs_all_bytes": round(allb / t / 1e6, 1),
            "routing": "caller logits", "blocks_timed": reps}


def run_profile_case(args):
    """Small case for `ncu --set full`: the Kimi-shaped layer on one row with router-GEMV
    routing, but a pool holding only the 32 experts with the largest float32 logits
    (about 0.6 GB on the device instead of 15.7 GB); four layers, L2 flushed before each."""
    import torch

    from mxfp4_mixture_experts_router_gb300 import build as build_mod
    from mxfp4_mixture_experts_router_gb300.layer import MoeLayer
    build_mod.build()
    sh = syn.KIMI
    rows = list(range(args.profile_rows))
    x = syn.x_rows(SEED, rows, sh.d_model)
    router = syn.router_weight(SEED, sh)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    wf = (router.astype(np.uint32) << 16).view(np.float32)
    lo = xf @ wf.T
    experts = sorted(set(np.argsort(-lo, axis=1)[:, :32].ravel().tolist()))
    lay = MoeLayer(sh.d_model, sh.d_ff, sh.n_experts, sh.top_k, n_rows_max=16, n_shared=2)
    lay.set_router(torch.from_numpy(router.view(np.int16)).view(torch.uint16))
    lay.alloc_pool(len(experts))
    slots = np.zeros(sh.n_experts, dtype=np.int32)
    for i, (e, slab) in enumerate(syn.mxfp4_slabs_parallel(SEED, experts, sh)):
        lay.put_slab(i, slab)
        slots[e] = i
    lay.set_expert_slots(slots)
    lay.set_shared([syn.q8_0_shared_slab(SEED, s, sh) for s in range(2)])
    X = torch.from_numpy(x.view(np.int16)).cuda().view(torch.uint16)
    flush = L2Flush(torch, torch.device("cuda"))
    for _ in range(4):
        flush.zero_()
        lay.forward(X, X)
    torch.cuda.synchronize()
    assert lay.error_bits() == 0
    print(json.dumps({"profile_case": "ok", "rows": len(rows), "pool_experts": len(experts)}))


def run_spine_profile_case(args):
    """Small case for `ncu`: the Q8_0 spine matmul 7168 -> 1536 on one row (11.8 MB of
    weights, the first of SPINE_SHAPES), four calls, L2 flushed before each."""
    import torch

    from mxfp4_mixture_experts_router_gb300 import binding as B
    from mxfp4_mixture_experts_router_gb300 import build as build_mod
    build_mod.build()
    k_in, n_out = SPINE_SHAPES[0]
    n = args.profile_rows
    key = int(syn.stream_key(SEED, 77, k_in, n_out))
    q = torch.from_numpy(syn.u64(key, 0, n_out * k_in // 8).view(np.int8)).cuda()
    dq = torch.from_numpy(((1e-3 + 9e-3 * syn.uniform01(key + 1, 0, n_out * k_in // 32)).astype(np.float16))
                          .view(np.int16)).cuda()
    x = torch.from_numpy(syn.x_rows(SEED, range(n), k_in).view(np.int16)).cuda().view(torch.uint16)
    ws = torch.zeros(B.q8_0_workspace_size(n, k_in, n_out), dtype=torch.uint8, device="cuda")
    y = torch.empty((n, n_out), dtype=torch.float32, device="cuda")
    flush = L2Flush(torch, torch.device("cuda"))
    for _ in range(4):
        flush.zero_()
        B.q8_0_block_matmul(n, k_in, n_out, x, B.MOE_DTYPE_BF16, q, dq, None, None, B.MOE_EPI_NONE, y, ws)
    torch.cuda.synchronize()
    assert B.moe_get_error(ws) == 0
    print(json.dumps({"spine_profile_case": "ok", "shape": [k_in, n_out], "rows": n}))


def gpu_body_pool(torch, n_bodies: int, seed: int):
    """n_bodies synthetic MXFP4 expert slabs in a pinned host pool, drawn on the GPU
    from a seeded generator: uniform code bytes, E8M0 scale bytes 120 + (byte mod 8)
    (the exponent range of the seeded slabs), then copied to pinned host memory."""
    sh = syn.KIMI
    d, f = sh.d_model, sh.d_ff
    per = f * d // 2 + f * d // 32
    planes = [(f * d // 2, f * d // 32), (per + f * d // 2, f * d // 32), (2 * per + d * f // 2, d * f // 32)]
    host = torch.empty((n_bodies, SLAB), dtype=torch.uint8).pin_memory()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    for b0 in range(0, n_bodies, 16):
        m = min(16, n_bodies - b0)
        buf = torch.randint(0, 256, (m, SLAB), dtype=torch.uint8, device="cuda", generator=gen)
        for off, cnt in planes:
            buf[:, off:off + cnt] = 120 + (buf[:, off:off + cnt] & 7)
        host[b0:b0 + m].copy_(buf)
    torch.cuda.synchronize()
    return host


class StackedDecode:
    """92 stacked Kimi-shaped MoE layers (routed experts only) served from a device
    expert cache through the real decode flow (GPU routing -> host slot requests ->
    resident-first expert kernel).  (layer, expert) maps to one of n_bodies slabs of a
    pinned host pool; router logits per layer = a fixed per-layer popularity N(0,1) + a
    block base drifting as AR(1) (rho 0.9) + per-row noise N(0, 0.5)."""

    def __init__(self, torch, args):
        from mxfp4_mixture_experts_router_gb300.layer import MoeLayer
        sh = syn.KIMI
        self.torch = torch
        self.L, self.NB, self.slots = args.cache_layers, args.cache_bodies, args.cache_slots
        self.E, self.k, self.d = sh.n_experts, sh.top_k, sh.d_model
        t0 = time.perf_counter()
        self.host = gpu_body_pool(torch, self.NB, SEED + 5)
        base = np.uint64(self.host.data_ptr())
        body = np.array([[syn.body_of(l, e, self.NB) for e in range(self.E)] for l in range(self.L)], dtype=np.uint64)
        self.body_ptr = lambda l, ex: (base + body[l, np.asarray(ex, dtype=np.int64)] * np.uint64(SLAB)).astype(np.uint64)
        self.lay = MoeLayer(self.d, sh.d_ff, self.E, self.k, n_rows_max=16, n_shared=0)
        self.x = torch.from_numpy(syn.x_rows(SEED, range(16), self.d).view(np.int16)).cuda().view(torch.uint16)
        self.setup_s = time.perf_counter() - t0

    def logits_stream(self, seed):
        rng = np.random.default_rng(seed)
        bias = rng.normal(size=(self.L, self.E)).astype(np.float32)
        state = rng.normal(size=(self.L, self.E)).astype(np.float32)
        rho = 0.9

        def next_block(n):
            nonlocal state
            state = (rho * state + np.sqrt(1 - rho * rho) * rng.normal(size=(self.L, self.E))).astype(np.float32)
            lg = bias[:, None, :] + state[:, None, :] + 0.5 * rng.normal(size=(self.L, n, self.E))
            return self.torch.from_numpy(np.ascontiguousarray(lg, dtype=np.float32)).cuda()
        return next_block

    def run(self, policy, prefetch, n, warm, timed, seed=SEED + 1, plain_rows=None):
        """Blocks of n rows through all layers; returns seconds per block (median), the
        cache's counters over the timed blocks and the unique experts per layer."""
        from mxfp4_mixture_experts_router_gb300.cache import CachedLayerRunner, DeviceExpertCache
        torch = self.torch
        cache = DeviceExpertCache(self.d, syn.KIMI.d_ff, self.E, self.k, n_slots=self.slots, n_streams=8,
                                  policy=policy)
        runner = CachedLayerRunner(cache, self.lay, self.body_ptr, prefetch=prefetch)
        nxt = self.logits_stream(seed)
        secs, unique, st0 = [], 0, None
        try:
            for blk in range(warm + timed):
                lg = nxt(n)
                torch.cuda.synchronize()
                cache.sync()
                if blk == warm:
                    st0 = cache.stats()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for l in range(self.L):
                    u, _ = runner.run_layer(l, n, self.x, lg[l], self.L)
                    if blk >= warm:
                        unique += u
                b.record()
                torch.cuda.synchronize()
                cache.sync()
                if blk >= warm:
                    secs.append(a.elapsed_time(b) * 1e-3)
            st = cache.stats()
            err = self.lay.error_bits()
        finally:
            cache.close()
        d = {k: st[k] - st0[k] for k in ("hits", "misses", "bytes_uploaded")}
        t = statistics.median(secs)
        return {"s_per_block": t, "sum_s": sum(secs), "hits": d["hits"], "misses": d["misses"],
                "hit_rate": round(d["hits"] / max(1, d["hits"] + d["misses"]), 4),
                "h2d_gbs": round(d["bytes_uploaded"] / sum(secs) / 1e9, 1),
                "hbm_expert_gbs": round(unique * SLAB / sum(secs) / 1e9, 1),
                "unique_experts_per_layer": round(unique / (timed * self.L), 1), "error_bits": err,
                "prefetched": runner.prefetched, "prefetch_uploads": runner.prefetch_uploads}


def run_stacked_legs(torch, args):
    """The device-expert-cache leg (8-row blocks, both eviction policies, with and
    without the shallow next-layer prefetch) and the block-verification harness
    (16-row blocks with synthetic accept-up-to-first-disagreement against 16 plain
    1-row steps), all through the real decode flow."""
    from mxfp4_mixture_experts_router_gb300 import binding as B
    sd = StackedDecode(torch, args)
    out = {"workload": f"{sd.L} Kimi K3.1 MoE layers (routed experts only), {sd.NB} seeded bodies in a pinned "
                       f"host pool ({sd.NB * SLAB / 1e9:.1f} GB), {sd.slots}-slot device cache "
                       f"({sd.slots * SLAB / 1e9:.1f} GB), 8 upload streams; per layer: GPU routing -> host "
                       f"slot requests -> resident-first expert kernel", "setup_s": round(sd.setup_s, 1)}
    cache = {}
    for policy, pname in ((B.MOE_CACHE_LRU, "lru"), (B.MOE_CACHE_KEEP_MULTI_ROW, "keep_multi_row")):
        for pf in (0, 8):
            r = sd.run(policy, pf, 8, warm=args.cache_warmup, timed=args.cache_blocks)
            r["tok_s"] = round(8 / r["s_per_block"], 2)
            cache[f"{pname}{'+prefetch8' if pf else ''}"] = r
    out["cache_8row_blocks_all_accepted"] = cache
    # block verification: 16-row blocks, each draft row accepted with probability 0.7 up
    # to the first rejection (+1 token the block itself yields), against plain steps
    rng = np.random.default_rng(SEED + 11)
    blocks = sd.run(B.MOE_CACHE_KEEP_MULTI_ROW, 8, 16, warm=1, timed=args.verify_blocks, seed=SEED + 21)
    accepted = []
    for _ in range(max(200, args.verify_blocks)):
        a = 0
        while a < 15 and rng.random() < 0.7:
            a += 1
        accepted.append(a + 1)
    tok_per_block = statistics.mean(accepted)
    plain = sd.run(B.MOE_CACHE_KEEP_MULTI_ROW, 8, 1, warm=2, timed=args.verify_plain_steps, seed=SEED + 21)
    out["block_verification"] = {
        "block_rows": 16, "accept_rule": "each draft row accepted with probability 0.7 up to the first rejection",
        "tokens_per_block_mean": round(tok_per_block, 2),
        "block_s": round(blocks["s_per_block"], 4), "plain_step_s": round(plain["s_per_block"], 4),
        "sixteen_plain_steps_s": round(16 * plain["s_per_block"], 4),
        "tok_s_blocks": round(tok_per_block / blocks["s_per_block"], 2),
        "tok_s_plain": round(1 / plain["s_per_block"], 2),
        "block_hit_rate": blocks["hit_rate"], "plain_hit_rate": plain["hit_rate"],
        "blocks_timed": args.verify_blocks, "plain_steps_timed": args.verify_plain_steps,
        # the block's cost does not depend on how many drafts are accepted: tokens per block
        # for other acceptance probabilities p, in closed form (sum of p^j, j = 0..15)
        "tok_s_blocks_by_acceptance": {
            str(q): round(sum(q ** j for j in range(16)) / blocks["s_per_block"], 2) for q in (0.5, 0.7, 0.8, 0.9)}}
    return out


def run_prefill_bench(args, pool=None):
    """Prefill blocks of 270 and 1,533 rows through the whole layer (routing, routed
    experts on the block-scaled tcgen05 path, the 2 Q8_0 shared experts, combine), all
    896 experts resident, independent N(0,1) router logits per row, L2 flushed before
    every block outside the events.  pool: (tensor, slot_bytes, n_slots) of an
    existing resident pool to reuse."""
    import torch

    from mxfp4_mixture_experts_router_gb300 import binding as B
    from mxfp4_mixture_experts_router_gb300 import build as build_mod
    from mxfp4_mixture_experts_router_gb300.layer import MoeLayer

    build_mod.build()
    sh = syn.KIMI
    E, k, d = sh.n_experts, sh.top_k, sh.d_model
    sizes = [int(v) for v in args.prefill_rows.split(",")]
    nmax = max(sizes)
    lay = MoeLayer(d, sh.d_ff, E, k, n_rows_max=nmax, n_shared=2)
    if pool is None:
        lay.alloc_pool(E)
        threads = max(2, min(16, os.cpu_count() or 2))
        for e, slab in syn.mxfp4_slabs_parallel(SEED, range(E), sh, threads=threads):
            lay.put_slab(e, slab)
    else:  # the decode layer's resident pool
        lay.attach_pool(*pool)
    lay.set_expert_slots(np.arange(E, dtype=np.int32))
    lay.set_shared([syn.q8_0_shared_slab(SEED, s, sh) for s in range(2)])
    flush = L2Flush(torch, torch.device("cuda"))
    peak, peak_kind = load_peaks()
    res = {}
    for n in sizes:
        rng = np.random.default_rng(SEED + n)
        x = torch.from_numpy(syn.x_rows(SEED, range(n), d).view(np.int16)).cuda().view(torch.uint16)
        ts, us = [], []
        for rep in range(args.prefill_warmup + args.prefill_steps):
            lg = torch.from_numpy(rng.normal(size=(n, E)).astype(np.float32)).cuda()
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            lay.forward(x, x, logits_in=lg, mode=B.MOE_MODE_PREFILL)
            b.record()
            torch.cuda.synchronize()
            if rep >= args.prefill_warmup:
                ts.append(a.elapsed_time(b) * 1e-3)
                us.append(int(lay.ws_view(lay.offsets.n_unique, 1, torch.int32).item()))
        assert lay.error_bits() == 0
        t = statistics.median(ts)
        u = statistics.mean(us)
        gbs = u * SLAB / t / 1e9
        res[str(n)] = {"ms_median": round(t * 1e3, 3), "unique_experts": u, "gbs_unique": round(gbs, 1),
                       "frac_of_hbm_peak": round(gbs / peak, 4),
                       "gbs_all_bytes": round((u * SLAB + 2 * Q8_SLAB) / t / 1e9, 1),
                       "tflops": round(2 * 3 * n * (k + 2) * d * sh.d_ff / t / 1e12, 1)}
    return {"metric": "prefill layer ms and GB/s on unique MXFP4 expert bytes",
            "unit": "GB/s", "value": res[str(nmax)]["gbs_unique"], "n_gpus": 1,
            "config": {"workload": "Kimi K3.1 MoE layer prefill: routing, 16 routed experts per row, 2 Q8_0 shared "
                                   "experts, combine; all 896 experts resident, independent N(0,1) logits per row",
                       "rows": sizes, "steps": args.prefill_steps,
                       "l2": "flushed before every block, outside the events"},
            "peak_gbs": peak, "peak_kind": peak_kind, "blocks": res, "data": "synthetic"}


def run_prefill_profile_case(args):
    """Small prefill case for ncu: 270 rows whose router logits favour 160 of the 896
    experts (+8 on those), so each selected expert gets about 27 (row, slot) pairs, as in
    the 1,533-row block with all experts; a pool of those 160 experts (2.8 GB).  Four
    blocks, L2 flushed before each."""
    import torch

    from mxfp4_mixture_experts_router_gb300 import binding as B
    from mxfp4_mixture_experts_router_gb300 import build as build_mod
    from mxfp4_mixture_experts_router_gb300.layer import MoeLayer

    build_mod.build()
    sh = syn.KIMI
    E, k, d, n = sh.n_experts, sh.top_k, sh.d_model, 270
    rng = np.random.default_rng(SEED + 7)
    hot = np.sort(rng.choice(E, size=160, replace=False))
    lg = rng.normal(size=(n, E)).astype(np.float32)
    lg[:, hot] += 8.0
    lay = MoeLayer(d, sh.d_ff, E, k, n_rows_max=n, n_shared=0)
    lay.alloc_pool(len(hot))
    slots = np.zeros(E, dtype=np.int32)
    threads = max(2, min(16, os.cpu_count() or 2))
    for i, (e, slab) in enumerate(syn.mxfp4_slabs_parallel(SEED, hot.tolist(), sh, threads=threads)):
        lay.put_slab(i, slab)
        slots[e] = i
    lay.set_expert_slots(slots)
    x = torch.from_numpy(syn.x_rows(SEED, range(n), d).view(np.int16)).cuda().view(torch.uint16)
    L = torch.from_numpy(lg).cuda()
    flush = L2Flush(torch, torch.device("cuda"))
    for _ in range(4):
        flush.zero_()
        lay.forward(x, x, logits_in=L, mode=B.MOE_MODE_PREFILL)
    torch.cuda.synchronize()
    assert lay.error_bits() == 0
    u = int(lay.ws_view(lay.offsets.n_unique, 1, torch.int32).item())
    print(json.dumps({"prefill_profile_case": "ok", "rows": n, "unique_experts": u, "pairs": n * k}))


def run_reference(args):
    """The CPU oracle timed on this host's cores: each step is the oracle's expert MLP
    of one (row, selected expert) pair of the workload (17,547,264 expert bytes)."""
    K, W = args.steps, args.warmup
    pairs = oracle_pairs(K + W)
    secs = oracle_step_seconds(pairs)[W:]
    total = sum(secs)
    value = K * SLAB / total / 1e9
    cores = 1  # BLAS pinned to one thread before numpy was imported
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
            "steps": K, "warmup": W, "ms_per_step": total / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "rows_per_step": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "cpu": cpu_model(),
                             "sample": "each step one (row, selected expert) fp64 expert MLP of the workload "
                                       "(17,547,264 expert bytes); the metric's unit scaled from it"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-blocks", action="store_true")
    ap.add_argument("--block-reps", type=int, default=10)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-stacked", action="store_true")
    ap.add_argument("--verify-blocks", type=int, default=2)
    ap.add_argument("--verify-plain-steps", type=int, default=8)
    ap.add_argument("--_oracle-rows", default="", dest="oracle_rows")
    ap.add_argument("--profile-case", action="store_true",
                    help="run the small ncu case (a few layers, <1 GB on the device) and exit")
    ap.add_argument("--profile-rows", type=int, default=1)
    ap.add_argument("--cache-bench", action="store_true",
                    help="only the stacked legs (device expert cache, block verification; one JSON line) and exit")
    ap.add_argument("--cache-layers", type=int, default=92)
    ap.add_argument("--cache-bodies", type=int, default=1024)
    ap.add_argument("--cache-slots", type=int, default=1567)
    ap.add_argument("--cache-blocks", type=int, default=2)
    ap.add_argument("--cache-warmup", type=int, default=1)
    ap.add_argument("--prefill-bench", action="store_true",
                    help="prefill blocks through the layer (one JSON line) and exit")
    ap.add_argument("--prefill-rows", default="270,1533")
    ap.add_argument("--prefill-steps", type=int, default=5)
    ap.add_argument("--prefill-warmup", type=int, default=2)
    ap.add_argument("--spine-profile-case", action="store_true",
                    help="run the small Q8_0 spine matmul case for ncu and exit")
    ap.add_argument("--prefill-profile-case", action="store_true",
                    help="run the small prefill ncu case (270 rows over 160 experts, 2.8 GB) and exit")
    args = ap.parse_args()

    if args.spine_profile_case:
        run_spine_profile_case(args)
        return
    if args.prefill_profile_case:
        run_prefill_profile_case(args)
        return

    if args.prefill_bench:
        print(json.dumps(run_prefill_bench(args)))
        return

    if args.cache_bench:
        import torch
        from mxfp4_mixture_experts_router_gb300 import build as build_mod
        build_mod.build()
        print(json.dumps({"metric": "stacked decode through the device expert cache", "unit": "tok/s",
                          "n_gpus": 1, "data": "synthetic", "stacked": run_stacked_legs(torch, args)}))
        return

    if args.profile_case:
        run_profile_case(args)
        return

    if args.oracle_rows:
        gbs, secs = oracle_layer_rows([int(v) for v in args.oracle_rows.split(",")])
        print(json.dumps({"gbs": round(gbs, 5), "seconds": round(secs, 2)}))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(max(1, min(16, os.cpu_count() or 1)))
        print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
