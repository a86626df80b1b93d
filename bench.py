"""Benchmark: FP8 W8A8 MoE grouped GEMM, decode sweep, on GB300.

Workload: K=4096, N=14336, E=8, top_k=2, M in {64, 128, 256, 512}; A bf16
N(0,1), W N(0,1/K) quantised per output channel to e4m3, router logits N(0,1)
-> softmax -> top-2 (renormalised).  One step = one pass of the whole path for
each M: moe_align_quant_fp8 (moe_align_block_size and the per-token e4m3
quantisation, rows written in padded sorted order, in one launch) ->
moe_gemm_w8a8 (PADDED activation tiles by TMA, SLOT output [M, 2, N] bf16 with
the routing-weight multiply).  Weights (470 MB of e4m3)
exceed the 129 MB L2, so every GEMM streams them from HBM.

value  = algorithmic bytes of the four GEMMs / device time of the timed steps
         (bytes: weights of the experts hit + their scales + A codes and scales
         + routing + bf16 output), in GB/s; the line also carries TFLOPS.
e2e    = the same metric through the public API with pinned host buffers: per
         step the activations and routing go host -> device and the outputs
         device -> host inside the timed region (copies on their own streams,
         overlapping the kernels of other shapes); the calls of up to 100 steps are
         captured into a CUDA graph that is replayed (the figure with every call
         enqueued by the host as it runs is reported beside it).
roofline = the grouped GEMM kernel alone (CUDA events around each launch).
layers = the compute-bound M=4096 up and down GEMMs of the Mixtral-8x7B- and
         8x22B-shaped layers, each timed alone (median of 20 launches after an
         L2 flush, own clock record), as fractions of the dense FP8 rate that
         cuBLAS reaches on the same GPU in the same run (8192^3, burst).
cpu_baseline / --impl reference = the CPU oracle on a bounded sample of slots.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       python bench.py --suite [--only TEXT]        (every other kernel, timed alone)
       python bench.py --tile-sweep [--only TEXT]   (one-SM against CTA-pair GEMM tiles)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

K_DIM, N_DIM, E, TOP_K = 4096, 14336, 8, 2
SWEEP_M = (64, 128, 256, 512)
METRIC = "MoE grouped GEMM TFLOPS & GB/s (M,K,N,E=8,top2) vs GB300 roofline, 1 GPU"
WORKLOAD = "decode fp8 w8a8 sweep M={64,128,256,512} K=4096 N=14336 E=8 top2"
# "Tianxing/moe quantization" FP8_W8A8 table rows for this sweep: (M, TFLOPS, GB/s)
PAGE_ROWS = ((64, 47.124442, 1480.603863), (128, 93.602312, 1478.376964),
             (256, 166.424183, 1358.410607), (512, 314.778601, 1296.118960))


def slot_tile(M: int) -> int:
    """Slot tile (BM) per M: 64 or 128, the smaller when it holds twice the mean
    slots per expert (both run the wide tile: 256 weight rows against 64 or 128
    slots; the swapped tiles of BM 16 and 32 measured slower at decode)."""
    mean = 2 * M * TOP_K // E
    return 64 if mean <= 64 else 128


def algorithmic_bytes(M: int, ids: np.ndarray) -> int:
    T = M * TOP_K
    hit = len(np.unique(ids))
    return (hit * N_DIM * K_DIM          # e4m3 weights of the experts hit
            + hit * N_DIM * 4            # their per-channel scales
            + M * K_DIM + M * 4          # e4m3 activations + per-token scales
            + T * 8                      # topk ids + weights
            + T * N_DIM * 2)             # bf16 output


def flops(M: int) -> float:
    return 2.0 * M * TOP_K * K_DIM * N_DIM


def page_aggregate():
    t = [flops(m) / (tf * 1e12) for m, tf, _ in PAGE_ROWS]
    b = [gbs * 1e9 * ti for (_, _, gbs), ti in zip(PAGE_ROWS, t)]
    return sum(b) / sum(t) / 1e9, sum(flops(m) for m in SWEEP_M) / sum(t) / 1e12


def recorded_traffic():
    """DRAM bytes per step of the GEMM launches from the committed ncu record,
    or None when the kernel sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gemm_fp8_decode_sweep_traffic.json")
    try:
        rec = json.load(open(path))
        h = hashlib.sha256()
        for src in rec["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return int(rec["traffic_bytes_per_step"])
    except Exception:
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------- clocks ---
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"qmoe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ GPU setup ---
def setup(dev, seed_base=1000):
    import torch

    import quantized_moe_grouped_gb300 as q
    from quantized_moe_grouped_gb300 import inputs

    q.load_library()
    wq = torch.empty(E, N_DIM, K_DIM, dtype=torch.uint8, device=dev)
    ws = torch.empty(E, N_DIM, dtype=torch.float32, device=dev)
    for e in range(E):                      # weights shared by the sweep (seed of the first shape)
        we = torch.from_numpy(inputs.expert_weight_f32(N_DIM, K_DIM, seed_base, e)).to(dev)
        qe, se = q.quant_weight_fp8(we)
        wq[e].copy_(qe)
        ws[e].copy_(se)
        del we
    shapes = []
    for i, M in enumerate(SWEEP_M):
        seed = seed_base + i
        a_bits = inputs.activations_bf16(M, K_DIM, seed)
        ids, tw = inputs.routing(M, E, TOP_K, seed)
        BM = slot_tile(M)
        T = M * TOP_K
        sh = dict(M=M, BM=BM, ids_np=ids, tw_np=tw, a_np=a_bits,
                  a=torch.from_numpy(a_bits.view(np.int16)).to(dev).view(torch.bfloat16),
                  ids=torch.from_numpy(ids).to(dev), tw=torch.from_numpy(tw).to(dev),
                  align=q.alloc_align_outputs(T, E, BM, dev),
                  aq=torch.empty(q.align_max_padded(T, E, BM), K_DIM, dtype=torch.uint8, device=dev),
                  sa=torch.empty(q.align_max_padded(T, E, BM), dtype=torch.float32, device=dev),
                  out=torch.empty(T, N_DIM, dtype=torch.bfloat16, device=dev),
                  bytes=algorithmic_bytes(M, ids), flops=flops(M))
        # pinned host buffers for the end-to-end leg
        sh["a_h"] = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        sh["ids_h"] = torch.from_numpy(ids).pin_memory()
        sh["tw_h"] = torch.from_numpy(tw).pin_memory()
        sh["out_h"] = torch.empty(T, N_DIM, dtype=torch.bfloat16).pin_memory()
        shapes.append(sh)
    return q, wq, ws, shapes


def run_path(q, wq, ws, sh, stream, ev=None):
    """One pass of the path for one shape; ev = (before_gemm, after_gemm) events or None."""
    q.moe_align_quant_fp8(sh["a"], sh["ids"], E, sh["BM"], align=sh["align"], q=sh["aq"], scale=sh["sa"],
                          stream=stream)
    if ev is not None:
        ev[0].record(stream)
    q.moe_gemm_w8a8(sh["aq"], sh["sa"], wq, ws, sh["align"], sh["tw"], M=sh["M"], top_k=TOP_K, BM=sh["BM"],
                    a_layout=q.A_PADDED, out=sh["out"], stream=stream)
    if ev is not None:
        ev[1].record(stream)


# ---------------------------------------------------------- CPU oracle ---
class OracleBench:
    """The CPU oracle (dense per-token expert loop in fp64, as it stands) on a
    bounded random sample of slots of the M=64 shape; the measured per-slot time
    is extrapolated to every slot of the sweep (the oracle's cost per slot does
    not depend on M)."""

    def __init__(self, seed_base=1000):
        import oracle
        from quantized_moe_grouped_gb300 import inputs
        self.oracle = oracle
        self.cores = oracle.num_threads()
        self.rwq = np.empty((E, N_DIM, K_DIM), dtype=np.uint8)
        self.rws = np.empty((E, N_DIM), dtype=np.float32)
        for e in range(E):
            self.rwq[e], self.rws[e] = oracle.quant_rows_fp8_f32(inputs.expert_weight_f32(N_DIM, K_DIM, seed_base, e))
        M = SWEEP_M[0]
        a = inputs.activations_bf16(M, K_DIM, seed_base)
        self.ids, self.tw = inputs.routing(M, E, TOP_K, seed_base)
        self.raq, self.rsa = oracle.quant_rows_fp8_bf16(a)
        self.T = M * TOP_K
        self.sweep_slots = sum(m * TOP_K for m in SWEEP_M)
        self.sweep_bytes = sum(algorithmic_bytes(m, inputs.routing(m, E, TOP_K, seed_base + i)[0])
                               for i, m in enumerate(SWEEP_M))
        self.rng = np.random.default_rng(0)

    def run(self, seconds: float):
        """Batches of one slot per thread, drawn at random from the M=64 shape's
        slots, until `seconds` of oracle time have passed (at least one batch)."""
        o = self.oracle
        n, elapsed, done = min(max(self.cores, 1), self.T), 0.0, 0
        while done == 0 or elapsed < seconds:
            slots = self.rng.choice(self.T, n, replace=False)
            t0 = time.perf_counter()
            o.moe_gemm(a_kind=o.A_FP8_TOKEN, a=self.raq, a_scale=self.rsa, w_kind=o.W_FP8, w=self.rwq,
                       w_scale=self.rws, topk_ids=self.ids, topk_w=self.tw, E=E, slots=slots)
            elapsed += time.perf_counter() - t0
            done += n
        t_sweep = self.sweep_slots * elapsed / done
        sample = (f"{done} slots drawn at random from the {self.T} of the M=64 shape (K=4096, N=14336; fp64 "
                  f"dense per-slot loop) in {elapsed:.1f} s on {self.cores} threads; per-slot time extrapolated "
                  f"to the {self.sweep_slots} slots of the sweep")
        return self.sweep_bytes / t_sweep / 1e9, t_sweep, sample


def dist_env() -> tuple[int, int, int]:
    """(world size, rank, local rank) from torchrun's environment; (1, 0, 0) without it."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's);
    x itself on one rank.  Every rank must call it."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds: float, world: int) -> float:
    """Units per second of the whole job: every rank processes units_per_rank
    (weak scaling) in at most `seconds` (the max over ranks)."""
    return world * units_per_rank / seconds


def run_reference(args) -> None:
    _, rank, _ = dist_env()
    if rank != 0:  # the oracle runs on rank 0 alone; the other ranks exit without work
        return
    steps, warmup = args.steps, args.warmup
    per_step = min(6.0, 120.0 / max(1, steps + warmup))  # one slot batch at least
    ob = OracleBench()
    vals, times = [], []
    sample = None
    for i in range(warmup + steps):
        v, t_sweep, sample = ob.run(per_step)
        if i >= warmup:
            vals.append(v)
            times.append(t_sweep)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": statistics.median(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "oracle": "CPU fp64 dense per-token expert loop"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": ob.cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------- prefill layers ---
def fp8_dense_peak(dev, seconds: float = 2.0) -> dict:
    """Dense FP8 tensor-core rate of the library GEMM on this GPU: cuBLAS
    through torch._scaled_mm, e4m3 x e4m3 -> bf16 with unit tensor-wise scales,
    8192^3 (2 * 8192^3 FLOPs per call).  Burst = best of 10 calls timed one by
    one with CUDA events; sustained = calls back to back for `seconds`."""
    import torch
    n = 8192
    try:
        g = torch.Generator(device=dev).manual_seed(7)
        a = (torch.randn(n, n, device=dev, generator=g) * 0.05).to(torch.float8_e4m3fn)
        b = (torch.randn(n, n, device=dev, generator=g) * 0.05).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev, dtype=torch.float32)

        def mm():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        calls = max(10, int(seconds * 1e3 / best))
        e0.record()
        for _ in range(calls):
            mm()
        e1.record()
        torch.cuda.synchronize()
        sustained_ms = e0.elapsed_time(e1) / calls
        fl = 2.0 * n ** 3
        del a, b
        return {"burst_tflops": fl / (best * 1e-3) / 1e12, "sustained_tflops": fl / (sustained_ms * 1e-3) / 1e12,
                "how": "cuBLAS via torch._scaled_mm, e4m3 x e4m3 -> bf16, 8192^3: best of 10 (burst), "
                       f"{calls} calls back to back (sustained)"}
    except Exception as exc:  # reported, not hidden: the fractions then use the nominal ratio
        return {"burst_tflops": None, "sustained_tflops": None, "how": f"unavailable: {type(exc).__name__}: {exc}"}


def layer_gemm_timings(dev, reps: int = 20, fp8_peak: float | None = None, hbm: float | None = None) -> list:
    """The M=4096 FP8 grouped GEMMs of the Mixtral-8x7B- and 8x22B-shaped
    layers (the compute-bound shapes), each timed alone: median of `reps`
    launches, each after a 512 MB L2 flush.  Weights N(0, 1/K) from torch's
    seeded device generator (timing only; the parity tests check these
    launches against the oracle).  Returns one dict per GEMM."""
    import torch

    import quantized_moe_grouped_gb300 as q
    from quantized_moe_grouped_gb300 import inputs

    g = torch.Generator(device=dev).manual_seed(11)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def weights_fp8(E_, N_, K_):
        wq = torch.empty(E_, N_, K_, dtype=torch.uint8, device=dev)
        ws = torch.empty(E_, N_, dtype=torch.float32, device=dev)
        for e in range(E_):
            w = torch.randn(N_, K_, device=dev, generator=g) * (1.0 / np.sqrt(K_))
            wq[e], ws[e] = q.quant_weight_fp8(w)
        return wq, ws

    rows = []

    def record(wl, kernel, ms, nbytes, nflops, M, N, K):
        tf = nflops / (ms * 1e-3) / 1e12
        r = {"layer": wl.name, "gemm": kernel, "M": M, "N": N, "K": K, "us": ms * 1e3, "TFLOPS": tf,
             "GBps": nbytes / (ms * 1e-3) / 1e9, "flops": nflops, "algorithmic_bytes": nbytes}
        if fp8_peak:
            roof_ms = max(nflops / (fp8_peak * 1e12), nbytes / (hbm * 1e9) if hbm else 0.0) * 1e3
            r["frac"] = roof_ms / ms
        rows.append(r)

    for wl in (inputs.mixtral_8x7b_layer(), inputs.mixtral_8x22b_layer()):
        M, K, I, Nd = wl.M, wl.K, wl.inter, wl.N
        T, BM = M * TOP_K, 128
        ids, tw = inputs.routing(M, E, TOP_K, wl.seed, wl.zipf_s)
        hit = len(np.unique(ids))
        idsd, twd = torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev)
        a = torch.from_numpy(inputs.activations_bf16(M, K, wl.seed).view(np.int16)).to(dev).view(torch.bfloat16)
        al = q.moe_align_block_size(idsd, E, BM)
        aq, sa = q.quant_act_fp8_sorted(a, al, TOP_K)
        w1q, w1s = weights_fp8(E, 2 * I, K)
        up = torch.empty(T, 2 * I, dtype=torch.bfloat16, device=dev)
        ms = _timed(lambda: q.moe_gemm_w8a8(aq, sa, w1q, w1s, al, None, M=M, top_k=TOP_K, BM=BM,
                                            a_layout=q.A_PADDED, out_layout=q.OUT_GROUPED, out=up), reps, flush)
        record(wl, "up: moe_gemm_w8a8, padded A -> grouped out", ms,
               hit * 2 * I * K + hit * 2 * I * 4 + T * (K + 4) + T * 2 * I * 2, 2.0 * T * K * 2 * I, M, 2 * I, K)
        del w1q, w1s
        w2q, w2s = weights_fp8(E, Nd, I)
        out = torch.empty(M, Nd, dtype=torch.bfloat16, device=dev)
        acc = torch.empty(M, Nd, dtype=torch.float32, device=dev)
        if wl.act_scale == "token":
            hq, hs = q.silu_mul_quant(up)
            ms = _timed(lambda: q.moe_gemm_w8a8(hq, hs, w2q, w2s, al, twd, M=M, top_k=TOP_K, BM=BM,
                                                a_layout=q.A_GROUPED, out_layout=q.OUT_TOKEN_SUM, out=out,
                                                accum=acc), reps, flush)
            record(wl, "down: moe_gemm_w8a8, grouped A -> routing-weighted sum over top_k", ms,
                   hit * Nd * I + hit * Nd * 4 + T * (I + 4) + T * 8 + M * Nd * 2, 2.0 * T * I * Nd, M, Nd, I)
        else:
            hq, sf = q.silu_mul_quant(up, q.SCALE_MX_1X32, expert_offsets=al["expert_offsets"],
                                      sf_padded_offsets=al["padded_offsets"], sf_rows=q.align_max_padded(T, E, 128))
            ms = _timed(lambda: q.moe_gemm_w8a8(hq, None, w2q, w2s, al, twd, M=M, top_k=TOP_K, BM=BM,
                                                a_layout=q.A_GROUPED, out_layout=q.OUT_TOKEN_SUM, out=out,
                                                accum=acc, a_scale_mode=q.SCALE_MX_1X32, a_sf=sf,
                                                a_sf_padded_offsets=al["padded_offsets"]), reps, flush)
            record(wl, "down: moe_gemm_w8a8, MXFP8 grouped A -> routing-weighted sum over top_k", ms,
                   hit * Nd * I + hit * Nd * 4 + T * (I + I // 32) + T * 8 + M * Nd * 2, 2.0 * T * I * Nd, M, Nd, I)
        del w2q, w2s, up, out, acc
    del flush
    torch.cuda.empty_cache()
    return rows


# ----------------------------------------------------------------- suite ---
def _timed(fn, reps, flush=None, warmup=5):
    """Median device time (ms) of fn() over reps runs after `warmup` untimed
    runs, each timed run after an L2 flush.  A 30 us device sleep before the
    start event keeps the GPU busy while the host enqueues fn's launches, so
    short kernels are timed without the host's launch latency."""
    import torch
    for _ in range(warmup):
        fn()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        torch.cuda._sleep(60000)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def run_suite(reps: int = 50, only: str | None = None) -> None:
    """Per-entry-point timings of the other workloads (not the bench line):
    INT8 W8A16 sweep, Mixtral-8x7B- and 8x22B-shaped FP8 layers.  Weights are
    N(0, 1/K) drawn with torch's seeded device generator (timing only); every
    kernel is timed after a 512 MB L2 flush."""
    import torch

    import quantized_moe_grouped_gb300 as q
    from quantized_moe_grouped_gb300 import inputs

    q.load_library()
    dev = torch.device("cuda", 0)
    torch.manual_seed(0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    hbm, _ = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        bf16_peak = 1900.0
    # FP8 roofline: the library FP8 GEMM's rate measured here (burst); the
    # nominal fp8:bf16 ratio of 2 only when that measurement is unavailable
    pk = fp8_dense_peak(dev)
    fp8_peak = pk["burst_tflops"] or 2.0 * bf16_peak
    print(json.dumps({"suite": "fp8 dense peak", **pk}), flush=True)

    def line(workload, kernel, ms, nbytes, nflops, bound):
        gbs = nbytes / (ms * 1e-3) / 1e9
        tfl = nflops / (ms * 1e-3) / 1e12
        roof_ms = max(nbytes / (hbm * 1e9), nflops / ((fp8_peak if bound == "fp8" else bf16_peak) * 1e12)) * 1e3
        print(json.dumps({"suite": workload, "kernel": kernel, "us": ms * 1e3, "GBps": gbs, "TFLOPS": tfl,
                          "roofline_us": roof_ms * 1e3, "frac_of_roofline": roof_ms / ms}), flush=True)

    def weights_fp8(E_, N_, K_):
        wq = torch.empty(E_, N_, K_, dtype=torch.uint8, device=dev)
        ws = torch.empty(E_, N_, dtype=torch.float32, device=dev)
        for e in range(E_):
            w = torch.randn(N_, K_, device=dev) * (1.0 / np.sqrt(K_))
            wq[e], ws[e] = q.quant_weight_fp8(w)
        return wq, ws

    def weights_int8(E_, N_, K_):
        wq = torch.empty(E_, N_, K_, dtype=torch.int8, device=dev)
        ws = torch.empty(E_, N_, dtype=torch.float32, device=dev)
        for e in range(E_):
            w = torch.randn(N_, K_, device=dev) * (1.0 / np.sqrt(K_))
            wq[e], ws[e] = q.quant_weight_int8(w)
        return wq, ws

    # FP8 decode GEMM by activation layout: token rows gathered by the GEMM's
    # cp.async warps against rows quantised into padded sorted order
    for wl in inputs.decode_fp8_sweep():
        if only and only not in wl.name:
            continue
        if wl.M not in (64, 512):
            continue
        wq8, ws8 = weights_fp8(E, wl.N, wl.K)
        a = torch.from_numpy(inputs.activations_bf16(wl.M, wl.K, wl.seed).view(np.int16)).to(dev).view(torch.bfloat16)
        ids, tw = inputs.routing(wl.M, E, TOP_K, wl.seed)
        BM = 32 if wl.M <= 64 else 128
        al = q.moe_align_block_size(torch.from_numpy(ids).to(dev), E, BM)
        twd = torch.from_numpy(tw).to(dev)
        out = torch.empty(wl.M * TOP_K, wl.N, dtype=torch.bfloat16, device=dev)
        hit = len(np.unique(ids))
        nbytes = hit * wl.N * wl.K + hit * wl.N * 4 + wl.M * (wl.K + 4) + wl.M * TOP_K * (8 + 2 * wl.N)
        aq, sa = q.quant_act_fp8(a)
        ms = _timed(lambda: q.moe_gemm_w8a8(aq, sa, wq8, ws8, al, twd, M=wl.M, top_k=TOP_K, BM=BM, out=out), reps,
                    flush)
        line(wl.name, f"moe_gemm_w8a8 BM={BM} token-gather A", ms, nbytes,
             2.0 * wl.M * TOP_K * wl.K * wl.N, "fp8")
        aqp, sap = q.quant_act_fp8_sorted(a, al, TOP_K)
        ms = _timed(lambda: q.moe_gemm_w8a8(aqp, sap, wq8, ws8, al, twd, M=wl.M, top_k=TOP_K, BM=BM,
                                            a_layout=q.A_PADDED, out=out), reps, flush)
        line(wl.name, f"moe_gemm_w8a8 BM={BM} padded A", ms, nbytes, 2.0 * wl.M * TOP_K * wl.K * wl.N, "fp8")
        del wq8, ws8

    # INT8 W8A16 sweep
    for wl in inputs.int8_w8a16_sweep():
        if only and only not in wl.name:
            continue
        wq, ws = weights_int8(E, wl.N, wl.K)
        a = torch.from_numpy(inputs.activations_bf16(wl.M, wl.K, wl.seed).view(np.int16)).to(dev).view(torch.bfloat16)
        ids, tw = inputs.routing(wl.M, E, TOP_K, wl.seed)
        # the wide tile: more weight bytes per bf16 MMA than the swapped one, also at decode; 64 slots
        # when every expert's slots fit one such tile (the weights are still read once, the bf16
        # activation tile per stage halves)
        BM = 64 if np.bincount(ids.ravel(), minlength=E).max() <= 64 else 128
        al = q.moe_align_block_size(torch.from_numpy(ids).to(dev), E, BM)
        twd = torch.from_numpy(tw).to(dev)
        out = torch.empty(wl.M * TOP_K, wl.N, dtype=torch.bfloat16, device=dev)
        hit = len(np.unique(ids))
        nbytes = hit * wl.N * wl.K + hit * wl.N * 4 + wl.M * wl.K * 2 + wl.M * TOP_K * (8 + 2 * wl.N)
        ms = _timed(lambda: q.moe_gemm_w8a16(a, wq, ws, al, twd, M=wl.M, top_k=TOP_K, BM=BM, out=out), reps, flush)
        line(wl.name, f"moe_gemm_w8a16 BM={BM} token-gather A", ms, nbytes, 2.0 * wl.M * TOP_K * wl.K * wl.N, "bf16")
        ap = q.gather_sorted_bf16(a, al, TOP_K)
        ms = _timed(lambda: q.gather_sorted_bf16(a, al, TOP_K, out=ap), reps, flush)
        line(wl.name, "gather_sorted_bf16", ms, wl.M * wl.K * 2 + wl.M * TOP_K * wl.K * 2, 0, "bf16")
        ms = _timed(lambda: q.moe_gemm_w8a16(ap, wq, ws, al, twd, M=wl.M, top_k=TOP_K, BM=BM, a_layout=q.A_PADDED,
                                             out=out), reps, flush)
        line(wl.name, f"moe_gemm_w8a16 BM={BM} padded A", ms, nbytes, 2.0 * wl.M * TOP_K * wl.K * wl.N, "bf16")
        del wq, ws

    # INT4 W4A16 (int4wo, groups of 128 along K) on the same shapes
    for wl in inputs.int8_w8a16_sweep():
        if only and only not in wl.name.replace("int8 w8a16", "int4 w4a16"):
            continue
        wq = torch.empty(E, wl.N, wl.K // 2, dtype=torch.uint8, device=dev)
        ws = torch.empty(E, wl.N, wl.K // 128, dtype=torch.float32, device=dev)
        for e in range(E):
            w = torch.randn(wl.N, wl.K, device=dev) * (1.0 / np.sqrt(wl.K))
            q.quant_weight_int4(w, q=wq[e], scale=ws[e])
        a = torch.from_numpy(inputs.activations_bf16(wl.M, wl.K, wl.seed).view(np.int16)).to(dev).view(torch.bfloat16)
        ids, tw = inputs.routing(wl.M, E, TOP_K, wl.seed)
        BM = 64 if np.bincount(ids.ravel(), minlength=E).max() <= 64 else 128
        al = q.moe_align_block_size(torch.from_numpy(ids).to(dev), E, BM)
        twd = torch.from_numpy(tw).to(dev)
        out = torch.empty(wl.M * TOP_K, wl.N, dtype=torch.bfloat16, device=dev)
        hit = len(np.unique(ids))
        nbytes = hit * wl.N * wl.K // 2 + hit * wl.N * (wl.K // 128) * 4 + wl.M * wl.K * 2 + wl.M * TOP_K * (8 + 2 * wl.N)
        ap = q.gather_sorted_bf16(a, al, TOP_K)
        ms = _timed(lambda: q.moe_gemm_w4a16(ap, wq, ws, al, twd, M=wl.M, top_k=TOP_K, BM=BM, a_layout=q.A_PADDED,
                                             out=out), reps, flush)
        line(wl.name.replace("int8 w8a16", "int4 w4a16"), f"moe_gemm_w4a16 BM={BM} padded A", ms, nbytes,
             2.0 * wl.M * TOP_K * wl.K * wl.N, "bf16")
        del wq, ws

    # Fused activation + MXFP8 on the TransformerEngine GroupedLinear page's input
    # (8 experts x 4000 rows, width 4096): SReLU on [32000, 4096]; SwiGLU on the
    # same input read as gate|up, [32000, 2 x 2048].  Page: ~142 us (SReLU) and
    # ~343 us (SwiGLU) fused, plus 75 / 84 us of scale-factor padding kernels,
    # on unnamed hardware -- context only.
    if not only or "activation" in only:
        rows, width = 8 * 4000, 4096
        y = (torch.randn(rows, width, device=dev)).to(torch.bfloat16)
        eoff = torch.arange(0, rows + 1, 4000, dtype=torch.int32, device=dev)
        soff = torch.arange(0, 8 * 4096 + 1, 4096, dtype=torch.int32, device=dev)
        for name, fn, I in (("srelu_quant mxfp8 [32000, 4096]", q.srelu_quant, width),
                            ("silu_mul_quant mxfp8 [32000, 2x2048]", q.silu_mul_quant, width // 2)):
            hq, sf = fn(y, q.SCALE_MX_1X32, expert_offsets=eoff, sf_padded_offsets=soff, sf_rows=8 * 4096)
            ms = _timed(lambda: fn(y, q.SCALE_MX_1X32, expert_offsets=eoff, sf_padded_offsets=soff, q=hq, sf=sf),
                        reps, flush)
            line("activation + MXFP8 8x4000x4096", name, ms, rows * width * 2 + rows * I + 8 * 4096 * (I // 32), 0,
                 "fp8")
        # plain MXFP8 input (rowwise, per-expert padded factors) and columnwise factors
        xq, xsf = q.quant_mxfp8(y, expert_offsets=eoff, sf_padded_offsets=soff, sf_rows=8 * 4096)
        ms = _timed(lambda: q.quant_mxfp8(y, expert_offsets=eoff, sf_padded_offsets=soff, q=xq, sf=xsf), reps, flush)
        line("MXFP8 quantisation 8x4000x4096", "quant_mxfp8 rowwise", ms, rows * width * 3 + 8 * 4096 * (width // 32),
             0, "fp8")
        cq, csf = q.quant_mxfp8_colwise(y)
        ms = _timed(lambda: q.quant_mxfp8_colwise(y, q=cq, sf=csf), reps, flush)
        line("MXFP8 quantisation 8x4000x4096", "quant_mxfp8_colwise", ms, rows * width * 3 + csf.numel(), 0, "fp8")
        del y, xq, cq

    # Router front: fp32 logits [M, 8] -> top-2 -> align -> sorted e4m3 rows,
    # fused into one launch at decode sizes, against the separate launches.
    if not only or "router" in only:
        for M in (64, 512, 4096):
            K = 4096
            lg = torch.randn(M, E, device=dev)
            a = torch.randn(M, K, device=dev).to(torch.bfloat16)
            ids, tw = q.moe_router_topk(lg, TOP_K)
            ms = _timed(lambda: q.moe_router_topk(lg, TOP_K, topk_ids=ids, topk_weights=tw), reps)
            line(f"router M={M} E={E} top_k={TOP_K}", "moe_router_topk", ms, M * E * 4 + M * TOP_K * 8, 0, "fp8")
            BM = 32 if M <= 64 else 128
            ids2, tw2, al, aq, sa = q.moe_route_align_quant_fp8(lg, a, TOP_K, BM)
            ms = _timed(lambda: q.moe_route_align_quant_fp8(lg, a, TOP_K, BM, align=al, topk_ids=ids2,
                                                            topk_weights=tw2, q=aq, scale=sa), reps, flush)
            line(f"router M={M} E={E} top_k={TOP_K}", f"moe_route_align_quant_fp8 BM={BM}", ms,
                 M * E * 4 + M * TOP_K * 8 + M * K * 2 + M * TOP_K * (K + 8), 0, "fp8")

            def separate():
                q.moe_router_topk(lg, TOP_K, topk_ids=ids, topk_weights=tw)
                q.moe_align_quant_fp8(a, ids, E, BM, align=al, q=aq, scale=sa)
            ms = _timed(separate, reps, flush)
            line(f"router M={M} E={E} top_k={TOP_K}", f"moe_router_topk + moe_align_quant_fp8 BM={BM}", ms,
                 M * E * 4 + M * TOP_K * 8 + M * K * 2 + M * TOP_K * (K + 8), 0, "fp8")

    # FP8 layers
    for wl in (inputs.mixtral_8x7b_layer(), inputs.mixtral_8x22b_layer()):
        if only and only not in wl.name:
            continue
        M, K, I, Nd = wl.M, wl.K, wl.inter, wl.N
        T = M * TOP_K
        BM = 128
        ids, tw = inputs.routing(M, E, TOP_K, wl.seed, wl.zipf_s)
        hit = len(np.unique(ids))
        idsd, twd = torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev)
        a = torch.from_numpy(inputs.activations_bf16(M, K, wl.seed).view(np.int16)).to(dev).view(torch.bfloat16)
        w1q, w1s = weights_fp8(E, 2 * I, K)
        al = q.moe_align_block_size(idsd, E, BM)
        ms = _timed(lambda: q.moe_align_block_size(idsd, E, BM, out=al), reps)
        line(wl.name, "moe_align_block_size", ms, T * 4 + al["sorted_ids"].numel() * 4, 0, "fp8")
        aq, sa = q.quant_act_fp8_sorted(a, al, TOP_K)
        ms = _timed(lambda: q.quant_act_fp8_sorted(a, al, TOP_K, q=aq, scale=sa), reps, flush)
        line(wl.name, "quant_act_fp8_sorted", ms, M * K * 2 + T * (K + 4), 0, "fp8")
        up = torch.empty(T, 2 * I, dtype=torch.bfloat16, device=dev)
        ms = _timed(lambda: q.moe_gemm_w8a8(aq, sa, w1q, w1s, al, None, M=M, top_k=TOP_K, BM=BM,
                                            a_layout=q.A_PADDED, out_layout=q.OUT_GROUPED, out=up), reps, flush)
        line(wl.name, "moe_gemm_w8a8 up (padded A -> grouped out)", ms,
             hit * 2 * I * K + hit * 2 * I * 4 + T * (K + 4) + T * 2 * I * 2, 2.0 * T * K * 2 * I, "fp8")
        if wl.act_scale == "token":  # the same projection with SwiGLU in its epilogue + the per-token pass
            fq = torch.empty(T, I, dtype=torch.uint8, device=dev)
            fs = torch.empty(T, dtype=torch.float32, device=dev)
            hs_scr = torch.empty(T * I + T, dtype=torch.float32, device=dev)
            ms = _timed(lambda: q.moe_gemm_w8a8_silu_fp8_token(aq, sa, w1q, w1s, al, M=M, top_k=TOP_K,
                                                               a_layout=q.A_PADDED, q=fq, scale=fs,
                                                               h_scratch=hs_scr), reps, flush)
            line(wl.name, "moe_gemm_w8a8 up + SwiGLU epilogue + per-token FP8 pass (2 launches + memset)", ms,
                 hit * 2 * I * K + hit * 2 * I * 4 + T * (K + 4) + 2 * T * I * 4 + T * (I + 4), 2.0 * T * K * 2 * I,
                 "fp8")
            del fq, fs, hs_scr
        if wl.act_scale == "mx":  # the same projection with SwiGLU + MXFP8 in its epilogue
            fq = torch.empty(T, I, dtype=torch.uint8, device=dev)
            fsf = torch.empty(q.align_max_padded(T, E, 128), q.mx_sf_ld(I), dtype=torch.uint8, device=dev)
            ms = _timed(lambda: q.moe_gemm_w8a8_silu_mxfp8(aq, sa, w1q, w1s, al, M=M, top_k=TOP_K,
                                                           a_layout=q.A_PADDED, q=fq, sf=fsf), reps, flush)
            line(wl.name, "moe_gemm_w8a8 up + SwiGLU + MXFP8 epilogue (padded A -> grouped e4m3 + E8M0)", ms,
                 hit * 2 * I * K + hit * 2 * I * 4 + T * (K + 4) + T * I + T * (I // 32), 2.0 * T * K * 2 * I, "fp8")
            del fq, fsf
        del w1q, w1s
        if wl.act_scale == "token":
            hq, hs = q.silu_mul_quant(up)
            ms = _timed(lambda: q.silu_mul_quant(up, q=hq, scale=hs), reps, flush)
            line(wl.name, "silu_mul_quant per-token", ms, T * 2 * I * 2 + T * (I + 4), 0, "fp8")
            w2q, w2s = weights_fp8(E, Nd, I)
            out = torch.empty(M, Nd, dtype=torch.bfloat16, device=dev)
            acc = torch.empty(M, Nd, dtype=torch.float32, device=dev)
            ms = _timed(lambda: q.moe_gemm_w8a8(hq, hs, w2q, w2s, al, twd, M=M, top_k=TOP_K, BM=BM,
                                                a_layout=q.A_GROUPED, out_layout=q.OUT_TOKEN_SUM, out=out,
                                                accum=acc), reps, flush)
            line(wl.name, "moe_gemm_w8a8 down (grouped A -> token sum)", ms,
                 hit * Nd * I + hit * Nd * 4 + T * (I + 4) + T * 8 + M * Nd * 2, 2.0 * T * I * Nd, "fp8")
            del w2q, w2s
        else:
            sf_rows = q.align_max_padded(T, E, 128)
            hq, sf = q.silu_mul_quant(up, q.SCALE_MX_1X32, expert_offsets=al["expert_offsets"],
                                      sf_padded_offsets=al["padded_offsets"], sf_rows=sf_rows)
            ms = _timed(lambda: q.silu_mul_quant(up, q.SCALE_MX_1X32, expert_offsets=al["expert_offsets"],
                                                 sf_padded_offsets=al["padded_offsets"], q=hq, sf=sf), reps, flush)
            line(wl.name, "silu_mul_quant mxfp8", ms, T * 2 * I * 2 + T * I + T * (I // 32), 0, "fp8")
            w2q, w2s = weights_fp8(E, Nd, I)
            out = torch.empty(M, Nd, dtype=torch.bfloat16, device=dev)
            acc = torch.empty(M, Nd, dtype=torch.float32, device=dev)
            ms = _timed(lambda: q.moe_gemm_w8a8(hq, None, w2q, w2s, al, twd, M=M, top_k=TOP_K, BM=BM,
                                                a_layout=q.A_GROUPED, out_layout=q.OUT_TOKEN_SUM, out=out,
                                                accum=acc, a_scale_mode=q.SCALE_MX_1X32, a_sf=sf,
                                                a_sf_padded_offsets=al["padded_offsets"]), reps, flush)
            line(wl.name, "moe_gemm_w8a8 down mxfp8 (grouped A -> token sum)", ms,
                 hit * Nd * I + hit * Nd * 4 + T * (I + I // 32) + T * 8 + M * Nd * 2, 2.0 * T * I * Nd, "fp8")
            del w2q, w2s
            # the same down projection with MXFP8 weights too (both operands block-scaled)
            w2mq = torch.empty(E, Nd, I, dtype=torch.uint8, device=dev)
            w2msf = torch.empty(E * Nd, q.mx_sf_ld(I), dtype=torch.uint8, device=dev)
            for e in range(E):
                w = torch.randn(Nd, I, device=dev) * (1.0 / np.sqrt(I))
                q.quant_weight_mxfp8(w, q=w2mq[e], sf=w2msf[e * Nd:(e + 1) * Nd])
            w2mt = q.mx_weight_sf_tiled(w2msf, E, Nd, I)
            ms = _timed(lambda: q.moe_gemm_w8a8(hq, None, w2mq, None, al, twd, M=M, top_k=TOP_K, BM=BM,
                                                a_layout=q.A_GROUPED, out_layout=q.OUT_TOKEN_SUM, out=out,
                                                accum=acc, a_scale_mode=q.SCALE_MX_1X32, a_sf=sf,
                                                a_sf_padded_offsets=al["padded_offsets"],
                                                w_scale_mode=q.SCALE_MX_1X32, w_sf=w2mt), reps, flush)
            line(wl.name, "moe_gemm_w8a8 down, MXFP8 activations and weights (token sum)", ms,
                 hit * Nd * I + hit * Nd * (I // 32) + T * (I + I // 32) + T * 8 + M * Nd * 2, 2.0 * T * I * Nd, "fp8")
            del w2mq, w2msf, w2mt
        del up


# ------------------------------------------------------------ tile sweep ---
def run_tile_sweep(reps: int = 20, only: str | None = None, launches: int = 0) -> None:
    """One-SM against CTA-pair tiles of the grouped GEMMs (forced through the
    debug tile entry point) on the Mixtral-shaped projections and the W8A16 /
    W4A16 sweep: median µs of `reps` launches each after a 512 MB L2 flush, one
    JSON line per shape.  Weights are random codes with random scales (timing
    only).  launches > 0: instead of timing, run that many launches of each
    family per shape (a fixed launch list for a profiler)."""
    import torch

    import quantized_moe_grouped_gb300 as q
    from quantized_moe_grouped_gb300 import inputs

    q.load_library()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(3)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    fp8 = [("fp8 up N=28672 K=4096", 28672, 4096, q.OUT_GROUPED, (1024, 2048, 4096), None),
           ("fp8 down N=4096 K=14336", 4096, 14336, q.OUT_TOKEN_SUM, (1024, 2048, 4096), None),
           ("fp8 up N=32768 K=6144 zipf1.2", 32768, 6144, q.OUT_GROUPED, (2048, 4096), 1.2),
           ("fp8 down N=6144 K=16384", 6144, 16384, q.OUT_TOKEN_SUM, (1024, 2048, 4096), None),
           ("fp8 decode N=14336 K=4096", 14336, 4096, q.OUT_SLOT, (256, 512, 1024), None)]
    a16 = [("a16 N=14336 K=4096", 14336, 4096, (64, 1024, 4096)), ("a16 N=7168 K=4096", 7168, 4096, (64, 1024, 4096))]

    def measure(fn):
        if launches > 0:
            for _ in range(launches):
                fn()
            torch.cuda.synchronize()
            return float("nan")
        return _timed(fn, reps, flush) * 1e3

    for name, N, K, ol, Ms, zipf in fp8:
        if only and only not in name:
            continue
        wq = torch.randint(0, 120, (E, N, K), device=dev, dtype=torch.uint8, generator=g)
        ws = torch.rand(E, N, device=dev, generator=g)
        for M in Ms:
            ids, tw = inputs.routing(M, E, TOP_K, 7000 + M, zipf)
            al = q.moe_align_block_size(torch.from_numpy(ids).to(dev), E, 128)
            twd = torch.from_numpy(tw).to(dev)
            a = torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16)
            aq, sa = q.quant_act_fp8_sorted(a, al, TOP_K)
            out = torch.empty(M if ol == q.OUT_TOKEN_SUM else M * TOP_K, N, dtype=torch.bfloat16, device=dev)
            acc = torch.empty(M, N, dtype=torch.float32, device=dev)
            r = {"tile_sweep": name, "M": M}
            for tile, key in ((q.TILE_ONE_SM, "one_sm_us"), (q.TILE_PAIR, "pair_us")):
                r[key] = measure(lambda: q.moe_gemm_w8a8(aq, sa, wq, ws, al, twd, M=M, top_k=TOP_K, BM=128,
                                                         a_layout=q.A_PADDED, out_layout=ol, out=out, accum=acc,
                                                         tile=tile))
            print(json.dumps(r), flush=True)
        del wq, ws
        torch.cuda.empty_cache()
    for name, N, K, Ms in a16:
        if only and only not in name:
            continue
        w8 = torch.randint(-127, 128, (E, N, K), device=dev, dtype=torch.int16, generator=g).to(torch.int8)
        s8 = torch.rand(E, N, device=dev, generator=g) * 1e-2
        w4 = torch.randint(0, 256, (E, N, K // 2), device=dev, dtype=torch.int16, generator=g).to(torch.uint8)
        s4 = torch.rand(E, N, K // 128, device=dev, generator=g) * 1e-2
        for M in Ms:
            ids, tw = inputs.routing(M, E, TOP_K, 2000 + M)
            al = q.moe_align_block_size(torch.from_numpy(ids).to(dev), E, 128)
            twd = torch.from_numpy(tw).to(dev)
            ap = q.gather_sorted_bf16(torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16), al, TOP_K)
            out = torch.empty(M * TOP_K, N, dtype=torch.bfloat16, device=dev)
            r = {"tile_sweep": name, "M": M}
            for kind, fn, ww, ss in (("w8a16", q.moe_gemm_w8a16, w8, s8), ("w4a16", q.moe_gemm_w4a16, w4, s4)):
                for tile, key in ((q.TILE_ONE_SM, "one_sm_us"), (q.TILE_PAIR, "pair_us")):
                    r[f"{kind}_{key}"] = measure(lambda: fn(ap, ww, ss, al, twd, M=M, top_k=TOP_K, BM=128,
                                                            a_layout=q.A_PADDED, out=out, tile=tile))
            print(json.dumps(r), flush=True)
        del w8, w4
        torch.cuda.empty_cache()


# ------------------------------------------------------------------ main ---
def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--suite", action="store_true", help="per-kernel timings of the other workloads instead")
    ap.add_argument("--only", default=None, help="--suite: workloads whose name contains this text")
    ap.add_argument("--reps", type=int, default=50, help="--suite: timed repetitions per kernel (median)")
    ap.add_argument("--no-layers", action="store_true", help="skip the M=4096 layer GEMM timings")
    ap.add_argument("--tile-sweep", action="store_true",
                    help="one-SM against CTA-pair tiles of the grouped GEMMs (--only filters the shapes)")
    ap.add_argument("--launches", type=int, default=0,
                    help="--tile-sweep: run this many launches per family and shape instead of timing")
    ap.add_argument("--layer-reps", type=int, default=20, help="timed launches per M=4096 layer GEMM (median)")
    args = ap.parse_args()
    if args.suite:
        run_suite(args.reps, args.only)
        return
    if args.tile_sweep:
        run_tile_sweep(args.reps if args.reps != 50 else 20, args.only, args.launches)
        return
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    q, wq, ws, shapes = setup(dev)
    stream = torch.cuda.current_stream(dev)
    n_sh = len(shapes)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        for sh in shapes:
            run_path(q, wq, ws, sh, stream)
    torch.cuda.synchronize()

    # device-timed steps (inputs resident in HBM): the K steps run back to back
    # with nothing between the kernels (an event between two kernels would
    # stop the next one from launching under the previous one); then the same
    # K steps again with events around every GEMM on its stream, which give the
    # GEMM's own launch duration for the roofline object.
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sh)]
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(args.steps):
        for i, sh in enumerate(shapes):
            run_path(q, wq, ws, sh, stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    for s in range(args.steps):
        for i, sh in enumerate(shapes):
            run_path(q, wq, ws, sh, stream, evs[s][i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    gemm_ms = [sum(evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps)) / args.steps
               for i in range(n_sh)]
    ms = max_over_ranks(ms, world, dev)

    # end-to-end through the public API with pinned host buffers
    h2d = sum(sh["a_h"].numel() * 2 + sh["ids_h"].numel() * 4 + sh["tw_h"].numel() * 4 for sh in shapes)
    d2h = sum(sh["out_h"].numel() * 2 for sh in shapes)
    # Copies run on their own streams and overlap the kernels: a shape's inputs
    # go host -> device once the previous step's kernels of that shape are done
    # with them, its kernels wait for that copy and for the previous copy-out
    # of its output buffer, and outputs go device -> host on two alternating
    # streams (two copy engines).
    h2d_stream = torch.cuda.Stream(dev)
    d2h_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    ev_in = [torch.cuda.Event() for _ in shapes]
    ev_gemm = [torch.cuda.Event() for _ in shapes]
    ev_done = [torch.cuda.Event() for _ in shapes]

    def enqueue_e2e(cs, n_steps):
        """n_steps of the path with their host copies, issued on compute stream cs
        (the copy streams fork from it and join it again at the end)."""
        fork = torch.cuda.Event()
        fork.record(cs)
        for st_ in (h2d_stream, *d2h_streams):
            st_.wait_event(fork)
        for i in range(n_sh):
            ev_gemm[i].record(cs)
            ev_done[i].record(d2h_streams[i % 2])
        for _ in range(n_steps):
            for i, sh in enumerate(shapes):
                h2d_stream.wait_event(ev_gemm[i])
                with torch.cuda.stream(h2d_stream):
                    sh["a"].copy_(sh["a_h"], non_blocking=True)
                    sh["ids"].copy_(sh["ids_h"], non_blocking=True)
                    sh["tw"].copy_(sh["tw_h"], non_blocking=True)
                ev_in[i].record(h2d_stream)
                cs.wait_event(ev_in[i])
                cs.wait_event(ev_done[i])
                run_path(q, wq, ws, sh, cs)
                ev_gemm[i].record(cs)
                out_stream = d2h_streams[i % 2]
                out_stream.wait_event(ev_gemm[i])
                with torch.cuda.stream(out_stream):
                    sh["out_h"].copy_(sh["out"], non_blocking=True)
                ev_done[i].record(out_stream)
        for ev in ev_done:
            cs.wait_event(ev)

    def timed_e2e(run, n_steps):
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n_steps

    e2e_steps = max(3, min(args.steps, 200))
    # (a) every call enqueued by the host as it runs
    enqueue_e2e(stream, 2)
    e2e_eager_ms = timed_e2e(lambda: enqueue_e2e(stream, e2e_steps), e2e_steps)
    # (b) the same calls captured once into a CUDA graph of G steps and replayed:
    # what a serving loop does to take the host's enqueue time off the GPU's path
    e2e_mode = "cuda graph"
    graph_steps = min(e2e_steps, 100)
    replays = max(1, e2e_steps // graph_steps)
    try:
        cap = torch.cuda.Stream(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            enqueue_e2e(cap, graph_steps)
        graph.replay()
        torch.cuda.synchronize()

        def replay_all():
            for _ in range(replays):
                graph.replay()
        e2e_ms = timed_e2e(replay_all, replays * graph_steps)
    except Exception as exc:  # reported in the line, not hidden
        e2e_mode = f"host-enqueued (graph capture failed: {type(exc).__name__}: {exc})"
        e2e_ms = e2e_eager_ms
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_eager_ms = max_over_ranks(e2e_eager_ms, world, dev)

    # the compute-bound M=4096 layer GEMMs, timed alone with their own clock record
    layers = None
    if rank == 0 and not args.no_layers:
        hbm_peak, _ = measured_peaks()
        lclk = ClockSampler(local)
        lclk.start()
        time.sleep(0.3)
        pk = fp8_dense_peak(dev)
        rows = layer_gemm_timings(dev, reps=args.layer_reps, fp8_peak=pk["burst_tflops"], hbm=hbm_peak)
        layers = {"fp8_peak": {**pk, "unit": "TFLOP/s"}, "gemms": rows, "clocks": lclk.stop(),
                  "frac_against": "measured FP8 burst rate of the library GEMM above, roofline time = "
                                  "max(flops / peak, algorithmic bytes / measured HBM copy rate)",
                  "timing": f"median of {args.layer_reps} launches, each after a 512 MB L2 flush"}

    step_bytes = sum(sh["bytes"] for sh in shapes)
    step_flops = sum(sh["flops"] for sh in shapes)
    ms_step = ms / args.steps
    value = whole_job_rate(step_bytes, ms_step * 1e-3, world) / 1e9
    tflops = whole_job_rate(step_flops, ms_step * 1e-3, world) / 1e12
    peak, peak_kind = measured_peaks()
    gemm_total_ms = sum(gemm_ms)
    achieved = step_bytes / (gemm_total_ms * 1e-3) / 1e9
    page_gbs, page_tflops = page_aggregate()

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            ob = OracleBench()
            v, _, sample = ob.run(12.0)
            cpu = {"value": v, "unit": "GB/s", "cores": ob.cores, "kind": "oracle", "sample": sample}
        sweep = [{"M": sh["M"], "BM": sh["BM"], "gemm_us": g * 1e3, "gemm_GBps": sh["bytes"] / (g * 1e-3) / 1e9,
                  "gemm_TFLOPS": sh["flops"] / (g * 1e-3) / 1e12,
                  "gemm_frac_hbm": sh["bytes"] / (g * 1e-3) / 1e9 / peak, "bytes": sh["bytes"]}
                 for sh, g in zip(shapes, gemm_ms)]
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "tflops": tflops, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": value / world / page_gbs, "dtype": "fp8_e4m3 (fp32 accumulate)",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "BM": [sh["BM"] for sh in shapes], "l2": "inputs larger than L2 "
                       "(470 MB of e4m3 weights streamed by every GEMM)", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "grouped GEMM (moe_gemm_kernel<fp8> at M=64..256, "
                         "moe_gemm_pair_kernel at M=512)", "achieved": achieved, "peak": peak,
                         "peak_kind": f"{peak_kind} (hbm_gbs, burst)", "unit": "GB/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(), "algorithmic_bytes": step_bytes,
                         "per": "one step = the four GEMM launches of the sweep"},
            "sweep": sweep,
            "vs_baseline_note": f"page aggregate over the same sweep: {page_gbs:.0f} GB/s, {page_tflops:.0f} TFLOPS "
                                "(ROCm GPU, unnamed)",
            "e2e": {"value": whole_job_rate(step_bytes, e2e_ms * 1e-3, world) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "how": e2e_mode,
                    "host_enqueued_value": whole_job_rate(step_bytes, e2e_eager_ms * 1e-3, world) / 1e9},
            "gpu_launches": 2 * n_sh * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "layers": layers,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
