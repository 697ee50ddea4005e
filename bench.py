"""Benchmark of the LM-head contraction + consumer-surface projection on GB300.

Default workload (the decode token-only shape): H [16, 5120] bf16, W [151936, 5120] bf16,
k = 4 contiguous vocabulary lane shards (S = 37984), surface TOKEN_LOGPROB (argmax token +
chosen log-prob + logsumexp).  One step = one projection call = the fused GEMM + record
epilogue kernel followed by the record combine kernel.  W (1.56 GB) is larger than the
129 MB L2, so every step streams it from HBM and no L2 flush is needed between steps.

Prints one JSON line (rank 0):
  value       rows/s over K back-to-back projection calls (sb_lmhead_project, inputs
              resident in HBM), CUDA events at the step boundaries on the launching stream,
              barrier + synchronize on both sides, max over ranks;
  roofline    the GEMM kernel's algorithmic bytes (W + H read once, outputs written) divided
              by its average duration, from K further launches of that kernel alone with
              CUDA events around each (sb_lmhead_records), against the measured HBM copy
              bandwidth (kernel timed alone: the burst figure);
  e2e         the same metric through the public C-ABI call with host buffers
              (sb_lmhead_project_from_host): each step the call copies H from pinned host
              memory, runs the projection and copies token and log-prob back, and the step
              waits for them;
  cpu_baseline  the fp64 oracle (plain C, OpenMP over the host cores) on a bounded sample of
              the same workload (rank 0, N = 1 only).
``--impl reference`` times that oracle alone as the reference arm.  With N > 1 (torchrun),
each rank runs its own batch of rows against its own replica of W (weak scaling, no
collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# w_layout: how the workload stores W (packed once with sb_pack_weights where that streams
# faster: the d = 5120 decode and 256-row shapes; row-major for the 64-row shape, whose
# full-logit surface streams 2.8 % slower packed and its token surface no faster, and for
# prefill scoring, where the layout makes no difference)
WORKLOADS = {
    "decode16": dict(M=16, d=5120, V=151936, k=4, surface="token_logprob",
                     w_layout="packed", desc="decode token-only: H[16,5120] x W[151936,5120] bf16, k=4 shards of 37984, TOKEN + chosen log-prob"),
    "decode64": dict(M=64, d=4096, V=151936, k=2, surface="full_logits",
                     desc="decode full-logit: H[64,4096] x W[151936,4096] bf16, k=2, FULL_LOGITS"),
    "prefill": dict(M=4096, d=6144, V=200064, k=4, surface="token_logprob", targets=True,
                    desc="prefill scoring: H[4096,6144] x W[200064,6144] bf16, k=4, lse + target log-prob"),
    "decode64_token": dict(M=64, d=4096, V=151936, k=2, surface="token_logprob",
                           desc="decode token-only at the full-logit shape: H[64,4096] x W[151936,4096] bf16, k=2"),
    "sampling": dict(M=256, d=5120, V=151936, k=4, surface="gumbel_token", T=0.7, seed=1234,
                     w_layout="packed", desc="seeded sampling: H[256,5120] x W[151936,5120] bf16, k=4, GUMBEL_TOKEN T=0.7"),
    "decode16_sample": dict(M=16, d=5120, V=151936, k=4, surface="gumbel_token", T=0.7,
                            seed=1234,
                            w_layout="packed", desc="decode seeded sampling: H[16,5120] x W[151936,5120] bf16, k=4, GUMBEL_TOKEN T=0.7"),
    "tiny": dict(M=4, d=256, V=4096, k=2, surface="token_logprob",
                 w_layout="packed", desc="tiny: H[4,256] x W[4096,256] bf16, k=2"),
    "decode16_topk": dict(M=16, d=5120, V=151936, k=4, surface="topk_logprob", topk=8,
                          w_layout="packed", desc="decode top-8 log-probs: H[16,5120] x W[151936,5120] bf16, k=4"),
    "sampling_topk": dict(M=256, d=5120, V=151936, k=4, surface="topk_logprob", topk=8,
                          w_layout="packed", desc="256-row batch, top-8 log-probs: H[256,5120] x W[151936,5120] bf16, k=4"),
    "sampling_token": dict(M=256, d=5120, V=151936, k=4, surface="token_logprob",
                           w_layout="packed", desc="256-row decode batch: H[256,5120] x W[151936,5120] bf16, k=4, TOKEN + log-prob"),
    "sampling_full": dict(M=256, d=5120, V=151936, k=4, surface="full_logits",
                          w_layout="packed", desc="256-row batch, full logits: H[256,5120] x W[151936,5120] bf16, k=4, FULL_LOGITS"),
    "mlp_down": dict(kind="partial", M=64, N=5120, K=17408, lanes=2,
                     desc="row-parallel MLP down projection: X[64,17408] x W[5120,17408] bf16, 2 lanes, partials summed, bf16 out"),
    "mlp_down8": dict(kind="partial", M=8, N=5120, K=17408, lanes=2,
                      desc="row-parallel MLP down projection, 8 tokens"),
    "mlp_down_small": dict(kind="partial", M=64, N=2048, K=17408, lanes=2,
                           desc="profiling case: X[64,17408] x W[2048,17408] bf16, 2 lanes"),
    # smaller cases of the same kernels for ncu captures (inputs still larger than L2)
    "decode16_small": dict(M=16, d=1024, V=151936, k=4, surface="token_logprob",
                           desc="profiling case: H[16,1024] x W[151936,1024] bf16, k=4"),
    "prefill_small": dict(M=1024, d=2048, V=65536, k=4, surface="token_logprob", targets=True,
                          desc="profiling case: H[1024,2048] x W[65536,2048] bf16, k=4"),
    "sampling_token_small": dict(M=256, d=5120, V=65536, k=4, surface="token_logprob",
                                 desc="profiling case: H[256,5120] x W[65536,5120] bf16, k=4"),
    "decode16_topk_small": dict(M=16, d=1024, V=151936, k=4, surface="topk_logprob", topk=8,
                                desc="profiling case: H[16,1024] x W[151936,1024] bf16, k=4, top-8"),
    "sampling_token_mid": dict(M=256, d=5120, V=77824, k=4, surface="token_logprob",
                               desc="profiling case: H[256,5120] x W[77824,5120] bf16, k=4 (4 W tiles per CTA pair)"),
    "sampling_mid": dict(M=256, d=5120, V=77824, k=4, surface="gumbel_token", T=0.7, seed=1234,
                         desc="profiling case: H[256,5120] x W[77824,5120] bf16, k=4, GUMBEL (4 W tiles per CTA pair)"),
    "decode64_small": dict(M=64, d=1024, V=151936, k=2, surface="full_logits",
                           desc="profiling case: H[64,1024] x W[151936,1024] bf16, k=2, FULL_LOGITS"),
    "decode64_token_small": dict(M=64, d=1024, V=151936, k=2, surface="token_logprob",
                                 desc="profiling case: H[64,1024] x W[151936,1024] bf16, k=2, TOKEN_LOGPROB"),
    "sampling_topk_small": dict(M=256, d=1024, V=151936, k=4, surface="topk_logprob", topk=8,
                                desc="profiling case: H[256,1024] x W[151936,1024] bf16, k=4, top-8"),
    "sampling_full_small": dict(M=256, d=1024, V=151936, k=4, surface="full_logits",
                                desc="profiling case: H[256,1024] x W[151936,1024] bf16, k=4, FULL_LOGITS"),
    "sampling_small": dict(M=256, d=1024, V=151936, k=4, surface="gumbel_token", T=0.7,
                           seed=1234,
                           desc="profiling case: H[256,1024] x W[151936,1024] bf16, k=4, GUMBEL"),
}
METRIC = "LM-head+projection rows/s; % of HBM GB/s (decode) or bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal GB300 figures, reported beside the measured-peak fraction: ~8 TB/s HBM3e and
# 2.25 PFLOP/s dense bf16
NOMINAL_PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}

# DRAM traffic of the GEMM kernel per launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), with the hash of the kernel source it was taken on; reported as
# null once the source differs.
KERNEL_TRAFFIC = {
    # decode16: dram__bytes_read.sum + dram__bytes_write.sum of one full-size launch
    # with W packed (1,557,352,448 + 2,670,592 B; W + H are 1,555,988,480 B, and the packed
    # W pads each shard's last 96-column tile to 128 rows, 1.3 MB more).
    "decode16": {"bytes": 1560023040, "src_sha": "cafe303e71c1a23a", "w_layout": "packed"},
}


def kernel_src_hash() -> str:
    h = hashlib.sha256()
    for f in ("lmhead.cu", "sb_ptx.cuh", "sb_pipe.cuh", "sb_gumbel.cuh", "sb_internal.h"):
        with open(os.path.join(ROOT, "gemm_epilogue_reduction_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def l2_bytes() -> int:
    """L2 size of the current device (129 MB on GB300 if the property is missing)."""
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return int(getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20)


class L2Flush:
    """Writes a buffer of twice the L2 size between timed steps of workloads whose inputs fit
    in L2, so every step starts with its inputs in HBM only."""

    def __init__(self):
        import torch
        self.buf = torch.empty(2 * l2_bytes(), dtype=torch.uint8, device="cuda")
        self.v = 0

    def __call__(self):
        self.v ^= 1
        self.buf.fill_(self.v)


def timed_steps(step, K, stream, flush):
    """K steps on `stream`; returns the mean ms per step from CUDA events.  Without a flush
    the steps run back to back between one start and one end event (an event between two
    steps would cut the programmatic overlap of one step's first kernel with the previous
    step's last); with one, each step is timed alone between two events and the flush runs
    outside them."""
    import torch
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for a, b in evs:
        flush()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / K


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_rows_seed(rank: int) -> int:
    """Seed of the H batch a rank projects (rank 0 uses the workload's seed-0 inputs)."""
    return 0 if rank == 0 else 1000 + rank


def max_over_ranks(x: float, device) -> float:
    """The maximum of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(world: int, rows_per_rank: int, max_ms_per_step: float) -> float:
    """Whole-job throughput: the rows every rank projected per step over the slowest rank."""
    return world * rows_per_rank / (max_ms_per_step * 1e-3)


def oracle_rows_per_s(Hb, Wb, k, cfg, rows_per_call, min_seconds, max_calls=None):
    """Time the oracle (as it stands) on `rows_per_call`-row samples until min_seconds."""
    import numpy as np
    import oracle
    gumbel = cfg["surface"] == "gumbel_token"
    T = cfg.get("T", 1.0)
    seed = cfg.get("seed", 0)
    M = Hb.shape[0]
    done, calls, t0 = 0, 0, time.perf_counter()
    while True:
        r0 = (calls * rows_per_call) % M
        rows = [(r0 + i) % M for i in range(rows_per_call)]
        oracle.project(Hb[rows], Wb, k, gumbel=gumbel, temperature=T, seed=seed,
                       row_ids=np.array(rows))
        done += rows_per_call
        calls += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or (max_calls and calls >= max_calls):
            return done / el, done, el, oracle.num_threads()


def run_reference(args, cfg, world, rank):
    """The reference arm: the fp64 oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np
    import torch
    import oracle
    from gemm_epilogue_reduction_gb300 import synth
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    H, W = synth.make_hw(cfg["M"], cfg["d"], cfg["V"], seed=0, device=dev)
    Hb, Wb = synth.bf16_bits(H), synth.bf16_bits(W)
    del H, W
    rows_per_step = max(1, min(cfg["M"], 2))
    gumbel = cfg["surface"] == "gumbel_token"
    for i in range(args.warmup):
        oracle.project(Hb[:rows_per_step], Wb, cfg["k"], gumbel=gumbel,
                       temperature=cfg.get("T", 1.0), seed=cfg.get("seed", 0))
    times = []
    for i in range(args.steps):
        rows = [(i * rows_per_step + j) % cfg["M"] for j in range(rows_per_step)]
        t0 = time.perf_counter()
        oracle.project(Hb[rows], Wb, cfg["k"], gumbel=gumbel, temperature=cfg.get("T", 1.0),
                       seed=cfg.get("seed", 0), row_ids=np.array(rows))
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = rows_per_step * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, **{k: cfg[k] for k in ("M", "d", "V", "k")},
                   "surface": cfg["surface"], "desc": cfg["desc"]},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} of the workload's {cfg['M']} rows per step "
                                   f"against the full W (fp64 C oracle, OpenMP)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# the layout of W the projection calls read (--w-layout): "row", "packed", or "auto" = the
# workload's own choice (its "w_layout", else row-major)
W_LAYOUT = {"layout": "auto"}


def layout_for(cfg) -> str:
    lay = W_LAYOUT["layout"]
    return cfg.get("w_layout", "row") if lay == "auto" else lay


def make_projection(cfg, rank=0):
    """Inputs (seed 0; targets seed 1; rank r > 0 draws its own rows), caller-owned outputs
    and the three step closures of one projection workload on the current device."""
    import types
    import torch
    import gemm_epilogue_reduction_gb300 as sb
    from gemm_epilogue_reduction_gb300 import synth
    M, d, V, k = cfg["M"], cfg["d"], cfg["V"], cfg["k"]
    w = types.SimpleNamespace(M=M, d=d, V=V, k=k, surface=sb.SURFACES[cfg["surface"]],
                              T=cfg.get("T", 1.0), gseed=cfg.get("seed", 0))
    w.H, w.W = synth.make_hw(M, d, V, seed=0, device="cuda")
    if rank:
        w.H = synth.make_hw(M, d, 1, seed=rank_rows_seed(rank), device="cuda")[0]
    w.targets = synth.make_targets(M, V, seed=1, device="cuda") if cfg.get("targets") else None
    w.out, w.bufs = sb.make_outputs(M, V, k, w.surface, targets=w.targets,
                                    topk=cfg.get("topk", 0))
    w.tps = sb.sb_tiles_per_shard(M, V, k)
    w.stream = torch.cuda.current_stream()
    # W as the calls read it: row-major, or packed once here (a model parameter is laid out
    # when it is loaded, not per call)
    w.layout = layout_for(cfg)
    if w.layout == "packed":
        w.Warg, w.wsurf = sb.pack_weights(w.W, k, w.stream), w.surface | sb.SB_W_PACKED
        torch.cuda.synchronize()
    else:
        w.Warg, w.wsurf = w.W, w.surface

    def records():
        st = sb.sb_lmhead_records(w.H, w.Warg, M, d, V, k, w.wsurf, w.T, w.gseed, w.out,
                                  w.stream)
        if st != sb.SB_OK:
            raise sb.SbError(st, "sb_lmhead_records")

    def combine():
        st = sb.sb_combine_shard_records(w.bufs["workspace"], M, k, w.tps, w.surface, w.T, w.out,
                                         w.stream)
        if st != sb.SB_OK:
            raise sb.SbError(st, "sb_combine_shard_records")

    def project():
        st = sb.sb_lmhead_project(w.H, w.Warg, M, d, V, k, w.wsurf, w.T, w.gseed, w.out,
                                  w.stream)
        if st != sb.SB_OK:
            raise sb.SbError(st, "sb_lmhead_project")

    w.records, w.combine, w.project = records, combine, project
    w.in_bytes = V * d * 2 + M * d * 2
    return w


def kernel_times(w, K):
    """Average ms of the GEMM kernel alone and of the combine alone: K launches each, CUDA
    events around every launch on the launching stream."""
    import torch
    evk = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    res = []
    for fn in (w.records, w.combine):
        for i in range(K):
            evk[2 * i].record(w.stream)
            fn()
            evk[2 * i + 1].record(w.stream)
        torch.cuda.synchronize()
        res.append(sum(evk[2 * i].elapsed_time(evk[2 * i + 1]) for i in range(K)) / K)
    return res[0], res[1]


def projection_roofline(w, gemm_ms, comb_ms, peaks, peak_src, tensor_bound, traffic=None):
    """Roofline of the GEMM kernel: algorithmic bytes (W and H read once, 12 B of outputs per
    row, bf16 logits for FULL_LOGITS) or flops (2 M V d) over its event-timed duration."""
    import gemm_epilogue_reduction_gb300 as sb
    M, d, V = w.M, w.d, w.V
    alg_bytes = V * d * 2 + M * d * 2 + M * 12 + (M * V * 2 if w.surface == sb.SB_FULL_LOGITS
                                                   else 0)
    alg_flops = 2.0 * M * V * d
    gbs = alg_bytes / (gemm_ms * 1e-3) / 1e9
    tfs = alg_flops / (gemm_ms * 1e-3) / 1e12
    if not tensor_bound:
        return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": f"{peak_src} (HBM copy, burst)", "kernel": "lmhead_kernel",
                "kernel_ms": gemm_ms, "combine_ms": comb_ms, "algorithmic_bytes": alg_bytes,
                "tensor_tflops": tfs,
                "tensor_frac": tfs / peaks["bf16_tflops"],
                "nominal": {"peak": NOMINAL_PEAKS["hbm_gbs"],
                            "frac": gbs / NOMINAL_PEAKS["hbm_gbs"]}}
    sus = peaks.get("bf16_tflops_sustained")
    return {"bound": "tensor", "achieved": tfs, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": tfs / peaks["bf16_tflops"], "traffic": traffic,
            "peak_source": f"{peak_src} (cuBLAS bf16, burst)", "kernel": "lmhead_kernel",
            "kernel_ms": gemm_ms, "combine_ms": comb_ms, "algorithmic_flops": alg_flops,
            "hbm_gbs": gbs,
            "sustained": ({"peak": sus, "frac": tfs / sus} if sus else None),
            "nominal": {"peak": NOMINAL_PEAKS["bf16_tflops"],
                        "frac": tfs / NOMINAL_PEAKS["bf16_tflops"]}}


def steps_for(step, stream, seconds, lo=5, hi=4000, flush=None):
    """Steps that fill about `seconds` of device time (from three timed steps)."""
    est = timed_steps(step, 3, stream, flush)
    return max(lo, min(hi, int(seconds * 1e3 / max(est, 1e-3))))


def measure_workload(name, seconds, peaks, peak_src, gpu_index):
    """One workload of the per-configuration table: back-to-back projection steps for about
    `seconds` (clocks sampled meanwhile), then each kernel alone."""
    import torch
    import gemm_epilogue_reduction_gb300 as sb
    cfg = WORKLOADS[name]
    w = make_projection(cfg)
    flush = L2Flush() if w.in_bytes < l2_bytes() else None
    for _ in range(3):
        w.project()
    torch.cuda.synchronize()
    if sb.sb_last_device_status(w.out) != sb.SB_OK:
        raise RuntimeError(f"{name}: device status not OK after warm-up")
    K = steps_for(w.project, w.stream, seconds, flush=flush)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clocks:
        step_ms = timed_steps(w.project, K, w.stream, flush)
    if sb.sb_last_device_status(w.out) != sb.SB_OK:
        raise RuntimeError(f"{name}: device status not OK after the timed steps")
    gemm_ms, comb_ms = kernel_times(w, min(K, 200))
    roof = projection_roofline(w, gemm_ms, comb_ms, peaks, peak_src,
                               tensor_bound=name.startswith("prefill"))
    entry = {"desc": cfg["desc"], "surface": cfg["surface"], "w_layout": w.layout, "steps": K,
             "step_us": step_ms * 1e3, "rows_per_s": w.M / (step_ms * 1e-3),
             "gemm_us": gemm_ms * 1e3, "combine_us": comb_ms * 1e3,
             "bound": roof["bound"], "frac": roof["frac"], "achieved": roof["achieved"],
             "unit": roof["unit"], "clocks": clocks.summary()}
    if roof["bound"] == "tensor":
        entry["frac_sustained"] = roof["sustained"]["frac"] if roof["sustained"] else None
        entry["hbm_gbs"] = roof["hbm_gbs"]
    else:
        entry["tensor_frac"] = roof["tensor_frac"]
        entry["nominal_frac"] = roof["nominal"]["frac"]
    entry["payload_bytes"] = sb.sb_payload_bytes(w.M, w.k, w.surface) if w.surface in (
        sb.SB_TOKEN, sb.SB_TOKEN_LOGPROB, sb.SB_GUMBEL_TOKEN) else None
    del w
    torch.cuda.empty_cache()
    return entry


def measure_partial(name, seconds, peaks, peak_src, gpu_index, steps=None, warmup=3):
    """The row-parallel partial completion (both kernels) timed back to back; returns
    (ms per call, roofline dict, clocks summary)."""
    import torch
    import gemm_epilogue_reduction_gb300 as sb
    from gemm_epilogue_reduction_gb300 import synth
    cfg = WORKLOADS[name]
    M, N, K, lanes = cfg["M"], cfg["N"], cfg["K"], cfg["lanes"]
    X, W = synth.make_hw(M, K, N, seed=0, device="cuda")
    nbytes = sb.sb_partial_workspace_bytes(M, N, K, lanes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        st = sb.sb_partial_completion(X, W, M, N, K, lanes, Y, True, ws, nbytes, stream)
        if st != sb.SB_OK:
            raise sb.SbError(st, "sb_partial_completion")

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    in_bytes = N * K * 2 + M * K * 2
    flush = L2Flush() if in_bytes < l2_bytes() else None
    n = steps if steps else steps_for(step, stream, seconds, flush=flush)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clocks:
        ms = timed_steps(step, n, stream, flush)
    alg = N * K * 2 + M * K * 2 + M * N * 2
    ach = alg / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"], "traffic": None,
            "peak_source": f"{peak_src} (HBM copy, burst)",
            "kernel": "partial_kernel + complete_kernel", "algorithmic_bytes": alg,
            "nominal": {"peak": NOMINAL_PEAKS["hbm_gbs"], "frac": ach / NOMINAL_PEAKS["hbm_gbs"]}}
    flushed = flush is not None
    del X, W, ws, Y, flush
    torch.cuda.empty_cache()
    return ms, n, roof, clocks.summary(), in_bytes, flushed


# Links for the Equation (7) decision: the pages' 1-GbE testbed, a PCIe-class host link and an
# NVLink-class device link (payload bytes per second).
SELECTION_LINKS = {"1GbE": 1e9 / 8, "25GB/s": 25e9, "900GB/s": 900e9}


def plan_selection(M, V, k, local_proj_s, local_ref_s, frame_startup_s=0.0):
    """Equation (7) on measured local costs: plan r ships the complete bf16 logits (one frame
    per lane, 2 M V bytes), plan s each lane's shard-local projection record (one frame per
    lane, sb_payload_bytes of the token surface); L_s and L_r are the two plans' measured
    on-device step times.  Returns the decision per link and the threshold bandwidth (the
    link rate above which the complete logits would win: (B_r - B_s) / (L_s - L_r), or None
    when projecting costs no more on the device, so that it wins on every link)."""
    import gemm_epilogue_reduction_gb300 as sb
    B_r = 2.0 * M * V
    B_s = float(sb.sb_payload_bytes(M, k, sb.SB_TOKEN))
    F_r = F_s = float(k)
    out = {"bytes_ref": B_r, "bytes_proj": B_s, "frames_ref": F_r, "frames_proj": F_s,
           "local_proj_s": local_proj_s, "local_ref_s": local_ref_s,
           "frame_startup_s": frame_startup_s, "decisions": {}}
    for nm, beta in SELECTION_LINKS.items():
        dcs, margin = sb.sb_select_source_projection(B_r, B_s, F_r, F_s, beta, frame_startup_s,
                                                     local_proj_s, local_ref_s)
        out["decisions"][nm] = {"link_bytes_per_s": beta, "project": dcs,
                                "margin_s": margin}
    dl = local_proj_s - local_ref_s - frame_startup_s * (F_r - F_s)
    out["threshold_bytes_per_s"] = (B_r - B_s) / dl if dl > 0 else None
    return out


def measure_plan_costs(seconds, peaks, peak_src, gpu_index, ref="decode64",
                       proj="decode64_token"):
    """L_r and L_s of Equation (7) at a decode shape, measured on this device: the step time
    of the complete-logit surface and of the projected token surface on the same shape."""
    er = measure_workload(ref, seconds, peaks, peak_src, gpu_index)
    es = measure_workload(proj, seconds, peaks, peak_src, gpu_index)
    c = WORKLOADS[ref]
    sel = plan_selection(c["M"], c["V"], c["k"], es["step_us"] * 1e-6, er["step_us"] * 1e-6)
    sel["shape"] = {"M": c["M"], "d": c["d"], "V": c["V"], "k": c["k"]}
    sel["surfaces"] = {"ref": er["surface"], "proj": es["surface"]}
    return sel, er, es


PER_CONFIG = ("decode64", "decode64_token", "sampling", "prefill")
IDLE_BETWEEN_S = 0.5  # the GPU idles this long before each entry (power state of the last)


def per_config_table(seconds, peaks, peak_src, gpu_index):
    """The other configurations, each timed on its own for about `seconds` after a short idle
    gap (the power-capped prefill last, so it does not set the clocks of the others), plus
    the partial completion and the Equation (7) decision on the measured decode64 costs."""
    out = {}
    time.sleep(IDLE_BETWEEN_S)
    sel, out["decode64"], out["decode64_token"] = measure_plan_costs(seconds, peaks, peak_src,
                                                                     gpu_index)
    time.sleep(IDLE_BETWEEN_S)
    ms, n, roof, clk, _, _ = measure_partial("mlp_down", seconds, peaks, peak_src, gpu_index)
    out["mlp_down"] = {"desc": WORKLOADS["mlp_down"]["desc"], "steps": n, "step_us": ms * 1e3,
                       "rows_per_s": WORKLOADS["mlp_down"]["M"] / (ms * 1e-3),
                       "bound": "hbm", "frac": roof["frac"], "achieved": roof["achieved"],
                       "unit": "GB/s", "nominal_frac": roof["nominal"]["frac"], "clocks": clk}
    for name in PER_CONFIG[2:]:
        time.sleep(IDLE_BETWEEN_S)
        out[name] = measure_workload(name, seconds, peaks, peak_src, gpu_index)
    out["selection"] = sel
    return out


def run_partial(args, cfg, world, rank, local):
    """The row-parallel partial completion (lane partials + their ordered sum); under
    torchrun each rank runs its own replica (weak scaling, max-over-ranks timing)."""
    import torch
    import torch.distributed as dist
    from gemm_epilogue_reduction_gb300 import build as sbbuild
    sbbuild.build()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist.barrier()
    peaks, peak_src = load_peaks()
    ms, K_, roof, clk, in_bytes, flushed = measure_partial(
        args.workload, 0, peaks, peak_src, local, steps=args.steps, warmup=args.warmup)
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ms, "cuda")
    M = cfg["M"]
    line = {
        "metric": METRIC, "value": job_rows_per_s(world, M, ms), "unit": "rows/s", "n_gpus": world,
        "steps": K_, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": cfg["N"], "K": cfg["K"],
                   "lanes": cfg["lanes"], "desc": cfg["desc"],
                   "l2": ("inputs %.0f MB > L2, streamed every step" % (in_bytes / 1e6))
                   if not flushed else
                   ("inputs %.0f MB fit in L2: L2 flushed (2x L2 written) before every "
                    "step, outside its events" % (in_bytes / 1e6))},
        "roofline": roof,
        "cpu_baseline": None, "e2e": None, "clocks": clk, "gpu_launches": 2 * K_,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode16", choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--w-layout", default="auto", choices=["auto", "row", "packed"],
                    help="W as the calls read it: row-major [V, d], or packed once before "
                         "timing (sb_pack_weights, SB_W_PACKED); auto = the workload's layout")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--per-config-seconds", type=float, default=0.4,
                    help="device seconds of back-to-back steps per entry of the per_config "
                         "table (N = 1, default workload only; 0 leaves the table out)")
    args = ap.parse_args()
    W_LAYOUT["layout"] = args.w_layout
    cfg = WORKLOADS[args.workload]
    world, rank, local = dist_env()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
        return
    if cfg.get("kind") == "partial":
        run_partial(args, cfg, world, rank, local)
        return

    import torch
    import torch.distributed as dist

    import gemm_epilogue_reduction_gb300 as sb
    from gemm_epilogue_reduction_gb300 import build as sbbuild, synth

    sbbuild.build()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # each rank draws its own batch of rows (weak scaling) and the same W
    w = make_projection(cfg, rank)
    M, d, V, k = w.M, w.d, w.V, w.k
    H, W, out, stream = w.H, w.W, w.out, w.stream
    Wc = w.Warg  # W as the calls read it (row-major, or its packed copy)
    w_layout = w.layout
    surface, T, gseed = w.wsurf, w.T, w.gseed

    for _ in range(args.warmup):
        w.project()
    torch.cuda.synchronize()
    if sb.sb_last_device_status(out) != sb.SB_OK:
        raise RuntimeError("device status not OK after warm-up")

    # ---- timed region: the real call, back to back (its combine overlaps the GEMM's tail
    # as a programmatic dependent launch, and each call's GEMM the previous call's combine),
    # one event before the first step and one after the last
    K = args.steps
    flush = L2Flush() if w.in_bytes < l2_bytes() else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        total_ms = timed_steps(w.project, K, stream, flush) * K
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(total_ms, "cuda")
    if sb.sb_last_device_status(out) != sb.SB_OK:
        raise RuntimeError("device status not OK after the timed region")

    # ---- per-kernel durations: each kernel alone, K launches, events around each launch
    gemm_avg, comb_avg = kernel_times(w, K)

    # ---- the same steps on the row-major W, when the workload reads a packed one (reported
    # beside the line's value, which is the packed layout's)
    row_major = None
    if w_layout == "packed":
        def project_row():
            st = sb.sb_lmhead_project(H, W, M, d, V, k, w.surface, T, gseed, out, stream)
            if st != sb.SB_OK:
                raise sb.SbError(st, "sb_lmhead_project")
        for _ in range(3):
            project_row()
        torch.cuda.synchronize()
        row_ms = max_over_ranks(timed_steps(project_row, K, stream, flush), "cuda")
        def records_row():
            st = sb.sb_lmhead_records(H, W, M, d, V, k, w.surface, T, gseed, out, stream)
            if st != sb.SB_OK:
                raise sb.SbError(st, "sb_lmhead_records")
        import types
        row_gemm, _ = kernel_times(types.SimpleNamespace(records=records_row, combine=w.combine,
                                                         stream=stream), min(K, 200))
        row_major = {"ms_per_step": row_ms, "value": job_rows_per_s(world, M, row_ms),
                     "unit": "rows/s", "kernel_ms": row_gemm,
                     "frac": (V * d * 2 + M * d * 2 + 12 * M) / (row_gemm * 1e-3) /
                             (load_peaks()[0]["hbm_gbs"] * 1e9)}

    # ---- end to end through the public call with host buffers: H is copied from pinned
    # host memory and token + log-prob are copied back inside the call, every step
    # (token and log-prob back to back on both sides, so they come back in one copy)
    E = min(args.e2e_steps, K)
    H_host = H.cpu().pin_memory()
    res_host = torch.empty(2 * M, dtype=torch.int32).pin_memory()
    tok_host, lp_host = res_host[:M], res_host[M:].view(torch.float32)
    res_dev = torch.empty(2 * M, dtype=torch.int32, device="cuda")
    e2e_out = sb.sb_outputs(res_dev.data_ptr(), res_dev.data_ptr() + 4 * M, out.lse,
                            out.logits_bf16, out.target_ids, out.target_logprob, out.workspace,
                            out.workspace_bytes, out.topk_ids, out.topk_logprob, out.topk)
    H_dev = torch.empty_like(H)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        st = sb.sb_lmhead_project_from_host(H_host, H_dev, Wc, M, d, V, k, surface, T, gseed,
                                            e2e_out, tok_host, lp_host, stream)
        if st != sb.SB_OK:
            raise sb.SbError(st, "sb_lmhead_project_from_host")
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, "cuda")
    e2e_h2d = M * d * 2
    e2e_d2h = 2 * M * 4

    # ---- the same step as a serving loop would run it: captured once (sb_host_step_*),
    # one graph launch and one stream wait per step
    hstep = sb.HostStep(H_host, H_dev, Wc, M, d, V, k, surface, T, gseed, e2e_out, tok_host,
                        lp_host)
    for _ in range(3):
        hstep(stream)
        stream.synchronize()
    e0.record(stream)
    for _ in range(E):
        hstep(stream)
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_graph_ms = max_over_ranks(e0.elapsed_time(e1) / E, "cuda")
    hstep.close()

    ms_per_step = total_ms / K
    value = job_rows_per_s(world, M, ms_per_step)
    peaks, peak_src = load_peaks()
    tr = KERNEL_TRAFFIC.get(args.workload)
    traffic = (tr["bytes"] if tr and tr.get("src_sha") == kernel_src_hash() and
               tr.get("w_layout", "row") == w_layout else None)
    roof = projection_roofline(w, gemm_avg, comb_avg, peaks, peak_src,
                               tensor_bound=args.workload.startswith("prefill"), traffic=traffic)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        Hb, Wb = synth.bf16_bits(H), synth.bf16_bits(W)
        rows_per_call = max(1, min(M, 4))
        v, n, el, cores = oracle_rows_per_s(Hb, Wb, k, cfg, rows_per_call, args.cpu_seconds)
        cpu = {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} rows in {el:.1f} s ({rows_per_call}-row calls against the full W)"}

    per_cfg = None
    if world == 1 and args.workload == "decode16" and args.per_config_seconds > 0:
        del w, H, W, Wc, out, H_dev, H_host
        torch.cuda.empty_cache()
        per_cfg = per_config_table(args.per_config_seconds, peaks, peak_src, local)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "d": d, "V": V, "k": k,
                       "surface": cfg["surface"], "desc": cfg["desc"], "w_layout": w_layout,
                       "l2": ("inputs larger than L2 (W %.2f GB streamed every step)"
                              % (V * d * 2 / 1e9)) if flush is None else
                             ("inputs %.1f MB fit in L2: L2 flushed (2x L2 written) before "
                              "every step, outside its events" % (w_in_mb(V, d, M))),
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": M / (e2e_ms * 1e-3) * world, "unit": "rows/s",
                    "h2d_bytes_per_step": e2e_h2d, "d2h_bytes_per_step": e2e_d2h,
                    "ms_per_step": e2e_ms},
            "e2e_host_step": {"value": M / (e2e_graph_ms * 1e-3) * world, "unit": "rows/s",
                              "ms_per_step": e2e_graph_ms,
                              "api": "sb_host_step_create once, sb_host_step_launch per step"},
            "clocks": clocks.summary(),
            "gpu_launches": 2 * K,
            "row_major_w": row_major,
            "wall_s_timed": t_wall,
            "per_config": per_cfg,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def w_in_mb(V, d, M):
    return (V * d * 2 + M * d * 2) / 1e6


if __name__ == "__main__":
    main()
