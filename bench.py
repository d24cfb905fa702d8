"""Benchmark: sink-attention forward + backward on one GB300 (or N, weakly
scaled), reported as algorithmic bf16 TFLOP/s and as a fraction of the
measured dense bf16 tensor peak.

A step is one forward and one backward (every kernel of the path) over one
batch of the dense workload: B=4, T=2048, Hq=64, Hkv=8, d=64, causal, sinks
~ U(-2, 2), seeded synthetic bf16 tensors. FLOPs count only the (row, key)
pairs the mask allows: forward 4*d per pair and head, backward 10*d
(five products), so a step is 14*d*N_pairs*Hq.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload dense|window|varlen|long|long_window|tiny|decode|decode_window]

For N > 1 every rank (one process per GPU, under torch.distributed.run; a
plain ``python bench.py --gpus N`` starts that launcher itself) runs the step
on its own batch, data parallel: the only exchange is the all-reduce of the
per-head sink gradient dL/dS_h after each backward (NCCL). Timing is the max
over ranks and value the total over ranks (weak scaling). --impl reference times the fp64 CPU oracle on a
bounded sample of the same workload (rank 0 only).

The decode workloads time one decode step (a query row per sequence over a
paged KV cache) instead, reported as algorithmic HBM GB/s.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
# numpy's BLAS runs the decode oracle's products on one thread, so the CPU
# baseline's core count is known (the fwd/bwd oracle sets its own threads)
for _var in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
    os.environ.setdefault(_var, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "sink-attn fwd+bwd bf16 TFLOP/s on 1 GB300 and % of dense tensor peak"
UNIT = "TFLOP/s"
HEAD_DIM = 64
L2_FLUSH_BYTES = 512 << 20          # > 126 MB L2, written between timed steps
L2_CLEAN_BYTES = 256 << 20          # then read, so the written lines leave L2 before the step
L2_NOTE = ("flushed between timed steps: 512 MiB written, then 256 MiB read so that no dirty "
           "line of the flush is written back inside the step")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
THROTTLE = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


# ----------------------------------------------------------------- counting
def allowed_pairs(lengths, causal: bool, window: int) -> int:
    """Number of (row, key) pairs the mask allows, summed over sequences."""
    n = 0
    for L in lengths:
        L = int(L)
        if not causal:
            n += L * L
        elif window <= 0 or window >= L:
            n += L * (L + 1) // 2
        else:
            W = window
            n += W * (W + 1) // 2 + (L - W) * W
    return n


def step_flops(lengths, Hq, causal, window, d=HEAD_DIM):
    pairs = allowed_pairs(lengths, causal, window)
    return 4 * d * pairs * Hq, 10 * d * pairs * Hq


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(kernel_file: str):
    """Hash of a kernel's source together with the shared device headers it
    includes, so that a change to either invalidates recorded counters."""
    csrc = os.path.join(ROOT, "attention_learnable_sinks_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for fn in (kernel_file, "sm100.cuh", "internal.h"):
            h.update(open(os.path.join(csrc, fn), "rb").read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def traffic_record(key: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, valid only while the kernel source is unchanged. ``key`` is the
    kernel's source file, then "@<workload>" for a workload other than dense,
    then "#deterministic" for the main backward's deterministic-mode
    instantiation or "#exact" for the forward kernel's decode form."""
    kernel_file = key.split("#")[0].split("@")[0]
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    sha = kernel_source_sha(kernel_file)
    if sha is None:
        return None
    entry = rec.get(key)
    if not entry or entry.get("source_sha") != sha:
        return None
    return entry


class L2Flush:
    """Evicts the inputs from L2 between timed steps: a write larger than L2,
    then a read larger than L2 (which writes the dirty lines back before the
    step starts instead of during it)."""

    def __init__(self, device):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


# ----------------------------------------------------------------- clocks
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
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(THROTTLE, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- dist
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks (every rank gets it)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- oracle leg
ORACLE_SAMPLE = {"kv_groups": [0, 1], "seqs": [0, 1, 2, 3], "prefix": None}


def oracle_sample_run(w, kv_groups, seqs, prefix=None):
    """Time the fp64 oracle (as it stands) on complete GQA groups of whole
    sequences (or their first `prefix` tokens). Returns (seconds, flops)."""
    import oracle
    cu = w.cu_seqlens.numpy().astype(np.int64)
    G = w.Hq // w.Hkv
    qh = np.concatenate([np.arange(g * G, (g + 1) * G) for g in kv_groups])
    tok, lens = [], []
    for b in seqs:
        a, e = int(cu[b]), int(cu[b + 1])
        if prefix is not None:
            e = min(e, a + prefix)
        tok.append(np.arange(a, e))
        lens.append(e - a)
    tok = np.concatenate(tok)
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)

    def f64(t):
        return t.float().numpy().astype(np.float64)

    q, k, v = f64(w.q[tok][:, qh]), f64(w.k[tok][:, kv_groups]), f64(w.v[tok][:, kv_groups])
    do = f64(w.dout[tok][:, qh])
    s = w.sinks.numpy().astype(np.float64)[qh]
    t0 = time.perf_counter()
    oracle.sinkattn(q, k, v, s, sub_cu, causal=w.causal, window=w.window, scale=w.scale,
                    dout=do, want=("o", "lse", "dq", "dk", "dv", "dsinks"))
    dt = time.perf_counter() - t0
    f, b = step_flops(lens, len(qh), w.causal, w.window)
    return dt, f + b


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    import oracle
    from attention_learnable_sinks_gb300 import workloads
    oracle.build()
    w = workloads.config(args.workload)
    # bounded per-step sample: one GQA group, first sequence, first 768 tokens
    sample = {"kv_groups": [0], "seqs": [0], "prefix": min(768, w.max_seqlen)}
    for _ in range(args.warmup):
        oracle_sample_run(w, **sample)
    secs, flops = 0.0, 0
    for _ in range(args.steps):
        dt, f = oracle_sample_run(w, **sample)
        secs += dt
        flops += f
    value = flops / secs / 1e12
    cores = oracle.default_threads()
    desc = (f"fp64 oracle, kv group 0 ({w.Hq // w.Hkv} query heads), sequence 0, first "
            f"{sample['prefix']} tokens of {args.workload}, fwd+bwd per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(w, args.workload),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


def workload_config(w, name):
    from attention_learnable_sinks_gb300.workloads import DESCRIPTIONS
    return {"workload": f"{name}: {DESCRIPTIONS[name]}", "nseq": w.nseq, "total_tokens": w.total,
            "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": int(w.q.shape[2]), "causal": w.causal,
            "window": w.window, "l2": L2_NOTE,
            "flop_convention": "14*d*N_allowed_pairs*Hq (fwd 4*d, bwd 10*d)"}


# ----------------------------------------------------------------- gb300 leg
def run_gb300(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    from attention_learnable_sinks_gb300 import _binding, api, sharding, workloads
    _binding.lib()
    w = workloads.config(args.workload)
    lengths = w.meta["lengths"]
    hd = int(w.q.shape[2])
    fwd_flops, bwd_flops = step_flops(lengths, w.Hq, w.causal, w.window, hd)
    flops = fwd_flops + bwd_flops

    q, k, v, do = (t.to(device) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(device), w.cu_seqlens.to(device)
    maxlen = w.max_seqlen
    total, Hq, Hkv = w.total, w.Hq, w.Hkv
    o = torch.empty(total, Hq, hd, dtype=torch.bfloat16, device=device)
    lse = torch.empty(Hq, total, dtype=torch.float32, device=device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ds = torch.empty(Hq, dtype=torch.float32, device=device)
    ws_f = torch.empty(api.workspace_bytes("fwd", w.nseq, total, Hq, Hkv, head_dim=hd),
                       dtype=torch.uint8, device=device)
    ws_b = torch.empty(api.workspace_bytes("bwd", w.nseq, total, Hq, Hkv, head_dim=hd),
                       dtype=torch.uint8, device=device)
    flush = L2Flush(device)

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record()  # creates the CUDA event so the library can record into it
        return evs

    K = args.steps
    # head_dim 128 always takes dq from the fixed-order query-stationary pass
    det = args.deterministic or hd != HEAD_DIM
    step_ev = [new_events(2) for _ in range(K)]
    fwd_ev = [new_events(2) for _ in range(K)]
    bwd_ev = [new_events(2) for _ in range(K)]
    dq_ev = [new_events(2) for _ in range(K)] if det else None

    def step(i=None):
        # the forward clears the backward's dq accumulator (atomic mode)
        api.forward(q, k, v, s, cu, maxlen, causal=w.causal, window=w.window, scale=w.scale,
                    out=o, lse=lse, workspace=ws_f,
                    timing_events=None if i is None else fwd_ev[i],
                    bwd_workspace=None if det else ws_b)
        api.backward(q, k, v, s, cu, maxlen, o, lse, do, causal=w.causal, window=w.window,
                     scale=w.scale, dq=dq, dk=dk, dv=dv, dsinks=ds, workspace=ws_b,
                     timing_events=None if i is None else bwd_ev[i], deterministic=det,
                     timing_events_dq=None if i is None or not det else dq_ev[i],
                     workspace_cleared=not det)
        if world > 1:  # data parallel: sum the ranks' sink gradients
            sharding.all_reduce_sink_grad(ds)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert _binding.device_error() == 0, "device error word set during warm-up"

    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    n0 = _binding.launch_count()
    for i in range(K):
        flush()
        step_ev[i][0].record()
        step(i)
        step_ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    launches = _binding.launch_count() - n0
    clk = clocks.stop()
    assert _binding.device_error() == 0, "device error word set during the timed region"

    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_ev]
    bwd_ms = [a.elapsed_time(b) for a, b in bwd_ev]
    dq_ms = [a.elapsed_time(b) for a, b in dq_ev] if det else None
    total_ms = reduce_max(sum(step_ms), world, device)
    ms_per_step = total_ms / K
    value = flops * world * K / (total_ms / 1e3) / 1e12

    # ---- end to end through the public API with host buffers: HostPipeline
    # streams groups of whole sequences, overlapping each group's copies with
    # another group's kernels
    hq, hk, hv, hdo = (t.pin_memory() for t in (w.q, w.k, w.v, w.dout))
    hs = w.sinks.pin_memory()
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hdq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
    hdk = torch.empty(dk.shape, dtype=dk.dtype).pin_memory()
    hdv = torch.empty(dv.shape, dtype=dv.dtype).pin_memory()
    hds = torch.empty(ds.shape, dtype=ds.dtype).pin_memory()
    pipe = api.HostPipeline(w.cu_seqlens, w.Hq, w.Hkv, causal=w.causal, window=w.window,
                            scale=w.scale, groups=args.e2e_groups, device=device,
                            deterministic=det, head_dim=hd)
    h2d, d2h = pipe.h2d_bytes(), pipe.d2h_bytes()

    def e2e_step():
        pipe.run(hq, hk, hv, hdo, hs, ho, hdq, hdk, hdv, hds)

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [new_events(2) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush()
        e2e_ev[i][0].record()
        e2e_step()
        e2e_ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_total = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ev), world, device)
    e2e_value = flops * world * K / (e2e_total / 1e3) / 1e12

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    f_avg, b_avg = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    q_avg = statistics.mean(dq_ms) if det else None
    # the deterministic dq pass recomputes S and dP and forms dQ: three
    # products where the forward has two; in that mode the main backward's
    # algorithmic work is its dk / dv products (S, dP, dV, dK: 4 of 5)
    dq_flops = 1.5 * fwd_flops
    main_flops = 0.8 * bwd_flops if det else bwd_flops
    cands = [("fwd", f_avg, fwd_flops, "fwd.cu"),
             ("bwd main", b_avg, main_flops, "bwd.cu" if hd == HEAD_DIM else "bwd_wide.cu")]
    if det:
        cands.append(("dq pass", q_avg, dq_flops, "dq.cu"))
    dom, dom_ms, dom_flops, dom_file = max(cands, key=lambda c: c[1])
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    dom_key = dom_file + ("#deterministic" if det and dom_file == "bwd.cu" else "")
    # counters were taken on the dense workloads; other workloads have none
    tr = traffic_record(dom_key if args.workload == "dense" else f"{dom_key}@{args.workload}")
    if w.window > 0:
        # a band of W keys: about W flop per byte moved, below the ridge
        # (1910.8 TFLOP/s / 6786.6 GB/s = 282 flop/B), so HBM bounds it.
        # Algorithmic bytes per launch, per token (d = 64):
        #   forward:       read q, k, v; write o, LSE
        #   backward main: read q, dO, k, v, LSE, D; write dk, dv and the fp32
        #                  dq accumulator once (no accumulator when deterministic)
        #   dq pass:       read q, dO, k, v, LSE, D; write dq
        d, Hq, Hkv = hd, w.Hq, w.Hkv
        per_tok = {"fwd": 2 * Hq * d + 4 * Hkv * d + 2 * Hq * d + 4 * Hq,
                   "bwd main": 4 * Hq * d + 4 * Hkv * d + 8 * Hq + 4 * Hkv * d + (0 if det else 4 * Hq * d),
                   "dq pass": 4 * Hq * d + 4 * Hkv * d + 8 * Hq + 2 * Hq * d}[dom]
        gbs = per_tok * w.total / (dom_ms / 1e3) / 1e9
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roofline = {"bound": "hbm", "kernel": dom, "achieved": gbs, "peak": hbm, "unit": "GB/s",
                    "frac": gbs / hbm, "peak_source": f"{peak_src} HBM copy",
                    "algorithmic_bytes_per_launch": per_tok * w.total,
                    "tflops": achieved, "traffic": tr["dram_bytes_per_launch"] if tr else None}
    else:
        roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": f"{peak_src} bf16 dense (burst)",
                    "traffic": tr["dram_bytes_per_launch"] if tr else None}
    # nominal dense bf16 rate of this GPU for context: SMs x max SM clock x
    # 8192 flop/clk/SM (one M=128, N=256, K=16 product per 128 clk per SM)
    props_n = torch.cuda.get_device_properties(device)
    nominal = props_n.multi_processor_count * clk.get("sm_max_mhz", 0) * 1e6 * 8192 / 1e12 \
        if clk.get("sm_max_mhz") else None

    cfg = workload_config(w, args.workload)
    cfg["parallelism"] = (f"dp{world}: each rank its own batch, dL/dS_h all-reduced per step"
                          if world > 1 else "single GPU")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": cfg,
        "frac_of_peak": value / world / peak, "peak_tflops": peak, "peak_source": peak_src,
        "peak_nominal_tflops": nominal,
        "frac_of_nominal_peak": (value / world / nominal) if nominal else None,
        "fwd_ms": f_avg, "bwd_main_ms": b_avg,
        "fwd_tflops": fwd_flops / (f_avg / 1e3) / 1e12,
        "bwd_main_tflops": main_flops / (b_avg / 1e3) / 1e12,
        "deterministic_backward": det,
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_total / K},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if det:
        line["dq_pass_ms"] = q_avg
        line["dq_pass_tflops"] = dq_flops / (q_avg / 1e3) / 1e12
        line["config"]["backward"] = "deterministic: dq from a fixed-order query-stationary pass"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, f = oracle_sample_run(w, **ORACLE_SAMPLE)
        import oracle
        line["cpu_baseline"] = {
            "value": f / secs / 1e12, "unit": UNIT, "cores": oracle.default_threads(),
            "kind": "oracle", "seconds": secs,
            "sample": f"fp64 oracle fwd+bwd, kv groups {ORACLE_SAMPLE['kv_groups']} ({2 * (w.Hq // w.Hkv)} query heads), "
                      f"sequences {ORACLE_SAMPLE['seqs']} of {args.workload}"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------- decode
DECODE_METRIC = "sink-attn paged decode, algorithmic HBM GB/s on 1 GB300 and % of measured copy bandwidth"


def decode_bytes(w):
    """Algorithmic bytes of one decode step: the visible keys' K and V rows,
    q and o (bf16), LSE (fp32). Block rounding and the split partials are
    overhead, not counted."""
    d = int(w.q.shape[2])
    keys = sum(min(L, w.window) if w.window > 0 else L for L in w.meta["lengths"])
    return keys * w.Hkv * d * 2 * 2 + w.nseq * w.Hq * (2 * d * 2 + 4)


def decode_config_record(w, name):
    from attention_learnable_sinks_gb300.workloads import DECODE_DESCRIPTIONS
    return {"workload": f"{name}: {DECODE_DESCRIPTIONS[name]}", "nseq": w.nseq,
            "cached_tokens": sum(w.meta["lengths"]), "Hq": w.Hq, "Hkv": w.Hkv,
            "head_dim": int(w.q.shape[2]), "block_size": w.block_size, "window": w.window,
            "l2": L2_NOTE,
            "byte_convention": "visible K,V rows + q + o + lse per step"}


_F64_CACHE = {}


def oracle_decode_sample(w, seqs):
    """Time the fp64 decode oracle on some sequences (the caches are converted
    to fp64 once, outside the timing). Returns (seconds, algorithmic bytes)."""
    from oracle import decode as odec

    def f64(t):
        return t.float().numpy().astype(np.float64)
    if id(w) not in _F64_CACHE:
        _F64_CACHE.clear()
        _F64_CACHE[id(w)] = (f64(w.k_cache), f64(w.v_cache))
    kc, vc = _F64_CACHE[id(w)]
    q = f64(w.q[seqs])
    t0 = time.perf_counter()
    odec.decode(q, kc, vc, w.block_table.numpy()[seqs], w.seqlens.numpy()[seqs], w.sinks.numpy(),
                window=w.window, scale=w.scale)
    dt = time.perf_counter() - t0
    d = int(w.q.shape[2])
    lens = [w.meta["lengths"][b] for b in seqs]
    keys = sum(min(L, w.window) if w.window > 0 else L for L in lens)
    return dt, keys * w.Hkv * d * 4 + len(seqs) * w.Hq * (4 * d + 4)


def run_decode(args):
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        from attention_learnable_sinks_gb300 import workloads
        w = workloads.decode_config(args.workload)
        seqs = [0, 1]
        for _ in range(args.warmup):
            oracle_decode_sample(w, seqs)
        secs, nbytes = 0.0, 0
        for _ in range(args.steps):
            dt, b = oracle_decode_sample(w, seqs)
            secs += dt
            nbytes += b
        value = nbytes / secs / 1e9
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded)", "config": decode_config_record(w, args.workload),
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"numpy fp64 decode oracle, sequences {seqs}"},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line))
        return 0
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from attention_learnable_sinks_gb300 import _binding, api, workloads
    _binding.lib()
    w = workloads.decode_config(args.workload)
    q, kc, vc = w.q.to(device), w.k_cache.to(device), w.v_cache.to(device)
    table, lens, s = w.block_table.to(device), w.seqlens.to(device), w.sinks.to(device)
    o = torch.empty_like(q)
    lse = torch.empty(w.Hq, w.nseq, dtype=torch.float32, device=device)
    ws = torch.empty(_binding.lib().sinkattn_decode_workspace_size_d(w.nseq, w.Hq, 64, int(w.q.shape[2])),
                     dtype=torch.uint8, device=device)
    flush = L2Flush(device)
    nbytes = decode_bytes(w)

    def step():
        api.decode(q, kc, vc, table, lens, s, window=w.window, scale=w.scale, out=o, lse=lse,
                   workspace=ws, exact=args.decode_exact)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert _binding.device_error() == 0, "device error word set during warm-up"
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    n0 = _binding.launch_count()
    for i in range(K):
        flush()
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    launches = _binding.launch_count() - n0
    clk = clocks.stop()
    assert _binding.device_error() == 0, "device error word set during the timed region"
    total_ms = reduce_max(sum(a.elapsed_time(b) for a, b in ev), world, device)
    ms = total_ms / K
    value = nbytes * world * K / (total_ms / 1e3) / 1e9

    # end to end: the cache is state that stays on the device; each step copies
    # the new query rows and lengths in and o, lse out through pinned buffers
    hq, hl = w.q.pin_memory(), w.seqlens.pin_memory()
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = hq.numel() * 2 + hl.numel() * 4
    d2h = ho.numel() * 2 + hlse.numel() * 4

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        lens.copy_(hl, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush()
        e2e_ev[i][0].record()
        e2e_step()
        e2e_ev[i][1].record()
    torch.cuda.synchronize()
    e2e_total = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ev), world, device)
    e2e_value = nbytes * world * K / (e2e_total / 1e3) / 1e9

    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # counters of the decode's dominant kernel: the split kernel, or the
    # forward kernel's decode form for the exact decode
    tr = traffic_record(f"fwd.cu@{args.workload}#exact" if args.decode_exact
                        else f"decode.cu@{args.workload}")
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": dict(decode_config_record(w, args.workload),
                       decode=("exact: each row computed as the training forward's last row "
                               "(bitwise equal), one unit per (sequence, kv head)")
                       if args.decode_exact else "split keys + sink-aware combine"),
        "sequences_per_s": w.nseq * world * K / (total_ms / 1e3),
        "roofline": {"bound": "hbm", "kernel": "decode (split + combine)", "achieved": value / world,
                     "peak": hbm, "unit": "GB/s", "frac": value / world / hbm,
                     "peak_source": f"{peak_src} HBM copy",
                     "algorithmic_bytes_per_launch": nbytes,
                     "traffic": tr["dram_bytes_per_launch"] if tr else None},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_total / K},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, b = oracle_decode_sample(w, [0, 1, 2, 3])
        line["cpu_baseline"] = {"value": b / secs / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "seconds": secs,
                                "sample": f"numpy fp64 decode oracle, sequences 0-3 of {args.workload}"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default="dense",
                    choices=("tiny", "dense", "window", "varlen", "long", "long_window",
                             "dense_d128", "decode", "decode_window", "decode_d128"))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward with dq summed in a fixed order (query-stationary dq pass)")
    ap.add_argument("--decode-exact", action="store_true",
                    help="decode workloads: the exact decode (bitwise equal to the training "
                         "forward's last row) instead of the split decode")
    ap.add_argument("--e2e-groups", type=int, default=2,
                    help="groups of whole sequences streamed by the end-to-end leg")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the launcher with this same command line
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               "--master-port", str(port), os.path.abspath(__file__),
               *(sys.argv[1:] if argv is None else argv)]
        return subprocess.call(cmd)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE={world} of the launcher")
    if args.workload.startswith("decode"):
        return run_decode(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
