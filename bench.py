#!/usr/bin/env python3
"""Stochastic Attention forward throughput on one GB300 (or N replicas).

Workload: the long-prefill GQA shape -- batch 1, n = 32768 tokens, 32 query
heads / 8 kv heads, head_dim 128, bf16, causal SA with w = 128, one seeded
sigma.  One step = one sa_forward call (the whole hot path: sigma gather,
windowed attention, sigma^-1 scatter) through the libsa C ABI.

Prints ONE JSON line (rank 0).  ``value`` is device-timed tokens/s with
inputs resident in HBM (L2 flushed between steps); ``e2e`` times the same
call with the host->device copies of Q/K/V/sigma from pinned memory and the
device->host copy of the output inside the timed region, two streams taking
alternate steps so that one step's output copy overlaps the next step's
input copy.  ``roofline``
compares the kernel's algorithmic bytes per launch (Q, K, V and Y once,
sigma once) over its CUDA-event duration with the measured HBM copy peak.

``--impl reference`` times the fp64 CPU oracle (the only reference
implementation of this method) on the host cores instead.

``--workload`` times one of the other shapes instead of the headline (the
pretraining layer, the very long context gated merge, the length sweep), with
``--window`` / ``--seq-len`` overrides; their ``roofline`` uses whichever leg
(HBM bytes or tensor FLOPs) bounds them.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(workload="long_prefill_gqa", batch=1, seq_len=32768, num_q_heads=32,
                num_kv_heads=8, head_dim=128, window=128, causal=True, path="sa", seed=0,
                std=None)
METRIC = "SA fwd tokens/s and % roofline (bf16, n=32K, w=128, GQA 32q/8kv, d=128)"
# The other workload shapes (--workload): causal SA or the causal gated SA+SWA
# merge (gate logits ~ N(0, 1)); the default above is the headline.
WORKLOADS = {
    "long_prefill_gqa": WORKLOAD,
    "pretrain_layer": dict(workload="pretrain_layer", batch=4, seq_len=2048, num_q_heads=16,
                           num_kv_heads=16, head_dim=64, window=128, causal=True, path="gated",
                           seed=0, std=1.0 / 8.0),
    "very_long_context": dict(workload="very_long_context", batch=1, seq_len=131072,
                              num_q_heads=32, num_kv_heads=4, head_dim=128, window=1024,
                              causal=True, path="gated", seed=0, std=None),
    "length_sweep": dict(workload="length_sweep", batch=1, seq_len=262144, num_q_heads=16,
                         num_kv_heads=16, head_dim=128, window=128, causal=True, path="sa",
                         seed=0, std=None),
}
# DRAM bytes per launch of the headline kernel from its ncu capture, with the
# sha256 of the kernel sources the capture was taken on (written beside the
# ncu summary, profiles/sa_ring_kernel_long_prefill_gqa_w128.md)
PROFILE = os.path.join(ROOT, "profiles", "sa_ring_kernel_long_prefill_gqa_w128.json")
# the ring kernel and the tcgen05 helpers it inlines: the profile's DRAM
# counters hold only while these files are unchanged
KERNEL_SOURCES = [os.path.join(ROOT, "stochastic_sliding_window_gb300", "csrc", f)
                  for f in ("sa_tc_ring.cu", "sa_tc_common.cuh")]

_G: dict = {}  # arrays shared with forked oracle workers


def causal_sa_pairs(n: int, window: int) -> int:
    """Attended (query, key) pairs of causal SA in one sequence: each token
    itself plus, of every unordered pair at permuted distance 1..h, exactly
    one edge."""
    h = min(window // 2, n - 1)
    return n + sum(n - d for d in range(1, h + 1))


def swa_pairs(n: int, window: int) -> int:
    """Attended pairs of SWA: keys [i - w + 1, i] clipped at 0."""
    w = min(window, n)
    return n * w - w * (w - 1) // 2


def algorithmic(wl) -> tuple[int, float]:
    """Bytes the path must move (Q, K, V and Y once, sigma, gate logits when
    gated) and FLOPs it must do (QK^T and PV, 2d each, per attended pair)."""
    b, n, hq, hkv, d = wl["batch"], wl["seq_len"], wl["num_q_heads"], wl["num_kv_heads"], wl["head_dim"]
    bytes_alg = 2 * b * n * d * (hq + 2 * hkv + hq) + 4 * b * n
    pairs = causal_sa_pairs(n, wl["window"])
    if wl["path"] == "gated":
        bytes_alg += 2 * 4 * b * n * hq
        pairs += swa_pairs(n, wl["window"])
    flops = 4.0 * d * hq * b * pairs
    return bytes_alg, flops


def algorithmic_bwd(wl) -> tuple[int, float]:
    """Backward pass: bytes it must move (Q, K, V, dY and sigma read once;
    dQ, dK, dV written once; the gate logits read and their gradients written
    when gated) and FLOPs it must do (QK^T, dY V^T, dS K, dS^T Q, P^T dY:
    2d each per attended pair; the recomputation of S and dP by the key-tile
    kernel is implementation overhead, not counted)."""
    b, n, hq, hkv, d = wl["batch"], wl["seq_len"], wl["num_q_heads"], wl["num_kv_heads"], wl["head_dim"]
    bytes_alg = 2 * b * n * d * (2 * hq + 2 * hkv) + 2 * b * n * d * (hq + 2 * hkv) + 4 * b * n
    pairs = causal_sa_pairs(n, wl["window"])
    if wl["path"] == "gated":
        bytes_alg += 4 * 4 * b * n * hq
        pairs += swa_pairs(n, wl["window"])
    return bytes_alg, 10.0 * d * hq * b * pairs


def metric_of(wl, bwd: bool = False) -> str:
    if wl is WORKLOAD and not bwd:
        return METRIC
    what = "gated SA+SWA" if wl["path"] == "gated" else "SA"
    return (f"{what} {'bwd' if bwd else 'fwd'} tokens/s and % roofline (bf16, n={wl['seq_len']}, "
            f"w={wl['window']}, {wl['num_q_heads']}q/{wl['num_kv_heads']}kv, d={wl['head_dim']})")


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


def kernel_source_sha256() -> str:
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic() -> int | None:
    """DRAM bytes per launch from the committed ncu capture, if it was taken
    on the current kernel source (null once the kernel has changed)."""
    try:
        with open(PROFILE) as f:
            rec = json.load(f)
        src = kernel_source_sha256()
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != src:
        return None
    return int(rec["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ oracle leg

def _oracle_rows(rows):
    import oracle
    if _G.get("bwd"):
        oracle.sa_dq_rows(_G["q"], _G["k"], _G["v"], _G["perm"], _G["dy"], _G["window"],
                          _G["causal"], rows)
        return
    if _G["path"] == "gated":
        oracle.gated_rows(_G["q"], _G["k"], _G["v"], _G["perm"], _G["ga"], _G["gw"], _G["window"],
                          None, _G["causal"], rows=rows)
    else:
        oracle.sa_rows(_G["q"], _G["k"], _G["v"], _G["perm"], _G["window"], _G["causal"], rows=rows)


def _oracle_chunk(rows):
    _oracle_rows(rows)
    return len(rows)


def publish_oracle_inputs(case, perm, wl, dy=None):
    """Make the inputs visible to oracle workers forked after this call.  With
    dy, the oracle times the backward pass per query token (its row's dQ and
    its contributions to dK and dV)."""
    _G.update(q=case.q, k=case.k, v=case.v, perm=perm, window=wl["window"], causal=wl["causal"],
              path=wl["path"], ga=case.gate_sa, gw=case.gate_swa, dy=dy, bwd=dy is not None)


def oracle_throughput(case, perm, wl, seconds: float, pool=None, cores: int = 1) -> dict:
    """Time the oracle on a seeded sample of query tokens (all heads of each).
    Workers in ``pool`` must have been forked after publish_oracle_inputs."""
    import numpy as np
    n = wl["seq_len"]
    rng = np.random.default_rng(1)
    calib = [(0, int(i)) for i in rng.integers(0, n, 16)]
    t0 = time.perf_counter()
    _oracle_rows(calib)
    per_row = max((time.perf_counter() - t0) / len(calib), 1e-6)
    count = int(max(cores * 4, min(n * wl["batch"], seconds * cores / per_row)))
    rows = [(0, int(i)) for i in rng.integers(0, n, count)]
    chunk = max(1, count // (cores * 4))
    chunks = [rows[i:i + chunk] for i in range(0, count, chunk)]
    t0 = time.perf_counter()
    if pool is None:
        done = sum(_oracle_chunk(c) for c in chunks)
    else:
        done = sum(pool.map(_oracle_chunk, chunks))
    wall = time.perf_counter() - t0
    return dict(value=done / wall, unit="tokens/s", cores=cores, kind="oracle",
                sample=f"{done} seeded query tokens (all {wl['num_q_heads']} heads each) of the "
                       f"n={n} workload, fp64 NumPy oracle, {cores} worker processes",
                seconds=wall)


def make_pool(cores: int):
    import multiprocessing as mp
    # Forked before any CUDA call in this process; workers see the inputs
    # copy-on-write.
    return mp.get_context("fork").Pool(cores)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=mx, reasons=sorted(reasons),
                    samples=len(sm))


# ------------------------------------------------------------------ main legs

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device) -> float:
    """The slowest rank's value (replicas run independently; the job's time is
    the longest one).  Identity when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch each step."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def make_inputs(wl):
    from sa_synth import make_case
    return make_case(wl["batch"], wl["seq_len"], wl["num_q_heads"], wl["num_kv_heads"],
                     wl["head_dim"], wl["seed"], std=wl["std"], gates=wl["path"] == "gated")


def config_of(wl) -> dict:
    """The workload keys both arms report (so that their configs compare
    equal), with how the GPU arm keeps L2 from serving a step's inputs."""
    b, n, hq, hkv, d = (wl[k] for k in ("batch", "seq_len", "num_q_heads", "num_kv_heads",
                                        "head_dim"))
    in_mb = 2 * b * n * d * (hq + 2 * hkv) / 1e6
    cfg = {k: wl[k] for k in ("workload", "batch", "seq_len", "num_q_heads", "num_kv_heads",
                              "head_dim", "window", "causal", "path")}
    cfg["l2"] = f"flushed between steps (256 MB write); inputs {in_mb:.0f} MB"
    return cfg


def run_reference(args, wl=WORKLOAD):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    case = make_inputs(wl)
    perm = np.stack([oracle.make_perm(wl["seed"], 0, b, wl["seq_len"]) for b in range(wl["batch"])])
    cores = len(os.sched_getaffinity(0))
    bwd = getattr(args, "pass_", "fwd") == "bwd"
    dy = (np.random.default_rng(wl["seed"] + 7).standard_normal(case.q.shape).astype(np.float32)
          if bwd else None)
    publish_oracle_inputs(case, perm, wl, dy)
    pool = make_pool(cores)
    per_step = max(0.5, min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_throughput(case, perm, wl, per_step / 4, pool, cores)
    runs = [oracle_throughput(case, perm, wl, per_step, pool, cores) for _ in range(args.steps)]
    pool.close()
    tokens = sum(r["value"] * r["seconds"] for r in runs)
    secs = sum(r["seconds"] for r in runs)
    value = tokens / secs
    line = dict(impl="reference", metric=metric_of(wl, bwd), value=value, unit="tokens/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * secs / args.steps,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic",
                config=config_of(wl),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=cores, kind="oracle",
                                  sample=runs[0]["sample"].split(",")[0] + " per step (seeded "
                                  "sample), fp64 NumPy oracle"),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0),
                gpu_launches=0)
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, wl=WORKLOAD):
    import numpy as np
    rank, world, local = dist_env()
    from sa_synth import bf16_bits
    case = make_inputs(wl)
    gated = wl["path"] == "gated"
    bwd = getattr(args, "pass_", "fwd") == "bwd"
    if bwd and gated and not args.no_cpu_baseline:
        args.no_cpu_baseline = True  # the oracle's per-row backward covers the SA path only
    dy_np = None
    if bwd:  # upstream gradient ~ N(0, 1), bf16
        dy_np = np.random.default_rng(wl["seed"] + 7).standard_normal(case.q.shape).astype(np.float32)

    import stochastic_sliding_window_gb300 as sa
    sa.load()
    perm_np = sa.make_perms(wl["seed"], 0, wl["batch"], wl["seq_len"])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = len(os.sched_getaffinity(0))
        publish_oracle_inputs(case, perm_np.astype(np.int64), wl, dy_np)
        pool = make_pool(cores)  # before the first CUDA call
        cpu = oracle_throughput(case, perm_np.astype(np.int64), wl, args.cpu_seconds, pool, cores)
        pool.close()
        pool.join()
        cpu.pop("seconds", None)

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def host_bf16(x):
        return torch.from_numpy(bf16_bits(x).view(np.int16)).view(torch.bfloat16)

    # Host inputs of one step, in call order; outputs are allocated per slot.
    hins = [host_bf16(case.q), host_bf16(case.k), host_bf16(case.v), torch.from_numpy(perm_np)]
    if gated:
        hins += [torch.from_numpy(case.gate_sa), torch.from_numpy(case.gate_swa)]
    if bwd:
        hins.append(host_bf16(dy_np))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kern = {"auto": sa.KERNEL_AUTO, "simt": sa.KERNEL_SIMT, "gather": sa.KERNEL_TCGEN05_GATHER,
            "ring": sa.KERNEL_TCGEN05_RING, "chunk": sa.KERNEL_TCGEN05_CHUNK}[args.kernel]

    def make_outs():
        q_, k_ = hins[0], hins[1]
        if not bwd:
            return [torch.empty(q_.shape, dtype=torch.bfloat16, device=dev)]
        outs = [torch.empty(q_.shape, dtype=torch.bfloat16, device=dev),
                torch.empty(k_.shape, dtype=torch.bfloat16, device=dev),
                torch.empty(k_.shape, dtype=torch.bfloat16, device=dev)]
        if gated:
            outs += [torch.empty(hins[4].shape, dtype=torch.float32, device=dev) for _ in range(2)]
        return outs

    def call(d, o, st=stream):
        w = wl["window"]
        if not bwd:
            if gated:
                sa.sa_swa_gated_forward(d[0], d[1], d[2], d[3], d[4], d[5], w, causal=wl["causal"],
                                        out=o[0], err=err, stream=st, kernel=kern)
            else:
                sa.sa_forward(d[0], d[1], d[2], d[3], w, causal=wl["causal"], out=o[0], err=err,
                              stream=st, kernel=kern)
        elif gated:
            sa.sa_swa_gated_backward(d[0], d[1], d[2], d[3], d[4], d[5], d[6], w,
                                     causal=wl["causal"], dq=o[0], dk=o[1], dv=o[2],
                                     dgate_sa=o[3], dgate_swa=o[4], err=err, stream=st)
        else:
            sa.sa_backward(d[0], d[1], d[2], d[3], d[4], w, causal=wl["causal"], dq=o[0], dk=o[1],
                           dv=o[2], err=err, stream=st)

    ins = [x.to(dev) for x in hins]
    outs = make_outs()

    def step():
        call(ins, outs)

    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    launches_per_step = sa.last_launch_count()
    kernel = sa.last_kernel()

    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_seconds:  # settle clocks before timing
        for _ in range(50 if not bwd else 5):
            step()
        torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    total_ms = max_over_ranks(float(sum(step_ms)), dev)
    status = sa.check_error(err)
    if status != sa.SA_OK:
        raise RuntimeError(f"device error word reports status {status}")

    # end to end: pinned host buffers in, results out, copies inside the timing.
    # Two streams take alternate steps, each with its own device buffers and
    # host result buffers, so one step's result copy overlaps the next step's
    # input copy (the host link is full duplex).  Every step still copies all
    # of its inputs in and its whole result out.
    hins = [t.pin_memory() for t in hins]
    h2d = sum(t.numel() * t.element_size() for t in hins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    slots = []
    for _ in range(2):
        souts = make_outs()
        slots.append(dict(stream=torch.cuda.Stream(dev),
                          dins=[torch.empty_like(x, device=dev) for x in hins], outs=souts,
                          houts=[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in souts]))

    def e2e_step(i):
        sl = slots[i & 1]
        with torch.cuda.stream(sl["stream"]):
            for dst, src in zip(sl["dins"], hins):
                dst.copy_(src, non_blocking=True)
            call(sl["dins"], sl["outs"], st=sl["stream"])
            for hdst, dsrc in zip(sl["houts"], sl["outs"]):
                hdst.copy_(dsrc, non_blocking=True)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_steps = max(4, min(args.steps, 50 if (wl is WORKLOAD and not bwd) else 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for sl in slots:
        sl["stream"].wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    for sl in slots:
        stream.wait_stream(sl["stream"])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    for sl in slots:
        for hres, dres in zip(sl["houts"], outs):
            if not torch.equal(hres.view(torch.uint8), dres.cpu().view(torch.uint8)):
                raise RuntimeError("end-to-end result differs from the device-resident run")

    if rank != 0:
        return 0
    tokens = wl["batch"] * wl["seq_len"]
    ms_per_step = total_ms / args.steps
    value = job_tokens_per_s(world, tokens, ms_per_step)
    bytes_alg, flops_alg = algorithmic_bwd(wl) if bwd else algorithmic(wl)
    peaks = load_peaks()
    secs = ms_per_step * 1e-3
    tensor_bound = flops_alg / (peaks["bf16_tflops"] * 1e12) > bytes_alg / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:  # the slower of the two roofline legs bounds the path
        roof = dict(bound="tensor", achieved=flops_alg / secs / 1e12, peak=peaks["bf16_tflops"],
                    unit="TFLOP/s", peak_source=f"{peaks['source']} bf16_tflops (burst)")
    else:
        roof = dict(bound="hbm", achieved=bytes_alg / secs / 1e9, peak=peaks["hbm_gbs"],
                    unit="GB/s", peak_source=f"{peaks['source']} hbm_gbs (copy, read+write)")
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic() if (wl is WORKLOAD and not bwd) else None
    roof.update(bytes_per_launch=bytes_alg, flops_per_launch=flops_alg,
                hbm_frac=bytes_alg / secs / 1e9 / peaks["hbm_gbs"],
                tensor_frac=flops_alg / secs / 1e12 / peaks["bf16_tflops"])
    kname = {sa.KERNEL_SIMT: "simt", sa.KERNEL_TCGEN05_GATHER: "tcgen05-gather",
             sa.KERNEL_TCGEN05_RING: "tcgen05-ring",
             sa.KERNEL_TCGEN05_CHUNK: "tcgen05-chunk"}.get(kernel, str(kernel))
    line = dict(
        metric=metric_of(wl, bwd), value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=ms_per_step, higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="bf16", data="synthetic",
        config=config_of(wl),
        run=dict(kernel="tcgen05-backward (dq, dkv)" if bwd else kname,
                 parallelism="replicas" if world > 1 else "single-gpu",
                 **({"pass": "backward"} if bwd else {})),
        roofline=roof,
        cpu_baseline=cpu,
        e2e=dict(value=job_tokens_per_s(world, tokens, e2e_ms), unit="tokens/s",
                 h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h),
        clocks=clocks,
        gpu_launches=args.steps * launches_per_step,
        wall_s_timed=wall,
    )
    print(json.dumps(line), flush=True)
    return 0


def run_receptive(args):
    """Receptive-field analytics of stacked SA layers at the length-sweep
    size: |R_l(t)| for l = 1..8 and a seeded sample of target tokens, each
    layer with its own sigma.  One step = one sa_receptive_field call."""
    import numpy as np
    import torch
    import stochastic_sliding_window_gb300 as sa
    rank, world, local = dist_env()
    n, w, layers, ntargets = args.seq_len or 262144, args.window or 128, 8, 4096
    causal = args.causal_rf
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    perms = torch.from_numpy(np.stack([sa.make_perm(0, l, 0, n) for l in range(layers)])).to(dev)
    targets = torch.from_numpy(np.random.default_rng(1).integers(0, n, ntargets).astype(np.int32)).to(dev)
    sizes = torch.empty((layers, ntargets), dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        sa.receptive_field(perms, w, targets, causal=causal, sizes=sizes, err=err)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        sa.receptive_field(perms, w, targets, causal=causal, sizes=sizes, err=err)
    e1.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    if sa.check_error(err) != sa.SA_OK:
        raise RuntimeError("device error word set")
    cov = (sizes.double().mean(dim=1) / n).cpu().tolist()
    # work: every layer application visits n positions x (2h + 1) window slots;
    # R_L costs L applications, for every group of 64 targets
    h = min(w // 2, n - 1)
    apps = (ntargets + 63) // 64 * layers * (layers + 1) // 2
    slots = apps * n * (2 * h + 1)
    if rank == 0:
        print(json.dumps(dict(
            metric=f"SA receptive-field analytics fields/s (n={n}, w={w}, {layers} layers, "
                   f"{'causal' if causal else 'non-causal'})",
            value=ntargets * layers / (ms * 1e-3), unit="target-layer fields/s", n_gpus=world,
            steps=args.steps, warmup=args.warmup, ms_per_step=ms, higher_is_better=True,
            scaling="weak", vs_baseline=None, dtype="int64", data="synthetic",
            config=dict(workload="receptive_field", seq_len=n, window=w, layers=layers,
                        targets=ntargets, causal=causal),
            window_slots_per_s=slots / (ms * 1e-3), mean_coverage_per_layer=cov,
            gpu_launches=args.steps * ((ntargets + 63) // 64) * (layers * 3 + layers * (layers + 1) // 2),
            clocks=clocks)), flush=True)
    return 0


def run_prologue(args, wl):
    """The prologue of one layer at a workload's shape: both gate logits of
    the layer input (d_model = Hq * d) in one GEMM, then RoPE of Q and K by
    original index.  One step = sa_gate_projection + two sa_rope calls."""
    import numpy as np
    import torch
    import stochastic_sliding_window_gb300 as sa
    rank, world, local = dist_env()
    b, n, hq, hkv, d = wl["batch"], wl["seq_len"], wl["num_q_heads"], wl["num_kv_heads"], wl["head_dim"]
    dm = hq * d
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn((b, n, dm), device=dev, generator=g).to(torch.bfloat16)
    w1 = (torch.randn((hq, dm), device=dev, generator=g) * dm ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn((hq, dm), device=dev, generator=g) * dm ** -0.5).to(torch.bfloat16)
    b1 = torch.zeros(hq, device=dev)
    b2 = torch.zeros(hq, device=dev)
    q = torch.randn((b, n, hq, d), device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn((b, n, hkv, d), device=dev, generator=g).to(torch.bfloat16)
    a1 = torch.empty((b, n, hq), device=dev)
    a2 = torch.empty((b, n, hq), device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        sa.gate_projection(x, w1, w2, b1, b2, gate_sa=a1, gate_swa=a2, err=err)
        sa.rope_(q)
        sa.rope_(k)

    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        starts[i].record()
        step()
        ends[i].record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps
    if sa.check_error(err) != sa.SA_OK:
        raise RuntimeError("device error word set")
    # algorithmic bytes: x and both weights read, both logit arrays written,
    # Q and K read and written once
    bytes_alg = 2 * b * n * dm + 2 * 2 * hq * dm + 2 * 4 * b * n * hq + 2 * 2 * b * n * d * (hq + hkv)
    peaks = load_peaks()
    ach = bytes_alg / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps(dict(
            metric=f"SA layer prologue tokens/s (gate projections d_model={dm} -> 2x{hq} logits, "
                   f"RoPE of Q and K; n={n})",
            value=b * n / (ms * 1e-3), unit="tokens/s", n_gpus=world, steps=args.steps,
            warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
            vs_baseline=None, dtype="bf16", data="synthetic", config=config_of(wl),
            roofline=dict(bound="hbm", achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s",
                          frac=ach / peaks["hbm_gbs"], traffic=None, bytes_per_launch=bytes_alg),
            gpu_launches=3 * args.steps, clocks=clocks)), flush=True)
    return 0


def run_shard(args, wl):
    """sigma-routed sequence sharding, measured on one GPU: every rank's local
    problem of the workload's sequence (its span's Q/K/V rows, already
    gathered, and its local permutation) through sa_forward, one rank after
    another.  One GPU cannot run the two all-to-all exchanges, so they are not
    in the number: `value` is the sequence's tokens over the slowest rank's
    local forward, the rate the ranks would reach if the exchanges overlapped
    perfectly.  The host plan (sa_shard_plan) is timed separately."""
    import numpy as np
    import torch
    import stochastic_sliding_window_gb300 as sa
    from stochastic_sliding_window_gb300 import shard
    rank0, world_procs, local = dist_env()
    b, n, hq, hkv, d = wl["batch"], wl["seq_len"], wl["num_q_heads"], wl["num_kv_heads"], wl["head_dim"]
    if b != 1:
        raise SystemExit("sequence sharding splits one sequence: the workload needs batch 1")
    w, W = wl["window"], args.shard_world
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    perm = sa.make_perms(wl["seed"], 0, 1, n)[0]
    t0 = time.perf_counter()
    ps = shard.plans(perm, w, W)
    plan_ms = (time.perf_counter() - t0) * 1e3 / W
    g = torch.Generator(device=dev).manual_seed(0)
    q = torch.randn((n, hq, d), device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn((n, hkv, d), device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn((n, hkv, d), device=dev, generator=g).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    per_rank, spans = [], []
    kernels = set()
    # every rank's local inputs (the rows gather_local would deliver), then a
    # warm-up of all of them before any is timed
    local_in = []
    for pl in ps:
        tok = torch.from_numpy(pl.tokens.astype(np.int64)).to(dev)
        ql, kl, vl = (x.index_select(0, tok)[None].contiguous() for x in (q, k, v))
        lp = torch.from_numpy(pl.local_perm[None, :].copy()).to(dev)
        local_in.append((ql, kl, vl, lp, torch.empty_like(ql)))
        spans.append(int(pl.tokens.shape[0]))
    for _ in range(args.warmup):
        for ql, kl, vl, lp, yl in local_in:
            sa.sa_forward(ql, kl, vl, lp, w, causal=wl["causal"], out=yl, err=err)
            kernels.add(sa.last_kernel())
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    for ql, kl, vl, lp, yl in local_in:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            starts[i].record()
            sa.sa_forward(ql, kl, vl, lp, w, causal=wl["causal"], out=yl, err=err)
            ends[i].record()
        torch.cuda.synchronize(dev)
        per_rank.append(sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps)
    clocks = sampler.stop()
    if sa.check_error(err) != sa.SA_OK:
        raise RuntimeError("device error word set")
    ms = max(per_rank)
    peaks = load_peaks()
    # a rank's local bytes: its span's Q/K/V rows and output rows once, and its local sigma
    bytes_rank = [sp * (2 * (hq + 2 * hkv) * d + 2 * hq * d + 4) for sp in spans]
    slow = per_rank.index(ms)
    ach = bytes_rank[slow] / (ms * 1e-3) / 1e9
    if rank0 == 0:
        print(json.dumps(dict(
            metric=f"sharded SA tokens/s over {W} ranks' local forwards, measured one rank at a "
                   f"time on one GPU (exchanges not included; n={n}, w={w})",
            value=n / (ms * 1e-3), unit="tokens/s", n_gpus=1, steps=args.steps,
            warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="strong",
            vs_baseline=None, dtype="bf16", data="synthetic",
            config=dict(config_of(wl), world=W),
            shard=dict(per_rank_ms=per_rank, span_rows=spans, halo_overhead=sum(spans) / n,
                       plan_ms_per_rank=plan_ms, kernels=sorted(kernels)),
            roofline=dict(bound="hbm", achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s",
                          frac=ach / peaks["hbm_gbs"], traffic=None,
                          bytes_per_launch=bytes_rank[slow]),
            gpu_launches=W * args.steps, clocks=clocks)), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--soak-seconds", type=float, default=1.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long_prefill_gqa",
                    help="shape to time (default: the long-prefill GQA headline)")
    ap.add_argument("--window", type=int, default=0, help="override the workload's window")
    ap.add_argument("--seq-len", type=int, default=0, help="override the workload's length")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "receptive", "prologue", "shard"],
                    default="fwd",
                    help="time the forward pass (default), the backward pass, or the "
                         "receptive-field analytics of stacked layers")
    ap.add_argument("--shard-world", type=int, default=8,
                    help="ranks of the sequence-sharding pass (--pass shard)")
    ap.add_argument("--causal-rf", action="store_true",
                    help="receptive fields of causal SA (default: non-causal)")
    ap.add_argument("--kernel", choices=["auto", "simt", "gather", "ring", "chunk"],
                    default="auto", help="force one of the library's kernels (default: its choice)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]
    if args.window or args.seq_len:
        wl = dict(wl, window=args.window or wl["window"], seq_len=args.seq_len or wl["seq_len"])
    if args.pass_ == "receptive":
        return run_receptive(args)
    if args.pass_ == "prologue":
        return run_prologue(args, wl)
    if args.pass_ == "shard":
        return run_shard(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
