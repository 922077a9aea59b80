"""Benchmark: S3D8 W2.7A8 linear layers of a Llama-3.2-11B text decoder layer at M = 1.

One step is one pass of the whole hot path over one token: per-token INT8
quantisation of the four distinct activations of a decoder layer (attention
input, attention output, MLP input, MLP hidden) and the seven S3D8 linears
(q, k, v, o, gate, up, down), through the library's C ABI.  The headline
step is one grouped launch (s3d8_linear_batch, quantisation fused); the JSON
also reports the four-launch structure of a real decoder layer and the
eleven-launch form (separate quantisation + single-matrix linears).  Weights are
synthetic (seeded recipe in s3d8_inputs) and resident in HBM; the step cycles
through 8 independent copies of the layer (582 MB of packed weights, well
above the 129 MB L2) so that every step streams its weights from HBM.

Printed JSON (one line, rank 0):
  value      weight GB/s = (packed bytes + bf16 channel scales + tables) per
             step / device time per step, over all ranks (weak scaling);
  roofline   the grouped GEMV kernel's algorithmic bytes (weights, tables,
             scales, bf16 activations, outputs) per launch / its average launch
             time, measured with CUDA events recorded inside captured graphs,
             against the measured HBM copy bandwidth;
  e2e        the same metric with per-step host->device copies of the
             activations from pinned memory and device->host copies of the
             seven outputs, through the Python binding;
  prefill    INT8 tensor-op rate of the same library at M = 512 and 2048 on
             the gate/up and down shapes, with the fraction of the measured
             bf16 tensor peak (the engine the path runs on);
  decode_sweep  the batched-decode sizes (M = 8..64) with their roofline
             fractions;
  cpu_baseline  the plain CPU oracle, timed on this host on a bounded sample.

`--impl reference` times the CPU oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import s3d8_inputs as si  # noqa: E402

METRIC = "S3D8 linear weight GB/s (M=1) & INT8 TOPS (prefill), % of roofline"
UNIT = "GB/s"
COPIES = 8
# Longest run of headline steps captured in one CUDA graph: a timed region of at
# most this many steps is exactly one graph replay; longer regions replay it and
# then a graph holding the remainder.
MAX_GRAPH_STEPS = 512
WORKLOAD = ("Llama-3.2-11B text decoder layer, decode M=1: S3D8 linears q 4096->4096, "
            "k/v 4096->1024, o 4096->4096, gate/up 4096->14336, down 14336->4096")


def weight_bytes(K, N):
    """Packed bytes + bf16 channel scales + the 32x3 int8 table."""
    return si.groups(N) * K + 2 * N + 96


def linear_bytes(M, K, N):
    """Algorithmic bytes of one linear launch: weights, xq, xscale, output."""
    return weight_bytes(K, N) + M * K + 4 * M + 2 * M * N


LAYER_WEIGHT_BYTES = sum(weight_bytes(K, N) for _, K, N in si.LLAMA_11B_LAYER)
ACT_K = {"attn": 4096, "o": 4096, "mlp": 4096, "down": 14336}
# The workload both arms print, word for word: step i streams layer copy i mod 8.
CONFIG = {"workload": WORKLOAD, "M": 1, "weight_bytes_per_step": LAYER_WEIGHT_BYTES,
          "weight_copies": COPIES,
          "l2": f"inputs larger than L2: step i streams layer copy i mod {COPIES} "
                f"({COPIES * LAYER_WEIGHT_BYTES / 1e6:.0f} MB of weights in all, over 4x the "
                "129 MB L2), so no flush"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def gemv_source_sha():
    h = hashlib.sha256()
    for name in ("gemv_tma.cu", "common.cuh", "tma.cuh"):
        with open(os.path.join(ROOT, "s3d8_a8_linear_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch():
    """DRAM bytes per GEMV launch from the committed ncu summary, or None when
    the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("source_sha") != gemv_source_sha():
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def to_dev_bf16(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


class LayerCopy:
    def __init__(self, layer, dev, seed=0):
        import torch
        self.mats = []
        for mat in si.layer_matrices(layer=layer, seed=seed):
            self.mats.append(dict(
                name=mat.name, K=mat.K, N=mat.N,
                packed=torch.from_numpy(mat.packed).to(dev),
                C=torch.from_numpy(mat.C).to(dev),
                cs=to_dev_bf16(mat.chan_scale, dev)))


class Step:
    """Device buffers of one decoder-layer step at M tokens, and the three ways
    the library can run it:
      group1    one grouped launch for all seven projections, activation
                quantisation fused (the inputs of the synthetic step are
                independent, so they can stream together);
      group4    the launch structure a real decoder layer allows: q/k/v, o,
                gate/up and down as four grouped launches with fused quantisation;
      separate  four quantisation launches and seven single-matrix launches."""

    GROUP4 = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))

    def __init__(self, M, dev, seed=0):
        import torch
        self.M = M
        self.x = {k: to_dev_bf16(si.acts(M, K, seed=seed, index=i), dev)
                  for i, (k, K) in enumerate(ACT_K.items())}
        self.xq = {k: torch.empty((M, K), dtype=torch.int8, device=dev) for k, K in ACT_K.items()}
        self.xs = {k: torch.empty((M,), dtype=torch.float32, device=dev) for k in ACT_K}
        self.out = {n: torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                    for n, _, N in si.LLAMA_11B_LAYER}

    def job(self, m):
        a = si.LLAMA_11B_INPUT_OF[m["name"]]
        return dict(packed=m["packed"], centroids=m["C"], chan_scale=m["cs"], N=m["N"],
                    x=self.x[a], out=self.out[m["name"]])

    def run(self, s3d8, copy, mode="group1", events=None):
        mats = {m["name"]: m for m in copy.mats}
        if mode == "group1":
            groups_ = (tuple(mats),)
        elif mode == "group4":
            groups_ = self.GROUP4
        else:
            groups_ = None
        if groups_ is not None:
            for gi, names in enumerate(groups_):
                if events is not None:
                    events[gi][0].record()
                s3d8.linear_batch([self.job(mats[n]) for n in names], self.M)
                if events is not None:
                    events[gi][1].record()
            return
        for k in ACT_K:
            s3d8.quantize_act(self.x[k], self.xq[k], self.xs[k])
        for j, m in enumerate(copy.mats):
            a = si.LLAMA_11B_INPUT_OF[m["name"]]
            if events is not None:
                events[j][0].record()
            s3d8.linear(m["packed"], m["C"], m["cs"], self.xq[a], self.xs[a], m["N"],
                        out=self.out[m["name"]])
            if events is not None:
                events[j][1].record()


def n_launches(mode):
    return {"group1": 1, "group4": 4, "separate": len(ACT_K) + len(si.LLAMA_11B_LAYER)}[mode]


def group_bytes(names, M=1):
    """Algorithmic bytes of one grouped launch: weights, scales and tables, each
    distinct bf16 activation once, the bf16 outputs."""
    shapes = {n: (K, N) for n, K, N in si.LLAMA_11B_LAYER}
    acts = {si.LLAMA_11B_INPUT_OF[n] for n in names}
    total = sum(weight_bytes(*shapes[n]) + 2 * M * shapes[n][1] for n in names)
    return total + sum(2 * M * ACT_K[a] + 4 * M for a in acts)


def rank_env():
    """(world, rank, local rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(torch, value, device, world):
    """The largest per-rank step time: every rank runs its own replica of the
    step (no exchange on the data path), so the job is as slow as its slowest
    rank.  Collective only when more than one rank runs."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(world, ms_step, bytes_per_step=LAYER_WEIGHT_BYTES):
    """Whole-job weight GB/s: every rank streams its own copy of the layer per
    step (weak scaling), over the slowest rank's step time."""
    return world * bytes_per_step / (ms_step * 1e-3) / 1e9


def capture(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def make_timing_events(torch, n):
    try:
        return [(torch.cuda.Event(enable_timing=True, external=True),
                 torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n)]
    except TypeError:
        return None


def cpu_model():
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def gpu_arm(args):
    import torch

    import s3d8_a8_linear_gb300 as s3d8

    world, rank, local = rank_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    s3d8.load(build_if_missing=True)

    copies = [LayerCopy(r, dev) for r in range(COPIES)]
    step = Step(1, dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):       # eager warm-up of every path
        for mode in ("group1", "group4", "separate"):
            for r in range(COPIES):
                step.run(s3d8, copies[r], mode)
    stream.synchronize()

    # The timed region is exactly args.steps headline steps: one graph of
    # consecutive grouped launches (step i on layer copy i mod 8) if that is at
    # most MAX_GRAPH_STEPS, else replays of a MAX_GRAPH_STEPS graph and one graph
    # with the remainder.  Inside a graph consecutive launches overlap through
    # programmatic dependent launch; at a graph boundary they cannot.
    def run_steps(mode, n):
        for i in range(n):
            step.run(s3d8, copies[i % COPIES], mode)

    per_graph = min(args.steps, MAX_GRAPH_STEPS)
    full, rest = divmod(args.steps, per_graph)
    main_g = capture(torch, stream, lambda: run_steps("group1", per_graph))
    rest_g = capture(torch, stream, lambda: run_steps("group1", rest)) if rest else None
    torch.cuda.synchronize()

    def timed_replays(graphs):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for g in graphs:
                g.replay()
            t1.record(stream)
        t1.synchronize()
        return t0.elapsed_time(t1)

    # warm-up: at least args.warmup steps of the same graph
    with torch.cuda.stream(stream):
        for _ in range((args.warmup + per_graph - 1) // per_graph):
            main_g.replay()
    stream.synchronize()

    # ---- timed region: exactly args.steps steps of the headline structure ----
    # The step's inputs (8 layer copies, 582 MB) are larger than L2, so no flush
    # is needed.  One more warm-up replay is queued just before the start event,
    # so that the GPU is still busy with it while the host submits the timed
    # graph: the region then starts with the first timed launch, not with the
    # host's submission latency.  (An L2 flush there instead left ~129 MB of
    # dirty lines whose write-back slowed the first timed steps.)
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        main_g.replay()
    ms_step = timed_replays([main_g] * full + ([rest_g] if rest_g else [])) / args.steps
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()

    # ---- spread: replays of the same graph timed one by one, median and a 95 %
    # bootstrap interval of the per-step time (outside the timed region) ------
    spread = None
    if not args.layer_only:
        samples = [timed_replays([main_g]) / per_graph for _ in range(60)]
        spread = bootstrap_median(samples)
        spread["block_steps"] = per_graph

    # ---- other launch structures (same weights, same rotation) --------------
    variants = {}
    for mode in (() if args.layer_only else ("group4", "separate")):
        n = max(COPIES, min(per_graph, MAX_GRAPH_STEPS // 4) // COPIES * COPIES)
        g = capture(torch, stream, lambda mode=mode, n=n: run_steps(mode, n))
        timed_replays([g])
        ms = timed_replays([g]) / n
        variants[mode] = {"ms_per_step": round(ms, 6), "launches_per_step": n_launches(mode),
                          "steps_per_graph": n,
                          "value": round(LAYER_WEIGHT_BYTES / (ms * 1e-3) / 1e9, 1)}
        del g

    # ---- per-launch duration of the grouped kernel bracketed alone by events --
    launch_ms = []
    evgraphs = []
    for r in range(COPIES):
        ev = make_timing_events(torch, 1)
        if ev is None:
            break
        evgraphs.append((capture(torch, stream,
                                 lambda r=r, ev=ev: step.run(s3d8, copies[r], "group1", ev)), ev))
    if evgraphs:
        with torch.cuda.stream(stream):
            for rep in range(4):
                for g, _ in evgraphs:
                    g.replay()
                stream.synchronize()
                launch_ms += [ev[0][0].elapsed_time(ev[0][1]) for _, ev in evgraphs]
    status = s3d8.device_status()

    ms_step = max_over_ranks(torch, ms_step, dev, world)
    value = job_value(world, ms_step)
    hbm_peak, bf16_peak, peak_kind = load_peaks()
    # The timed region runs nothing but the grouped kernel, one launch per step, so
    # its average launch duration there is the region's event time / launches.
    # Launches bracketed one by one by events (no overlap with neighbours) are
    # reported beside it.
    step_bytes = group_bytes([n for n, _, _ in si.LLAMA_11B_LAYER])
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
                "traffic": traffic_per_launch(),
                "kernel": "gemv_group_kernel<1>: one launch, 7 projections, fused quantisation",
                "bytes_per_launch": step_bytes, "avg_launch_us": round(ms_step * 1e3, 3),
                "launches_timed": args.steps, "peak_kind": peak_kind,
                "method": "CUDA events around the timed region on the launching stream / launches"}
    if launch_ms:
        iso_ms = sum(launch_ms) / len(launch_ms)
        roofline["isolated_launch_us"] = round(iso_ms * 1e3, 3)
        roofline["isolated_achieved"] = round(step_bytes / (iso_ms * 1e-3) / 1e9, 1)

    e2e = prefill = unpack = quant = sweep = stack = encode = fit = None
    if not args.layer_only:
        e2e = e2e_measure(torch, s3d8, copies, dev, args.steps, per_graph)
        if not args.skip_prefill:
            psampler = ClockSampler(local)
            psampler.start()
            prefill = prefill_measure(torch, s3d8, dev, bf16_peak)
            prefill["clocks"] = psampler.stop()
        unpack = unpack_measure(torch, s3d8, dev)
        quant = quant_measure(torch, s3d8, dev)
        sweep = decode_sweep_measure(torch, s3d8, dev, hbm_peak, bf16_peak)
        stack = stack_measure(torch, s3d8, dev)
        encode = encode_measure(torch, s3d8, dev)
        fit = fit_measure(torch, s3d8, dev)

    if rank != 0:
        return
    cpu = None if args.skip_cpu else cpu_baseline(args.cpu_seconds)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded S3D8 fields, bf16 N(0,1) activations; no trained weights)",
        "config": dict(CONFIG),
        "parallelism": f"replicas x{world}",
        "launch": (f"one grouped launch per step (7 projections, activation quantisation fused); "
                   f"the {args.steps} timed steps are "
                   + (f"one CUDA graph of {per_graph} consecutive launches" if full == 1 and not rest
                      else f"{full} replays of a {per_graph}-step CUDA graph"
                      + (f" and one {rest}-step graph" if rest else ""))
                   + ", consecutive launches overlapping by programmatic dependent launch"),
        "gpu_launches": args.steps * n_launches("group1"),
        "device_status": status,
        "roofline": roofline, "variants": variants, "e2e": e2e, "prefill": prefill,
        "decode_sweep": sweep, "text_stack": stack, "spread": spread,
        "unpack": unpack, "quantize": quant, "encode": encode, "fit": fit, "clocks": clocks, "cpu_baseline": cpu,
    }
    print(json.dumps(line))


def e2e_measure(torch, s3d8, copies, dev, steps, per_graph, group=4, sets=3):
    """Same metric through the Python binding, with each step's four activations
    copied in from pinned host memory and its seven outputs copied back to
    pinned host memory (one copy each way per step), over exactly `steps` steps
    in the same graph structure as the headline (graphs of `per_graph` steps,
    step i on layer copy i mod 8).  Each graph runs on three streams (copies in,
    layer launches, copies out), in groups of `group` steps with `sets` rotating
    buffer sets per group: the layer stream waits for a group's copy-ins (issued
    while the previous group computes) once per group, and the copy-outs follow
    each group, so consecutive launches inside a group still overlap through
    programmatic dependent launch (a stream wait or event record between two
    launches stops that overlap).  The synthetic steps are independent, so a
    group's inputs may be copied before the previous group ends.  Every step's
    copies are inside the timed region."""
    nbuf = group * sets
    xk = list(ACT_K.items())
    kx = sum(K for _, K in xk)
    no = sum(N for _, _, N in si.LLAMA_11B_LAYER)
    steps_b, x_all, o_all, host_x, host_out = [], [], [], [], []
    for b in range(nbuf):
        st = Step(1, dev)
        xa = torch.empty((kx,), dtype=torch.bfloat16, device=dev)
        hx = torch.empty((kx,), dtype=torch.bfloat16).pin_memory()
        off = 0
        for i, (k, K) in enumerate(xk):
            st.x[k] = xa[off:off + K].view(1, K)
            hx[off:off + K] = torch.from_numpy(
                si.acts(1, K, seed=5 + b, index=i).view(np.int16)).view(torch.bfloat16)[0]
            off += K
        oa = torch.empty((no,), dtype=torch.bfloat16, device=dev)
        ho = torch.empty((no,), dtype=torch.bfloat16).pin_memory()
        off = 0
        for n, _, N in si.LLAMA_11B_LAYER:
            st.out[n] = oa[off:off + N].view(1, N)
            off += N
        steps_b.append(st)
        x_all.append(xa)
        o_all.append(oa)
        host_x.append(hx)
        host_out.append(ho)
    ks, cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    with torch.cuda.stream(ks):
        for b in range(nbuf):
            for r in range(COPIES):
                steps_b[b].run(s3d8, copies[r], "group1")
    ks.synchronize()

    def capture_steps(n):
        """A graph of n steps with their copies (groups of `group` steps)."""
        groups_ = [list(range(i, min(n, i + group))) for i in range(0, n, group)]
        ev_in = [torch.cuda.Event() for _ in groups_]
        ev_k = [torch.cuda.Event() for _ in groups_]
        ev_out = [torch.cuda.Event() for _ in groups_]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=ks):
            cin.wait_stream(ks)
            cout.wait_stream(ks)
            for gi, idx in enumerate(groups_):
                bufs = [(gi % sets) * group + j for j in range(len(idx))]
                with torch.cuda.stream(cin):
                    if gi >= sets:
                        cin.wait_event(ev_k[gi - sets])     # the set's last group has read its inputs
                    for b in bufs:
                        x_all[b].copy_(host_x[b], non_blocking=True)
                    ev_in[gi].record(cin)
                ks.wait_event(ev_in[gi])
                if gi >= sets:
                    ks.wait_event(ev_out[gi - sets])        # the set's last outputs are copied out
                for i, b in zip(idx, bufs):
                    steps_b[b].run(s3d8, copies[i % COPIES], "group1")
                ev_k[gi].record(ks)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_k[gi])
                    for b in bufs:
                        host_out[b].copy_(o_all[b], non_blocking=True)
                    ev_out[gi].record(cout)
            ks.wait_stream(cin)
            ks.wait_stream(cout)
        return g

    full, rest = divmod(steps, per_graph)
    main_g = capture_steps(per_graph)
    rest_g = capture_steps(rest) if rest else None
    h2d = host_x[0].numel() * 2
    d2h = host_out[0].numel() * 2
    with torch.cuda.stream(ks):
        for _ in range(2):
            main_g.replay()
    ks.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(ks):
        main_g.replay()         # keeps the GPU busy while the timed graphs are submitted
        t0.record(ks)
        for _ in range(full):
            main_g.replay()
        if rest_g is not None:
            rest_g.replay()
        t1.record(ks)
    t1.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return {"value": round(LAYER_WEIGHT_BYTES / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 5),
            "steps": steps,
            "path": "Python binding (grouped launch); per step one pinned host->device copy of "
                    "the four activations and one device->host copy of the seven outputs, on their "
                    f"own streams, synchronised with the layer stream once per group of {group} steps "
                    f"(launches inside a group overlap); the same {per_graph}-step graphs as the "
                    "headline"}


def prefill_measure(torch, s3d8, dev, bf16_peak, Ms=None, reps=20, copies=2):
    """The tensor-core path at the prefill sizes (M = 512 and 2048) on the gate/up
    and down shapes, through s3d8_linear (automatic algorithm), alternating
    between `copies` weight copies; 3 warm-up calls, then `reps` calls timed
    with CUDA events.  Roofline: the tensor engine the path runs on (bf16
    tcgen05.mma kind::f16, exact int32 sums from fp32 chunks), against the
    measured bf16 dense peak (burst: the calls are timed without a long
    sustained load); the fraction of the INT8 library GEMM rate measured on the
    same shapes (the pages' two-step method's GEMM) is reported beside it."""
    Ms = si.PREFILL_M if Ms is None else Ms
    two_step = two_step_measure(torch, s3d8, dev, max(Ms), 3)
    # the chip's INT8 tensor rate as the library GEMM reaches it on these shapes
    int8_peak = max(2 * max(Ms) * K * N / (two_step[name]["int8_gemm_us"] * 1e-6) / 1e12
                    for name, K, N in si.SWEEP_SHAPES)
    res = {"unit": "TOPS (int8 multiply-adds x2)", "engine": "tcgen05.mma kind::f16 (fp16 operands below the expansion size, bf16 above), exact int32",
           "peak_tflops": bf16_peak, "int8_library_peak_tops": round(int8_peak, 1),
           "int8_library": "torch._int_mm (PyTorch's CUTLASS int8 x int8 -> int32 mma.sync GEMM) on the same shapes at "
                           f"M = {max(Ms)}, the fastest of the two"}
    for M in Ms:
        tot_ops, tot_ms = 0, 0.0
        for name, K, N in si.SWEEP_SHAPES:
            mats = [si.matrix(name, K, N, seed=3, index=i) for i in range(copies)]
            w = [dict(packed=torch.from_numpy(m.packed).to(dev), C=torch.from_numpy(m.C).to(dev),
                      cs=to_dev_bf16(m.chan_scale, dev)) for m in mats]
            x = to_dev_bf16(si.acts(M, K, seed=3), dev)
            xq, xs = s3d8.quantize_act(x)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty((max(1, s3d8.workspace_size(M, N, K)),), dtype=torch.uint8, device=dev)

            def call(i):
                m = w[i % copies]
                s3d8.linear(m["packed"], m["C"], m["cs"], xq, xs, N, out=out, workspace=ws)

            for i in range(3):
                call(i)
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for i in range(reps):
                call(i)
            t1.record()
            t1.synchronize()
            ms = t0.elapsed_time(t1) / reps
            ops = 2 * M * N * K
            tops = ops / (ms * 1e-3) / 1e12
            res[f"{name}_M{M}"] = {"M": M, "K": K, "N": N, "us": round(ms * 1e3, 1),
                                   "tops": round(tops, 2),
                                   "roofline": {"bound": "tensor", "achieved": round(tops, 1),
                                                "peak": bf16_peak, "unit": "TFLOP/s",
                                                "frac": round(tops / bf16_peak, 4),
                                                "frac_of_int8_library": round(tops / int8_peak, 2)}}
            tot_ops += ops
            tot_ms += ms
            del w, mats
        tops = tot_ops / (tot_ms * 1e-3) / 1e12
        res[f"M{M}"] = {"tops": round(tops, 2), "frac": round(tops / bf16_peak, 4)}
    res["tops"] = res[f"M{max(Ms)}"]["tops"]
    res["two_step"] = two_step
    return res


def two_step_measure(torch, s3d8, dev, M, reps):
    """The pages' prefill method, for comparison: a standalone unpack to dense
    int8 weights (s3d8_decode), then a library GEMM on the dense weights, either
    INT8 x INT8 -> int32 (torch._int_mm, a CUTLASS mma.sync GEMM) or the same codes as bf16
    (torch.matmul, cuBLAS).  The epilogue is left out, so these times are lower
    bounds for the two-step layer."""
    out = {}
    for name, K, N in si.SWEEP_SHAPES:
        mat = si.matrix(name, K, N, seed=3)
        packed = torch.from_numpy(mat.packed).to(dev)
        C = torch.from_numpy(mat.C).to(dev)
        xq = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev)
        w = torch.empty((N, K), dtype=torch.int8, device=dev)
        xb = xq.to(torch.bfloat16)
        wb = torch.empty((N, K), dtype=torch.bfloat16, device=dev)

        def timed(fn):
            fn()
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(reps):
                fn()
            t1.record()
            t1.synchronize()
            return t0.elapsed_time(t1) / reps

        dec_ms = timed(lambda: s3d8.decode(packed, C, N, w))
        i8_ms = timed(lambda: torch._int_mm(xq, w.t()))
        cvt_ms = timed(lambda: wb.copy_(w))
        bf_ms = timed(lambda: torch.matmul(xb, wb.t()))
        ops = 2 * M * N * K
        out[name] = {"decode_us": round(dec_ms * 1e3, 1),
                     "int8_gemm_us": round(i8_ms * 1e3, 1),
                     "int8_two_step_tops": round(ops / ((dec_ms + i8_ms) * 1e-3) / 1e12, 1),
                     "to_bf16_us": round(cvt_ms * 1e3, 1),
                     "bf16_gemm_us": round(bf_ms * 1e3, 1),
                     "bf16_two_step_tops": round(
                         ops / ((dec_ms + cvt_ms + bf_ms) * 1e-3) / 1e12, 1)}
    return out


def device_matrix(torch, dev, gen, K, N):
    """Random S3D8 fields of the recipe's distribution, drawn on the device with a
    seeded generator (uniform bytes, table entries 1..127, |N(0, 0.02)|/127
    channel scales): for timing copies whose values nothing checks."""
    G = si.groups(N)
    return dict(K=K, N=N,
                packed=torch.randint(0, 256, (G, K), dtype=torch.uint8, device=dev, generator=gen),
                C=torch.randint(1, 128, (32, 3), dtype=torch.int8, device=dev, generator=gen),
                cs=(torch.randn((N,), device=dev, generator=gen).abs() * (0.02 / 127)).to(
                    torch.bfloat16))


def decode_sweep_measure(torch, s3d8, dev, hbm_peak, bf16_peak, copies=28, reps=56, replays=5):
    """Batched decode (M = 8..64) on the gate/up and down shapes through
    s3d8_linear (automatic algorithm choice), rotating `copies` weight copies
    (28 x 19.6 MB = 549 MB, over four times the 129 MB L2, so that every launch
    streams its weights from HBM).
    The `reps` launches are captured in one CUDA graph and replayed, so that the
    time is the device's and not the Python binding's per-call overhead.
    Roofline per entry: the larger of the HBM time of the algorithmic bytes
    (weights, scales, table, codes, token scales, bf16 outputs) at the measured
    copy bandwidth and the tensor time of 2 M N K operations at the measured
    bf16 dense peak (the engine of the tensor-core paths); frac = that bound /
    the measured time."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    res = {}
    stream = torch.cuda.Stream(dev)
    for name, K, N in si.SWEEP_SHAPES:
        mats = [device_matrix(torch, dev, gen, K, N) for _ in range(copies)]
        for M in si.DECODE_SWEEP_M:
            x = to_dev_bf16(si.acts(M, K, seed=7, outliers=True), dev)
            xq, xs = s3d8.quantize_act(x)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty((max(1, s3d8.workspace_size(M, N, K)),), dtype=torch.uint8, device=dev)
            for m in mats:   # eager warm-up (kernel attributes, first-touch)
                s3d8.linear(m["packed"], m["C"], m["cs"], xq, xs, N, out=out, workspace=ws)
            torch.cuda.synchronize()

            def body():
                for i in range(reps):
                    m = mats[i % copies]
                    s3d8.linear(m["packed"], m["C"], m["cs"], xq, xs, N, out=out, workspace=ws)
            g = capture(torch, stream, body)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g.replay()
                t0.record(stream)
                for _ in range(replays):
                    g.replay()
                t1.record(stream)
            t1.synchronize()
            ms = t0.elapsed_time(t1) / (reps * replays)
            hbm_us = linear_bytes(M, K, N) / (hbm_peak * 1e9) * 1e6
            tensor_us = 2 * M * N * K / (bf16_peak * 1e12) * 1e6
            bound_us = max(hbm_us, tensor_us)
            res[f"{name}_M{M}"] = {"us": round(ms * 1e3, 2),
                                   "weight_gbs": round(weight_bytes(K, N) / (ms * 1e-3) / 1e9, 1),
                                   "tops": round(2 * M * N * K / (ms * 1e-3) / 1e12, 2),
                                   "bound": "hbm" if hbm_us >= tensor_us else "tensor",
                                   "bound_us": round(bound_us, 3),
                                   "frac": round(bound_us / (ms * 1e3), 4)}
        del mats
    return res


def stack_measure(torch, s3d8, dev, reps=5):
    """The whole 40-layer text stack plus the LM head at M = 1 (3.08 GB of
    packed weights): one grouped launch per layer with fused quantisation and
    one for the head, captured as one graph of 41 launches."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    layers = [[dict(name=n, **device_matrix(torch, dev, gen, K, N)) for n, K, N in si.LLAMA_11B_LAYER]
              for _ in range(si.LLAMA_11B_LAYERS)]
    _, hK, hN = si.LLAMA_11B_HEAD
    head = device_matrix(torch, dev, gen, hK, hN)
    x = {k: to_dev_bf16(si.acts(1, K, seed=11, index=i), dev) for i, (k, K) in enumerate(ACT_K.items())}
    outs = {n: torch.empty((1, N), dtype=torch.bfloat16, device=dev) for n, _, N in si.LLAMA_11B_LAYER}
    hout = torch.empty((1, hN), dtype=torch.bfloat16, device=dev)
    total = sum(weight_bytes(m["K"], m["N"]) for L in layers for m in L) + weight_bytes(hK, hN)

    def run():
        for L in layers:
            s3d8.linear_batch([dict(packed=m["packed"], centroids=m["C"], chan_scale=m["cs"],
                                    N=m["N"], x=x[si.LLAMA_11B_INPUT_OF[m["name"]]],
                                    out=outs[m["name"]]) for m in L], 1)
        s3d8.linear_batch([dict(packed=head["packed"], centroids=head["C"], chan_scale=head["cs"],
                                N=hN, x=x["attn"], out=hout)], 1)

    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    g = capture(torch, stream, run)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
    t1.synchronize()
    ms = t0.elapsed_time(t1) / reps
    del layers, head
    return {"workload": "40 decoder layers x 7 S3D8 linears + LM head 4096->128256, M=1",
            "weight_bytes": total, "launches": si.LLAMA_11B_LAYERS + 1, "ms": round(ms, 4),
            "value": round(total / (ms * 1e-3) / 1e9, 1), "unit": UNIT}


def unpack_measure(torch, s3d8, dev, reps=20):
    name, K, N = "gate", 4096, 14336
    mats = [si.matrix(name, K, N, seed=4, index=i) for i in range(COPIES)]
    packed = [torch.from_numpy(m.packed).to(dev) for m in mats]
    Cs = [torch.from_numpy(m.C).to(dev) for m in mats]
    w = torch.empty((N, K), dtype=torch.int8, device=dev)
    s3d8.decode(packed[0], Cs[0], N, w)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(reps):
        s3d8.decode(packed[i % COPIES], Cs[i % COPIES], N, w)
    t1.record()
    t1.synchronize()
    ms = t0.elapsed_time(t1) / reps
    rd = si.groups(N) * K
    return {"shape": "4096x14336 (gate)", "us": round(ms * 1e3, 2),
            "read_gbs": round(rd / (ms * 1e-3) / 1e9, 1),
            "total_gbs": round((rd + N * K) / (ms * 1e-3) / 1e9, 1)}


def quant_measure(torch, s3d8, dev, M=2048, K=14336, copies=4, reps=20):
    """Standalone per-token activation quantisation at the prefill size of the
    down projection's input (bf16 [2048, 14336], 58.7 MB in), rotating over
    four input copies (235 MB, above L2).  Algorithmic bytes: 2MK read, MK + 4M
    written."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    xs = [torch.randn((M, K), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
          for _ in range(copies)]
    xq = torch.empty((M, K), dtype=torch.int8, device=dev)
    xscale = torch.empty((M,), dtype=torch.float32, device=dev)
    for i in range(copies):
        s3d8.quantize_act(xs[i], xq, xscale)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(reps):
        s3d8.quantize_act(xs[i % copies], xq, xscale)
    t1.record()
    t1.synchronize()
    ms = t0.elapsed_time(t1) / reps
    nbytes = 2 * M * K + M * K + 4 * M
    del xs
    return {"shape": f"bf16 [{M}, {K}]", "us": round(ms * 1e3, 2),
            "algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def encode_measure(torch, s3d8, dev, reps=3):
    """Direct-cast encoder over the seven matrices of one 11B decoder layer
    (218 M bf16 weights, 436 MB, larger than L2), weights N(0, 0.02) drawn on
    the device.  Algorithmic traffic: the bf16 weights once, the packed bytes
    and the scales written once; the fp32 work is 32 three-component squared
    distances (8 operations each) per packed byte."""
    gen = torch.Generator(device=dev).manual_seed(9)
    mats = []
    for name, K, N in si.LLAMA_11B_LAYER:
        w = (torch.randn((N, K), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        C = torch.randint(1, 128, (32, 3), dtype=torch.int8, device=dev, generator=gen)
        p = torch.empty((si.groups(N), K), dtype=torch.uint8, device=dev)
        cs = torch.empty((N,), dtype=torch.bfloat16, device=dev)
        mats.append((w, C, p, cs))
    ws = torch.empty((s3d8.ENCODE_WORKSPACE_BYTES,), dtype=torch.uint8, device=dev)

    def run():
        for w, C, p, cs in mats:
            s3d8.encode(w, C, p, cs, ws)

    run()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        run()
    t1.record()
    t1.synchronize()
    ms = t0.elapsed_time(t1) / reps
    params = sum(N * K for _, K, N in si.LLAMA_11B_LAYER)
    codes = sum(si.groups(N) * K for _, K, N in si.LLAMA_11B_LAYER)
    nbytes = 2 * params + codes + 2 * sum(N for _, _, N in si.LLAMA_11B_LAYER)
    # the QAT fake-quant forward on the same matrices (bf16 in, bf16 out)
    hats = [torch.empty_like(w) for w, _, _, _ in mats]
    for (w, C, _, cs), h in zip(mats, hats):
        s3d8.fake_quant(w, C, h, cs, ws)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(reps):
        for (w, C, _, cs), h in zip(mats, hats):
            s3d8.fake_quant(w, C, h, cs, ws)
    t1.record()
    t1.synchronize()
    fq_ms = t0.elapsed_time(t1) / reps
    return {"workload": "one 11B decoder layer's 7 bf16 matrices -> S3D8", "params": params,
            "ms": round(ms, 3), "gparams_s": round(params / (ms * 1e-3) / 1e9, 2),
            "algorithmic_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "fp32_tflops": round(codes * 32 * 8 / (ms * 1e-3) / 1e12, 2),
            "launches": 2 * len(mats) * reps,
            "fake_quant_ms": round(fq_ms, 3),
            "fake_quant_algorithmic_gbs": round((4 * params + 2 * sum(
                N for _, _, N in si.LLAMA_11B_LAYER)) / (fq_ms * 1e-3) / 1e9, 1)}


def fit_measure(torch, s3d8, dev, iters=25, reps=2):
    """Centroid fit (k-means++ then `iters` Lloyd iterations) on the gate
    matrix (4096 -> 14336, 19.6 M points), weights N(0, 0.02) drawn on the
    device.  The Lloyd assignment is the dominant cost: 32 squared distances
    (8 fp32 operations each) per point and iteration."""
    gen = torch.Generator(device=dev).manual_seed(11)
    N, K = 14336, 4096
    w = (torch.randn((N, K), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    draws = torch.randint(-2 ** 31, 2 ** 31 - 1, (32,), dtype=torch.int32, device=dev,
                          generator=gen)
    ws = torch.empty((s3d8.fit_workspace_size(N, K),), dtype=torch.uint8, device=dev)
    s3d8.fit_centroids(w, draws, iters, ws)
    torch.cuda.synchronize()
    res = {}
    for it in (0, iters):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            s3d8.fit_centroids(w, draws, it, ws)
        t1.record()
        t1.synchronize()
        res[it] = t0.elapsed_time(t1) / reps
    points = si.groups(N) * K
    per_iter = (res[iters] - res[0]) / iters
    return {"workload": "gate matrix 4096 -> 14336, 19.6 M points, 32 centroids",
            "iters": iters, "ms": round(res[iters], 3), "kmeanspp_ms": round(res[0], 3),
            "lloyd_ms_per_iter": round(per_iter, 4),
            "lloyd_gpoints_s": round(points / (per_iter * 1e-3) / 1e9, 1),
            "lloyd_fp32_tflops": round(points * 32 * 8 / (per_iter * 1e-3) / 1e12, 2)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def oracle_layer_step(oracle, mats, xs_bits):
    q = {k: oracle.quantize_act(xs_bits[k]) for k in ACT_K}
    for m in mats:
        xq, xsc = q[si.LLAMA_11B_INPUT_OF[m.name]]
        oracle.linear(m.packed, m.C, m.chan_scale, xq, xsc, m.N)


def bootstrap_median(samples, draws=2000, seed=0):
    """Median of per-step times (ms) with a 95 % percentile-bootstrap interval."""
    import numpy as np
    a = np.asarray(samples, np.float64)
    rng = np.random.default_rng(seed)
    meds = np.median(a[rng.integers(0, len(a), size=(draws, len(a)))], axis=1)
    return {"median_ms_per_step": round(float(np.median(a)), 6),
            "ci95_ms_per_step": [round(float(np.percentile(meds, 2.5)), 6),
                                 round(float(np.percentile(meds, 97.5)), 6)],
            "samples": len(a)}


def oracle_layer_step_threads(oracle, mats, xs_bits, pool, slices):
    """The same layer step with the unmodified oracle called concurrently on
    packed-row slices of every matrix (the C calls run outside the interpreter
    lock)."""
    q = {k: oracle.quantize_act(xs_bits[k]) for k in ACT_K}
    futs = []
    for m in mats:
        xq, xsc = q[si.LLAMA_11B_INPUT_OF[m.name]]
        G = m.packed.shape[0]
        step = (G + slices - 1) // slices
        for g0 in range(0, G, step):
            g1 = min(G, g0 + step)
            n1 = min(3 * g1, m.N)
            futs.append(pool.submit(oracle.linear, m.packed[g0:g1], m.C,
                                    m.chan_scale[3 * g0:n1], xq, xsc, n1 - 3 * g0))
    for f in futs:
        f.result()


def cpu_baseline(seconds, max_steps=None):
    import oracle
    mats = si.layer_matrices(layer=0, seed=0)
    xs_bits = {k: si.acts(1, K, seed=0, index=i) for i, (k, K) in enumerate(ACT_K.items())}
    oracle.lib()
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle_layer_step(oracle, mats, xs_bits)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_steps and n >= max_steps):
            break
    single = n * LAYER_WEIGHT_BYTES / el / 1e9
    # all host cores: the same oracle calls spread over a thread pool
    import concurrent.futures as cf
    import platform
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        oracle_layer_step_threads(oracle, mats, xs_bits, pool, cores)
        m = 0
        t1 = time.perf_counter()
        while True:
            oracle_layer_step_threads(oracle, mats, xs_bits, pool, cores)
            m += 1
            el2 = time.perf_counter() - t1
            if el2 >= seconds / 2 or (max_steps and m >= max_steps):
                break
    multi = m * LAYER_WEIGHT_BYTES / el2 / 1e9
    return {"value": round(multi, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "seconds": round(el + el2, 2),
            "single_thread_value": round(single, 4),
            "host": f"{cpu_model()} ({platform.machine()}), {cores} cores",
            "sample": f"{m} full layer steps at M=1 (4 activation quantisations + 7 linears) with "
                      f"the plain C oracle on {cores} threads (each linear split into {cores} "
                      f"packed-row slices); single-threaded: {n} steps"}


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    # the same workload as the GPU arm: step i streams layer copy i mod 8
    copies = [si.layer_matrices(layer=r, seed=0) for r in range(COPIES)]
    xs_bits = {k: si.acts(1, K, seed=0, index=i) for i, (k, K) in enumerate(ACT_K.items())}
    oracle.lib()
    import concurrent.futures as cf
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for i in range(args.warmup):
            oracle_layer_step_threads(oracle, copies[i % COPIES], xs_bits, pool, cores)
        t0 = time.perf_counter()
        for i in range(args.steps):
            oracle_layer_step_threads(oracle, copies[i % COPIES], xs_bits, pool, cores)
        el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = LAYER_WEIGHT_BYTES / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded S3D8 fields, bf16 N(0,1) activations; no trained weights)",
        "config": dict(CONFIG),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "host": f"{cpu_model()}, {cores} cores",
                         "sample": f"{args.steps} full layer steps at M=1, the plain C oracle "
                                   f"on {cores} threads (each linear split into {cores} "
                                   "packed-row slices)"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=("s3d8", "reference"), default="s3d8")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--layer-only", action="store_true",
                    help="time the headline step only (no variants, e2e, sweeps); for profiling")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill tensor-core measurement and print it; for profiling")
    ap.add_argument("--prefill-tokens", type=int, nargs="+", default=None,
                    help="token counts for --prefill-only (default: 512 and 2048)")
    ap.add_argument("--sweep-only", action="store_true",
                    help="run only the batched-decode sweep (M = 8..64) and print it; for profiling")
    ap.add_argument("--aux-only", action="store_true",
                    help="run only the standalone unpack and quantisation measurements and print "
                         "them; for profiling")
    ap.add_argument("--encode-only", action="store_true",
                    help="run only the encoder and centroid-fit measurements and print them; "
                         "for profiling")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = 10 if args.steps is None else args.steps
        args.warmup = 3 if args.warmup is None else args.warmup
        reference_arm(args)
        return
    if args.prefill_only:
        import torch

        import s3d8_a8_linear_gb300 as s3d8
        s3d8.load(build_if_missing=True)
        _, bf16_peak, _ = load_peaks()
        print(json.dumps(prefill_measure(torch, s3d8, torch.device("cuda:0"), bf16_peak,
                                         Ms=args.prefill_tokens)))
        return
    if args.sweep_only:
        import torch

        import s3d8_a8_linear_gb300 as s3d8
        s3d8.load(build_if_missing=True)
        hbm_peak, bf16_peak, _ = load_peaks()
        print(json.dumps(decode_sweep_measure(torch, s3d8, torch.device("cuda:0"), hbm_peak,
                                              bf16_peak)))
        return
    if args.aux_only:
        import torch

        import s3d8_a8_linear_gb300 as s3d8
        s3d8.load(build_if_missing=True)
        dev = torch.device("cuda:0")
        print(json.dumps({"unpack": unpack_measure(torch, s3d8, dev),
                          "quantize": quant_measure(torch, s3d8, dev)}))
        return
    if args.encode_only:
        import torch

        import s3d8_a8_linear_gb300 as s3d8
        s3d8.load(build_if_missing=True)
        print(json.dumps(encode_measure(torch, s3d8, torch.device("cuda:0"),
                                        reps=3 if args.steps is None else args.steps)))
        print(json.dumps(fit_measure(torch, s3d8, torch.device("cuda:0"))))
        return
    args.steps = 40000 if args.steps is None else args.steps
    args.warmup = 400 if args.warmup is None else args.warmup
    if args.warmup < 3:
        args.warmup = 3
    gpu_arm(args)


if __name__ == "__main__":
    main()
