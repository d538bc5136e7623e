#!/usr/bin/env python
"""Throughput of the ZeRO++ data-parallel codec path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input
with every simulated rank's buffers resident in HBM:

    qwZ quant (all ranks' weight shards) -> qwZ dequant (the all-gather
    receiver) -> qgZ reorder + one-shot quant (all ranks' buckets) -> hop 1
    [-> hop 2] -> x 1/N_d fused into the sharded Adam step.

Default workload: the 7B model, the largest configuration (qwZ int8 B=2048
over 7e9 bf16 weights in 27 calls of up to 2^28 elements; qgZ over N_d = 64
simulated as 8 nodes x 8 GPUs with a 2^26-element int4 B=256 bucket per rank
and the Adam step fused on the final hop; standalone Adam over the rest of
the 109,375,000-parameter owned shard).  `--config llama` is the llama-layer
bucket (Phi = 202,375,168, N_d = 8 as 1 node x 8 GPUs, int8/int4 B=512).  `value` is algorithmic bytes moved per step (the bytes
each kernel must read and write, summed over the pass) divided by the step
time, in GB/s; `qgz_bucket_elems_per_s` is N_d * bucket / (qgZ kernels' time).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...      # the CPU oracle, same metric

Multi-GPU (torchrun, one process per GPU): every rank runs an independent
replica of the whole simulated job (the path has no real collective on one
device); `value` = bytes of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
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

METRIC = "codec+Adam GB/s and % of GB300 HBM peak; qgZ bucket elements/s at N_d"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
KERNEL_OF = {  # launch name -> CUDA kernel (for the roofline and the ncu summaries)
    "qwz_quant": "quant_tiled_kernel<BITS, false, LOGB, false>",
    "qwz_dequant": "dequant_kernel<BITS, LOGB>",
    "qgz_reorder_quant": "quant_tiled_kernel<BITS, true, LOGB, false>",
    "qgz_hop1": "hop1_kernel<BITS, LOGB, SCH>",
    "qgz_final_hop": "hop_tiled_kernel<BITS, kFinalAdam, LOGB, WIDE, SCH>",
    "qgz_final_hop_qwz": "hop_tiled_kernel<BITS, kFinalAdamQwz, LOGB, WIDE, SCH>",
    "grad_accumulate": "accumulate_kernel",
    "qgz_reorder_quant_acc": "quant_tiled_kernel<BITS, true, LOGB, true>",
    "shard_adam": "adam_kernel<WIDE>",
    "hpz_gather": "dequant_kernel<BITS, LOGB> (G secondary sources)",
    "ring_step": "ring1_kernel<BITS, LOGB, MODE, WIDE>",
    "ring_adam": "adam_kernel<WIDE>",
}


def kernel_label(name, wl):
    """The CUDA kernel a launch runs on this workload: hop 1 picks its kernel by
    width, sources per node and whether every destination row is whole warp units,
    as the library's launcher does."""
    g = wl.qgz
    if name != "qgz_hop1" or g is None:
        return KERNEL_OF[name]
    whole = (g.nodes * (g.bucket // g.nd)) % max(1024, g.block) == 0
    if whole and g.gpus_per_node % 4 == 0:
        return ("hop1_staged_kernel<LOGB>" if g.bits == 4 and g.gpus_per_node == 8
                else "hop1_kernel<BITS, LOGB, SCH>")
    return ("hop_tiled_kernel<BITS, kRequant, LOGB, false, SCH>" if whole
            else "hop_kernel<BITS, kRequant, LOGB>")


KERNEL_SRC = {"qwz_quant": "quant.cu", "qwz_dequant": "quant.cu", "qgz_reorder_quant": "quant.cu",
              "qgz_hop1": "hop.cu", "qgz_final_hop": "hop.cu", "qgz_final_hop_qwz": "hop.cu",
              "grad_accumulate": "quant.cu", "qgz_reorder_quant_acc": "quant.cu",
              "shard_adam": "adam.cu", "hpz_gather": "quant.cu", "ring_step": "ring.cu",
              "ring_adam": "adam.cu"}


# ---- workload -> algorithmic bytes ------------------------------------------------

def codes_bytes(n, bits):
    return (n * bits + 7) // 8


def msg_bytes(n, block, bits):
    return codes_bytes(n, bits) + 4 * (-(-n // block))


def ring_launch_bytes(g, fused_adam):
    """[(launch, bytes)] of the quantized ring over qgZ workload `g`: at every
    step each rank reads its bf16 chunk, the incoming message after the first
    step, and writes the outgoing message (or the fp32 chunk at the last);
    then the Adam step on the reduced gradient (30 B a parameter)."""
    nd, L = g.nd, g.slice_elems
    m = msg_bytes(L, g.block, g.bits)
    out = []
    for step in range(nd):
        b = 2 * L + (m if step > 0 else 0) + (m if step < nd - 1 else 4 * L)
        out.append(("ring_step", nd * b))
    if fused_adam:
        out.append(("ring_adam", 30 * g.bucket))
    return out


def launch_bytes(wl, fuse_qwz=False, microbatches=1, hpz=False, ring=False):
    """[(launch name, algorithmic bytes)] of one pass, in launch order.  With
    fuse_qwz the weights' qwZ message is written by the final hop's Adam pass
    (the next step's message), so the pass has no separate quantize launch.
    With M > 1 micro-batches, M-1 accumulate launches (bf16 in, fp32
    accumulator read except the first, fp32 written) precede a one-shot
    quantizer that reads the accumulator and the last micro-batch.  With hpz
    the backward gather reads the node's secondary partitions (the whole
    message) and writes the bf16 weights again."""
    out = []
    q, g = wl.qwz, wl.qgz
    if q is not None and fuse_qwz:
        m = q.nranks * msg_bytes(q.shard, q.block, q.bits)
        out.append(("qwz_dequant", m + 2 * q.nranks * q.shard))
    elif q is not None:
        shards = [q.shard] * q.calls
        if q.tail_shard:
            shards[-1] = q.tail_shard
        for s in shards:
            m = q.nranks * msg_bytes(s, q.block, q.bits)
            out.append(("qwz_quant", 2 * q.nranks * s + m))
            out.append(("qwz_dequant", m + 2 * q.nranks * s))
    if q is not None and hpz:
        out.append(("hpz_gather", q.nranks * msg_bytes(q.shard, q.block, q.bits)
                    + 2 * q.nranks * q.shard))
    if g is not None and ring:
        out += ring_launch_bytes(g, wl.fused_adam)
    elif g is not None:
        nd, b = g.nd, g.bucket
        m1 = nd * msg_bytes(b, g.block, g.bits)
        if microbatches > 1:
            for k in range(microbatches - 1):
                out.append(("grad_accumulate", (6 if k == 0 else 10) * nd * b))
            out.append(("qgz_reorder_quant_acc", 6 * nd * b + m1))
        else:
            out.append(("qgz_reorder_quant", 2 * nd * b + m1))
        final_extra = (26 * b) if wl.fused_adam else 4 * b
        name = "qgz_final_hop"
        if fuse_qwz:
            final_extra += nd * msg_bytes(g.slice_elems, g.block, 8)
            name = "qgz_final_hop_qwz"
        if g.nodes == 1:
            out.append((name, m1 + final_extra))
        else:
            m2 = nd * msg_bytes(g.nodes * g.slice_elems, g.block, g.bits)
            out.append(("qgz_hop1", m1 + m2))
            out.append((name, m2 + final_extra))
    if wl.standalone_adam:   # g, master, m, v in; master, m, v, bf16 param out
        out.append(("shard_adam", 30 * wl.standalone_adam))
    return out


def workload_config(wl, name, fuse_qwz=False, microbatches=1, hpz=False, ring=False):
    q, g = wl.qwz, wl.qgz
    cfg = {"workload": wl.name, "name": name}
    if ring:
        cfg["reduce_scatter"] = ("comparator: quantized ring (a requantization at every hop, "
                                 "N_d launches) + Adam on the reduced gradient, instead of qgZ")
    if hpz:
        cfg["hpz"] = ("backward weight gather from the node's secondary partitions "
                      f"({hpz_nodes(wl)} node(s) x {q.nranks // hpz_nodes(wl)} GPUs)")
    if microbatches > 1:
        cfg["microbatches"] = microbatches
        cfg["accumulation"] = ("fp32 accumulator over the first M-1 micro-batches; the one-shot "
                               "quantizer adds the last")
    if fuse_qwz:
        cfg["qwz_fused"] = "the weights' int8 qwZ message is written by the final hop's Adam pass"
    if q is not None:
        cfg.update(qwz_phi=q.phi, qwz=f"int{q.bits} B={q.block}", qwz_nranks=q.nranks,
                   qwz_calls=q.calls)
    if g is not None:
        cfg.update(N_d=g.nd, topology=f"{g.nodes}x{g.gpus_per_node}", bucket_per_rank=g.bucket,
                   qgz=f"int{g.bits} B={g.block}", adam="fused on the final hop" if wl.fused_adam
                   else "none")
    if wl.standalone_adam:
        cfg["standalone_adam_params"] = wl.standalone_adam
    per_step = sum(b for _, b in launch_bytes(wl, fuse_qwz, microbatches, hpz, ring))
    if per_step > 4 * L2_BYTES:
        cfg["l2"] = (f"inputs larger than L2: {per_step / 1e9:.2f} GB moved per step vs "
                     f"{L2_BYTES / 2**20:.0f} MiB L2; no flush")
    else:
        cfg["l2"] = (f"L2-resident: {per_step / 1e6:.1f} MB moved per step fits the "
                     f"{L2_BYTES / 2**20:.0f} MiB L2; not a roofline configuration")
    cfg["arithmetic"] = "bf16 in, int8/int4 codes + fp32 scales, fp32 sums and Adam"
    return cfg


def hpz_nodes(wl):
    """hpZ node count of the qwZ ranks: the qgZ topology's when they coincide."""
    q, g = wl.qwz, wl.qgz
    if g is not None and q.nranks == g.nd:
        return g.nodes
    return 1


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_table():
    """ncu DRAM bytes per launch recorded in profiles/traffic.txt, keyed by
    launch name, workload name and the sha1 of the kernel's source file; a
    row whose source hash no longer matches is ignored (null traffic)."""
    import hashlib
    rows = {}
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return rows
    for line in open(p):
        line = line.split("#", 1)[0].split()
        if len(line) >= 4:
            name, wname, sha, byts = line[:4]
            rows[(name, wname)] = (sha, float(byts))
    cur = {}
    for name, src in KERNEL_SRC.items():
        path = os.path.join(ROOT, "gradient_comm_codecs_gb300", "csrc", src)
        h = hashlib.sha1(open(path, "rb").read())
        h.update(open(os.path.join(ROOT, "gradient_comm_codecs_gb300", "csrc",
                                   "zpp_device.cuh"), "rb").read())
        cur[name] = h.hexdigest()[:12]
    return {k: v[1] for k, v in rows.items() if cur.get(k[0]) == v[0]}


# ---- multi-rank helpers ------------------------------------------------------------------

def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: int, world: int, ms_step_max: float) -> float:
    """Whole-job throughput: bytes every replica moved per step / slowest step time."""
    return bytes_per_rank_step * world / (ms_step_max * 1e-3) / 1e9


# ---- clocks --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", device_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if len(inside) < 2:
            inside = [p for t, p in self.samples if t0 - 0.5 <= t <= t1 + 0.5]
            note = "timed region shorter than the sampling period: samples within 0.5 s of it"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        pw = [num(p[3]) for p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ---- the GPU arm ------------------------------------------------------------------------

def fill_inputs(path, wl):
    import torch
    import synth
    from synth import workloads as W
    chunk = 1 << 27
    if wl.qwz is not None:
        synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, path.qwz.phi, out=path.w, chunk=chunk)
    if wl.qgz is not None:
        g = wl.qgz
        for k, grads in enumerate(path.grads_mb):
            for r in range(g.nd):
                synth.fill(g.grad, wl.seed, synth.grad_stream(r, k), 0, g.bucket,
                           out=grads[r * g.bucket:(r + 1) * g.bucket], chunk=chunk)
        if path.adam is not None:
            synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, 0, g.bucket, out=path.param,
                       chunk=chunk)
            path.master.copy_(path.param.float())
        if path.standalone_adam:
            n = path.standalone_adam
            t = synth.fill(W.GRAD_NORMAL, wl.seed, synth.SHARD_GRAD, 0, n, device=path.device,
                           chunk=chunk)
            path.sa_grad.copy_(t.float())
            synth.fill(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, g.bucket, n, out=t, chunk=chunk)
            path.sa_master.copy_(t.float())
            del t
    torch.cuda.synchronize()


def run_gpu(args, wl, rank, world, device):
    import torch
    import gradient_comm_codecs_gb300 as Z
    from gradient_comm_codecs_gb300 import _build
    _build.build()

    q, g = wl.qwz, wl.qgz
    qs = Z.QwzSpec(q.nranks, q.shard, q.block, q.bits, chunks=q.calls, tail_shard=q.tail_shard,
                   nodes=hpz_nodes(wl) if args.hpz else 1) if q else None
    gs = Z.QgzSpec(g.nodes, g.gpus_per_node, g.bucket, g.block, g.bits) if g else None
    a = wl.adam
    adam = Z.AdamSpec(a.lr, a.beta1, a.beta2, a.eps, a.step) if (g and wl.fused_adam) else None
    path = Z.CodecPath(qs, gs, adam, device=device, keep_grad=False, fuse_qwz=args.fuse_qwz,
                       microbatches=args.microbatches,
                       standalone_adam=wl.standalone_adam if adam is not None else 0,
                       hpz=args.hpz, ring=args.ring)
    fill_inputs(path, wl)
    stream = torch.cuda.current_stream(device)
    if args.fuse_qwz:
        path.prime_fused_qwz(stream)
    lb = launch_bytes(wl, args.fuse_qwz, args.microbatches, args.hpz, args.ring)
    step_bytes = sum(b for _, b in lb)

    def one_step(i, events=None):
        mark = None
        if events is not None:
            def mark(name):
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(stream)
                events.append((name, ev))
        path.run(stream, adam_step=1 + i, mark=mark)

    for i in range(args.warmup):
        one_step(i)
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(device)
    dev_id = str(getattr(props, "uuid", "")) or str(device.index)
    if dev_id and not dev_id.startswith("GPU-") and "-" in dev_id:
        dev_id = "GPU-" + dev_id
    sampler = ClockSampler(dev_id)
    time.sleep(0.3)

    events = []
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        events.append(("__step__", None))
        one_step(args.warmup + i, events)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    total_ms = start.elapsed_time(end)
    # per-launch durations from consecutive events
    per = {}
    prev = start
    for name, ev in events:
        if name == "__step__":
            continue
        per.setdefault(name, []).append(prev.elapsed_time(ev))
        prev = ev
    ms_step = max_over_ranks(total_ms / args.steps, device)

    # the same steps once more with events only around them (after the timed region, for
    # information): what the events between kernels cost the step
    bare = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    bare[0].record(stream)
    for i in range(args.steps):
        one_step(args.warmup + args.steps + i)
    bare[1].record(stream)
    torch.cuda.synchronize()
    ms_step_bare = bare[0].elapsed_time(bare[1]) / args.steps

    peak, peak_kind = measured_peak()
    kernels = {}
    bytes_of = {}
    for name, b in lb:
        bytes_of.setdefault(name, []).append(b)
    for name, ts in per.items():
        nb = sum(bytes_of[name]) / len(bytes_of[name])
        avg = sum(ts) / len(ts)
        kernels[name] = {"kernel": kernel_label(name, wl), "launches": len(ts), "avg_ms": avg,
                         "bytes_per_launch": nb, "gbs": nb / (avg * 1e-3) / 1e9,
                         "frac_of_peak": nb / (avg * 1e-3) / 1e9 / peak,
                         "share": sum(ts) / total_ms}
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    traffic = traffic_table().get((dom, args.config + ("+fuse_qwz" if args.fuse_qwz else "")
                                   + (f"+mb{args.microbatches}" if args.microbatches > 1 else "")
                                   + ("+hpz" if args.hpz else "") + ("+ring" if args.ring else "")))
    dk = kernels[dom]
    roofline = {"bound": "hbm", "kernel": dk["kernel"], "launch": dom,
                "achieved": dk["gbs"], "peak": peak, "unit": "GB/s",
                "frac": dk["gbs"] / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "traffic": traffic, "algorithmic_bytes": dk["bytes_per_launch"]}

    value = whole_job_gbs(step_bytes, world, ms_step)
    qgz_ms = sum(sum(per[n]) for n in per if n.startswith("qgz") or n.startswith("ring")) \
        / args.steps
    qgz_eps = (g.nd * g.bucket / (qgz_ms * 1e-3)) if g else None

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, path, wl, stream, step_bytes, world, device)

    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic: seeded counter-based generator (lowbias32 hash -> "
        "2^20-entry quantile table), weights N(0,0.02), grads per the workload",
        "config": workload_config(wl, args.config, args.fuse_qwz, args.microbatches, args.hpz,
                                  args.ring),
        "pct_hbm_peak_measured": 100.0 * value / world / peak,
        "pct_hbm_peak_nominal": 100.0 * value / world / NOMINAL_HBM_GBS,
        "qgz_bucket_elems_per_s": qgz_eps * world if qgz_eps else None,
        "bytes_per_step": step_bytes,
        "ms_per_step_without_kernel_events": ms_step_bare,
        "gpu_launches": sum(len(v) for v in per.values()),
        "kernels": kernels, "roofline": roofline, "clocks": clocks, "e2e": e2e,
        "impl": "ours",
    }
    del path
    return res


def run_e2e(args, path, wl, stream, step_bytes, world, device):
    import torch
    steps = max(3, min(args.steps, 30))
    # fused mode: the step's weight message comes from the previous step on the device
    w_host = path.w.cpu().pin_memory() if (path.qwz is not None and not path.fuse_qwz) else None
    g_host = [t.cpu().pin_memory() for t in path.grads_mb] if path.qgz is not None else None
    p_host = None
    if path.qgz is not None and path.adam is not None:
        p_host = torch.empty(path.qgz.bucket, dtype=torch.bfloat16).pin_memory()
    sa_g = sa_p = None
    if path.standalone_adam:
        sa_g = path.sa_grad.cpu().pin_memory()
        sa_p = torch.empty(path.standalone_adam, dtype=torch.bfloat16).pin_memory()
    for i in range(2):
        path.run_from_host(w_host, g_host, p_host, stream, adam_step=1 + i, sa_grad_host=sa_g,
                           sa_param_host=sa_p)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    h2d = d2h = 0
    for i in range(steps):
        h2d, d2h = path.run_from_host(w_host, g_host, p_host, stream, adam_step=3 + i,
                                      sa_grad_host=sa_g, sa_param_host=sa_p)
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t0) / steps, device)
    return {"value": whole_job_gbs(step_bytes, world, dt * 1e3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": steps,
            "note": "pinned host inputs copied in and bf16 parameters copied out every step, "
                    "wall clock around the steps; value counts the same algorithmic bytes"}


# ---- the oracle (CPU baseline and reference arm) --------------------------------------------

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: the first `nbw`
    blocks of every rank's weight shard (first qwZ call) and the first `nbg`
    blocks of every slice of every rank's bucket -- a self-contained smaller
    instance of the same pass (same topology, block, bits, Adam, micro-batches)."""

    def __init__(self, wl, nbw, nbg, microbatches=1, hpz=False, ring=False):
        import numpy as np
        import synth
        from synth import workloads as W
        self.wl = wl
        self.steps_bytes = 0
        q, g = wl.qwz, wl.qgz
        self.q = self.g = None
        if q is not None:
            nbw = max(1, min(nbw, -(-q.shard // q.block)))
            n = min(q.shard, nbw * q.block)
            idx = (np.arange(q.nranks)[:, None] * q.shard + np.arange(n)[None, :]).reshape(-1)
            self.wx = synth.bf16_to_u16(synth.at(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, idx))
            self.q = (q.nranks, n, q.block, q.bits)
            m = q.nranks * msg_bytes(n, q.block, q.bits)
            self.steps_bytes += 2 * (2 * q.nranks * n + m)
            self.hpz = hpz_nodes(wl) if hpz else 0
            if hpz:
                self.steps_bytes += 2 * q.nranks * n + m
        if g is not None:
            nbg = max(1, min(nbg, g.slice_elems // g.block))
            Lm = nbg * g.block
            nd = g.nd
            pos = (np.arange(nd)[:, None] * g.slice_elems + np.arange(Lm)[None, :]).reshape(-1)
            self.mbs = [np.concatenate([synth.bf16_to_u16(
                synth.at(g.grad, wl.seed, synth.grad_stream(r, k), pos)) for r in range(nd)])
                for k in range(microbatches)]
            self.gx = self.mbs[-1]
            bucket = nd * Lm
            self.g = (g.nodes, g.gpus_per_node, bucket, g.block, g.bits)
            self.ring = ring
            gidx = (np.arange(nd)[:, None] * g.slice_elems + np.arange(Lm)[None, :]).reshape(-1)
            import oracle
            self.master = oracle.bf16_bits_to_f32(synth.bf16_to_u16(
                synth.at(W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS, gidx)))
            self.zero = np.zeros(bucket, np.float32)
            m1 = nd * msg_bytes(bucket, g.block, g.bits)
            if ring:   # the same accounting as the GPU ring, on the sample's bucket
                import dataclasses
                gm = dataclasses.replace(g, bucket=bucket)
                b = sum(x for _, x in ring_launch_bytes(gm, wl.fused_adam))
            else:
                b = m1 + 2 * nd * bucket
                if microbatches > 1:
                    b += 4 * nd * bucket + sum(6 if k == 0 else 10
                                               for k in range(microbatches - 1)) * nd * bucket
                if g.nodes == 1:
                    b += m1
                else:
                    m2 = nd * msg_bytes(g.nodes * Lm, g.block, g.bits)
                    b += m1 + m2 + m2
                b += (26 if wl.fused_adam else 4) * bucket
            self.steps_bytes += b
            self.elems = nd * bucket
        self.sa = None
        if wl.standalone_adam and wl.fused_adam:   # a bounded slice of the standalone shard
            n = min(wl.standalone_adam, max(4096, nbg * 2048))
            t = synth.at(W.GRAD_NORMAL, wl.seed, synth.SHARD_GRAD, np.arange(n))
            import oracle
            self.sa = (oracle.bf16_bits_to_f32(synth.bf16_to_u16(t)),
                       oracle.bf16_bits_to_f32(synth.bf16_to_u16(synth.at(
                           W.WEIGHT_RECIPE, wl.seed, synth.WEIGHTS,
                           np.arange(n) + (g.bucket if g is not None else 0)))),
                       np.zeros(n, np.float32))
            self.steps_bytes += 30 * n

    def run(self):
        import oracle
        if self.q is not None:
            c, s = oracle.qwz_quant(self.wx, *self.q)
            oracle.qwz_dequant(c, s, *self.q)
            if self.hpz:
                nr, n, block, bits = self.q
                N, G = self.hpz, nr // self.hpz
                cb, nb = oracle.codes_bytes(n, bits), oracle.num_blocks(n, block)
                oracle.hpz_gather([(c[l * N * cb:(l + 1) * N * cb], s[l * N * nb:(l + 1) * N * nb])
                                   for l in range(G)], N, n, block, bits)
        if self.g is not None:
            if self.ring:
                N, G, bucket, block, bits = self.g
                gr = oracle.ring_reduce_scatter(self.gx, N * G, bucket, block, bits)
            elif len(self.mbs) > 1:
                N = self.g[0]
                c1, s1 = oracle.qgz_reorder_quant_f32(oracle.grad_accumulate(self.mbs), *self.g)
                if N == 1:
                    gr = oracle.qgz_hop1(c1, s1, *self.g)
                else:
                    gr = oracle.qgz_hop2(*oracle.qgz_hop1(c1, s1, *self.g), *self.g)
            else:
                gr = oracle.qgz_reduce_scatter(self.gx, *self.g)
            if self.wl.fused_adam:
                a = self.wl.adam
                oracle.adam_step(gr, self.master, self.zero, self.zero, a.lr, a.beta1, a.beta2,
                                 a.eps, a.step)
        if self.sa is not None:
            a = self.wl.adam
            g, p, z = self.sa
            oracle.adam_step(g, p, z, z, a.lr, a.beta1, a.beta2, a.eps, a.step)


def host_cpu():
    """CPU model and online core count of this host."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip().lower() in ("model name", "cpu model"):
                    model = v.strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                k, _, v = line.partition(":")
                if k.strip() == "Model name":
                    model = v.strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "nproc": os.cpu_count()}


def sized_sample(wl, seconds, microbatches=1, hpz=False, ring=False):
    """Calibrate the sample so one oracle pass takes about `seconds`."""
    s = OracleSample(wl, 4, 2, microbatches, hpz, ring)
    t = time.perf_counter()
    s.run()
    dt = max(time.perf_counter() - t, 1e-4)
    scale = max(1.0, seconds / dt)
    return OracleSample(wl, int(4 * scale), int(2 * scale), microbatches, hpz, ring)


def cpu_baseline(wl, seconds=12.0, microbatches=1, hpz=False, ring=False):
    s = sized_sample(wl, seconds / 2, microbatches, hpz, ring)
    t = time.perf_counter()
    n = 0
    while True:
        s.run()
        n += 1
        if time.perf_counter() - t >= seconds / 2 and n >= 1:
            break
    dt = (time.perf_counter() - t) / n
    return {"value": s.steps_bytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            **host_cpu(),
            "sample": f"{s.steps_bytes / 1e6:.1f} MB of algorithmic traffic per pass: the first "
                      f"blocks of every shard and of every slice of every rank (same topology, "
                      f"block, bits, Adam), {n} passes, single-threaded C oracle",
            "seconds": dt * n}


def run_reference(args, wl):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    budget = 150.0
    per_step = max(0.2, min(5.0, budget / max(1, args.steps + args.warmup)))
    s = sized_sample(wl, per_step, args.microbatches, args.hpz, args.ring)
    for _ in range(args.warmup):
        s.run()
    t = time.perf_counter()
    for _ in range(args.steps):
        s.run()
    dt = (time.perf_counter() - t) / args.steps
    value = s.steps_bytes / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded counter-based generator, bounded sample of the workload",
        "config": workload_config(wl, args.config, microbatches=args.microbatches, hpz=args.hpz,
                                  ring=args.ring),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         **host_cpu(),
                         "sample": f"{s.steps_bytes / 1e6:.1f} MB of algorithmic traffic per "
                                   "step: the first blocks of every shard and slice of every "
                                   "rank, single-threaded C oracle"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---- the ring comparator sweep (precision and time against qgZ) -------------------------------

RING_SWEEP_ND = (2, 4, 8, 16, 32, 64, 128)


def run_ring_sweep(args):
    """For N_d = 2..128 ranks of a 2^22-element bucket (N(0, 1e-3) bf16
    gradients, int4, block 256): the quantized ring and the qgZ chain (1 x N_d
    up to 8 ranks, N_d/8 nodes x 8 beyond) on the same data, their errors
    against the float64 average of the bf16 inputs (relative RMS, max over
    the RMS of the average) and their CUDA-event times.  One JSON line per
    N_d."""
    import torch
    import gradient_comm_codecs_gb300 as Z
    from gradient_comm_codecs_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    bucket_per_rank, block, bits = 1 << 22, 256, 4
    for nd in RING_SWEEP_ND:
        N, G = (1, nd) if nd <= 8 else (nd // 8, 8)
        b = bucket_per_rank
        torch.manual_seed(nd)
        qgz = Z.CodecPath(None, Z.QgzSpec(N, G, b, block, bits), None, device=dev, keep_grad=True)
        qgz.grads.normal_(0.0, 1e-3)
        ring = Z.CodecPath(None, Z.QgzSpec(N, G, b, block, bits), None, device=dev,
                           keep_grad=True, ring=True)
        ring.grads = qgz.grads          # the same gradients
        exact = qgz.grads.view(nd, nd, b // nd).double().sum(0).reshape(-1) / nd
        rms = exact.pow(2).mean().sqrt().item()
        rec = {"N_d": nd, "topology": f"{N}x{G}", "bucket_per_rank": b, "block": block,
               "bits": bits}
        for name, path in (("qgz", qgz), ("ring", ring)):
            path.run_qgz(st)
            torch.cuda.synchronize()
            err = path.grad_out.double() - exact
            rec[f"{name}_rel_rmse"] = err.pow(2).mean().sqrt().item() / rms
            rec[f"{name}_max_over_rms"] = err.abs().max().item() / rms
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(10):
                path.run_qgz(st)
            e1.record(st)
            torch.cuda.synchronize()
            rec[f"{name}_ms"] = e0.elapsed_time(e1) / 10
        rec["rmse_ratio_ring_over_qgz"] = rec["ring_rel_rmse"] / rec["qgz_rel_rmse"]
        rec["time_ratio_ring_over_qgz"] = rec["ring_ms"] / rec["qgz_ms"]
        print(json.dumps(rec), flush=True)
        del qgz, ring, exact
        torch.cuda.empty_cache()


# ---- the sweep (small-message efficiency) -----------------------------------------------------

def run_sweep(args):
    """Every sweep point: qgZ chain (reorder+quant, hop 1, hop 2 / final, no
    Adam) and qwZ quant+dequant on N_d shards of the same size, timed with
    CUDA events (plain launches back to back, so points smaller than L2 run
    from L2) and, for the qgZ chain, as a CUDA-graph replay, and once more
    with L2 flushed before every pass (a read of twice L2's size) and an
    event after every kernel (the per-kernel split, in microseconds).  The
    first line is the launch floor: a one-element kernel's time on the
    stream.  Timing inputs are filled in place by torch's normal_ (bf16,
    N(0, 1e-3) gradients, N(0, 0.02) weights); parity of sweep points is
    covered by the tests.  Points whose buffers do not fit in free memory are
    skipped and reported as such."""
    import torch
    import gradient_comm_codecs_gb300 as Z
    from gradient_comm_codecs_gb300 import _build
    from synth import workloads as W
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    out = []
    flush = None
    # the launch floor: a one-element kernel, back to back, timed the same way
    st0 = torch.cuda.current_stream(dev)
    one = torch.zeros(1, device=dev)
    for _ in range(10):
        one.add_(1)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(st0)
    for _ in range(200):
        one.add_(1)
    a1.record(st0)
    torch.cuda.synchronize()
    floor = {"launch_floor_us": 1e3 * a0.elapsed_time(a1) / 200,
             "note": "a one-element torch kernel launched 200 times back to back: the time a "
                     "launch takes on the stream when there is no work"}
    print(json.dumps(floor), flush=True)
    for i, wl in W.sweep_points():
        q, g = wl.qwz, wl.qgz
        if g.bucket * 2 > args.sweep_max_mib << 20:
            continue
        rec = {"index": i, "block": g.block, "bits": g.bits, "N_d": g.nd,
               "topology": f"{g.nodes}x{g.gpus_per_node}", "mib_per_rank": g.bucket * 2 >> 20}
        nd, b = g.nd, g.bucket
        c = g.bits / 8 + 4 / g.block
        need = nd * b * (2 + c) + nd * g.nodes * g.slice_elems * c + 4 * b
        free, _ = torch.cuda.mem_get_info(dev)
        if need > 0.85 * free:
            rec["skipped"] = f"needs {need / 2**30:.0f} GiB"
            out.append(rec)
            print(json.dumps(rec), flush=True)
            continue
        torch.manual_seed(i)
        path = Z.CodecPath(None, Z.QgzSpec(g.nodes, g.gpus_per_node, b, g.block, g.bits), None,
                           device=dev, keep_grad=True)
        path.grads.normal_(0.0, 1e-3)  # in place: no temporary
        qgz_bytes = sum(x for n, x in launch_bytes(wl) if n.startswith("qgz"))
        st = torch.cuda.current_stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        path.run_qgz(st)
        torch.cuda.synchronize()
        e0.record(st)
        path.run_qgz(st)
        e1.record(st)
        torch.cuda.synchronize()
        once = e0.elapsed_time(e1)
        iters = max(3, min(200, int(200.0 / max(once, 1e-3))))
        e0.record(st)
        for _ in range(iters):
            path.run_qgz(st)
        e1.record(st)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        rec.update(qgz_ms=ms, qgz_gbs=qgz_bytes / (ms * 1e-3) / 1e9,
                   qgz_elems_per_s=nd * b / (ms * 1e-3))
        # per-kernel split, and the chain again with L2 flushed before every pass
        # (a read of twice L2's size, so L2 holds only clean lines of another
        # buffer when the chain starts), the chain timed alone
        per = {}
        if flush is None:
            flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
        reps = max(3, min(50, iters))
        t_flushed = 0.0
        for _ in range(reps):
            flush.sum()
            marks = [torch.cuda.Event(enable_timing=True)]
            marks[0].record(st)

            def mark(name, marks=marks):
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(st)
                marks.append((name, ev))
            path.run_qgz(st, mark=mark)
            torch.cuda.synchronize()
            prev = marks[0]
            for name, ev in marks[1:]:
                per.setdefault(name, []).append(prev.elapsed_time(ev))
                prev = ev
            t_flushed += marks[0].elapsed_time(marks[-1][1])
        rec["qgz_flushed_ms"] = t_flushed / reps
        rec["qgz_flushed_gbs"] = qgz_bytes / (t_flushed / reps * 1e-3) / 1e9
        rec["kernels_flushed_us"] = {n: 1e3 * sum(v) / len(v) for n, v in per.items()}
        # CUDA-graph replay of the same chain (launch overhead removed)
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(st)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            path.run_qgz(gs)
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=gs):
                path.run_qgz(gs)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        e0.record(st)
        for _ in range(iters):
            graph.replay()
        e1.record(st)
        torch.cuda.synchronize()
        gms = e0.elapsed_time(e1) / iters
        rec.update(qgz_graph_ms=gms, qgz_graph_gbs=qgz_bytes / (gms * 1e-3) / 1e9)
        del graph, path
        torch.cuda.empty_cache()
        # qwZ on N_d shards of the same size
        if nd * b * (4 + c) < 0.85 * torch.cuda.mem_get_info(dev)[0]:
            qp = Z.CodecPath(Z.QwzSpec(q.nranks, q.shard, q.block, q.bits), None, None, device=dev)
            qp.w.normal_(0.0, 0.02)
            qwz_bytes = sum(x for n, x in launch_bytes(wl) if n.startswith("qwz"))
            qp.run_qwz(st)
            torch.cuda.synchronize()
            e0.record(st)
            for _ in range(iters):
                qp.run_qwz(st)
            e1.record(st)
            torch.cuda.synchronize()
            qms = e0.elapsed_time(e1) / iters
            rec.update(qwz_ms=qms, qwz_gbs=qwz_bytes / (qms * 1e-3) / 1e9)
            del qp
            torch.cuda.empty_cache()
        out.append(rec)
        print(json.dumps(rec), flush=True)
    return out


# ---- main ------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="7b", choices=["tiny", "llama", "two_hop", "7b"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fuse-qwz", action="store_true",
                    help="produce the weights' qwZ message inside the final hop's Adam pass")
    ap.add_argument("--ring", action="store_true",
                    help="comparator: reduce the gradients with the quantized ring instead of qgZ")
    ap.add_argument("--ring-sweep", action="store_true",
                    help="ring vs qgZ error and time over N_d = 2..128 (GPU), one JSON line each")
    ap.add_argument("--hpz", action="store_true",
                    help="add the hpZ backward weight gather from the secondary partitions")
    ap.add_argument("--microbatches", type=int, default=1,
                    help="gradient accumulation: micro-batches summed before the qgZ reduce")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="run the 144-point block/bits/topology/message-size sweep instead")
    ap.add_argument("--sweep-max-mib", type=int, default=1024)
    ap.add_argument("--scale", type=int, default=1,
                    help="divide the workload's shard and bucket by this (small profiling cases)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    from synth import workloads as W
    wl = W.WORKLOADS[args.config]
    if args.scale > 1:
        wl = W.scaled(wl, args.scale)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.sweep:
        run_sweep(args)
        return
    if args.ring_sweep:
        run_ring_sweep(args)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        res = run_gpu(args, wl, rank, world, device)
        if rank == 0 and world == 1 and not args.no_cpu:
            res["cpu_baseline"] = cpu_baseline(wl, microbatches=args.microbatches, hpz=args.hpz,
                                               ring=args.ring)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
