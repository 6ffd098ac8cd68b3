"""Benchmark: causal linear-attention forward, tokens/s and roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step is one forward pass (one la_forward call) over the whole workload,
inputs already resident in HBM.  The default workload is the causal,
per-head-decayed one at N = 16384, D = Dv = 128, bf16 (B = 2, H = 16); its
Q, K, V and O (537 MB) exceed the 129 MB L2, so no flush is needed between
iterations.  Under torchrun each rank runs its own replica (independent
batches, no collective on the data path: weak scaling); the time is the max
over ranks and the value the tokens of all ranks over that time.

Rank 0 prints one JSON line.  `--impl reference` times the fp64 CPU oracle
instead (the one other place this script runs oracle/), on a bounded sample
of the same workload.
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

METRIC = ("causal linear-attn fwd tokens/s and % roofline "
          "(TFLOP/s or HBM GB/s), 1×GB300")
# metrics of the other workloads (same unit, their own roofline)
METRICS = {
    "noncausal": "non-causal linear-attn fwd tokens/s and % HBM roofline, 1×GB300",
    "decode": "recurrent decode step tokens/s and % HBM roofline, 1×GB300",
    "decode_gated": "gated recurrent decode step tokens/s and % HBM roofline, 1×GB300",
    "gated": "gated linear-attn fwd tokens/s and % roofline (HBM, or fp32 ALU on CUDA cores), 1×GB300",
    "favor": "Performer (FAVOR+) causal linear-attn fwd tokens/s and % HBM roofline, 1×GB300",
    "backward": "causal linear-attn bwd (dq, dk, dv) tokens/s and % roofline (HBM on tensor cores, fp32 ALU on CUDA cores), 1×GB300",
}


def workload_metric(w):
    if w.steps:
        return METRICS["decode_gated"] if w.gated else METRICS["decode"]
    if w.gated:
        return METRICS["gated"]
    if w.favor_r:
        return METRICS["favor"]
    if w.backward:
        return METRICS["backward"]
    return METRIC if w.causal else METRICS["noncausal"]
DEFAULT_WORKLOAD = "causal_decay_bf16_n16384"
FALLBACK_HBM_GBS = 6800.0  # profiling recipe fallback, used only if absent
L2_BYTES = 129 * 1024 * 1024   # GB300 L2
FALLBACK_BF16_TFLOPS = 1900.0
# fp32 CUDA-core peak of a GB300, from its unit counts and clock: 152 SMs x
# 128 fp32 lanes x 2 flops (one FMA) x 2070 MHz maximum SM clock
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2070e6 / 1e12

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from an
# ncu capture, keyed by workload, with the hash of the kernel source the
# capture was taken on; reported only while that source is unchanged.
NCU_TRAFFIC = {
    # dram__bytes_read.sum 556.580608 MB + dram__bytes_write.sum 113.448960 MB
    # in one launch of the full workload (relay split, phase-A-only prefetch)
    "causal_decay_bf16_n16384": {"bytes": 670029568, "source": "99a80a2e9216e568"},
}

# the other configurations of the method, timed in the same process as the
# default workload and reported in its line under "workloads"
EXTRA_WORKLOADS = ("causal_f32_n256", "causal_bf16_n4096", "noncausal_bf16_n65536",
                   "decode_bf16_h32", "gla_bf16_n16384", "favor_bf16_n16384",
                   "backward_bf16_n4096")


# ---------------------------------------------------------------------------
# host-side helpers (also exercised by the CPU multi-process tests)

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(ms_per_step_max: float, tokens_per_rank_step: int, world: int):
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_rank_step / (ms_per_step_max / 1e3)


def decode_work(w):
    """Algorithmic bytes and flops of one decode step over all B*H units:
    the fp32 state (S and z) read and written once, q, k, v read and o
    written once; flops per unit 4 D Dv + 3 D + Dv as in the forward."""
    import torch
    es = torch.tensor([], dtype=w.dtype).element_size()
    units = w.B * w.H
    byts = units * (2 * 4 * (w.D * w.Dv + w.D) + (2 * w.D + 2 * w.Dv) * es)
    flops = units * (4 * w.D * w.Dv + 3 * w.D + w.Dv)
    if w.gated:  # the fp32 gates read once; one more multiply per state entry
        byts += units * w.D * 4
        flops += units * (w.D * w.Dv + w.D)
    return byts, flops


def algorithmic_work(w):
    """Algorithmic bytes and flops of one forward pass over the workload.

    Bytes: Q, K, V read and O written once, in their dtype (the state never
    leaves the chip).  Flops per (b, h, token), recurrent form: 2 D Dv state
    update + 2 D Dv read-out + 2 D denominator + D normaliser update + Dv
    divides (the chunked kernel's extra intra-chunk work is not counted)."""
    import torch
    es = torch.tensor([], dtype=w.dtype).element_size()
    units = w.B * w.H * w.N
    byts = units * (2 * w.D + 2 * w.Dv) * es
    flops = units * (4 * w.D * w.Dv + 3 * w.D + w.Dv)
    if w.gated:
        # plus the fp32 gates read once; the gate multiplies one more flop
        # per state and normaliser entry
        byts += units * w.D * 4
        flops += units * (w.D * w.Dv + w.D)
    if w.favor_r:
        # r features in place of D: the projections of q and k (2 D r flops
        # each, plus the norm and the exponential) and the attention over r
        r = w.favor_r
        byts += r * w.D * es
        flops = units * (2 * (2 * w.D * r + 2 * w.D + r) + 4 * r * w.Dv + 3 * r + w.Dv)
    if w.backward:
        # read q, k, v, dL/do, write dq, dk, dv; recurrent-form flops: the
        # forward (4 D Dv) plus dphi(q) = S gt - c z, the reverse state
        # U = sum phi(q) gt^T, dv = U^T phi(k), dphi(k) = U v - u (2 D Dv each)
        byts = units * (4 * w.D + 3 * w.Dv) * es
        flops = units * (12 * w.D * w.Dv + 10 * w.D + 4 * w.Dv)
    return byts, flops


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# device sources of the 128-token causal kernel (the benchmark workload's)
KERNEL_SOURCES = ("chunk128.cu", "tc_common.cuh", "common.cuh")
# sources of the gated CUDA-core kernel
GATED_SOURCES = ("gla_simt.cu", "chunk128.cu", "tc_common.cuh", "common.cuh")
# sources of the Performer path (feature kernel, then the causal kernel)
FAVOR_SOURCES = ("favor.cu", "chunk128.cu", "tc_common.cuh", "common.cuh")
# sources of the backward pass
BACKWARD_SOURCES = ("backward_tc.cu", "chunk_tc.cu", "backward_simt.cu", "tc_common.cuh", "common.cuh")
# sources of the decode step, the 64-token tensor-core kernel (causal with
# D or Dv = 64; the non-causal sums and read-out with its part scan) and the
# fp32 CUDA-core kernels
DECODE_SOURCES = ("decode.cu", "common.cuh")
CHUNK_TC_SOURCES = ("chunk_tc.cu", "tc_common.cuh", "common.cuh")
NONCAUSAL_SOURCES = ("noncausal_tc.cu", "part_scan.cu", "tc_common.cuh", "common.cuh")
SIMT_SOURCES = ("causal_simt.cu", "common.cuh")
NONCAUSAL_SIMT_SOURCES = ("kv_state_simt.cu", "common.cuh")


def workload_sources(w):
    """The device sources whose hash identifies the timed kernels of ``w``."""
    if w.steps:
        return DECODE_SOURCES
    if w.gated:
        return GATED_SOURCES
    if w.favor_r:
        return FAVOR_SOURCES
    if w.backward:
        return BACKWARD_SOURCES
    fp32 = w.dtype.itemsize == 4
    if not w.causal:
        return NONCAUSAL_SIMT_SOURCES if fp32 else NONCAUSAL_SOURCES
    if fp32:
        return SIMT_SOURCES
    return KERNEL_SOURCES if w.D == 128 and w.Dv == 128 else CHUNK_TC_SOURCES


def ncu_traffic(w, src_hash, final_state=False):
    """The captured DRAM bytes of one launch for ``w``, or None when there is
    no capture, the kernel source has changed since it was taken, or the run
    does extra work (the final-state write) that the capture did not."""
    tr = NCU_TRAFFIC.get(w.name)
    if tr and tr.get("source") == src_hash and not final_state:
        return tr["bytes"]
    return None


def kernel_source_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kernelized_sequence_mixing_gb300", "csrc")
    for name in sources:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    """Median SM clock, maximum SM clock and the throttle reasons seen in
    ``nvidia-smi --format=csv,noheader,nounits`` lines of ClockSampler.FIELDS
    (index, sm, max sm, power, active mask, then one Active/Not Active column
    per reason).  Lines that do not parse are skipped."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, val in zip(names, parts[5:9]):
            if val.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)

def oracle_sample(w, heads_per_pass):
    """A bounded sample of the workload for the fp64 oracle: the first
    `heads_per_pass` (b, h) units, every token."""
    from kernelized_sequence_mixing_gb300.workloads import workload_gates, workload_inputs
    import numpy as np
    q, k, v = workload_inputs(w)
    f = lambda t: t.float().reshape(-1, w.N, t.shape[-1])[:heads_per_pass].numpy()  # noqa: E731
    if w.gated:  # the gates in place of per-head decays
        return f(q), f(k), f(v), f(workload_gates(w))
    if w.favor_r:  # the random directions in place of per-head decays
        from kernelized_sequence_mixing_gb300.workloads import workload_favor_matrix
        return f(q), f(k), f(v), workload_favor_matrix(w).float().numpy()
    if w.backward:  # the upstream gradient in place of per-head decays
        from kernelized_sequence_mixing_gb300.workloads import workload_upstream
        return f(q), f(k), f(v), f(workload_upstream(w))
    g = w.gamma()
    gu = None
    if g is not None:
        gu = np.tile(g.numpy(), w.B)[:heads_per_pass]
    return f(q), f(k), f(v), gu


def time_oracle(w, heads_per_pass, passes):
    import oracle
    qs, ks, vs, gu = oracle_sample(w, heads_per_pass)
    # the C oracle starts at most one thread per unit; the Performer and
    # gradient oracles are numpy, whose BLAS may use every host thread
    threads = oracle.default_threads()
    if not (w.favor_r or w.backward):
        threads = min(threads, qs.shape[0])
    times = []
    for _ in range(passes):
        t0 = time.perf_counter()
        if w.gated:
            oracle.gated(qs, ks, vs, gu, eps=w.eps, nthreads=threads)
        elif w.favor_r:
            from oracle import favor as fv
            fv.favor(qs, ks, vs, gu, causal=True, eps=w.eps)
        elif w.backward:
            from oracle import backward as bw
            for u in range(qs.shape[0]):
                bw.causal_backward(qs[u], ks[u], vs[u], gu[u], None, w.eps)
        elif w.causal:
            oracle.causal(qs, ks, vs, gamma=gu, eps=w.eps, nthreads=threads)
        else:
            oracle.noncausal(qs, ks, vs, eps=w.eps, nthreads=threads)
        times.append(time.perf_counter() - t0)
    # tokens/s of the workload's metric: a token is one position of one
    # sequence across all H heads, so the sample covers heads/H of N tokens.
    tokens = heads_per_pass / w.H * w.N
    return tokens, times, threads


def time_oracle_decode(w, units, passes):
    """The oracle's decode step on the first `units` (sequence, head) units,
    from a zero state (the work per step does not depend on the state); for
    the gated workload, one step of the oracle's gated recurrence."""
    import numpy as np
    import oracle
    from kernelized_sequence_mixing_gb300.workloads import decode_step_inputs
    qt, kt, vt = decode_step_inputs(w, 0)
    f = lambda t: t.float().reshape(-1, t.shape[-1])[:units].numpy()  # noqa: E731
    q, k, v = f(qt), f(kt), f(vt)
    S = np.zeros((units, w.D, w.Dv))
    z = np.zeros((units, w.D))
    threads = min(oracle.default_threads(), units)
    times = []
    if w.gated:
        from kernelized_sequence_mixing_gb300.workloads import decode_step_gates
        ag = decode_step_gates(w, 0).reshape(-1, w.D)[:units].numpy()[:, None, :]
    for _ in range(passes):
        t0 = time.perf_counter()
        if w.gated:
            oracle.gated(q[:, None, :], k[:, None, :], v[:, None, :], ag, eps=w.eps,
                         nthreads=threads)
        else:
            oracle.decode_step(q, k, v, S, z, eps=w.eps, nthreads=threads)
        times.append(time.perf_counter() - t0)
    # a token is one position of one sequence across all H heads
    return units / w.H, times, threads


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    if w.steps:
        heads = min(1024, w.B * w.H)
        for _ in range(args.warmup):
            time_oracle_decode(w, heads, 1)
        tokens, times, threads = time_oracle_decode(w, heads, args.steps)
    else:
        # one unit per host thread (the oracle runs at most one thread per unit)
        import oracle
        heads = max(1, min(oracle.default_threads(), w.B * w.H))
        for _ in range(args.warmup):
            time_oracle(w, heads, 1)
        tokens, times, threads = time_oracle(w, heads, args.steps)
    total = sum(times)
    value = tokens * len(times) / total
    line = {
        "impl": "reference", "metric": workload_metric(w), "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle",
                         "sample": (f"{heads} of {w.B * w.H} (b,h) units, one "
                                    "decode step per step") if w.steps else
                                   (f"{heads} of {w.B * w.H} (b,h) units, all "
                                    f"{w.N} tokens, per step")},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
           "Dv": w.Dv, "causal": w.causal, "global_batch": w.B,
           "seq_len": w.N, "parallelism": "replicas (independent batches)"}
    if w.decayed:
        cfg["gamma"] = "per head 1 - 2^(-5 - h/4)"
    if w.gated:
        cfg["gates"] = (f"fp32 a [B][H][D] per step, uniform in [{w.gate_lo}, 1)" if w.steps else
                        f"fp32 a [B][H][N][D] uniform in [{w.gate_lo}, 1), one per key "
                        "feature and token")
    if w.backward:
        cfg["pass"] = "backward: dq, dk, dv from q, k, v and dL/do ~ N(0, 1)"
    if w.favor_r:
        cfg["features"] = (f"Performer, r = {w.favor_r} block-orthogonal directions; q, k "
                           f"~ N(0, 1) * {w.scale:.4f} (D^-1/4)")
    if w.steps:
        cfg.update(seq_len=1, prefill_len=w.N, state="fp32 S [D][Dv] and z [D] "
                   "per (sequence, head), from the prefill",
                   step=("one la_decode_gated" if w.gated else "one la_decode_step") +
                   " over all B*H units")
    return cfg


# ---------------------------------------------------------------------------
# our arm

def run_ours(args, w):
    import torch
    import kernelized_sequence_mixing_gb300 as la
    from kernelized_sequence_mixing_gb300 import build as labuild
    from kernelized_sequence_mixing_gb300.workloads import make_qkv

    ws, rank, local = dist_env()
    gated_tc = False
    bwd_tc = False
    final_state = bool(getattr(args, "final_state", False))
    if final_state and (w.steps or not w.causal or w.gated or w.favor_r or w.backward):
        raise SystemExit("--final-state applies to the causal forward workloads")
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        labuild.build()
    barrier(ws)
    la.load_library()

    # this rank's replica: an independent batch of the same shape
    g = w.gamma()
    seed = w.seed + 7919 * rank
    if w.steps:
        # decode: the state comes from a prefill of N tokens (not timed);
        # every timed step is one la_decode_step over all B*H units
        from kernelized_sequence_mixing_gb300.workloads import decode_step_inputs
        _, kp, vp = make_qkv(w.B, w.H, w.N, w.D, w.Dv, w.dtype, seed, w.scale)
        S, z = la.prefill_state(kp.to(dev), vp.to(dev), gamma=g)
        del kp, vp
        q, k, v = decode_step_inputs(w, 7919 * rank)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        od = torch.empty((w.B, w.H, w.Dv), dtype=w.dtype, device=dev)
        launches_per_step = 1
        if w.gated:
            # gated: a fresh fp32 gate per key feature; the prefill above is
            # the ungated state (the work of a step does not depend on it)
            from kernelized_sequence_mixing_gb300.workloads import decode_step_gates
            a = decode_step_gates(w, 7919 * rank)
            ad = a.to(dev)

            def step():
                la.decode_gated(qd, kd, vd, ad, S, z, eps=w.eps, out=od)
        else:
            def step():
                la.decode_step(qd, kd, vd, S, z, gamma=g, eps=w.eps, out=od)

        def e2e_step(qh, kh, vh, oh, ah=None):
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            if ah is not None:
                ad.copy_(ah, non_blocking=True)
            step()
            oh.copy_(od, non_blocking=True)
        tokens_rank = w.B
    elif w.gated:
        # gated forward: the state pass and the scan over sequence parts,
        # then the output pass (one launch when the sequence is one part)
        from kernelized_sequence_mixing_gb300.workloads import make_gates
        q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.Dv, w.dtype, seed, w.scale)
        a = make_gates(w.B, w.H, w.N, w.D, seed + 1, w.gate_lo)
        qd, kd, vd, ad = q.to(dev), k.to(dev), v.to(dev), a.to(dev)
        od = torch.empty((w.B, w.H, w.N, w.Dv), dtype=w.dtype, device=dev)
        ncopy = 1
        step_bytes = sum(t.numel() * t.element_size() for t in (qd, kd, vd, ad, od))
        assert step_bytes > L2_BYTES, "gated workloads are sized above L2"
        # the CUDA-core form: three launches whenever the sequence splits into
        # parts, which the library does for every gated workload here (long
        # sequences, fewer (b, h) x Dv-slice CTAs than two per SM); the
        # tensor-core form adds its prep kernel and the causal kernel in
        # front (the CUDA-core launches then return at once unless some
        # chunk forgot too hard)
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        launches_per_step = 3 if w.B * w.H * (w.Dv // 32) < 2 * nsm and w.N > 64 else 1
        gated_tc = la.gated_kernel(w.B, w.H, w.N, w.D, w.Dv, w.dtype) == "tensor-core"
        if gated_tc:
            launches_per_step += 2

        def step():
            la.forward_gated(qd, kd, vd, ad, eps=w.eps, out=od)

        def e2e_step(qh, kh, vh, oh, ah=None):
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            ad.copy_(ah, non_blocking=True)
            step()
            oh.copy_(od, non_blocking=True)
        tokens_rank = w.B * w.N
    elif w.backward:
        # backward: operand preparation, the forward's n and d (one chunked
        # causal product), the middle elementwise kernel, the three gradient
        # products in one launch, the final elementwise kernel
        from kernelized_sequence_mixing_gb300.workloads import workload_upstream
        q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.Dv, w.dtype, seed, w.scale)
        do = workload_upstream(w)
        qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
        grads = (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd))
        od = grads[2]
        ncopy = 1
        launches_per_step = la.backward_launches(w.B, w.H, w.N, w.D, w.Dv, gamma=g, dtype=w.dtype)
        bwd_tc = la.backward_kernel(w.B, w.H, w.N, w.D, w.Dv, gamma=g, dtype=w.dtype) == "tensor-core"

        def step():
            la.backward(qd, kd, vd, dod, eps=w.eps, dq=grads[0], dk=grads[1], dv=grads[2])

        grads_host = []

        def e2e_step(qh, kh, vh, oh, doh=None):
            # all three gradients come back to pinned host memory
            if not grads_host:
                grads_host.extend(torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                                  for t in grads)
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            dod.copy_(doh, non_blocking=True)
            step()
            for hst, dvc in zip(grads_host, grads):
                hst.copy_(dvc, non_blocking=True)
        tokens_rank = w.B * w.N
    elif w.favor_r:
        # Performer: the feature kernel (q and k in one launch), then the
        # causal kernel over the features; the directions stay resident
        from kernelized_sequence_mixing_gb300.workloads import favor_matrix
        q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.Dv, w.dtype, seed, w.scale)
        Wd = favor_matrix(w.favor_r, w.D, w.seed + 2, True, w.dtype).to(dev)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        od = torch.empty((w.B, w.H, w.N, w.Dv), dtype=w.dtype, device=dev)
        ncopy = 1
        launches_per_step = 2

        def step():
            la.forward_favor(qd, kd, vd, Wd, causal=True, eps=w.eps, out=od)

        def e2e_step(qh, kh, vh, oh):
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            step()
            oh.copy_(od, non_blocking=True)
        tokens_rank = w.B * w.N
    else:
        q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.Dv, w.dtype, seed, w.scale)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        od = torch.empty((w.B, w.H, w.N, w.Dv), dtype=w.dtype, device=dev)
        # causal: one chunk kernel (after a small memset of its flags);
        # non-causal: state pass, scan, apply
        launches_per_step = 1 if w.causal else 3
        # a working set that fits in L2 is rotated over enough copies that
        # every step reads its inputs from HBM (no flush needed otherwise)
        step_bytes = sum(t.numel() * t.element_size() for t in (qd, kd, vd, od))
        ncopy = 1 if step_bytes > L2_BYTES else -(-2 * L2_BYTES // step_bytes)
        copies = [(qd, kd, vd, od)] + [
            (qd.clone(), kd.clone(), vd.clone(), torch.empty_like(od))
            for _ in range(ncopy - 1)]
        rot = [0]

        if final_state:
            Sd = torch.empty((w.B, w.H, w.D, w.Dv), dtype=torch.float32, device=dev)
            zd = torch.empty((w.B, w.H, w.D), dtype=torch.float32, device=dev)

            def step():
                qc, kc, vc, oc = copies[rot[0] % ncopy]
                rot[0] += 1
                la.forward_state(qc, kc, vc, gamma=g, eps=w.eps, out=oc, S=Sd, z=zd)

            def e2e_step(qh, kh, vh, oh):
                qd.copy_(qh, non_blocking=True)
                kd.copy_(kh, non_blocking=True)
                vd.copy_(vh, non_blocking=True)
                la.forward_state(qd, kd, vd, gamma=g, eps=w.eps, out=od, S=Sd, z=zd)
                oh.copy_(od, non_blocking=True)
        else:
            def step():
                qc, kc, vc, oc = copies[rot[0] % ncopy]
                rot[0] += 1
                la.forward(qc, kc, vc, causal=w.causal, gamma=g, eps=w.eps, out=oc)

            def e2e_step(qh, kh, vh, oh):
                la.forward(qh, kh, vh, causal=w.causal, gamma=g, eps=w.eps, out=oh)
        tokens_rank = w.B * w.N
    stream = torch.cuda.current_stream(dev)
    if w.steps:
        ncopy = 1

    # a bounded device wait that gave up leaves its CTA's output incomplete
    # (and the launch faster): the count is checked after the timed work
    torch.cuda.synchronize(dev)
    la.device_wait_timeouts(reset=True)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    roll = 0.0 if args.quick else 0.5
    if not args.quick:
        sampler.start()
    # keep the GPU under the same load before and after the timed region so
    # the clock sampler sees it even when the timed region is short
    t_end = time.perf_counter() + roll
    while time.perf_counter() < t_end:
        step()
        torch.cuda.synchronize(dev)

    barrier(ws)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    per_launch = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms = ev[0].elapsed_time(ev[-1]) / args.steps

    t_end = time.perf_counter() + roll
    while time.perf_counter() < t_end:
        step()
        torch.cuda.synchronize(dev)
    clocks = sampler.stop() if not args.quick else None

    ms_max = reduce_max(ms, ws)
    value = aggregate(ms_max, tokens_rank, ws)

    # end to end through the public API with host buffers: pinned inputs
    # copied in, result copied out, every step
    e2e_s = None
    if not args.quick:
        qh, kh, vh = (t.pin_memory() for t in (q, k, v))
        oh = torch.empty(od.shape, dtype=od.dtype, pin_memory=True)
        extra = ({"ah": a.pin_memory()} if w.gated else
                 {"doh": do.pin_memory()} if w.backward else {})
        e2e_step(qh, kh, vh, oh, **extra)
        torch.cuda.synchronize(dev)
        e2e_steps = max(1, min(args.steps, 10))
        barrier(ws)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step(qh, kh, vh, oh, **extra)
        torch.cuda.synchronize(dev)
        e2e_s = reduce_max((time.perf_counter() - t0) / e2e_steps, ws)
    es = q.element_size()
    h2d = (q.numel() + k.numel() + v.numel()) * es + (a.numel() * 4 if w.gated else 0) + (
        do.numel() * es if w.backward else 0)
    d2h = (sum(t.numel() for t in grads) if w.backward else od.numel()) * es

    torch.cuda.synchronize(dev)
    gave_up = la.device_wait_timeouts(reset=True)
    if gave_up:
        print(json.dumps({"metric": workload_metric(w), "invalid":
                          f"{gave_up} bounded device wait(s) gave up during the run; "
                          "the timed outputs are incomplete"}), flush=True)
        return 1
    if rank != 0:
        return 0

    hbm_peak, tc_peak, peak_src = measured_peaks()
    extra = None
    if ws == 1 and w.name == DEFAULT_WORKLOAD and not args.no_extra:
        extra = {}
        for name in EXTRA_WORKLOADS:
            extra[name] = time_extra(la, name, dev, hbm_peak, args.quick)
            torch.cuda.empty_cache()
        torch.cuda.synchronize(dev)
        gave_up = la.device_wait_timeouts(reset=True)
        if gave_up:
            print(json.dumps({"metric": workload_metric(w), "invalid":
                              f"{gave_up} bounded device wait(s) gave up in the other "
                              "configurations; their outputs are incomplete"}), flush=True)
            return 1
    byts, flops = decode_work(w) if w.steps else algorithmic_work(w)
    if final_state:  # the state written once at the end, fp32
        byts += w.B * w.H * (w.D * w.Dv + w.D) * 4
    launch_ms = statistics.mean(per_launch)  # the whole step's launches
    achieved_gbs = byts / (launch_ms / 1e3) / 1e9
    src_hash = kernel_source_hash(workload_sources(w))
    traffic = ncu_traffic(w, src_hash, final_state)

    # CPU baseline: the fp64 oracle on the host cores, one pass over a bounded
    # sample (all 32 heads of the default workload, ~20 s of CPU work)
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        if w.steps:
            heads = min(w.B * w.H, 2048)
            tokens, times, threads = time_oracle_decode(w, heads, 3)
            t = min(times)
            sample = (f"{heads} of {w.B * w.H} (sequence, head) units, one decode "
                      f"step, best of 3 ({t:.2f} s wall)")
        else:
            # the quadratic gradient oracle is O(N^2) per unit: 4 units
            heads = min(w.B * w.H, 4 if w.backward else 32)
            tokens, times, threads = time_oracle(w, heads, 1)
            t = times[0]
            sample = (f"{heads} of {w.B * w.H} (b,h) units, all {w.N} "
                      f"tokens, one pass ({t:.1f} s wall)")
        cpu = {"value": tokens / t, "unit": "tokens/s", "cores": threads,
               "kind": "oracle", "sample": sample}

    line = {
        "metric": workload_metric(w), "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": compute_dtype(w, gated_tc, bwd_tc),
        "data": "synthetic",
        "config": dict(workload_config(w), **({"final_state": "S [B][H][D][Dv] and z [B][H][D] "
                                               "fp32 written after the last token"}
                                              if final_state else {}),
                       l2=(f"working set larger than L2 ({byts / 1e6:.0f} MB "
                           "read and written per step), no flush")
                       if w.steps or ncopy == 1 else
                          (f"working set {byts / 1e6:.0f} MB < L2: steps rotate "
                           f"over {ncopy} input/output copies")),
        "roofline": roofline_entry(w, byts, flops, launch_ms, hbm_peak, peak_src,
                                   tc_peak, traffic, launches_per_step,
                                   gated_tc=bool(w.gated and gated_tc), bwd_tc=bwd_tc),
        "cpu_baseline": cpu,
        "e2e": None if e2e_s is None else {
            "value": tokens_rank * ws / e2e_s, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "kernel_source": src_hash,
    }
    if extra is not None:
        line["workloads"] = extra
    print(json.dumps(line), flush=True)
    return 0


def device_inputs(w, gen, dev, N=None):
    """q, k, v of workload ``w`` drawn on the device (N(0, 1) times the
    workload's scale, rounded once to its dtype) from a seeded CUDA
    generator: the shapes and distribution of the workload's recipe, for
    timing only (the parity tests use the CPU recipe itself)."""
    import torch
    N = w.N if N is None else N
    out = []
    for width in (w.D, w.D, w.Dv):
        t = torch.randn((w.B, w.H, N, width), generator=gen, device=dev, dtype=torch.float32)
        out.append((t * w.scale).to(w.dtype))
    return out


def time_extra(la, name, dev, hbm_peak, quick):
    """Time one more configuration in this process: warm-up, then CUDA events
    around each step on the launching stream; clocks sampled around it.
    Forward configurations run ``steps`` forward passes (rotating input
    copies when the working set fits in L2), captured once in a CUDA graph
    and replayed, so that a short step measures the GPU's work rather than
    the host's call overhead; the decode configuration runs its whole loop
    of single-token steps, each with fresh inputs, as plain launches (each
    step is long enough to hide the host)."""
    import torch
    from kernelized_sequence_mixing_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    stream = torch.cuda.current_stream(dev)
    gated_tc = bwd_tc = False  # the tensor-core forms, where the workload has one
    if w.steps:
        _, kp, vp = device_inputs(w, gen, dev)
        S, z = la.prefill_state(kp, vp, gamma=w.gamma())
        del kp, vp
        steps_in = [device_inputs(w, gen, dev, N=1) for _ in range(w.steps)]
        steps_in = [tuple(t[:, :, 0].contiguous() for t in x) for x in steps_in]
        od = torch.empty((w.B, w.H, w.Dv), dtype=w.dtype, device=dev)
        S0, z0 = S.clone(), z.clone()

        def run(i):
            qd, kd, vd = steps_in[i % w.steps]
            la.decode_step(qd, kd, vd, S, z, eps=w.eps, out=od)
        nsteps, warm = w.steps, 3
        byts, flops = decode_work(w)
        tokens = w.B
    else:
        q, k, v = device_inputs(w, gen, dev)
        od = torch.empty((w.B, w.H, w.N, w.Dv), dtype=w.dtype, device=dev)
        # the gated forward's fp32 gates U[gate_lo, 1), the Performer's
        # directions, the backward's upstream gradient N(0, 1) and its
        # three gradients
        extra = []
        if w.gated:
            extra = [torch.rand((w.B, w.H, w.N, w.D), generator=gen, device=dev) * (1.0 - w.gate_lo)
                     + w.gate_lo]
            gated_tc = la.gated_kernel(w.B, w.H, w.N, w.D, w.Dv, w.dtype) == "tensor-core"
        elif w.backward:
            extra = [torch.randn((w.B, w.H, w.N, w.Dv), generator=gen, device=dev).to(w.dtype),
                     torch.empty_like(q), torch.empty_like(k)]
            bwd_tc = la.backward_kernel(w.B, w.H, w.N, w.D, w.Dv, dtype=w.dtype) == "tensor-core"
        if w.favor_r:
            from kernelized_sequence_mixing_gb300.workloads import favor_matrix
            Wd = favor_matrix(w.favor_r, w.D, w.seed + 2, True, w.dtype).to(dev)
        step_bytes = sum(t.numel() * t.element_size() for t in [q, k, v, od] + extra)
        ncopy = 1 if step_bytes > L2_BYTES else -(-2 * L2_BYTES // step_bytes)
        copies = [[q, k, v, od] + extra] + [[t.clone() for t in [q, k, v, od] + extra]
                                            for _ in range(ncopy - 1)]

        def run(i):
            c = copies[i % ncopy]
            if w.gated:
                la.forward_gated(c[0], c[1], c[2], c[4], eps=w.eps, out=c[3])
            elif w.favor_r:
                la.forward_favor(c[0], c[1], c[2], Wd, causal=w.causal, eps=w.eps, out=c[3])
            elif w.backward:
                la.backward(c[0], c[1], c[2], c[4], eps=w.eps, dq=c[5], dk=c[6], dv=c[3])
            else:
                la.forward(c[0], c[1], c[2], causal=w.causal, gamma=w.gamma(), eps=w.eps, out=c[3])
        nsteps = 20 if w.N * w.B * w.H >= (1 << 22) else 100
        warm = 5
        byts, flops = algorithmic_work(w)
        tokens = w.B * w.N
    for i in range(warm):
        run(i)
    torch.cuda.synchronize(dev)
    graph = None
    if not w.steps:
        # one graph over a whole rotation of the input copies (at least
        # `nsteps` launches); replayed until nsteps steps have run
        per_graph = ncopy * max(1, -(-nsteps // ncopy)) if ncopy < nsteps else ncopy
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(per_graph):
                    run(i)
            graph.replay()
            torch.cuda.synchronize(dev)
            nsteps = per_graph
        except RuntimeError:
            graph = None
            torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    roll = 0.0 if quick else 0.5
    if not quick:
        sampler.start()
    t_end = time.perf_counter() + roll
    i = 0
    while time.perf_counter() < t_end:
        run(i)
        i += 1
        torch.cuda.synchronize(dev)
    if w.steps:  # the decode loop starts from the prefill state
        S.copy_(S0)
        z.copy_(z0)
        torch.cuda.synchronize(dev)
    if graph is not None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        total = e0.elapsed_time(e1)
        per = [total / nsteps]
    else:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps + 1)]
        ev[0].record(stream)
        for i in range(nsteps):
            run(i)
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(nsteps)]
        total = ev[0].elapsed_time(ev[-1])
    t_end = time.perf_counter() + roll
    i = 0
    while time.perf_counter() < t_end:
        run(i)
        i += 1
        torch.cuda.synchronize(dev)
    clocks = sampler.stop() if not quick else None
    ms = total / nsteps
    gbs = byts / (ms / 1e3) / 1e9
    entry = {"ms_per_step": ms, "value": tokens / (ms / 1e3), "unit": "tokens/s",
             "steps": nsteps, "dtype": compute_dtype(w, gated_tc, bwd_tc),
             "config": workload_config(w),
             "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                          "frac": gbs / hbm_peak, "algorithmic_bytes": byts,
                          "tflops": flops / (ms / 1e3) / 1e12},
             "clocks": clocks,
             "timing": ("one CUDA graph of the steps, replayed between two events" if graph is not None
                        else "CUDA events around each plain launch"),
             "inputs": "device-drawn from a seeded CUDA generator, same shapes and N(0,1) x "
                       f"{w.scale} distribution as the recipe"}
    if w.steps:
        med = statistics.median(per)
        entry.update(ms_per_step_median=med, ms_total=total,
                     note=f"{nsteps} single-token steps over all {w.B}x{w.H} units, fresh "
                          f"inputs per step, from a {w.N}-token prefill state")
        entry["roofline"]["frac_median_step"] = byts / (med / 1e3) / 1e9 / hbm_peak
    else:
        entry["l2"] = ("working set larger than L2, no flush" if ncopy == 1 else
                       f"working set below L2: steps rotate over {ncopy} input/output copies")
    return entry


def compute_dtype(w, gated_tc=False, bwd_tc=False):
    """The arithmetic type the timed path computes in: bf16 tensor-core
    operands (fp32 accumulation) for the bf16 forward kernels and the
    tensor-core backward, fp32 for the CUDA-core paths (fp32 inputs, the
    decode steps' fp32 state update, the CUDA-core gated form and backward)."""
    if w.backward:
        return "bf16" if bwd_tc else "f32"
    if w.steps:
        return "f32"
    if w.gated and not gated_tc:
        return "f32"
    return "bf16" if w.dtype.itemsize == 2 else "f32"


def roofline_entry(w, byts, flops, launch_ms, hbm_peak, peak_src, tc_peak, traffic,
                   launches, gated_tc=False, bwd_tc=False):
    """HBM roofline for the forward, decode and tensor-core backward kernels;
    for the gated and backward CUDA-core kernels, the fp32 ALU roofline
    (their bound), with the HBM figure beside it.  Timed over the whole step
    (all of its launches)."""
    achieved_gbs = byts / (launch_ms / 1e3) / 1e9
    tflops = flops / (launch_ms / 1e3) / 1e12
    hbm_src = (f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
               else "fallback")
    if (w.gated and not w.steps and not gated_tc) or (w.backward and not bwd_tc):
        return {"bound": "alu", "achieved": tflops, "peak": ALU_FP32_TFLOPS,
                "unit": "TFLOP/s", "frac": tflops / ALU_FP32_TFLOPS, "traffic": traffic,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                "algorithmic_flops": flops, "algorithmic_bytes": byts,
                "hbm_achieved_gbs": achieved_gbs, "hbm_frac": achieved_gbs / hbm_peak,
                "hbm_peak_source": hbm_src, "launches_per_step": launches}
    return {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved_gbs / hbm_peak, "traffic": traffic, "peak_source": hbm_src,
            "algorithmic_bytes": byts, "tflops": tflops, "tensor_peak_tflops": tc_peak}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--final-state", action="store_true",
                    help="causal workloads: time la_forward_state (the forward "
                         "plus the state after the last token) instead")
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload only: skip timing the other "
                         "configurations reported under 'workloads'")
    ap.add_argument("--quick", action="store_true",
                    help="skip the clock-sampling window and the end-to-end "
                         "leg (few launches, for profiler runs)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    from kernelized_sequence_mixing_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
