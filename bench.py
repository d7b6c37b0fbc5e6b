"""Benchmark of the multi-LoRA path (metadata + shrink + expand) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the fp64 CPU oracle, timed

One step = one pass of the whole path over one batch: metadata, shrink and
expand through the C ABI (lora_linear), or metadata and the expand of a
bf16 input for the embedding workload, on inputs already resident in HBM.
Input sets (ids, x, A, B, bias, y, buffer) are replicated until they total
at least 4x the L2 cache, and consecutive steps rotate through them, so
every step reads from HBM.  Steps are captured in CUDA graphs (one graph per
rotation).

With no --workload the headline is the large workload (16384 tokens,
hidden 8192, rank 128, three slices: the largest configuration): W warm-up
steps, then exactly K steps timed with CUDA events between a barrier +
synchronize on both sides, clocks sampled meanwhile; then the end-to-end
figure through the public API with host copies, and each kernel alone.
Every other workload of the layer (tiny, decode, prefill, mlp, the all -1
batch) is then timed the same way, step and kernels, and reported under
per_workload.  Rank 0 prints one JSON line.  N > 1 (torchrun) runs
independent replicas, one per GPU, and reports the aggregate over ranks
with the max time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "LoRA shrink+expand tokens/s and effective HBM GB/s (% of roofline), 1 GB300"
FALLBACK_HBM_GBS = 6800.0
E2E_GRAPH_STEPS = 8

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum of an
# ncu capture of the bench command), keyed by (kernel, workload), with the
# hash of the kernel's sources the capture was taken on; a stale hash
# reports null.
NCU_TRAFFIC = {
    # expand_tc_kernel<8, 0> and shrink_umma_kernel, one launch each at full
    # size (dram__bytes_read.sum + dram__bytes_write.sum, one single-pass capture)
    ("expand", "large"): ("efc2bfc911fdb557", 664651776),
    ("shrink", "large"): ("960e6f1709e55feb", 450486272),
    # linear_tc_kernel<0>, the step's kernel after the metadata kernel
    ("linear_tc", "large"): ("530c5a60b03f1ca4", 1117510400),
}

# The source files each reported kernel is built from.
KERNEL_SOURCES = {
    "expand": ("lora_expand.cu", "lora_expand.cuh", "lora_expand_tc.cu", "lora_umma.cuh",
               "lora_common.cuh"),
    "shrink": ("lora_shrink.cu", "lora_shrink_umma.cu", "lora_umma.cuh", "lora_common.cuh"),
    "linear_coop": ("lora_linear_coop.cu", "lora_expand.cuh", "lora_common.cuh"),
    "linear_fused": ("lora_fused.cu", "lora_common.cuh"),
    "linear_tc": ("lora_linear_tc.cu", "lora_umma.cuh", "lora_common.cuh"),
}


def _src_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "expand_gemm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


HEADLINE = "large"
# Workloads of one LoRA layer timed by a default run: the headline first,
# then the rest (each reported under per_workload).
LAYER_WORKLOADS = ["large", "tiny", "decode", "prefill", "mlp", "none"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(W.WORKLOADS),
                    help="time this workload alone (default: the large workload as the "
                         "headline, then every other workload of the layer)")
    ap.add_argument("--num-tokens", type=int, default=None,
                    help="a smaller case of the workload (profiling captures)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--kernel-seconds", type=float, default=0.25,
                    help="minimum timed seconds per kernel in the per-kernel loops")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args(argv)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured hbm_gbs (burst copy, MEASURED_PEAKS.json)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def _padded_rank(r: int) -> int:
    rp = 16
    while rp < r:
        rp *= 2
    return rp


def coop_path(w) -> bool:
    """lora_linear's rule for its single cooperative kernel (lora_linear_coop.cu)."""
    mode = os.environ.get("LORA_PUNICA_COOP", "")
    wanted = mode == "1" or (mode != "0" and w.num_tokens * w.num_slices <= 256)
    return (wanted and 1 <= w.num_tokens <= 512 and w.max_loras <= 256 and w.rank <= 64
            and w.hidden % 8 == 0)


def fused_path(w) -> bool:
    """lora_linear's rule for its single fused kernel (include/lora_punica.h)."""
    if coop_path(w):
        return False
    mode = os.environ.get("LORA_PUNICA_FUSED", "")
    limit = 512 if mode == "1" else int(os.environ.get("LORA_PUNICA_FUSED_MAX_TOKENS", "128"))
    return (w.num_tokens <= limit and w.max_loras <= 256 and _padded_rank(w.rank) <= 64
            and w.num_slices * _padded_rank(w.rank) <= 128 and mode != "0")


def linear_tc_path(w, sms: int = 152) -> bool:
    """lora_linear's rule for its rank-128 tensor-core kernel (metadata
    kernel + one kernel for the shrink and expand of every tile) on a GPU of
    `sms` SMs."""
    if coop_path(w) or fused_path(w) or w.kind == "embedding":
        return False
    mode = os.environ.get("LORA_PUNICA_LINEAR_TC", "-1")
    min_t = int(os.environ.get("LORA_PUNICA_LINEAR_TC_MIN_TOKENS", "0")) or 72 * sms
    return (mode != "0" and (mode == "1" or w.num_tokens >= min_t) and w.rank == 128
            and w.num_slices <= 3 and all(n % 64 == 0 for n in w.slices)
            and w.hidden >= 64 and w.hidden % 8 == 0)


def umma_shrink_path(w) -> bool:
    """lora_shrink's rule for taking its tensor-core kernel (which covers the
    whole batch, or only the whole tiles with LORA_PUNICA_UMMA_PARTIAL=0, the
    remainders then on the mma.sync kernel)."""
    return (w.num_tokens >= int(os.environ.get("LORA_PUNICA_UMMA_MIN_TOKENS", "1024"))
            and w.num_slices * w.rank >= int(os.environ.get("LORA_PUNICA_UMMA_MIN_COLS", "256"))
            and os.environ.get("LORA_PUNICA_UMMA", "1") != "0")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is under load."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.uuid = gpu_uuid
        self.rows = []
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            cmd = ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
        self.file.close()
        self.proc = None

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------ multi-rank host logic

def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest `value` over all ranks (the timed region of the slowest
    replica); the value itself when there is no process group."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the step, so
    the job processes world x tokens per step in the slowest rank's time."""
    return world * tokens_per_step * steps / (elapsed_ms / 1e3)


# ------------------------------------------------------------ GPU arm

class DeviceSet:
    """One resident copy of a workload's inputs and outputs."""

    def __init__(self, inp: W.Inputs, dev, eg):
        import torch
        w = inp.workload

        def bf16(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
                torch.bfloat16).to(dev)
        self.ids = torch.from_numpy(inp.ids).to(dev)
        self.x = bf16(inp.x)
        self.A = [bf16(a) for a in inp.lora_a]
        self.B = [bf16(b) for b in inp.lora_b]
        self.bias = None if inp.lora_bias is None else [bf16(b) for b in inp.lora_bias]
        self.y = bf16(inp.y)
        self.buf = torch.zeros(inp.buf.shape, dtype=torch.float32, device=dev)
        self.meta = eg.LoRAKernelMeta.make(w.max_loras, w.num_tokens, dev)
        self.nbytes = sum(t.numel() * t.element_size() for t in
                          [self.ids, self.x, self.y, self.buf] + self.A + self.B
                          + (self.bias or []))

    def clone(self, eg):
        import torch
        c = object.__new__(DeviceSet)
        c.ids = self.ids.clone()
        c.x = self.x.clone()
        c.A = [a.clone() for a in self.A]
        c.B = [b.clone() for b in self.B]
        c.bias = None if self.bias is None else [b.clone() for b in self.bias]
        c.y = self.y.clone()
        c.buf = torch.zeros_like(self.buf)
        c.meta = eg.LoRAKernelMeta.make(self.meta.max_loras, self.meta.max_num_tokens,
                                        self.meta.device)
        c.nbytes = self.nbytes
        return c


def _workload(name, args):
    w = W.WORKLOADS[name]
    if args.num_tokens is not None:
        from dataclasses import replace
        w = replace(w, num_tokens=args.num_tokens, n_decode=min(w.n_decode, args.num_tokens))
    return w


class Measured:
    """One workload measured on the GPU: the step timed over a rotation of
    resident input sets, then each kernel alone."""

    def __init__(self, name, args, dev, eg, stream, props, dist, headline, clocks):
        import torch
        w = _workload(name, args)
        inp = W.generate(w)
        ub = W.unique_bytes(w, inp.ids)
        l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
        base = DeviceSet(inp, dev, eg)
        n_sets = max(2, -(-4 * l2 // base.nbytes))
        sets = [base] + [base.clone(eg) for _ in range(n_sets - 1)]
        emb = w.kind == "embedding"

        def step(s: DeviceSet):
            if emb:
                # metadata + expand of the looked-up bf16 rows (embedding LoRA)
                s.meta.prepare_tensors(s.ids)
                eg.add_lora_embedding(s.y, s.x, s.B[0], s.meta, w.add_inputs)
            else:
                # metadata + shrink + expand of one layer (or of the logits):
                # one C-ABI call (one kernel for small batches, three otherwise)
                eg.lora_linear(s.ids, s.x, s.A, s.B, s.bias, w.scale, s.buf, s.y, s.meta)

        # eager pass first: configures kernels (smem attributes, occupancy) before capture
        with torch.cuda.stream(stream):
            for s in sets:
                step(s)
        torch.cuda.synchronize(dev)

        def capture(fn_list):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for fn in fn_list:
                    fn()
            return g

        def graphs_for(n_steps, make):
            """Graphs covering exactly n_steps steps: full rotations + a tail."""
            rot = capture([make(s) for s in sets])
            tail_n = n_steps % n_sets
            tail = capture([make(s) for s in sets[:tail_n]]) if tail_n else None
            return [rot] * (n_steps // n_sets) + ([tail] if tail else [])

        def mk_step(s):
            return lambda: step(s)

        def time_kernel(make, min_s):
            """ms per call of make(s)'s work: graphs of one rotation, replayed
            (after at least three warm-up calls) until min_s seconds pass."""
            g = capture([make(s) for s in sets])
            with torch.cuda.stream(stream):
                for _ in range(-(-3 // n_sets)):
                    g.replay()
            torch.cuda.synchronize(dev)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            reps = 1
            while True:
                with torch.cuda.stream(stream):
                    a.record(stream)
                    for _ in range(reps):
                        g.replay()
                    b.record(stream)
                torch.cuda.synchronize(dev)
                ms = a.elapsed_time(b)
                if ms >= min_s * 1e3 or reps >= 1 << 16:
                    return ms / (reps * n_sets)
                reps *= 2 if ms <= 0 else max(2, min(16, int(min_s * 1e3 / ms) + 1))

        self.elapsed_ms = None
        self.wall = None
        if headline:
            # exactly K timed steps after W warm-up steps, barrier + synchronize
            # on both sides, clocks sampled meanwhile
            warm = graphs_for(args.warmup, mk_step)
            timed = graphs_for(args.steps, mk_step)
            with torch.cuda.stream(stream):
                for g in warm:
                    g.replay()
            torch.cuda.synchronize(dev)
            clocks.start()
            time.sleep(0.3)
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            if dist:
                dist.barrier()
            torch.cuda.synchronize(dev)
            t_wall = time.perf_counter()
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for g in timed:
                    g.replay()
                ev1.record(stream)
            torch.cuda.synchronize(dev)
            self.wall = time.perf_counter() - t_wall
            if dist:
                dist.barrier()
            self.elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)

        ks = args.kernel_seconds
        k_step = time_kernel(mk_step, ks)
        k_meta = time_kernel(lambda s: (lambda: s.meta.prepare_tensors(s.ids)), ks)
        if emb:
            k_shrink = 0.0
            k_expand = time_kernel(lambda s: (lambda: eg.lora_expand(
                s.x.unsqueeze(0), s.B, s.y, s.meta, w.offset_start, w.add_inputs, s.bias)), ks)
        else:
            k_shrink = time_kernel(lambda s: (lambda: eg.lora_shrink(s.x, s.A, s.buf, s.meta,
                                                                     w.scale)), ks)
            k_expand = time_kernel(lambda s: (lambda: eg.lora_expand(
                s.buf, s.B, s.y, s.meta, w.offset_start, w.add_inputs, s.bias)), ks)
        if headline:
            clocks.stop()
        self.w, self.inp, self.ub, self.emb, self.step = w, inp, ub, emb, step
        self.n_sets, self.set_bytes, self.l2 = n_sets, base.nbytes, l2
        self.k = {"meta": k_meta, "shrink": k_shrink, "expand": k_expand, "step": k_step}
        self.coop = coop_path(w) and not emb
        self.fused = (fused_path(w) and not emb) or self.coop
        self.linear_tc = linear_tc_path(w, props.multi_processor_count) and not self.fused
        self.launches_per_step = (2 if emb or self.linear_tc else 1 if self.fused else 3 + (
            1 if umma_shrink_path(w) and os.environ.get("LORA_PUNICA_UMMA_PARTIAL", "1") == "0"
            else 0))
        del sets, base
        torch.cuda.synchronize(dev)

    def path(self):
        if self.emb:
            return "metadata + expand of a bf16 input (add_lora_embedding): two kernels"
        return "lora_linear (metadata + shrink + expand): %s" % (
            "one cooperative kernel" if self.coop else
            "one fused cluster kernel" if self.fused else
            "metadata kernel + one tensor-core shrink/expand kernel" if self.linear_tc else
            "three kernels")

    def summary(self, args, step_ms=None):
        """The workload's figures: the step and each kernel, with the
        dominant kernel's roofline.  step_ms: the step time to report (the
        exact-K timed region for the headline; else the per-kernel loop's)."""
        w, ub, k = self.w, self.ub, self.k
        step_ms = k["step"] if step_ms is None else step_ms
        hbm, peak_src = peaks()
        step_bytes = ub["shrink"] + ub["expand"]
        if self.coop:
            # the whole step is one kernel: its bytes are the step's bytes
            dominant, dom_bytes, dom_ms = "linear_coop", step_bytes, k["step"]
        elif self.fused:
            dominant, dom_bytes, dom_ms = "linear_fused", step_bytes, k["step"]
        elif self.linear_tc:
            # the step is the metadata kernel + this one: its time is the
            # step's less the metadata kernel's, both timed the same way; its
            # bytes are the shrink's and the expand's without the expand's
            # re-read of the buffer (the tile's rows stay on chip)
            dominant, dom_bytes = "linear_tc", ub["linear"]
            dom_ms = k["step"] - k["meta"]
        else:
            dominant = "expand" if k["expand"] >= k["shrink"] else "shrink"
            dom_bytes, dom_ms = ub[dominant], k[dominant]
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
        tr = NCU_TRAFFIC.get((dominant, w.name))
        traffic = tr[1] if (tr and tr[0] == _src_hash(dominant)
                            and args.num_tokens is None) else None
        kern_us = {"meta": k["meta"] * 1e3, "shrink": k["shrink"] * 1e3,
                   "expand": k["expand"] * 1e3,
                   ("embedding_step" if self.emb else "lora_linear"): k["step"] * 1e3}
        if self.emb:
            del kern_us["shrink"]
        step_gbps = step_bytes / (step_ms * 1e-3) / 1e9
        return {
            "workload": w.name,
            "step": self.path(),
            "num_tokens": w.num_tokens, "active_tokens": ub["t_active"],
            "distinct_loras": ub["distinct"],
            "step_us": step_ms * 1e3,
            "tokens_per_s": w.num_tokens / (step_ms * 1e-3),
            "step_unique_bytes": step_bytes,
            "step_gbps": step_gbps,
            "step_frac": step_gbps / hbm,
            # the metric's other reading: tokens over the shrink and expand
            # kernels' standalone times, metadata (once per forward) left out
            "tokens_per_s_shrink_expand": (w.num_tokens / ((k["shrink"] + k["expand"]) * 1e-3)
                                           if k["shrink"] + k["expand"] > 0 else None),
            "kernels_us": kern_us,
            "kernels_gbps": {
                "shrink": (ub["shrink"] / (k["shrink"] * 1e-3) / 1e9
                           if k["shrink"] and ub["shrink"] else None),
                "expand": ub["expand"] / (k["expand"] * 1e-3) / 1e9 if ub["expand"] else None},
            "kernels_frac": {
                "shrink": (ub["shrink"] / (k["shrink"] * 1e-3) / 1e9 / hbm
                           if k["shrink"] and ub["shrink"] else None),
                "expand": (ub["expand"] / (k["expand"] * 1e-3) / 1e9 / hbm
                           if ub["expand"] else None)},
            "roofline": {
                "bound": "hbm", "kernel": "lora_" + dominant,
                "note": ("single kernel: algorithmic bytes of shrink + expand per launch"
                         if self.fused else
                         "shrink + expand kernel (the buffer read once, written once); "
                         "launch time = step - metadata kernel" if self.linear_tc else
                         "the step's longest kernel"),
                "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic,
                "algorithmic_bytes_per_launch": dom_bytes,
                "launch_us": dom_ms * 1e3,
                "peak_source": peak_src + " (of measured)" if "measured" in peak_src
                else peak_src,
            },
            "l2": "inputs larger than L2: %d resident input sets of %.1f MB rotated "
                  "(%.0f MB total, L2 %.0f MB)" % (self.n_sets, self.set_bytes / 1e6,
                                                   self.n_sets * self.set_bytes / 1e6,
                                                   self.l2 / 1e6),
        }


def run_ours(args, rank, world):
    import torch
    import expand_gemm_gb300 as eg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    eg.library()                                        # fail loudly if not built
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    props = torch.cuda.get_device_properties(dev)
    gpu_uuid = getattr(props, "uuid", None)
    gpu_uuid = ("GPU-" + str(gpu_uuid)) if gpu_uuid is not None else None
    clocks = ClockSampler(gpu_uuid)
    stream = torch.cuda.Stream(dev)

    names = [args.workload] if args.workload else LAYER_WORKLOADS
    head = Measured(names[0], args, dev, eg, stream, props, dist, True, clocks)
    w, inp = head.w, head.inp
    # ---- end to end through the public API, host buffers, copies timed
    e2e = None if args.no_e2e else run_e2e(args, inp, w, dev, eg, stream, head.step)
    torch.cuda.empty_cache()
    per = {}
    for name in names[1:]:
        m = Measured(name, args, dev, eg, stream, props, None, False, clocks)
        per[name] = m.summary(args)
        del m
        torch.cuda.empty_cache()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None

    T = w.num_tokens
    ms_per_step = head.elapsed_ms / args.steps
    value = job_tokens_per_s(world, T, args.steps, head.elapsed_ms)
    hs = head.summary(args, step_ms=ms_per_step)
    per = {names[0]: hs, **per}
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; no dataset or weights)",
        "config": {
            **workload_config(w, head.ub, args),
            "l2": hs["l2"],
            "timing": "CUDA graphs of one rotation of steps, CUDA events on the launch stream",
            "step": head.path(),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "tokens_per_s_shrink_expand": hs["tokens_per_s_shrink_expand"],
        "effective_gbps": hs["step_gbps"],
        "step_unique_bytes": hs["step_unique_bytes"],
        "hbm_frac_step": hs["step_frac"],
        "kernels_us": hs["kernels_us"],
        "kernels_gbps": hs["kernels_gbps"],
        "roofline": hs["roofline"],
        "gpu_launches": args.steps * head.launches_per_step,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "wall_s_timed": head.wall,
        "per_workload": per,
    }
    # the oracle's CPU baseline is timed at N = 1 only
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(w, inp, target_s=10.0)
    if dist:
        dist.destroy_process_group()
    return out


def run_e2e(args, inp, w, dev, eg, stream, step):
    """Same step through the public API from pinned host buffers: every
    step's H2D of its ids, x and y, the step's calls, and the D2H of its y,
    all inside the timed region.  Steps are pipelined as a serving loop
    would run them: two device buffer sets, the copies in on one stream,
    the step on another, the read-back on a third, so that step i's copies
    overlap step i - 1's compute and step i - 2's read-back.  The pipeline
    of E2E_GRAPH_STEPS steps is captured in one CUDA graph (copies as
    memcpy nodes), so the host's issue rate does not set the pace."""
    import torch
    ids_h = torch.from_numpy(inp.ids).pin_memory()
    x_h = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).pin_memory()
    y_h = torch.from_numpy(np.ascontiguousarray(inp.y).view(np.int16)).pin_memory()
    outs_h = [torch.empty_like(y_h).pin_memory() for _ in range(2)]
    sets = [DeviceSet(inp, dev, eg) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def one(i):
        b = i % 2
        s = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_free[b])          # step i - 2 has read this set back
            s.ids.copy_(ids_h, non_blocking=True)
            s.x.view(torch.int16).copy_(x_h, non_blocking=True)
            s.y.view(torch.int16).copy_(y_h, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[b])
            step(s)
            ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            outs_h[b].copy_(s.y.view(torch.int16), non_blocking=True)
            ev_free[b].record(s_out)

    side = (s_in, s_out)

    def pipeline():
        for t in side:
            t.wait_stream(stream)
        for i in range(E2E_GRAPH_STEPS):
            one(i)
        for t in side:
            stream.wait_stream(t)

    with torch.cuda.stream(stream):
        pipeline()                                   # eager pass: kernels configured
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pipeline()
    reps = max(1, -(-max(3, args.e2e_steps) // E2E_GRAPH_STEPS))
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    n = reps * E2E_GRAPH_STEPS
    ms = a.elapsed_time(b) / n
    h2d = ids_h.numel() * 4 + x_h.numel() * 2 + y_h.numel() * 2
    return {"value": w.num_tokens / (ms * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": outs_h[0].numel() * 2,
            "ms_per_step": ms, "steps": n,
            "pipeline": "two buffer sets; H2D, step and D2H on three streams; CUDA graph "
                        "of %d steps" % E2E_GRAPH_STEPS}


# ------------------------------------------------------ oracle (CPU) arm

def _oracle_step(oracle, w, inp, sel):
    """One oracle pass: metadata on the whole map, shrink + expand (expand of
    the bf16 input for an embedding workload) on tokens sel."""
    oracle.meta_prepare(inp.ids, w.max_loras)
    ids = inp.ids[sel]
    if w.kind == "embedding":
        b = oracle.bf16_to_f64(inp.x[sel])[None]
    else:
        buf = np.zeros((w.num_slices, sel.size, w.rank), np.float32)
        b = oracle.shrink(inp.x[sel], inp.lora_a, ids, w.scale, buf)
    oracle.expand(b.astype(np.float32), inp.lora_b, ids, inp.y[sel], w.slices,
                  w.offset_start, w.add_inputs, inp.lora_bias)


def cpu_baseline(w, inp, target_s=10.0):
    import oracle
    oracle.build()
    T = w.num_tokens
    n = min(T, 64)
    sel = np.arange(n)
    t0 = time.perf_counter()
    _oracle_step(oracle, w, inp, sel)
    per_tok = (time.perf_counter() - t0) / n
    n = int(min(T, max(1, target_s / max(per_tok, 1e-9))))
    rng = np.random.default_rng(0)
    sel = np.sort(rng.choice(T, size=n, replace=False)) if n < T else np.arange(T)
    done, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(oracle, w, inp, sel)
        done += sel.size
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": done / el, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "%d of %d tokens of the %s batch per pass (metadata on the full map), "
                      "%d tokens in %.1f s" % (sel.size, T, w.name, done, el)}


def workload_config(w, ub, args):
    """The workload part of the line's config, shared by both arms."""
    return {
        "workload": "%s: %s%s" % (w.name, w.description,
                                  "" if args.num_tokens is None else
                                  " (this run: %d tokens)" % w.num_tokens),
        "num_tokens": w.num_tokens, "active_tokens": ub["t_active"],
        "distinct_loras": ub["distinct"], "hidden": w.hidden, "rank": w.rank,
        "max_loras": w.max_loras, "slices": list(w.slices), "bias": w.bias, "scale": w.scale,
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = _workload(args.workload or HEADLINE, args)
    inp = W.generate(w)
    T = w.num_tokens
    sel = np.arange(min(T, 16))
    t0 = time.perf_counter()
    _oracle_step(oracle, w, inp, sel)
    per_tok = (time.perf_counter() - t0) / sel.size
    budget = 90.0 / max(1, args.steps + args.warmup)      # seconds per step
    n = int(min(T, max(1, budget / max(per_tok, 1e-9))))
    sel = np.sort(np.random.default_rng(0).choice(T, size=n, replace=False))
    for _ in range(args.warmup):
        _oracle_step(oracle, w, inp, sel)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(oracle, w, inp, sel)
    el = time.perf_counter() - t0
    value = args.steps * n / el
    sample = ("%d of %d tokens of the %s batch per step (metadata on the full map)"
              % (n, T, w.name))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy PCG64)",
        "config": {**workload_config(w, W.unique_bytes(w, inp.ids), args),
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    out = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
