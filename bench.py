"""Benchmark of the structured-read denoise step on GB300 (one JSON line on rank 0).

Workload (default): the full-canvas denoise step -- one request, prompt 4096
tokens of encoder KV, 256-token canvas, 8 query / 2 KV heads of width 512,
window +-128, d_model 2816, vocabulary 262144 -- with the three answer slots
of the single structured read (2 / 26 / 5 labels, 4 noise reads) read in the
same step.  One step = attention, lm-head log-softmax/entropy over all 256
rows, the slot read (noise + one W pass + gate), the entropy commit,
self-conditioning and the next-step canvas update.  W and E (1.48 GB each)
are streamed every step, so every timed step reads inputs far larger than L2.
The step's slot finish, commit and attention run on a side stream beside the
self-conditioning GEMM (``--schedule serial``: every call on one stream).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload NAME] [--schedule concurrent|serial]
"""
import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "denoise steps/s per 256-tok canvas; slot reads/s; % of tensor/HBM roofline"
UNIT = "denoise steps/s"

LMHEAD_KINDS = ("lmhead", "lmhead_fp8", "lmhead_fp4", "lmhead_fp4mma")

# workload name -> (runner kind, shape name, overrides).  Kinds: "step" = the
# full denoise step, "read" = the read-only step (attention + one slot read),
# "two_stage" = the mixed batch of two-stage ask_if reads over paged prompt KV.
WORKLOADS = {
    "full_canvas_step": ("step", "FULL_CANVAS", {}),
    "single_structured_read": ("read", "SINGLE_READ", {}),
    "single_structured_read_nvfp4": ("read_fp4", "SINGLE_READ", {}),
    "mixed_batched_reads": ("two_stage", "MIXED_BATCH", {}),
    "long_context_read": ("read", "LONG_CONTEXT", {}),
    "wide_read_77": ("read", "SINGLE_READ", dict(slots=[(61, 77)])),
    "lmhead_bf16_m256": ("lmhead", "FULL_CANVAS", {}),
    "lmhead_fp8_m256": ("lmhead_fp8", "FULL_CANVAS", {}),
    "lmhead_bf16_m12": ("lmhead", "FULL_CANVAS", dict(C=12)),
    "lmhead_fp8_m12": ("lmhead_fp8", "FULL_CANVAS", dict(C=12)),
    "lmhead_nvfp4_m256": ("lmhead_fp4", "FULL_CANVAS", {}),
    "lmhead_nvfp4_m12": ("lmhead_fp4", "FULL_CANVAS", dict(C=12)),
    "lmhead_nvfp4_mma_m12": ("lmhead_fp4mma", "FULL_CANVAS", dict(C=12)),
    "lmhead_nvfp4_mma_m256": ("lmhead_fp4mma", "FULL_CANVAS", {}),
    "heads_bf16_m256": ("heads", "FULL_CANVAS", {}),
    "heads_fp8_m256": ("heads_fp8", "FULL_CANVAS", {}),
    "selfcond_bf16_m256": ("selfcond", "FULL_CANVAS", {}),
    "selfcond_fp8_m256": ("selfcond_fp8", "FULL_CANVAS", {}),
    "mixed_decode8_prefill2": ("mixed", "LONG_CONTEXT", dict(B=10, C=2048, P=4096)),
    "prefill_8192": ("prefill", "LONG_CONTEXT", dict(B=1, P=8192)),
    "prefill_long": ("prefill", "LONG_CONTEXT", {}),
    "sweep_read_b1": ("read", "LONG_CONTEXT", dict(B=1, P=8192)),
    "sweep_read_b8": ("read", "LONG_CONTEXT", dict(B=8, P=8192)),
    "sweep_read_b64": ("read", "LONG_CONTEXT", dict(B=64, P=8192)),
    "sweep_step_b1": ("step", "FULL_CANVAS", dict(B=1, P=8192)),
    "sweep_step_b8": ("step", "FULL_CANVAS", dict(B=8, P=8192)),
    "sweep_step_b64": ("step", "FULL_CANVAS", dict(B=64, P=8192)),
    # the full-canvas step and the single read with a 65536-entry vocabulary (W
    # 369 MB, still past L2): the small cases for whole-kernel profiler captures
    "step_v65536": ("step", "FULL_CANVAS", dict(V=65536)),
    "single_read_v65536": ("read", "SINGLE_READ", dict(V=65536)),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="headline line only (skip the single read, the mixed batch and the "
                         "long-context read that the default line also reports)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--schedule", default="concurrent", choices=["concurrent", "serial"],
                    help="step schedule: side stream beside the self-conditioning GEMM, "
                         "or every call on one stream")
    ap.add_argument("--workload", default="full_canvas_step", choices=list(WORKLOADS),
                    help="full_canvas_step is the headline line; the others measure the "
                         "remaining workloads (read-only steps, the mixed batch, the sweep)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world):
    """Max of a float over ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ms_max, steps, world):
    """Whole-job throughput: the units all ranks processed (each rank runs `steps`
    units of the same work) over the slowest rank's time."""
    return world * steps / (ms_max / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        sms.sort()
        med = sms[len(sms) // 2] if sms else None
        return {"sm_mhz": med, "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms)}


# --------------------------------------------------------------- roofline
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def traffic_from_profile(kernel_src, name):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b:
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, kernel_src), "rb").read()).hexdigest()
    return float(m_b.group(1)) if sha == m_sha.group(1) else None


# ------------------------------------------------------------ the GPU arm
def build_step(shape, device, concurrent=True):
    import torch

    from structured_slot_reads_gb300 import dg, inputs
    from structured_slot_reads_gb300.step import DenoiseStep
    torch.manual_seed(0)
    w = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 1, device)
    e = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 2, device)
    st = DenoiseStep(shape, w, e, device=device, seed=7, concurrent=concurrent)
    st.h0.copy_(inputs.device_normal_bf16(st.h0.shape, 1.0, 3, device))
    st.inv_t.copy_(1.0 / inputs.device_uniform(st.inv_t.shape, 0.5, 2.0, 4, device))
    for i, k in enumerate(("q", "kc", "vc", "kenc", "venc")):
        getattr(st, k).copy_(inputs.device_normal_bf16(getattr(st, k).shape, 1.0, 10 + i, device))
    st.cand.fill_(1)
    st.set_slots(*inputs.slot_table(shape, 0))
    st.reset_state()
    torch.cuda.synchronize()
    return st


class CallTimer:
    """CUDA events around each library call of a step, on the launching stream."""

    def __init__(self, names):
        import torch
        self.torch = torch
        self.names = names
        self.pairs = {n: [] for n in names}

    def wrap(self, st):
        from structured_slot_reads_gb300 import dg
        torch = self.torch
        timer = self
        orig = {}
        for n in self.names:
            fn = getattr(dg, n)
            orig[n] = fn

            def make(fn, n):
                def inner(*a, **k):
                    # the call's own stream: its last argument, else the current one
                    s = k.get("stream", a[-1] if a else None)
                    if not isinstance(s, torch.cuda.Stream):
                        s = torch.cuda.current_stream()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(s)
                    r = fn(*a, **k)
                    e1.record(s)
                    timer.pairs[n].append((e0, e1))
                    return r
                return inner
            setattr(dg, n, make(fn, n))
        self._orig = orig

    def unwrap(self):
        from structured_slot_reads_gb300 import dg
        for n, fn in self._orig.items():
            setattr(dg, n, fn)

    def mean_ms(self, n):
        ps = self.pairs[n]
        return sum(a.elapsed_time(b) for a, b in ps) / max(1, len(ps))


def gpu_arm(args, rank, world, local):
    import torch

    from structured_slot_reads_gb300 import configs, dg
    shape = configs.FULL_CANVAS
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    st = build_step(shape, device, concurrent=args.schedule == "concurrent")
    stream = torch.cuda.current_stream()
    # warm-up
    for i in range(args.warmup):
        st.run(step_idx=i)
    torch.cuda.synchronize()
    dg.dg_clear_status()
    calls = ["dg_attn_decode", "dg_lmhead_logsoftmax_entropy", "dg_slot_read", "dg_slot_noise",
             "dg_denoise_heads", "dg_slot_finish", "dg_commit", "dg_selfcond_embed",
             "dg_selfcond_from_probs", "dg_canvas_update"]
    timer = CallTimer(calls)
    timer.wrap(st)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.6)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # per-call times need one stream: the eager pass runs the one-stream schedule
    concurrent, st.concurrent = st.concurrent, False
    e0.record(stream)
    launches = 0
    for i in range(args.steps):
        launches += st.run(step_idx=args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_eager = max_over_ranks(e0.elapsed_time(e1), world)
    timer.unwrap()
    st.concurrent = concurrent
    per_call = {n: timer.mean_ms(n) for n in calls}

    # the same steps replayed as CUDA graphs (one per step index, captured before
    # the timed region): this is the reported throughput
    for i in range(args.steps):
        st.capture(args.warmup + i)
    torch.cuda.synchronize()
    barrier(world)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    launches = 0
    for i in range(args.steps):
        launches += st.replay(args.warmup + i)
    g1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(g0.elapsed_time(g1), world)
    clk = clocks.stop()
    status = dg.dg_get_status()

    # end to end through the public step API with host buffers: each step copies
    # all its inputs from pinned memory and reads its decisions back; the copies
    # of step i+1 run on their own streams while step i computes (HostPipeline)
    from structured_slot_reads_gb300.step import HostPipeline
    ins, outs = st.host_buffers()
    for k, t in ins.items():
        t.copy_(getattr(st, k).cpu())
    pipe = HostPipeline(st)
    pipe.prepare(range(args.e2e_steps))
    h2d = d2h = 0
    barrier(world)
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(args.e2e_steps):
        h2d, d2h = pipe.submit(i, ins, outs)
    pipe.join(stream)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world)
    e2e_value = job_rate(e2e_ms, args.e2e_steps, world) if args.e2e_steps > 0 else None

    value = job_rate(ms, args.steps, world)
    pk = peaks()
    work = call_work(shape, st)
    kernels = {}
    for n in calls:
        if not timer.pairs[n]:
            continue
        t_s = per_call[n] / 1e3
        b, f = work.get(n, (0.0, 0.0))
        kernels[n] = {"ms": round(per_call[n], 4), "bytes": b, "flops": f}
        if b:
            kernels[n]["hbm_frac"] = round(b / t_s / 1e9 / pk["hbm"], 4)
        if f:
            kernels[n]["tensor_frac_sustained"] = round(f / t_s / 1e12 / pk["bf16_sus"], 4)
    # the dominant kernel: the one W stream of the step (fused lm-head pass)
    dom = "dg_denoise_heads" if "dg_denoise_heads" in kernels else "dg_lmhead_logsoftmax_entropy"
    dom_ms = per_call[dom]
    dom_bytes, dom_flops = work[dom]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    src = ("structured_slot_reads_gb300/csrc/heads_tc.cu" if dom == "dg_denoise_heads"
           else "structured_slot_reads_gb300/csrc/gemm_tc.cu")
    spill = spill_bytes(shape) if dom == "dg_denoise_heads" else 0
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm"], 4),
            "traffic": traffic_from_profile(src, "denoise_heads_full_canvas"
                                            if dom == "dg_denoise_heads"
                                            else "lmhead_stats_full_canvas"),
            "kernel": dom, "peak_source": pk["source"] + " (burst copy)",
            "algorithmic_bytes": dom_bytes,
            "bytes_with_probability_spill": dom_bytes + spill,
            "frac_with_probability_spill": round((dom_bytes + spill) / (dom_ms / 1e3) / 1e9
                                                 / pk["hbm"], 4),
            "tensor_tflops": round(dom_flops / (dom_ms / 1e3) / 1e12, 1),
            "tensor_frac_sustained": round(dom_flops / (dom_ms / 1e3) / 1e12 / pk["bf16_sus"], 4)}

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "ms_per_step_eager": round(ms_eager / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "full_canvas_step: B=1, prompt 4096, canvas 256, Hq 8 / Hkv 2, "
                               "d_head 512, W 128, d_model 2816, vocab 262144, gamma 25.6, "
                               "3 answer slots (2/26/5 labels) x 4 noise reads",
                   "global_batch": world * shape.B, "seq_len": shape.C,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: W and E (1.48 GB each) streamed every step",
                   "launch": "each step replayed as a CUDA graph of its library kernels"
                             + (", slot finish, commit and attention on a side stream beside "
                                "the self-conditioning GEMM" if st.concurrent else "")
                             + " (per-call times from an eager one-stream pass of the same "
                               "steps)",
                   "schedule": args.schedule},
        "slot_reads_per_s": round(value, 3),
        "slot_decisions_per_s": round(value * len(shape.slots), 3),
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": round(e2e_value, 3) if e2e_value else None, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "each step's host copies run on their own streams, overlapping the "
                           "neighbouring steps' compute (double-buffered pinned-to-device "
                           "staging; each step's graph reads and writes its staging set)"},
        "gpu_launches": launches,
        "clocks": clk,
        "device_status": status,
    }
    return line, st


def slot_finish_bytes(shape, n_slots):
    """Algorithmic bytes of the slot finish from gathered label logits: the label
    logits of every draw read and rewritten as logprobs, the draw rows' lse, the
    label counts, and the per-slot outputs written."""
    rows = n_slots * shape.R
    return rows * 26 * 4 * 2 + rows * 4 + n_slots * 4 + n_slots * (26 * 4 + 4 + 4 + 1 + 4)


def commit_bytes(shape):
    """Algorithmic bytes of the commit: per position entropy, argmax, candidate
    flag and carried state read; accept flag, token and carried state written."""
    return shape.B * shape.C * (4 + 4 + 1 + 1 + 4 + 1 + 4 + 1 + 4) + shape.B * 8


def call_work(shape, st):
    """Algorithmic HBM bytes and FLOPs of each library call of one step.

    The fused heads pass counts what the method must move: W once, the canvas and
    draw rows, the row statistics.  The bf16 probabilities it also writes for the
    self-conditioning GEMM (and that GEMM reads back) are this design's hand-off
    between the two passes, not the method's work; ``spill`` gives them apart."""
    M, V, D = shape.B * shape.C, shape.V, shape.D
    W = V * D * 2
    nd = getattr(st, "n_draw", 0)
    S = getattr(st, "S", 0)
    sr = S * shape.R                          # draw rows of a dg_slot_read pass
    return {
        "dg_attn_decode": (attn_bytes(shape), attn_flops(shape)),
        "dg_lmhead_logsoftmax_entropy": (W + M * D * 2 + M * 16, 2.0 * M * V * D),
        "dg_slot_read": (W + sr * D * 4, 2.0 * sr * V * D),
        "dg_denoise_heads": (W + (M + nd) * D * 2 + M * 20 + nd * 4 + nd * 26 * 4,
                             2.0 * (M + nd) * V * D),
        "dg_selfcond_embed": (2 * W + M * D * 2 + M * 8 + M * D * 4, 4.0 * M * V * D),
        "dg_selfcond_from_probs": (W + M * D * 4, 2.0 * M * V * D),
        "dg_slot_noise": (3 * nd * D * 2, 0.0),
        "dg_slot_finish": (slot_finish_bytes(shape, S) if nd else 0.0, 0.0),
        "dg_commit": (commit_bytes(shape), 0.0),
        "dg_canvas_update": (M * D * (2 + 4 + 2), 0.0),
    }


def spill_bytes(shape):
    """The heads pass's bf16 probabilities: written once, read once by P.E."""
    return shape.B * shape.C * shape.V * 2


def attn_flops(shape, prompt_len=None):
    """Algorithmic attention FLOPs of one step (QK^T and PV over visible keys)."""
    C, W = shape.C, shape.W
    win = sum(min(C - 1, i + W) - max(0, i - W) + 1 for i in range(C))
    plens = [shape.P] * shape.B if prompt_len is None else [int(p) for p in prompt_len]
    vis = sum(C * p + win for p in plens)
    return 4.0 * shape.Hq * shape.d_head * vis


def configs_scaled(shape, **kw):
    from structured_slot_reads_gb300 import configs
    return configs.scaled(shape, **kw)


def prefill_flops(shape):
    """Causal prefill: QK^T and PV over the P (P + 1) / 2 visible (row, key) pairs."""
    return 4.0 * shape.B * shape.Hq * shape.d_head * shape.P * (shape.P + 1) / 2


def prefill_bytes(shape):
    """Q and O once, K and V read once and written once more into the page pool."""
    q = shape.B * shape.P * shape.Hq * shape.d_head * 2
    kv = shape.B * shape.P * shape.Hkv * shape.d_head * 2 * 2
    return 2 * q + 2 * kv


def attn_bytes(shape, prompt_len=None):
    """Algorithmic attention bytes: prompt + canvas K/V once, Q read and O written once."""
    plens = [shape.P] * shape.B if prompt_len is None else [int(p) for p in prompt_len]
    kv = (sum(plens) + shape.B * shape.C) * shape.Hkv * shape.d_head * 2 * 2
    return kv + 2 * shape.B * shape.C * shape.Hq * shape.d_head * 2


# ------------------------------------------------- the other workloads
def workload_shape(name):
    from structured_slot_reads_gb300 import configs
    kind, base, kw = WORKLOADS[name]
    shape = getattr(configs, base)
    if kw:
        shape = configs.scaled(shape, name=name, **kw)
    return kind, shape


def fill_common(st, shape, device, kv=("kenc", "venc")):
    """Synthetic device inputs: N(0,1) hidden rows and attention tensors, 1/T ~ 1/U(0.5, 2)."""
    from structured_slot_reads_gb300 import inputs
    h = st.h0 if hasattr(st, "h0") else st.h
    h.copy_(inputs.device_normal_bf16(h.shape, 1.0, 3, device))
    st.inv_t.copy_(1.0 / inputs.device_uniform(st.inv_t.shape, 0.5, 2.0, 4, device))
    for i, k in enumerate(("q", "kc", "vc") + tuple(kv)):
        getattr(st, k).copy_(inputs.device_normal_bf16(getattr(st, k).shape, 1.0, 10 + i, device))


def build_runner(kind, shape, device, concurrent=True):
    import torch

    from structured_slot_reads_gb300 import inputs
    from structured_slot_reads_gb300.read import ReadStep, TwoStageRead
    if kind == "step":
        return build_step(shape, device, concurrent=concurrent)
    if kind in LMHEAD_KINDS:
        from structured_slot_reads_gb300.read import LmHead
        w = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 1, device)
        st = LmHead(shape, w, shape.B * shape.C, fp8=kind == "lmhead_fp8", device=device,
                    fp4=kind == "lmhead_fp4", fp4_mma=kind == "lmhead_fp4mma")
        st.h.copy_(inputs.device_normal_bf16(st.h.shape, 1.0, 3, device))
        st.inv_t.copy_(1.0 / inputs.device_uniform(st.inv_t.shape, 0.5, 2.0, 4, device))
        torch.cuda.synchronize()
        return st
    if kind in ("heads", "heads_fp8"):
        # the fused pass alone: 256 canvas rows and the 12 draw rows of three slots
        from structured_slot_reads_gb300.read import Heads
        w = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 1, device)
        nd = len(shape.slots) * shape.R
        st = Heads(shape, w, shape.B * shape.C, nd, fp8=kind == "heads_fp8", device=device)
        st.h.copy_(inputs.device_normal_bf16(st.h.shape, 1.0, 3, device))
        st.draw_rows.copy_(inputs.device_normal_bf16(st.draw_rows.shape, 1.0, 5, device))
        st.inv_t.copy_(1.0 / inputs.device_uniform(st.inv_t.shape, 0.5, 2.0, 4, device))
        st.inv_t_draw.copy_(1.0 / inputs.device_uniform(st.inv_t_draw.shape, 0.5, 2.0, 6, device))
        torch.cuda.synchronize()
        return st
    if kind in ("selfcond", "selfcond_fp8"):
        from structured_slot_reads_gb300.read import SelfCond
        e = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 2, device)
        st = SelfCond(shape, e, shape.B * shape.C, fp8=kind == "selfcond_fp8", device=device)
        st.probs.copy_(inputs.device_normal_bf16(st.probs.shape, 1.0, 3, device).abs())
        st.prob_scale.fill_(1.0 / shape.V)
        torch.cuda.synchronize()
        return st
    if kind == "mixed":
        # 8 decoder requests (256-row canvas over a P-token prompt) and 2 encoder
        # requests of C prompt tokens, one launch
        from structured_slot_reads_gb300.read import MixedAttention
        mode = [0] * (shape.B - 2) + [1, 1]
        rows = [256] * (shape.B - 2) + [shape.C, shape.C]
        plen = [shape.P] * (shape.B - 2) + [0, 0]
        st = MixedAttention(mode, rows, plen, shape.C, shape.Hq, shape.Hkv, shape.d_head, shape.W,
                            device=device)
        for i, k in enumerate(("q", "kc", "vc", "kenc", "venc")):
            getattr(st, k).copy_(inputs.device_normal_bf16(getattr(st, k).shape, 1.0, 40 + i,
                                                           device))
        torch.cuda.synchronize()
        return st
    if kind == "prefill":
        from structured_slot_reads_gb300.read import Prefill
        st = Prefill(shape.B, shape.P, shape.Hq, shape.Hkv, shape.d_head, shape.page_size,
                     device=device, seed=5)
        for i, k in enumerate(("q", "k", "v")):
            getattr(st, k).copy_(inputs.device_normal_bf16(getattr(st, k).shape, 1.0, 30 + i,
                                                           device))
        torch.cuda.synchronize()
        return st
    w = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 1, device)
    e = inputs.device_normal_bf16((shape.V, shape.D), shape.D ** -0.5, 2, device)
    if kind in ("read", "read_fp4"):
        st = ReadStep(shape, w, e, device=device, seed=7, concurrent=concurrent,
                      fp4=kind == "read_fp4")
        fill_common(st, shape, device)
    else:
        plen = inputs.prompt_lengths(shape, 5)
        st = TwoStageRead(shape, w, e, inputs.two_stage_tables(shape, 5), plen, device=device,
                          seed=7)
        table, n_pages = inputs.page_table(plen, shape.page_size, 5)
        pool = (n_pages, shape.page_size, shape.Hkv, shape.d_head)
        st.set_kv(inputs.device_normal_bf16(pool, 1.0, 20, device),
                  inputs.device_normal_bf16(pool, 1.0, 21, device),
                  torch.from_numpy(table).to(device))
        st.prompt_lens_host = plen
        fill_common(st, shape, device, kv=())
    torch.cuda.synchronize()
    return st


def timed_steps(args, run, calls, local, world, sched=None):
    """W warm-up steps, then K steps timed with CUDA events on the launching stream.

    ``sched``: a DenoiseStep whose side-stream schedule is timed; its per-call
    times then come from a second pass of K steps on one stream (events around
    a call on a shared GPU would time the neighbours too).
    Returns (max-over-ranks ms for K steps, mean ms per library call, kernels
    launched, clock record)."""
    import torch
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        run(i)
    torch.cuda.synchronize()
    timer = CallTimer(calls)
    if sched is None:
        timer.wrap(None)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.6)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    launches = 0
    for i in range(args.steps):
        launches += run(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    if sched is not None:
        concurrent, sched.concurrent = sched.concurrent, False
        timer.wrap(None)
        for i in range(args.steps):
            run(args.warmup + args.steps + i)
        torch.cuda.synchronize()
        sched.concurrent = concurrent
    timer.unwrap()
    return ms, {n: timer.mean_ms(n) for n in calls if timer.pairs[n]}, launches, clk


def workload_arm(args, rank, world, local):
    """One JSON line for a workload other than the headline step."""
    import torch

    from structured_slot_reads_gb300 import dg
    kind, shape = workload_shape(args.workload)
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    st = build_runner(kind, shape, device, concurrent=args.schedule == "concurrent")
    if kind == "two_stage":
        run = lambda i: st.run()                        # noqa: E731
        calls = ["dg_attn_decode", "dg_slot_noise", "dg_lmhead_logsoftmax_entropy",
                 "dg_slot_finish", "dg_ask_if_select"]
    elif kind == "prefill":
        run = lambda i: st.run(step_idx=i)              # noqa: E731
        calls = ["dg_prefill_attn"]
    elif kind == "mixed":
        run = lambda i: st.run(step_idx=i)              # noqa: E731
        calls = ["dg_attn_mixed"]
    elif kind in LMHEAD_KINDS:
        run = lambda i: st.run(step_idx=i)              # noqa: E731
        calls = ["dg_lmhead_logsoftmax_entropy", "dg_quantize_rows_e4m3",
                 "dg_lmhead_logsoftmax_entropy_fp8", "dg_lmhead_logsoftmax_entropy_nvfp4",
                 "dg_lmhead_logsoftmax_entropy_nvfp4_mma"]
    elif kind in ("selfcond", "selfcond_fp8"):
        run = lambda i: st.run(step_idx=i)              # noqa: E731
        calls = ["dg_selfcond_from_probs", "dg_quantize_rows_e4m3", "dg_selfcond_from_probs8"]
    elif kind in ("heads", "heads_fp8"):
        run = lambda i: st.run(step_idx=i)              # noqa: E731
        calls = ["dg_denoise_heads", "dg_quantize_rows_e4m3", "dg_denoise_heads_fp8"]
    else:
        run = lambda i: st.run(step_idx=i)              # noqa: E731
        calls = ["dg_attn_decode", "dg_slot_read", "dg_slot_read_wide", "dg_slot_noise",
                 "dg_lmhead_logsoftmax_entropy_nvfp4_mma", "dg_denoise_heads",
                 "dg_slot_finish", "dg_commit", "dg_selfcond_from_probs", "dg_canvas_update"]
    dg.dg_clear_status()
    sched = (st if kind in ("step", "read", "read_fp4") and getattr(st, "concurrent", False)
             else None)
    ms, per_call, launches, clk = timed_steps(args, run, calls, local, world, sched)
    status = dg.dg_get_status()
    steps_per_s = job_rate(ms, args.steps, world)
    pk = peaks()
    V, D, R = shape.V, shape.D, shape.R
    Wb = V * D * 2
    plen = getattr(st, "prompt_lens_host", None)
    work = call_work(shape, st) if kind == "step" else {}
    work["dg_attn_decode"] = (attn_bytes(shape, plen), attn_flops(shape, plen))
    if kind == "prefill":
        work["dg_prefill_attn"] = (prefill_bytes(shape), prefill_flops(shape))
    if kind == "mixed":
        dec = configs_scaled(shape, B=1, C=256)
        enc = configs_scaled(shape, B=1, P=shape.C)
        fl = (shape.B - 2) * attn_flops(dec) + 2 * prefill_flops(enc)
        by = (shape.B - 2) * attn_bytes(dec) + 2 * prefill_bytes(enc)
        work["dg_attn_mixed"] = (by, fl)
    if kind in LMHEAD_KINDS:
        Mr = shape.B * shape.C
        esz = 1 if kind == "lmhead_fp8" else 2
        lm = (V * D * esz + Mr * D * esz + V * 4 * (esz == 1) + Mr * 16, 2.0 * Mr * V * D)
        work["dg_lmhead_logsoftmax_entropy"] = lm
        work["dg_lmhead_logsoftmax_entropy_fp8"] = lm
        # NVFP4 weights: half a byte per element plus one e4m3 scale per 16; bf16 rows
        work["dg_lmhead_logsoftmax_entropy_nvfp4"] = (V * D // 2 + V * D // 16 + Mr * D * 2
                                                      + Mr * 16, 2.0 * Mr * V * D)
        # both NVFP4: the weights' codes and scales, the rows read once (bf16) and
        # quantised (their codes and scales written and read back)
        work["dg_lmhead_logsoftmax_entropy_nvfp4_mma"] = (
            V * D // 2 + V * D // 16 + Mr * D * 2 + 2 * (Mr * D // 2 + Mr * D // 16) + Mr * 16,
            2.0 * Mr * V * D)
        work["dg_quantize_rows_e4m3"] = (Mr * D * 3 + Mr * 4, 0.0)
    if kind in ("selfcond", "selfcond_fp8"):
        Mr = shape.B * shape.C
        pe = 2.0 * Mr * V * D
        work["dg_selfcond_from_probs"] = (V * D * 2 + Mr * V * 2 + Mr * D * 4, pe)
        work["dg_quantize_rows_e4m3"] = (Mr * V * 3 + Mr * 4, 0.0)
        work["dg_selfcond_from_probs8"] = (V * D + D * 4 + Mr * V + Mr * D * 4, pe)
    if kind in ("heads", "heads_fp8"):
        # algorithmic bytes: W (bf16, or e4m3 and its row scales) and the rows;
        # the probabilities this design writes are not counted
        Mr, nd = st.M, st.n_draw
        fl = 2.0 * (Mr + nd) * V * D
        work["dg_denoise_heads"] = (Wb + (Mr + nd) * D * 2 + Mr * 16, fl)
        work["dg_denoise_heads_fp8"] = (V * D + V * 4 + (Mr + nd) * (D + 4) + Mr * 16, fl)
        work["dg_quantize_rows_e4m3"] = ((Mr + nd) * D * 3 + (Mr + nd) * 4, 0.0)
    if kind == "read":
        work["dg_slot_read"] = (Wb + st.S * R * D * 4, 2.0 * st.S * R * V * D)
        work["dg_slot_read_wide"] = work["dg_slot_read"]
        decisions = st.S
    elif kind == "read_fp4":
        nd = st.S * R
        work["dg_lmhead_logsoftmax_entropy_nvfp4_mma"] = (
            V * D // 2 + V * D // 16 + nd * D * 2 + 2 * (nd * D // 2 + nd * D // 16) + nd * 16,
            2.0 * nd * V * D)
        work["dg_slot_noise"] = (3 * nd * D * 2, 0.0)
        decisions = st.S
    elif kind == "two_stage":
        rows = (st.S1 + st.S2) * R                      # draw rows of both stages, one W pass
        work["dg_lmhead_logsoftmax_entropy"] = (Wb + rows * D * 2 + rows * 16,
                                                2.0 * rows * V * D)
        decisions = st.decisions()
    else:
        decisions = getattr(st, "S", 0)
    kernels, best = {}, None
    n_calls = {"dg_slot_noise": 2, "dg_slot_finish": 2} if kind == "two_stage" else {}
    # 8- and 4-bit contractions against their own peak: the measured bf16 figure
    # times the nominal ratio (dense: e4m3 4.5, NVFP4 13.5 against bf16 2.25
    # PFLOP/s); the widened NVFP4 pass multiplies in bf16 / f16 and keeps bf16's
    e4m3 = ("dg_lmhead_logsoftmax_entropy_fp8", "dg_selfcond_from_probs8", "dg_denoise_heads_fp8")
    nvf4 = ("dg_lmhead_logsoftmax_entropy_nvfp4_mma",)
    ratio = lambda n: 2.0 if n in e4m3 else 6.0 if n in nvf4 else 1.0   # noqa: E731
    tpeak = lambda n: pk["bf16_sus"] * ratio(n)   # noqa: E731
    for n, t in per_call.items():
        b, f = work.get(n, (0.0, 0.0))
        kernels[n] = {"ms": round(t, 4), "bytes": b, "flops": f}
        if b:
            kernels[n]["hbm_frac"] = round(b / (t / 1e3) / 1e9 / pk["hbm"], 4)
        if f:
            kernels[n]["tensor_frac_sustained"] = round(f / (t / 1e3) / 1e12 / tpeak(n), 4)
        share = t * n_calls.get(n, 1)
        if (b or f) and (best is None or share > best[1]):
            best = (n, share)
    roof = None
    if best:
        n = best[0]
        t_s = per_call[n] / 1e3
        b, f = work[n]
        tensor_bound = f / max(b, 1.0) > tpeak(n) * 1e3 / pk["hbm"]
        if tensor_bound:
            ach, peak, unit = f / t_s / 1e12, tpeak(n), "TFLOP/s"
        else:
            ach, peak, unit = b / t_s / 1e9, pk["hbm"], "GB/s"
        roof = {"bound": "tensor" if tensor_bound else "hbm", "achieved": round(ach, 1),
                "peak": peak, "unit": unit, "frac": round(ach / peak, 4), "traffic": None,
                "kernel": n, "peak_source": pk["source"] + (
                    " (bf16 sustained x 2, the nominal e4m3 ratio)"
                    if tensor_bound and n in e4m3 else
                    " (bf16 sustained x 6, the nominal NVFP4 ratio)"
                    if tensor_bound and n in nvf4 else "")}
    if kind == "step":
        unit, value = UNIT, steps_per_s * shape.B
    elif kind == "prefill":
        unit, value = "prompt tokens/s", steps_per_s * shape.B * shape.P
    elif kind == "mixed":
        unit, value = "attention launches/s", steps_per_s
    elif kind in LMHEAD_KINDS:
        unit, value = "lm-head passes/s", steps_per_s
    elif kind in ("selfcond", "selfcond_fp8"):
        unit, value = "self-conditioning passes/s", steps_per_s
    elif kind in ("heads", "heads_fp8"):
        unit, value = "fused heads passes/s", steps_per_s
    else:
        unit, value = "slot decisions/s", steps_per_s * decisions
    return {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3" if kind.endswith("_fp8") else
                  "nvfp4 weights x bf16 rows" if kind.endswith("_fp4") else
                  "nvfp4 weights x nvfp4 rows" if kind.endswith(("_fp4mma", "read_fp4")) else
                  "bf16"),
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: kind {kind}, B={shape.B}, prompt "
                               f"{'U[512, %d] paged' % shape.P if kind == 'two_stage' else shape.P}"
                               f", canvas {shape.C}, Hq {shape.Hq} / Hkv {shape.Hkv}, d_head "
                               f"{shape.d_head}, W {shape.W}, d_model {D}, vocab {V}",
                   "global_batch": world * shape.B, "seq_len": shape.C,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("inputs larger than L2: E (1.48 GB bf16, 0.74 GB e4m3) streamed "
                          "every pass" if kind.startswith("selfcond") else
                          "inputs larger than L2: NVFP4 W (0.42 GB) streamed every step"
                          if kind in ("lmhead_fp4", "lmhead_fp4mma", "read_fp4") else
                          "inputs larger than L2: e4m3 W (0.74 GB) streamed every pass"
                          if kind == "heads_fp8" else
                          "inputs larger than L2: W (1.48 GB) streamed every step"),
                   "launch": ("eager; " + ("slot finish, commit and attention on a side "
                                           "stream beside the self-conditioning GEMM"
                                           if kind == "step" else
                                           "attention on a side stream beside the slot "
                                           "read's W pass")
                              + " (per-call times from a second, one-stream pass of as many "
                                "steps)" if sched is not None else "eager, one stream")},
        "steps_per_s": round(steps_per_s, 3),
        "canvases_per_s": round(steps_per_s * shape.B, 3),
        "slot_decisions_per_s": round(steps_per_s * decisions, 3),
        "slot_decisions_per_step": decisions,
        "roofline": roof, "kernels": kernels, "e2e": None, "gpu_launches": launches,
        "clocks": clk, "device_status": status,
    }


# --------------------------------------------------------- the CPU oracle
def oracle_inputs(shape, st=None):
    """Host copies of one step's inputs for the oracle (weights held in float64)."""
    import numpy as np

    from structured_slot_reads_gb300 import inputs
    if st is not None:
        w = st.w.float().cpu().numpy().astype(np.float64)
        e = st.e.float().cpu().numpy().astype(np.float64)
        h = st.h0.float().cpu().numpy()
        inv_t = st.inv_t.cpu().numpy()
    else:
        w32, e32 = inputs.weights(shape.V, shape.D, 1)
        w, e = w32.astype(np.float64), e32.astype(np.float64)
        del w32, e32
        h = inputs.hidden(shape.B * shape.C, shape.D, 3)
        inv_t = inputs.inv_temperature(shape.B * shape.C, 4)
    x = inputs.attention_inputs(shape, 5)
    slots = inputs.slot_table(shape, 0)
    return dict(w=w, e=e, h=h, inv_t=inv_t, att=x, slots=slots)


def oracle_step(shape, data, step_idx=0):
    """One whole denoise step of the workload in the float64 oracle, as it stands:
    attention of every row and head over the whole prompt, the lm-head statistics
    of every canvas row, the slot read (noise draws, their full-vocabulary
    log-normalisers, label logits, gate and average), the commit, the expected
    embedding of every row and the next canvas input.  Returns (seconds, parts)."""
    import numpy as np

    import oracle
    w, e, h, inv_t, x = data["w"], data["e"], data["h"], data["inv_t"], data["att"]
    row, req, lab, n = data["slots"]
    B, C, R = shape.B, shape.C, shape.R
    parts = {}
    t_all = time.perf_counter()
    t0 = time.perf_counter()
    oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"], x["prompt_len"], shape.W)
    parts["attention"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    _, ent, _, arg = oracle.lmhead_stats(h, w, inv_t)
    parts["lmhead"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    rows_d, _ = oracle.slot_noise_rows(h, e, row, req, 7, step_idx, R, shape.V)
    inv_d = np.repeat(inv_t[row], R)
    lse_d, _, _, _ = oracle.lmhead_stats(rows_d, w, inv_d)
    zl = oracle.label_logits(rows_d, w, inv_d, np.repeat(lab, R, axis=0), np.repeat(n, R))
    oracle.slot_read(zl.reshape(len(row), R, -1), lse_d.reshape(len(row), R), n, R, shape.gate)
    parts["slot_read"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    cm, tk, _ = oracle.commit(ent.reshape(B, C), arg.reshape(B, C), np.ones((B, C), np.uint8),
                              np.full(B, shape.gamma))
    parts["commit"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    e_sc = oracle.selfcond_embed(h, w, e, inv_t)
    parts["selfcond"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.canvas_update(h, e_sc, e, tk.reshape(-1), cm.reshape(-1))
    parts["canvas_update"] = time.perf_counter() - t0
    return time.perf_counter() - t_all, parts


ORACLE_SAMPLE = ("one whole full-canvas step: attention of all 8 heads over the 4096-token "
                 "prompt and the window, lm-head statistics and self-conditioning of all 256 "
                 "rows over the 262144-entry vocabulary, the three slot reads (4 draws each), "
                 "the commit and the canvas update; no part sampled or scaled")


def reference_arm(args, rank, budget_s=150.0, shape=None):
    """The oracle as the reference implementation, timed on the host cores (rank 0 only).

    Each step is one whole float64 step (oracle_step).  Warm-up is at most two
    steps and the timed steps stop once ``budget_s`` of them have run, so the
    run ends in a few minutes; the line reports the steps actually timed."""
    from structured_slot_reads_gb300 import configs
    if rank != 0:
        return None
    shape = shape or configs.FULL_CANVAS
    data = oracle_inputs(shape)
    warm = min(args.warmup, 2)
    for i in range(warm):
        oracle_step(shape, data, i)
    times, parts = [], None
    for i in range(args.steps):
        dt, parts = oracle_step(shape, data, warm + i)
        times.append(dt)
        if sum(times) >= budget_s:
            break
    t = sum(times)
    value = len(times) / t
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": 1, "steps": len(times), "warmup": warm, "steps_requested": args.steps,
            "warmup_requested": args.warmup,
            "ms_per_step": round(1e3 * t / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "full_canvas_step (float64 CPU oracle, whole steps)",
                       "global_batch": 1, "seq_len": shape.C, "parallelism": "host cores"},
            "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "sample": ORACLE_SAMPLE,
                             "value": round(value, 6), "unit": UNIT,
                             "parts_s": {k: round(v, 3) for k, v in parts.items()}},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


EXTRA_WORKLOADS = ("single_structured_read", "mixed_batched_reads", "long_context_read",
                   "single_structured_read_nvfp4")


def extra_workloads(args, rank, world, local):
    """The single structured read, the mixed batch of two-stage reads and the
    long-context read, each timed as ``--workload`` times it (eager, 3 warm-up
    steps, at most 10 timed steps), summarised into the default line."""
    import torch
    out = {}
    for name in EXTRA_WORKLOADS:
        wargs = argparse.Namespace(**vars(args))
        wargs.workload = name
        wargs.warmup = max(3, min(args.warmup, 5))
        wargs.steps = min(args.steps, 10)
        ln = workload_arm(wargs, rank, world, local)
        out[name] = {k: ln[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup",
                                        "slot_decisions_per_s", "slot_decisions_per_step",
                                        "roofline", "kernels", "clocks", "device_status",
                                        "gpu_launches")}
        out[name]["workload"] = ln["config"]["workload"]
        torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        line = reference_arm(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if args.workload != "full_canvas_step":
        line = workload_arm(args, rank, world, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    line, st = gpu_arm(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        data = oracle_inputs(st.shape, st)
        dt, parts = oracle_step(st.shape, data)
        line["cpu_baseline"] = {"value": round(1.0 / dt, 6), "unit": UNIT,
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": ORACLE_SAMPLE, "steps_timed": 1,
                                "parts_s": {k: round(v, 3) for k, v in parts.items()}}
    if not args.no_extra_workloads:
        # the other headline workloads, each timed on its own (the step's buffers freed first)
        import torch
        del st
        torch.cuda.empty_cache()
        line["workloads"] = extra_workloads(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
