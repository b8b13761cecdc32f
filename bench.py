"""Benchmark of one MoE layer training step (dispatch build + forward +
backward) on synthetic inputs shaped like the workload, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` = tokens/s of the whole job with
inputs resident in HBM (device-timed with CUDA events, max over ranks, L2
flushed between steps); `e2e` = the same metric through the library's
pipelined step runner with host inputs/outputs (every step's pinned host ->
device copies of x, ids, gates, dY and device -> host copies of y and dX
inside the timed region, overlapped with the neighbouring steps); `roofline`
describes the dominant kernel, timed live from the library's stage events;
`cpu_baseline` times the CPU oracle on a bounded sample of the workload.
Beside the step: the router legs (timed first), the step replayed as one
captured CUDA graph (`graph_step`), the step without H / Hg temporaries
(`recompute_h`), and the dispatch build and identity gather/combine on the
2M-token routing stress case.  --tokens and --experts shrink the workload
for profiling captures.
With --gpus N > 1 every rank runs an independent replica on its own batch
(weak scaling; the step has no cross-rank exchange in the timed region).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_atomic_gb300 import binding as B  # noqa: E402
from mixture_experts_atomic_gb300 import inputs as I  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s (bf16), tensor-pipe %; dispatch-build HBM GB/s"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
L2_BYTES = 129 * 1024 * 1024
GEMM_SRC = "mixture_experts_atomic_gb300/csrc/gemm_tc.cu"
IDENTITY_SRC = "mixture_experts_atomic_gb300/csrc/identity.cu"


def peaks():
    """HBM copy GB/s and dense bf16 TFLOP/s (burst and sustained): the
    measured figures of this GPU pool when present, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            out = dict(FALLBACK)
            for k in FALLBACK:
                if isinstance(d.get(k), (int, float)):
                    out[k] = float(d[k])
            return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def code_sha256(path):
    """sha256 of a CUDA/C++ source with its comments and whitespace removed,
    so that a change of wording alone keeps a capture valid."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


def traffic_per_launch(workload, stage, source):
    """DRAM bytes (read + write) per launch of one kernel (`stage`) on one
    workload, from a committed ncu summary under profiles/ that names the
    kernel's source file and its code hash at capture (code_sha256); None
    when there is no such summary or the code has changed since."""
    sha = code_sha256(os.path.join(ROOT, source))
    key = ["traffic-per-launch", f"workload={workload}", f"file={source}", f"code-sha256={sha}"]
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        if not name.endswith(".md"):
            continue
        lines = open(os.path.join(ROOT, "profiles", name)).read().splitlines()
        for i, ln in enumerate(lines):
            if ln.split() == key:
                for row in lines[i + 1:]:
                    g = row.split()
                    if len(g) != 2:
                        break
                    if g[0] == stage:
                        return int(g[1])
    return None


# ------------------------------------------------------------------ algorithmic work

def stage_flops(cfg):
    """Algorithmic FLOPs of each GEMM stage (unpadded routed rows)."""
    LK, d, h = cfg.L * cfg.K, cfg.d, cfg.h
    sw = cfg.act == "swiglu"
    nb = 2 if sw else 1
    return {"up": 2 * nb * LK * d * h, "down": 2 * LK * h * d, "dh": 2 * LK * d * h,
            "dx": 2 * nb * LK * h * d, "dw12": 2 * nb * LK * d * h, "dw3": 2 * LK * h * d}


def dispatch_bytes(cfg):
    """Algorithmic bytes of the dispatch build (the per-token figure of the
    method's dispatch): ids read (4LK), D1, D3, D4 written (12LK), the
    offsets, and the bit-packed L x E bitmap written once and read twice
    (3LE/8).  These kernels keep each chunk's bitmap on chip, so they move
    none of the bitmap bytes; dispatch_kernel_bytes counts what they move."""
    LK = cfg.L * cfg.K
    return 4 * LK + 12 * LK + 4 * (cfg.E + 1) + 3 * (cfg.L * cfg.E // 8)


def dispatch_kernel_bytes(cfg):
    """Bytes the three dispatch kernels read and write: the ids (4LK), D3
    (4LK) and the packed (in-chunk rank, expert) slots (4LK) in K1; those
    slots again (4LK), D1 and D4 (8LK) in K3; and the per-(expert, chunk)
    counts: written, scanned in place (large layers) and read per chunk with
    the expert totals (about 16 E C)."""
    LK = cfg.L * cfg.K
    C = (cfg.L + 1023) // 1024
    return 24 * LK + 16 * cfg.E * C + 4 * (cfg.E + 1)


def materialising_bytes(cfg):
    """Activation bytes a materialising MoE layer keeps from the forward for
    the backward (MoEBlaze summary page, "问题与动机": the routing buffer is
    O(L*K*d), the first MLP's output O(L*h) per active expert, and SwiGLU adds
    several point-wise tensors).  Counted here as the routed copy of x
    (L*K*d) plus, per routed row, a, b, sigma(a), SiLU(a) and H (5*h) for
    SwiGLU or a and SiLU(a) (2*h) for SiLU; the identity expert keeps the
    routed buffer alone.  Elements of the layer dtype."""
    LK, s = cfg.L * cfg.K, cfg.elem_bytes
    per_row = {"swiglu": 5 * cfg.h, "silu": 2 * cfg.h, "identity": 0}[cfg.act]
    return LK * cfg.d * s + LK * per_row * s


def memory_report(cfg, layer, step_alloc_peak):
    """What this layer keeps from the forward for the backward (the saved A
    and B, padded expert-major, and the index structures), its scratch, and
    the same retained figure for a materialising layer.  step_alloc_peak:
    bytes the torch allocator handed out during one step on top of what was
    already allocated."""
    from mixture_experts_atomic_gb300 import binding as B
    sh = layer.shape

    def nb(t):
        return t.numel() * t.element_size()

    saved = B.moeblaze_saved_bytes(sh)
    d = layer.disp
    index = sum(nb(t) for t in (d.expert_token_indices, d.expert_token_offsets, d.token_expert_indices,
                                d.token_index_map, d.meta))
    mat = materialising_bytes(cfg)
    scratch = {"dispatch": B.moeblaze_dispatch_workspace_bytes(sh),
               "forward": B.moeblaze_forward_workspace_bytes(sh),
               "backward": B.moeblaze_backward_workspace_bytes(sh)}
    # what the layer holds at once at its high-water mark: the retained
    # checkpoint and indices plus the larger pass's scratch (the passes run
    # one after the other and each frees its scratch for the next)
    peak = saved + index + max(scratch["forward"], scratch["backward"])
    return {"retained_fwd_to_bwd_bytes": saved + index, "saved_activation_bytes": saved, "index_bytes": index,
            "scratch_bytes": scratch,
            "peak_activation_bytes": peak,
            "step_alloc_peak_bytes": int(step_alloc_peak),
            "materialising_retained_bytes": mat,
            "materialising_over_retained": mat / (saved + index),
            "materialising_retained_over_peak": mat / peak}


def identity_bytes(cfg):
    """Bytes one identity gather/combine pass must move: x read once (the K
    routed copies of a token's row are one row), y written once, and D1, D4
    and the gates read (12*L*K).  This is the roofline figure."""
    s = cfg.elem_bytes
    return 2 * cfg.L * cfg.d * s + 12 * cfg.L * cfg.K


def identity_routed_bytes(cfg):
    """The same pass counted with every routed row read on its own (L*K
    rows), as a routed buffer would be; the K reads of a row after the first
    come from L2, so this figure can exceed the HBM bandwidth."""
    s = cfg.elem_bytes
    return (cfg.L * cfg.K + cfg.L) * cfg.d * s + 12 * cfg.L * cfg.K


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int, keep: str | None = None):
        """keep: a path to keep the raw samples at (CSV); by default they go
        to a temporary file that is removed once summarised."""
        self.dev = device_index
        self.proc = None
        self.keep = keep
        self.path = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        if self.keep:
            os.makedirs(os.path.dirname(os.path.abspath(self.keep)), exist_ok=True)
            self.f = open(self.keep, "w")
        else:
            self.f = tempfile.NamedTemporaryFile("w", prefix=f"clocks_rank{self.dev}_", suffix=".csv", delete=False)
        self.path = self.f.name
        self.proc = subprocess.Popen([exe, "-i", str(self.dev), "--query-gpu=" + ",".join(self.FIELDS),
                                      "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                                     stderr=subprocess.DEVNULL)
        # the timed region starts once the sampler has written its first line
        t0 = time.time()
        while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.03)  # one more sampling interval
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.read().splitlines()
        if not self.keep:
            os.unlink(self.path)
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1])); mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle sample

class HostInputs:
    """The workload's inputs for the CPU oracle: the expert weights once, in
    fp64 (the oracle widens every input to fp64 itself; doing it once here
    keeps that copy out of each timed call), and the first rows of x, dY,
    ids and gates on demand.  x, dY and the routing are row-wise, so the
    first L' rows of the workload are the inputs of its first L' tokens.
    `src` holds the full workload's tensors (on any device), or is None to
    generate the rows and weights on the host."""

    def __init__(self, cfg, src=None):
        self.cfg = cfg
        self.src = src
        w = src if src is not None else I.make_weights(cfg, "cpu")
        self.W = {k: (None if w.get(k) is None else self._f64(w[k])) for k in ("W1", "W2", "W3")}

    @staticmethod
    def _f64(t):
        t = t.detach().cpu()
        return (t.float() if t.dtype == torch.bfloat16 else t).numpy().astype(np.float64)

    def rows(self, n):
        if self.src is not None:
            r = {k: self.src[k][:n].cpu() for k in ("ids", "gates", "x", "dY")}
        else:
            sub = self.cfg.scaled(L=n)
            x = I.make_x(sub, "cpu")
            ids, gates = I.make_routing(sub, x, "cpu")
            r = {"ids": ids, "gates": gates, "x": x, "dY": I.make_dy(sub, "cpu")}
        r.update(self.W)
        return r


def oracle_run(cfg, inp):
    """One forward + backward of the CPU oracle on a prepared sample."""
    import oracle.moe_oracle as O
    O.forward(inp["ids"], inp["gates"], inp["x"], inp["W1"], inp["W2"], inp["W3"], cfg.act, E=cfg.E)
    O.backward(inp["ids"], inp["gates"], inp["x"], inp["dY"], inp["W1"], inp["W2"], inp["W3"], cfg.act, E=cfg.E)


def oracle_sample(cfg, host, target_s=12.0, max_tokens=None):
    """Time the CPU oracle (forward + backward) on the first L' tokens of the
    workload, growing L' until one run takes about target_s / 3 seconds or
    more; returns (tokens/s, L', seconds) of that last run."""
    Lp = 64
    cap = min(max_tokens or cfg.L, cfg.L)
    while True:
        inp = host.rows(Lp)
        t0 = time.perf_counter()
        oracle_run(cfg, inp)
        dt = time.perf_counter() - t0
        if dt >= target_s / 3 or Lp >= cap:
            return Lp / dt, Lp, dt
        Lp = min(cap, Lp * max(2, int(target_s / 3 / max(dt, 1e-3))))


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ our arm

def max_over_ranks(ms, world, device):
    """The slowest rank's step time: every rank runs its own replica on its
    own batch, so the job advances at the pace of the slowest."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, ms):
    """Whole-job throughput: every rank's tokens in the slowest rank's step."""
    return world * tokens_per_rank / (ms * 1e-3)


def flush_l2(buf):
    buf.add_(1)


def run_ours(args, rank, world, local_rank):
    cfg = I.CONFIGS[args.config]
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from mixture_experts_atomic_gb300.layer import MoELayer
    inp = I.make_inputs(cfg, dev)
    # the step is the layer's dispatch, forward and backward (dX, dW1..dW3);
    # the optional gate gradients are not requested
    layer = MoELayer.for_config(cfg, dev, with_dgates=False)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    identity = cfg.act == "identity"
    nf, nbk = 4, 6

    def one_step(rec=None):
        s = torch.cuda.current_stream()
        if rec is not None:
            rec["e0"].record(s)
        layer.dispatch(inp["ids"])
        if rec is not None:
            rec["e1"].record(s)
            with rec["fw"]:
                layer.forward(inp["x"], inp["gates"], inp.get("W1"), inp.get("W2"), inp.get("W3"))
            rec["e2"].record(s)
            with rec["bw"]:
                layer.backward(inp["dY"], inp["x"], inp["gates"], inp.get("W1"), inp.get("W2"), inp.get("W3"))
            rec["e3"].record(s)
        else:
            layer.forward(inp["x"], inp["gates"], inp.get("W1"), inp.get("W2"), inp.get("W3"))
            layer.backward(inp["dY"], inp["x"], inp["gates"], inp.get("W1"), inp.get("W2"), inp.get("W3"))

    pk, src = peaks()
    # the router legs are timed first, before the layer steps heat the GPU
    # into its power cap (they are HBM-bound kernels of their own)
    router = run_router(cfg, inp, dev, flush, pk) if cfg.router in ("softmax", "softmax_bias") else None
    for _ in range(args.warmup):
        flush_l2(flush)
        one_step()
    torch.cuda.synchronize()
    assert layer.device_error() == 0, "device error during warm-up"
    # one more untimed step, watched by the torch allocator: every buffer of
    # the layer exists before the step, so this is what a step allocates
    alloc0 = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    one_step()
    torch.cuda.synchronize()
    step_alloc_peak = torch.cuda.max_memory_allocated(dev) - alloc0

    recs = [{"e0": torch.cuda.Event(enable_timing=True), "e1": torch.cuda.Event(enable_timing=True),
             "e2": torch.cuda.Event(enable_timing=True), "e3": torch.cuda.Event(enable_timing=True),
             "fw": B.StageEvents(nf), "bw": B.StageEvents(nbk)} for _ in range(args.steps)]
    clocks = ClockSampler(local_rank, args.clock_log.format(rank=rank) if args.clock_log else None)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = B.moeblaze_kernel_launches()
    for r in recs:
        flush_l2(flush)
        one_step(r)
    torch.cuda.synchronize()
    launches = B.moeblaze_kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    assert layer.device_error() == 0, "device error during the timed steps"

    step_ms = [r["e0"].elapsed_time(r["e3"]) for r in recs]
    disp_ms = [r["e0"].elapsed_time(r["e1"]) for r in recs]
    fwd_ms = [r["e1"].elapsed_time(r["e2"]) for r in recs]
    bwd_ms = [r["e2"].elapsed_time(r["e3"]) for r in recs]
    stages = {}
    if not identity:
        fw_names = ["up", "down", "convert_y"]
        bw_names = ["dh", "dx", "dw12", "dw3", "convert_dx"]
        per = {n: [] for n in fw_names + bw_names}
        for r in recs:
            for n, v in zip(fw_names, r["fw"].elapsed_ms()):
                per[n].append(v)
            for n, v in zip(bw_names, r["bw"].elapsed_ms()):
                per[n].append(v)
        stages = {n: statistics.mean(v) for n, v in per.items()}
    stages["dispatch"] = statistics.mean(disp_ms)
    stages["forward"] = statistics.mean(fwd_ms)
    stages["backward"] = statistics.mean(bwd_ms)
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    value = job_tokens_per_s(world, cfg.L, ms)

    # a kernel timed inside a step that ran power-capped is held to the
    # sustained tensor peak, otherwise to the burst peak
    capped = "sw_power_cap" in (clk or {}).get("reasons", [])
    tpk = pk["bf16_tflops_sustained"] if capped else pk["bf16_tflops"]
    tsrc = f"{src} ({'sustained, sw_power_cap seen' if capped else 'burst'})"
    if identity:
        roof = identity_roofline(cfg, statistics.mean(fwd_ms), pk, src)
    else:
        fl = stage_flops(cfg)
        dom = max(fl, key=lambda n: stages[n])
        ach = fl[dom] / (stages[dom] * 1e-3) / 1e12
        roof = {"kernel": f"moe_gemm_kernel<{dom}>", "bound": "tensor", "achieved": ach, "peak": tpk,
                "unit": "TFLOP/s", "frac": ach / tpk, "traffic": traffic_per_launch(cfg.name, dom, GEMM_SRC), "peak_source": tsrc,
                "algorithmic_flops": fl[dom],
                "gemm_tflops_all_stages": sum(fl.values()) / (sum(stages[n] for n in fl) * 1e-3) / 1e12}
    db = dispatch_bytes(cfg)
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded counter-based generator; random-init weights)",
        "config": {"workload": cfg.name, "L": cfg.L, "d": cfg.d, "h": cfg.h, "E": cfg.E, "K": cfg.K,
                   "act": cfg.act, "tokens_per_step_per_gpu": cfg.L, "l2": "flushed between steps (256 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "stages_ms": stages,
        "dispatch_build": {"ms": stages["dispatch"], "algorithmic_bytes": db,
                           "GB_per_s": db / (stages["dispatch"] * 1e-3) / 1e9},
        "roofline": roof,
        "gpu_launches": int(launches),
        "gpu_launches_per_step": launches / max(1, args.steps),
        "clocks": clk,
        "activation_memory": memory_report(cfg, layer, step_alloc_peak),
    }
    if router is not None:
        out["router"] = router
    if not args.no_graph_leg:
        out["graph_step"] = run_graph_leg(args, layer, inp, flush, statistics.mean(step_ms))
    if not args.no_e2e:
        out["e2e"] = run_e2e(args, cfg, layer, inp, dev, world)
    del layer
    torch.cuda.empty_cache()
    if not identity and cfg.dtype == "bf16" and not args.no_recompute_leg:
        out["recompute_h"] = run_recompute_leg(args, cfg, inp, dev, flush, pk, tpk)
    del flush
    return out, inp


def run_recompute_leg(args, cfg, inp, dev, flush, pk, tpk):
    """The same step with MOEBLAZE_RECOMPUTE_H (no H / Hg temporaries; the
    down projection and dW3 recompute them from the saved A, B): step time,
    GEMM stage times and activation memory, beside the default above."""
    from mixture_experts_atomic_gb300.layer import MoELayer
    layer = MoELayer.for_config(cfg, dev, with_dgates=False, recompute_h=True)
    W = (inp.get("W1"), inp.get("W2"), inp.get("W3"))

    def step():
        layer.dispatch(inp["ids"])
        layer.forward(inp["x"], inp["gates"], *W)
        layer.backward(inp["dY"], inp["x"], inp["gates"], *W)

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    n = min(args.steps, 10)
    # in this mode the backward runs its dW3 GEMM first (see moeblaze_set_stage_events)
    names_f, names_b = ["up", "down", "convert_y"], ["dw3", "dh", "dx", "dw12", "convert_dx"]
    per = {k: [] for k in names_f + names_b}
    tot = []
    for _ in range(n):
        flush_l2(flush)
        fw, bw = B.StageEvents(4), B.StageEvents(6)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.dispatch(inp["ids"])
        with fw:
            layer.forward(inp["x"], inp["gates"], *W)
        with bw:
            layer.backward(inp["dY"], inp["x"], inp["gates"], *W)
        e1.record()
        torch.cuda.synchronize()
        tot.append(e0.elapsed_time(e1))
        for k, v in zip(names_f, fw.elapsed_ms()):
            per[k].append(v)
        for k, v in zip(names_b, bw.elapsed_ms()):
            per[k].append(v)
    assert layer.device_error() == 0, "device error in the recompute leg"
    stages = {k: statistics.mean(v) for k, v in per.items()}
    fl = stage_flops(cfg)
    ms = statistics.mean(tot)
    out = {"ms_per_step": ms, "value": cfg.L / (ms * 1e-3), "unit": "tokens/s", "steps": n, "stages_ms": stages,
           "tflops": {k: fl[k] / (stages[k] * 1e-3) / 1e12 for k in fl},
           "frac_of_peak": {k: fl[k] / (stages[k] * 1e-3) / 1e12 / tpk for k in fl},
           "activation_memory": memory_report(cfg, layer, 0)}
    del layer
    torch.cuda.empty_cache()
    return out


def identity_roofline(cfg, t_ms, pk, src):
    """Roofline of one identity gather/combine pass against the HBM copy
    bandwidth, on the bytes the pass must move (identity_bytes); the
    every-routed-row figure is reported beside it."""
    nbytes = identity_bytes(cfg)
    ach = nbytes / (t_ms * 1e-3) / 1e9
    rb = identity_routed_bytes(cfg)
    return {"kernel": "identity_combine_kernel (forward pass)", "bound": "hbm", "achieved": ach,
            "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
            "traffic": traffic_per_launch(cfg.name, "identity_forward", IDENTITY_SRC),
            "peak_source": src, "algorithmic_bytes": nbytes, "ms": t_ms,
            "routed_row_bytes": rb, "routed_row_GB_per_s": rb / (t_ms * 1e-3) / 1e9}


def run_graph_leg(args, layer, inp, flush, eager_ms):
    """The same step captured once as a CUDA graph (layer.GraphStep) and
    replayed: what one graph launch saves over a host call per kernel."""
    from mixture_experts_atomic_gb300.layer import GraphStep
    g = GraphStep(layer, inp)
    ms = time_calls(g.replay, flush, args.warmup, min(args.steps, 10))
    torch.cuda.synchronize()
    assert layer.device_error() == 0, "device error in the graph leg"
    del g
    return {"ms": ms, "eager_ms": eager_ms, "saved_ms": eager_ms - ms}


def time_calls(fn, flush, warmup, iters):
    """Median CUDA-event time (ms) of fn() on the current stream, L2 flushed
    before every call."""
    for _ in range(warmup):
        flush_l2(flush)
        fn()
    ts = []
    for _ in range(iters):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def run_routing_stress(cfg, dev, warmup, iters, pk, src, flush, combine=True):
    """The dispatch build and the identity gather/combine on the routing
    stress workload (Zipf ids over 256 experts), measured on their own:
    the dispatch build from the ids alone, then one identity forward pass
    (gather through expert_token_indices, gate-weighted combine) over x."""
    ids, gates = I.make_routing(cfg, None, dev)
    shape = B.make_shape(cfg.L, cfg.d, cfg.h, cfg.E, cfg.K, cfg.torch_dtype, cfg.act)
    disp = B.alloc_dispatch(shape, dev)
    n0 = B.moeblaze_kernel_launches()
    ms = time_calls(lambda: B.dispatch_build(shape, ids, disp), flush, warmup, iters)
    per_build = (B.moeblaze_kernel_launches() - n0) / (warmup + iters)
    assert B.device_error(shape, disp) == 0
    nb = dispatch_bytes(cfg)
    kb = dispatch_kernel_bytes(cfg)
    ach = nb / (ms * 1e-3) / 1e9
    out = {"dispatch_build": {
        "workload": cfg.name, "ms": ms, "algorithmic_bytes": nb, "GB_per_s": ach, "launches_per_build": per_build,
        "kernel_bytes": kb, "kernel_GB_per_s": kb / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / pk["hbm_gbs"], "peak_source": src}}}
    if combine:
        x = I.make_x(cfg, dev)
        y = torch.empty_like(x)
        lb = B.alloc_layer(shape, dev)
        t = time_calls(lambda: B.forward(shape, x, gates, disp, None, None, None, y, lb), flush, warmup, iters)
        assert B.device_error(shape, disp) == 0
        out["identity_combine"] = identity_roofline(cfg, t, pk, src)
        out["identity_combine"]["workload"] = cfg.name
        del x, y
    del ids, gates, disp
    return out


def fp32_alu_tflops(pk):
    """CUDA-core fp32 peak: 152 SMs x 128 fp32 lanes x 2 FLOP (FMA) x the
    maximum SM clock (MEASURED_PEAKS' sm_max_mhz, else 2070 MHz)."""
    mhz = pk.get("sm_max_mhz", 2070.0)
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def run_router(cfg, inp, dev, flush, pk, iters=10):
    """The workload's softmax router (the step before the dispatch) and its
    backward, and the router followed by the dispatch build (two calls, and
    the fused call), timed outside the layer step with CUDA events, L2
    flushed before each call.  Algorithmic bytes: forward x read, ids and gates
    written, Wr read; backward x read, dx written, ids/gates/dgates read, Wr
    read, dWr written.  FLOPs 2LdE (forward) and 4LdE (backward)."""
    from mixture_experts_atomic_gb300 import binding as B
    x = inp["x"]
    Wr, b = I.router_weights(cfg, dev)
    sh = B.make_shape(cfg.L, cfg.d, cfg.h, cfg.E, cfg.K, cfg.torch_dtype, cfg.act)
    ids = torch.empty((cfg.L, cfg.K), dtype=torch.int32, device=dev)
    gates = torch.empty((cfg.L, cfg.K), dtype=torch.float32, device=dev)
    dg = torch.randn(cfg.L, cfg.K, device=dev)
    dWr, db, dx = torch.empty_like(Wr), torch.empty(cfg.E, device=dev), torch.empty_like(x)
    ws = torch.empty(B.moeblaze_router_backward_workspace_bytes(sh), dtype=torch.uint8, device=dev)
    disp = B.alloc_dispatch(sh, dev)
    rd_ws = torch.empty(B.moeblaze_router_dispatch_workspace_bytes(sh), dtype=torch.uint8, device=dev)
    calls = {"forward": lambda: B.router_forward(sh, x, Wr, b, ids, gates),
             "backward": lambda: B.router_backward(sh, x, Wr, ids, gates, dg, dWr, db, dx, ws),
             # the router and the dispatch build: two calls, and the fused call
             "forward_then_dispatch": lambda: (B.router_forward(sh, x, Wr, b, ids, gates),
                                               B.dispatch_build(sh, ids, disp)),
             "fused_router_dispatch": lambda: B.router_dispatch_build(sh, x, Wr, b, ids, gates, disp, rd_ws)}
    s_x = cfg.L * cfg.d * cfg.elem_bytes
    # router + dispatch: x read, ids and gates written, D1, D3, D4 written (the
    # bytes the pair must move; the dispatch's bitmap is not counted)
    rd = s_x + 8 * cfg.L * cfg.K + 4 * cfg.d * cfg.E + 12 * cfg.L * cfg.K
    work = {"forward": (s_x + 8 * cfg.L * cfg.K + 4 * cfg.d * cfg.E, 2 * cfg.L * cfg.d * cfg.E),
            "backward": (2 * s_x + 12 * cfg.L * cfg.K + 8 * cfg.d * cfg.E, 4 * cfg.L * cfg.d * cfg.E),
            "forward_then_dispatch": (rd, 2 * cfg.L * cfg.d * cfg.E),
            "fused_router_dispatch": (rd, 2 * cfg.L * cfg.d * cfg.E)}
    alu = fp32_alu_tflops(pk)
    ridge = alu * 1e12 / (pk["hbm_gbs"] * 1e9)  # FLOP per byte where the two bounds meet
    out = {"fp32_alu_peak_tflops": alu}
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        ts = []
        for _ in range(iters):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.median(ts)
        nbytes, flops = work[name]
        if flops / nbytes > ridge:
            ach = flops / (ms * 1e-3) / 1e12
            roof = {"bound": "alu", "achieved": ach, "peak": alu, "unit": "TFLOP/s", "frac": ach / alu}
        else:
            ach = nbytes / (ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"]}
        if name == "fused_router_dispatch" and cfg.dtype == "bf16" and cfg.E <= 64 and cfg.L >= 128:
            # the fused kernel (bf16 x, E <= 64, L >= 128) runs the logits on the tensor cores: its bound is HBM
            ach = nbytes / (ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"]}
        out[name] = {"ms": ms, "algorithmic_bytes": nbytes, "flops": flops, "roofline": roof}
    return out


def run_e2e(args, cfg, layer, inp, dev, world):
    """The same step through the library's pipelined step runner
    (layer.StepPipeline): every step's inputs come from pinned host memory
    and its y and dX go back to pinned host memory, all inside the timed
    region; the copies of neighbouring steps overlap the compute."""
    from mixture_experts_atomic_gb300.layer import StepPipeline
    keys = ("x", "ids", "gates", "dY")
    host = {k: inp[k].cpu().pin_memory() for k in keys}
    # one host output pair serves every step: the output stream copies into
    # it one step after another
    out = (torch.empty(layer.y.shape, dtype=layer.y.dtype).pin_memory(),
           torch.empty(layer.dX.shape, dtype=layer.dX.dtype).pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out)
    W = (inp.get("W1"), inp.get("W2"), inp.get("W3"))
    pipe = StepPipeline(layer, keys)

    def run(n):
        pipe.run([host] * n, [out] * n, W)

    run(max(2, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # at most 20 steps: on the largest layers each step moves ~100 GB over the host link
    n = min(args.steps, 20)
    e0.record()
    run(n)
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / n, world, dev)
    return {"value": job_tokens_per_s(world, cfg.L, ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n,
            "copies": "overlapped with the neighbouring steps' compute"}


def run_dispatch_only(args, local_rank):
    """The dispatch build alone on the workload's routing (ids only; no
    activations or weights are allocated), CUDA-event timed, L2 flushed."""
    cfg = I.CONFIGS[args.config]  # already scaled by --tokens
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ids, _ = I.make_routing(cfg, None, dev) if cfg.router == "zipf" else I.make_routing(cfg, I.make_x(cfg, dev), dev)
    shape = B.make_shape(cfg.L, cfg.d, cfg.h, cfg.E, cfg.K, cfg.torch_dtype, cfg.act)
    disp = B.alloc_dispatch(shape, dev)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    ms = time_calls(lambda: B.dispatch_build(shape, ids, disp), flush, args.warmup, args.steps)
    assert B.device_error(shape, disp) == 0
    nb = dispatch_bytes(cfg)
    kb = dispatch_kernel_bytes(cfg)
    pk, src = peaks()
    ach = nb / (ms * 1e-3) / 1e9
    return {"metric": "dispatch build HBM GB/s", "config": {"workload": cfg.name, "L": cfg.L, "E": cfg.E, "K": cfg.K},
            "ms": ms, "algorithmic_bytes": nb, "kernel_bytes": kb, "kernel_GB_per_s": kb / (ms * 1e-3) / 1e9,
            "steps": args.steps, "warmup": args.warmup,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / pk["hbm_gbs"], "peak_source": src}}


def run_reference(args, cfg):
    """The CPU oracle as the reference arm: each step runs it on a bounded
    sample of the workload's tokens (same shapes otherwise).  Its inputs are
    generated on the host (the weights once)."""
    # each step's sample is sized so that all warm-up and timed steps take
    # about 150 s together (at most 6 s a step)
    per_step = max(0.1, min(6.0, 150.0 / (args.steps + args.warmup)))
    host = HostInputs(cfg)
    tps, ntok, dt = oracle_sample(cfg, host, target_s=3 * per_step)
    inp = host.rows(ntok)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle_run(cfg, inp)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    v = ntok / statistics.mean(times)
    cores = cpu_cores()
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded counter-based generator; random-init weights)",
            "config": {"workload": cfg.name, "L": cfg.L, "d": cfg.d, "h": cfg.h, "E": cfg.E, "K": cfg.K,
                       "act": cfg.act},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "machine": platform.machine(),
                             "sample": f"first {ntok} tokens of the workload per step (same d, h, E, K)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3,
                    help="workload index (0..4); default: the Mixtral-like SwiGLU bf16 layer, the largest GEMM workload")
    ap.add_argument("--no-routing-stress", action="store_true",
                    help="skip the dispatch build and identity gather/combine measured on the routing stress workload")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the workload with this many tokens instead (smaller profiling captures)")
    ap.add_argument("--experts", type=int, default=None,
                    help="run the workload with this many experts instead (smaller profiling captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="keep the raw nvidia-smi clock samples of the timed region at this path ({rank} is replaced)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph-leg", action="store_true",
                    help="skip timing the step replayed as a captured CUDA graph")
    ap.add_argument("--no-recompute-leg", action="store_true",
                    help="skip timing the step again with MOEBLAZE_RECOMPUTE_H (no H / Hg temporaries)")
    ap.add_argument("--only", choices=["dispatch", "router"], default=None,
                    help="time only the dispatch build of the workload (allocates only its routing and index buffers), "
                         "or only its router legs (x, the router's weights and outputs, the index buffers)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = I.CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.scaled(L=args.tokens, name=f"{cfg.name}_tokens{args.tokens}")
        I.CONFIGS[args.config] = cfg
    if args.experts:
        cfg = cfg.scaled(E=args.experts, name=f"{cfg.name}_experts{args.experts}")
        I.CONFIGS[args.config] = cfg

    if args.only == "dispatch":
        if rank == 0:
            print(json.dumps(run_dispatch_only(args, local_rank)), flush=True)
        return
    if args.only == "router":
        if rank == 0:
            cfg = I.CONFIGS[args.config]
            torch.cuda.set_device(local_rank)
            dev = torch.device("cuda", local_rank)
            flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
            pk, _ = peaks()
            out = run_router(cfg, {"x": I.make_x(cfg, dev)}, dev, flush, pk, iters=args.steps)
            print(json.dumps({"metric": "router legs", "config": {"workload": cfg.name}, "router": out}), flush=True)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, cfg)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    B.lib()
    out, inp = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on the first tokens of the same inputs (copied to the host)
        host = HostInputs(cfg, inp)
        tps, ntok, dt = oracle_sample(cfg, host)
        del host
        out["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                               "machine": platform.machine(),
                               "sample": f"first {ntok} tokens of the workload (same d, h, E, K), "
                                         f"{dt:.1f} s of fp64 CPU work"}
    del inp
    torch.cuda.empty_cache()
    stress = I.CONFIGS[4]
    if not args.no_routing_stress and cfg.act != "identity":
        # the dispatch build and the gather/combine on the workload whose
        # index structures are largest (2M tokens, 256 experts, Zipf ids)
        dev = torch.device("cuda", local_rank)
        flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        pk, src = peaks()
        out["routing_stress"] = run_routing_stress(stress, dev, args.warmup, min(args.steps, 20), pk, src, flush)
        del flush
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
