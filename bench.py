"""Benchmark of the LoRA MLP forward + backward on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one lora_mlp_fwd + lora_mlp_bwd of the Llama-3-8B-shaped LoRA SwiGLU MLP
(T = 4 x 2048 tokens, d = 4096, n = 14336, r = 16, alpha = 32, bf16 base) on seeded synthetic
inputs already resident in HBM.  The working set (weights 336 MiB, activations > 1 GiB) is
larger than the 129 MB L2, so no flush is needed between steps.  Multi-GPU runs are replicas
(the path has no exchange step): every rank runs the same step on its own GPU and the value is
the tokens all ranks processed divided by the slowest rank's time.

--impl reference times the fp64 CPU oracle on the host cores (rank 0 only), each step a
bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
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

METRIC = "LoRA-MLP fwd+bwd tokens/s and TFLOP/s (frac. of BF16 roofline), 1×GB300"
METRICS = {"mlp": METRIC,
           "qkv": "LoRA-QKV fwd+bwd tokens/s and TFLOP/s (frac. of BF16 roofline), 1×GB300",
           "o": "LoRA-O fwd+bwd tokens/s and TFLOP/s (frac. of BF16 roofline), 1×GB300",
           "relu2": "LoRA ReLU^2-MLP fwd+bwd tokens/s and TFLOP/s (frac. of BF16 roofline), 1×GB300"}
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "llama3_8b_mlp_bf16"
NF4_WORKLOAD = "llama3_8b_mlp_nf4"
NOMINAL_BF16_TFLOPS = 2250.0  # dense bf16 tensor peak of one GB300, nominal (no sparsity)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def mlp_flops(T, d, n, r):
    """Algorithmic flops of one fwd+bwd: six base GEMMs (3 forward, dh, 2 in dX) and the rank-r
    products of the three projections (forward X A^T, (XA) B^T; backward G = dOut B, dA, dB, G A)."""
    return 12 * T * d * n + 18 * T * r * (d + n)


def proj_flops(T, d_in, d_out, r):
    """One LoRA projection fwd + bwd: base GEMMs X W^T and dOut W, rank-r products of both passes."""
    return 4 * T * d_in * d_out + 6 * T * r * (d_in + d_out)


def workload_flops(w):
    return sum(proj_flops(w.T, p.d_in, p.d_out, w.r) for p in w.projs)


def kernel_flops(tag, w):
    """Algorithmic flops of one launch of the tagged base-GEMM kernel (rank-r terms at rank r)."""
    T, r = w.T, w.r
    if w.kind == "mlp":
        d, n = w.projs[0].d_in, w.projs[0].d_out
        return {
            "mlp.gateup": 2 * T * d * 2 * n + 2 * 2 * T * r * n,
            "mlp.down": 2 * T * n * d + 2 * T * r * d,
            "mlp.dh": 2 * T * d * n + 2 * T * r * n,
            "mlp.dX": 2 * T * 2 * n * d + 2 * 2 * T * r * d,
        }.get(tag)
    base = sum(2 * T * p.d_in * p.d_out for p in w.projs)
    rank_out = sum(2 * T * r * p.d_out for p in w.projs)
    rank_in = sum(2 * T * r * p.d_in for p in w.projs)
    if w.kind == "relu2":
        d, n = w.projs[0].d_in, w.projs[0].d_out
        return {
            "relu2.up": 2 * T * d * n + 2 * T * r * n,
            "relu2.down": 2 * T * n * d + 2 * T * r * d,
            "relu2.dh": 2 * T * d * n + 2 * T * r * n,
            "relu2.dX": 2 * T * n * d + 2 * T * r * d,
        }.get(tag)
    return {"qkv.fwd": base + rank_out, "qkv.dX": base + rank_in,
            "o.fwd": base + rank_out, "o.dX": base + rank_in}.get(tag)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def step_roofline(tflops_per_gpu, peaks, peak_src):
    """The whole step's TFLOP/s per GPU against the burst bf16 figure (the headline fraction: the
    timed region lasts well under a second, short of the seconds-long loop the sustained figure
    was measured over), and against the sustained figure and the nominal dense bf16 peak."""
    return {"bound": "tensor", "achieved": tflops_per_gpu, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": tflops_per_gpu / peaks["bf16_tflops"],
            "peak_source": peak_src + " burst bf16",
            "frac_of_burst": tflops_per_gpu / peaks["bf16_tflops"],
            "frac_of_sustained": tflops_per_gpu / peaks["bf16_tflops_sustained"],
            "frac_of_nominal": tflops_per_gpu / NOMINAL_BF16_TFLOPS}


def src_digest():
    """Digest of the code of the GEMM kernel templates (the kernels the traffic figures are for):
    line comments, trailing blanks and blank lines are left out, so a comment edit keeps it."""
    h = hashlib.sha256()
    for f in [os.path.join(ROOT, "bwd_lora_mlp_gb300", "csrc", x) for x in ("lm_gemm.cuh", "lm_gemm2.cuh", "lm_gemm2_nf4.cuh", "lm_ptx.cuh")]:
        with open(f, encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(tag, workload):
    """DRAM bytes per launch of `tag` from the committed ncu summary, if it was taken on the
    current kernel sources; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rows = json.load(f)
    except Exception:
        return None
    dig = src_digest()
    for r in rows:
        if r.get("tag") == tag and r.get("workload") == workload and r.get("src_digest") == dig:
            return r.get("bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap",
              "enforced.power.limit"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_id)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        def num(i):
            out = []
            for r in rows:
                try:
                    out.append(float(r[i]))
                except ValueError:
                    pass
            return out
        plim = num(9)
        # the enforced power limit: tensor-bound kernels run at the power cap, so the limit of the
        # GPU at hand sets their clock (the sampled draw is a trailing average, too slow to follow a
        # sub-second timed region, and is not reported)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows), "power_limit_w": max(plim) if plim else None}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# the oracle on host cores (reference arm and cpu_baseline)

def oracle_step(w, inp64, Ts):
    from oracle import lora as O
    p = inp64["p"]
    X = inp64["X"][:Ts]
    dY = inp64["dY"][:Ts]
    O.mlp_backward(X, dY, p, w.act)


def oracle_inputs(w, inp):
    from oracle import lora as O
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = O.from_bf16(inp["W_" + t])
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    return {"p": p, "X": O.from_bf16(inp["X"]), "dY": O.from_bf16(inp["dY"])}


def pick_sample(w, inp64, budget_s):
    Ts = 64
    t0 = time.perf_counter()
    oracle_step(w, inp64, Ts)
    dt = time.perf_counter() - t0
    Ts = int(min(w.T, max(64, Ts * budget_s / max(dt, 1e-3))) // 64 * 64)
    return max(Ts, 64)


def cpu_baseline(w, inp, budget_s=12.0):
    inp64 = oracle_inputs(w, inp)
    Ts = pick_sample(w, inp64, budget_s)
    t0 = time.perf_counter()
    oracle_step(w, inp64, Ts)
    dt = time.perf_counter() - t0
    return {"value": Ts / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": "fp64 numpy oracle fwd+bwd of %d of the %d tokens, full d=%d, n=%d, r=%d; %.1f s"
                      % (Ts, w.T, w.projs[0].d_in, w.projs[0].d_out, w.r, dt)}


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    from bwd_lora_mlp_gb300 import synth
    inp = synth.make_inputs(w)
    inp64 = oracle_inputs(w, inp)
    # tokens per step sized so that the warm-up and timed steps together take about two minutes
    # (at most 2 s a step, at least the 64-token minimum sample)
    Ts = pick_sample(w, inp64, min(2.0, max(0.1, 120.0 / (args.steps + args.warmup))))
    for _ in range(args.warmup):
        oracle_step(w, inp64, Ts)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, inp64, Ts)
    dt = (time.perf_counter() - t0) / args.steps
    v = Ts / dt
    d, n = w.projs[0].d_in, w.projs[0].d_out
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "d": d, "n": n, "r": w.r, "alpha": w.alpha, "act": w.act,
                       "tokens_per_step": Ts},
            "tflops": mlp_flops(Ts, d, n, w.r) / dt / 1e12,
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": "%d tokens of %d per step" % (Ts, w.T)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the workload's shapes with this many tokens (small cases for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-nf4", action="store_true", help="skip the NF4-base step the default run adds")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from bwd_lora_mlp_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.tokens:
        w = synth.scaled_workload(w, T=args.tokens)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        assert w.kind == "mlp", "the reference arm times the MLP oracle"
        rc = run_reference(args, w, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc

    import torch
    import __graft_entry__
    __graft_entry__.build()

    rec = measure(w, args, world, local, e2e=True)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and w.kind == "mlp":
        cpu = cpu_baseline(w, rec.pop("_inputs"))
    rec.pop("_inputs", None)
    line = {
        "metric": METRICS[w.kind], "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded W~N(0,0.02), A~U(+-1/sqrt(in)), B~N(0,0.02), X~N(0,1), dY~N(0,0.01), bf16",
        "config": rec["config"],
        "tflops": rec["tflops"],
        "roofline_step": rec["roofline_step"],
        "roofline": rec["roofline"],
        "gpu_launches": rec["gpu_launches"],
        "kernels_ms_per_step": rec["kernels_ms_per_step"],
        "clocks": rec["clocks"],
        "e2e": rec["e2e"],
        "cpu_baseline": cpu,
    }
    # the default run also times the same MLP on an NF4-packed base (QLoRA), in the same process
    # after the headline: its own step time, roofline and kernel times, nested under "nf4"
    if args.workload == DEFAULT_WORKLOAD and not args.tokens and not args.no_nf4:
        wn = synth.WORKLOADS[NF4_WORKLOAD]
        rn = measure(wn, args, world, local, e2e=False)
        rn.pop("_inputs", None)
        line["nf4"] = {k: rn[k] for k in ("ms_per_step", "value", "tflops", "config", "roofline_step", "roofline",
                                          "gpu_launches", "kernels_ms_per_step", "clocks")}
        line["nf4"]["metric"] = METRICS["mlp"].replace("LoRA-MLP", "QLoRA-MLP (NF4 base)")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure(w, args, world, local, e2e=True):
    """Time args.steps steps of workload w (after args.warmup untimed ones) with CUDA events on the
    launching stream; then the same steps with the library's launch tracing for per-kernel times;
    then (e2e) the end-to-end figure through the C ABI from pinned host buffers."""
    import torch
    from bwd_lora_mlp_gb300 import lib as L
    from bwd_lora_mlp_gb300 import synth

    T, r = w.T, w.r
    inp = synth.make_inputs(w)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    def host_pinned(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()

    ab32 = synth.fp32_ab(w) if w.ab_f32 else None  # fp32 LoRA parameters: each call rounds them to bf16

    def mk(t):
        W = dev(inp["W_" + t])
        if w.nf4:  # quantise the frozen base on the device; packing is not part of the step
            W = L.nf4_pack(W)
        elif w.int4_group:
            W = L.int4_pack(W, w.int4_group)
        elif w.nvfp4:
            W = L.nvfp4_pack(W)
        if ab32 is not None:
            return L.Lora(W, torch.from_numpy(ab32["A_" + t]).cuda(), torch.from_numpy(ab32["B_" + t]).cuda(), w.s)
        return L.Lora(W, dev(inp["A_" + t]), dev(inp["B_" + t]), w.s)

    projs = {p.name: mk(p.name) for p in w.projs}
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # the step's inputs, in the order run() takes them
    in_names = ["X", "dY_q", "dY_k", "dY_v"] if w.kind == "qkv" else ["X", "dY"]
    ins = [dev(inp[k]) for k in in_names]

    if w.kind == "mlp":
        gate, up, down = projs["gate"], projs["up"], projs["down"]
        fw = L.lora_mlp_fwd(ins[0], gate, up, down, act=w.act)
        bw = L.lora_mlp_bwd(ins[0], ins[1], fw, gate, up, down, act=w.act)
        out_keys = ["y"]

        def run(xs, outs):
            L.lora_mlp_fwd(xs[0], gate, up, down, act=w.act, y=outs["y"], e=fw["e"], u=fw["u"], h=fw["h"],
                           saved=fw["saved"], ws=fw["ws"])
            L.lora_mlp_bwd(xs[0], xs[1], fw, gate, up, down, act=w.act, dX=outs["dX"],
                           grads={k: outs[k] for k in outs if k not in ("y", "dX")})
    elif w.kind == "relu2":
        up, down = projs["up"], projs["down"]
        fw = L.lora_relu2_mlp_fwd(ins[0], up, down)
        bw = L.lora_relu2_mlp_bwd(ins[0], ins[1], fw, up, down)
        out_keys = ["y"]

        def run(xs, outs):
            L.lora_relu2_mlp_fwd(xs[0], up, down, y=outs["y"], u=fw["u"], h=fw["h"], saved=fw["saved"], ws=fw["ws"])
            L.lora_relu2_mlp_bwd(xs[0], xs[1], fw, up, down, dX=outs["dX"],
                                 grads={k: outs[k] for k in outs if k not in ("y", "dX")})
    elif w.kind == "qkv":
        q, k_, v_ = projs["q"], projs["k"], projs["v"]
        fw = L.lora_qkv_fwd(ins[0], q, k_, v_)
        bw = L.lora_qkv_bwd(ins[0], ins[1], ins[2], ins[3], fw, q, k_, v_)
        out_keys = ["Q", "K", "V"]

        def run(xs, outs):
            L.lora_qkv_fwd(xs[0], q, k_, v_, out={t: outs[t] for t in ("Q", "K", "V")}, saved=fw["saved"],
                           ws=fw["ws"])
            L.lora_qkv_bwd(xs[0], xs[1], xs[2], xs[3], fw, q, k_, v_, dX=outs["dX"],
                           grads={t: outs[t] for t in ("dA_q", "dB_q", "dA_k", "dB_k", "dA_v", "dB_v")})
    else:
        o = projs["o"]
        fw = L.lora_o_fwd(ins[0], o)
        bw = L.lora_o_bwd(ins[0], ins[1], fw, o)
        out_keys = ["Y"]

        def run(xs, outs):
            L.lora_o_fwd(xs[0], o, Y=outs["Y"], saved=fw["saved"], ws=fw["ws"])
            L.lora_o_bwd(xs[0], xs[1], fw, o, dX=outs["dX"], dA=outs["dA"], dB=outs["dB"])

    dev_outs = {**{k: fw[k] for k in out_keys}, **bw}

    def step():
        run(ins, dev_outs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    L.lm_workspace_check(fw["ws"])

    # ---- timed region: inputs resident in HBM
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sampler = ClockSampler("GPU-" + str(props.uuid) if getattr(props, "uuid", None) else local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    L.lm_workspace_check(fw["ws"])
    ms = ev0.elapsed_time(ev1) / args.steps
    # ---- per-kernel times: the same steps again with the library's launch tracing on (an event
    # pair around every launch), kept out of the headline region above
    L.lm_profile_reset()
    L.lm_profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    L.lm_profile_enable(False)
    prof = L.lm_profile_summary()
    L.lm_workspace_check(fw["ws"])
    ms = max_over_ranks(ms, world)

    peaks, peak_src = load_peaks()
    flops = workload_flops(w)
    value = world * T / (ms / 1e3)
    tflops = world * flops / (ms / 1e3) / 1e12
    launches = sum(c for c, _ in prof.values())
    # dominant kernel: the tag with the largest share of the timed region
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    dom_tag, (dom_n, dom_ms) = dom
    per_launch_ms = dom_ms / dom_n
    kf = kernel_flops(dom_tag, w)
    roofline = None
    if kf is not None:
        ach = kf / (per_launch_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]  # burst: the timed region is far shorter than the sustained loop
        roofline = {"bound": "tensor", "kernel": dom_tag, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                    "frac": ach / peak, "traffic": committed_traffic(dom_tag, w.name),
                    "peak_source": peak_src + " burst bf16", "flops_per_launch": kf,
                    "ms_per_launch": per_launch_ms, "frac_of_burst": ach / peak,
                    "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                    "sustained_peak": peaks["bf16_tflops_sustained"]}

    e2e_rec = None
    if e2e:
        # ---- end to end through the C ABI from pinned host buffers: every step copies its inputs in
        # and its results out; the copies of neighbouring steps run on their own streams and overlap
        # the current step's kernels (inputs and outputs are double-buffered on the device)
        host_in = [host_pinned(inp[k]) for k in in_names]
        host_out = [{k: torch.empty_like(v, device="cpu").pin_memory() for k, v in dev_outs.items()} for _ in range(2)]
        dev_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
        dev_out = [{k: torch.empty_like(v) for k, v in dev_outs.items()} for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        for e_ in out_done + comp_done:
            e_.record(stream)

        def e2e_run(nsteps):
            for i in range(nsteps):
                b = i & 1
                with torch.cuda.stream(s_in):          # inputs of step i (after step i-2 stopped reading them)
                    s_in.wait_event(comp_done[b])
                    for dst, src in zip(dev_in[b], host_in):
                        dst.copy_(src, non_blocking=True)
                    in_done[b].record(s_in)
                stream.wait_event(in_done[b])           # step i's kernels
                stream.wait_event(out_done[b])          # after step i-2's results were copied out
                run(dev_in[b], dev_out[b])
                comp_done[b].record(stream)
                with torch.cuda.stream(s_out):         # results of step i
                    s_out.wait_event(comp_done[b])
                    for k, v in host_out[b].items():
                        v.copy_(dev_out[b][k], non_blocking=True)
                    out_done[b].record(s_out)

        # windows of up to 50 steps: the first step's copy-in and the last one's copy-out, which
        # nothing overlaps, are then a small part of a window
        e2e_steps = max(4, min(args.steps, 50))
        e2e_run(2)
        torch.cuda.synchronize()
        barrier(world)
        # five windows of e2e_steps steps each; the median window (the host-copy path shows
        # occasional slow windows)
        windows = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            s_in.wait_stream(stream)
            e2e_run(e2e_steps)
            stream.wait_stream(s_out)
            e1.record(stream)
            torch.cuda.synchronize()
            windows.append(e0.elapsed_time(e1) / e2e_steps)
        e2e_ms = max_over_ranks(statistics.median(windows), world)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
        # the same calls one at a time: a step's copy-in, kernels and copy-out back to back on the
        # launching stream, the host waiting for each step (what one synchronous call costs)
        sync = []
        for _ in range(e2e_steps):
            t0 = time.perf_counter()
            for dst, src in zip(dev_in[0], host_in):
                dst.copy_(src, non_blocking=True)
            run(dev_in[0], dev_out[0])
            for name, buf in host_out[0].items():  # (names that run()'s closure does not use)
                buf.copy_(dev_out[0][name], non_blocking=True)
            stream.synchronize()
            sync.append((time.perf_counter() - t0) * 1e3)
        sync_ms = max_over_ranks(statistics.median(sync), world)
        e2e_rec = {"value": world * T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                   "copies": "pipelined: step i's host copies overlap steps i-1 and i+1",
                   "sync_call": {"ms_per_step": sync_ms, "value": world * T / (sync_ms / 1e3),
                                 "how": "copy-in, fwd+bwd and copy-out of one step, then a host wait; median "
                                        "of %d calls" % e2e_steps}}

    d_in, d_out = w.projs[0].d_in, w.projs[-1].d_out
    cfg = {"workload": w.name, "T": T, "r": r, "alpha": w.alpha, "base": "nf4" if w.nf4 else ("int4_g%d" % w.int4_group if w.int4_group else ("nvfp4" if w.nvfp4 else "bf16")), "lora_params": "fp32" if w.ab_f32 else "bf16"}
    if w.kind in ("mlp", "relu2"):
        cfg.update(d=d_in, n=w.projs[0].d_out, act=w.act)
    else:
        cfg.update(projections={p.name: [p.d_in, p.d_out] for p in w.projs})
    cfg.update(parallelism="replicas" if world > 1 else "single",
               l2="no flush: the working set (weights, activations and saved tensors of the step) exceeds the "
                  "129 MB L2")
    if clocks and clocks.get("sm_mhz"):
        # the step in SM clock cycles at the median clock under load, to read clock dependence
        clocks["step_mcycles_at_median_clock"] = ms * clocks["sm_mhz"] / 1e3
    return {"value": value, "ms_per_step": ms, "tflops": tflops, "config": cfg,
            "roofline_step": step_roofline(tflops / world, peaks, peak_src), "roofline": roofline,
            "gpu_launches": launches, "kernels_ms_per_step": {k: v[1] / args.steps for k, v in prof.items()},
            "clocks": clocks, "e2e": e2e_rec, "_inputs": inp}


if __name__ == "__main__":
    sys.exit(main())
