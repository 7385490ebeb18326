"""Benchmark of the fused AttnRes + add2 + RMSNorm epilogue on GB300.

One step = one call of the whole op (fold, mixture, output norm) over one
batch: the bandwidth workload M=8192 tokens, N=12 snapshots, H=7168, both
addends, BF16 (about 2.0 GB moved per call; inputs larger than L2, so no L2
flush is needed between steps).  `value` is the achieved HBM throughput in
GB/s over all ranks (algorithmic bytes / max-over-ranks time).  The line also
carries the decode-window latencies (M <= 32, microseconds per call), the
roofline of the kernel, the end-to-end figure through the public API with
host buffers, the clocks seen under load, and the CPU oracle's throughput.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: one process per GPU; each rank runs its own batch of 8192 tokens
(tokens are independent, no collective on the data path), so scaling is
weak.  Under torchrun the ranks come from the environment; `--gpus N` with
N > 1 outside torchrun starts the N ranks itself (torch.distributed.run on
this node).  `--dry-run` runs the rank set-up, barriers, timing and
max-over-ranks on the host only (gloo, no GPU, no kernel) to check that
logic; its line says so and is not a measurement.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused AttnRes+add2+RMSNorm µs/call (M≤32) and HBM GB/s vs roofline (M=8192)"
UNIT = "GB/s"
WORKLOAD = "bandwidth-bound: M=8192 tokens, N=12 snapshots, H=7168, add2 present, BF16, N(0,1) inputs, eps=1e-6"
M_BW, N_BW, H = 8192, 12, 7168
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attnres_fused_M8192_N12_traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "kimi_k3_attention_gb300", "csrc", f)
                  for f in ("attnres_kernel.cuh", "attnres_launch.cuh", "attnres_api.cu")]


def algorithmic_bytes(M, N, H, has_add2=True):
    R = M * H * 2
    return (N + (3 if has_add2 else 2)) * R + 2 * R + 4 * H


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def free_port():
    import socket
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    return port


def launch_ranks(argv, gpus):
    """Start `gpus` ranks of this script on this node under
    torch.distributed.run (rendezvous on 127.0.0.1) with the same arguments;
    returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def rank_seed(rank):
    """Every rank draws its own 8192-token batch (weak scaling)."""
    return 4 + rank


def max_over_ranks(x, device):
    """Max of a host float over all ranks of the default process group (the
    timing rule: the slowest rank sets the time); identity when not
    distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(nbytes_per_call, world_size, steps, seconds):
    """Whole-job GB/s: every rank moved nbytes_per_call per step."""
    return nbytes_per_call * world_size * steps / seconds / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the kernel sources as they are now; else None."""
    try:
        kv = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_digest") != kernel_source_digest():
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), active=parts[4],
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8],
                                 util=float(parts[9])))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        load = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in load:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in load),
                "reasons": sorted(reasons), "samples": len(load)}


# ---------------------------------------------------------------- CPU oracle leg

def oracle_throughput(inp_cpu, budget_s, chunk=64, max_tokens=None):
    """Time the CPU oracle, as it stands, on whole chunks of tokens of `inp_cpu`
    until `budget_s` has elapsed.  Returns (GB/s, tokens, seconds, outputs)."""
    import numpy as np
    import torch
    from oracle import attnres_add_rmsnorm as oracle_op

    def u(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    arrs = [u(inp_cpu.prefix), u(inp_cpu.add), u(inp_cpu.add2), u(inp_cpu.bank),
            u(inp_cpu.w), u(inp_cpu.gamma)]
    M = inp_cpu.M
    done, t0 = 0, time.perf_counter()
    results = []
    while True:
        toks = np.arange(done, min(done + chunk, M))
        results.append((toks, oracle_op(*arrs, inp_cpu.eps, tokens=toks, chunk=chunk)))
        done = toks[-1] + 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= M or (max_tokens and done >= max_tokens):
            break
    bytes_ = algorithmic_bytes(done, inp_cpu.N, inp_cpu.H, inp_cpu.add2 is not None) - 4 * inp_cpu.H
    return bytes_ / el / 1e9, int(done), el, results


def oracle_per_config(reps=3):
    """The CPU oracle as it stands, on the host cores, per workload
    configuration: the PR reference case (M=4, N=3), all 96 decode-sweep
    cases, the bit-exactness stress case (M=32, N=12) and the 25-layer chain
    (M=8, bank growing 1 -> 12), each in full; median of `reps` runs, one
    thread.  Seconds per call (per chain for the chain) and GB/s of the
    algorithmic bytes."""
    import numpy as np
    import torch
    from kimi_k3_attention_gb300 import workloads as wl
    from oracle import attnres_add_rmsnorm as oop

    def u(t):
        return None if t is None else t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def args_of(inp):
        return (u(inp.prefix), u(inp.add), u(inp.add2), u(inp.bank), u(inp.w), u(inp.gamma), inp.eps)

    def med(fn):
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return statistics.median(ts)

    def row(seconds, nbytes, **kw):
        return dict(kw, s_per_call=round(seconds, 6), gbs=round(nbytes / seconds / 1e9, 4))

    res = {}
    pr = wl.pr_reference_case()
    a = args_of(pr)
    res["pr_reference_M4_N3"] = row(med(lambda: oop(*a)), algorithmic_bytes(4, 3, pr.H))
    cases = [(M, N, ad, args_of(wl.decode_sweep_inputs(i, M, N, ad)))
             for i, M, N, ad in wl.decode_sweep_cases()]
    t = med(lambda: [oop(*c[3]) for c in cases])
    nb = sum(algorithmic_bytes(M, N, H, ad) for M, N, ad, _ in cases)
    res["decode_sweep_96_cases"] = row(t / len(cases), nb / len(cases), cases=len(cases),
                                       s_all_cases=round(t, 4))
    st = wl.stress_inputs(special_prefix=True)
    a = args_of(st)
    res["stress_M32_N12"] = row(med(lambda: oop(*a)), algorithmic_bytes(32, 12, H))
    emb, p0, layers = wl.chain_inputs(M=8, H=H, layers=25)

    def chain():
        bank, P = [u(emb)], u(p0)
        for li, L in enumerate(layers):
            P, _, _ = oop(P, u(L.routed), u(L.shared), np.stack(bank), u(L.w), u(L.gamma), wl.EPS)
            if wl.chain_appends_after(li):
                bank.append(P.copy())
    nb, n = 0, 1
    for li in range(25):
        nb += algorithmic_bytes(8, n, H)
        n += 1 if wl.chain_appends_after(li) else 0
    res["chain_25_layers_M8"] = row(med(chain), nb, unit_of_s="per 25-layer chain")
    model, ncpu = cpu_info()
    res.update(threads=1, reps=reps, cpu=model, host_cpus=ncpu,
               note="reported baseline, not a target")
    return res


def cpu_info():
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
    except Exception:
        pass
    import platform
    return model or platform.processor() or platform.machine(), os.cpu_count()


def run_reference(args):
    """The reference arm: the CPU oracle on a bounded sample of the same
    workload, every step a fresh chunk of 32 tokens."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    from kimi_k3_attention_gb300 import workloads as wl
    tokens_per_step = 32
    total = tokens_per_step * (args.steps + args.warmup)
    inp = wl.make_inputs(total, N_BW, H, seed=4, add2=True)
    step_times = []
    for s in range(args.warmup + args.steps):
        sub = wl.Inputs(inp.prefix[s * tokens_per_step:(s + 1) * tokens_per_step],
                        inp.add[s * tokens_per_step:(s + 1) * tokens_per_step],
                        inp.add2[s * tokens_per_step:(s + 1) * tokens_per_step],
                        inp.bank[:, s * tokens_per_step:(s + 1) * tokens_per_step].contiguous(),
                        inp.w, inp.gamma, inp.eps)
        t0 = time.perf_counter()
        oracle_throughput(sub, 0.0, chunk=tokens_per_step)
        if s >= args.warmup:
            step_times.append(time.perf_counter() - t0)
    el = sum(step_times)
    bytes_ = algorithmic_bytes(tokens_per_step, N_BW, H) * args.steps
    value = bytes_ / el / 1e9
    model, ncpu = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{tokens_per_step} tokens per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{tokens_per_step} of the 8192 tokens per step, {args.steps} steps",
                         "cpu": model, "host_cpus": ncpu},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU legs

def after_current(*streams):
    """Order `streams` after the work already queued on the current stream.
    The inputs are drawn there, and the caching allocator may hand a block
    that a queued kernel of the current stream still reads (a float32
    temporary of the draws) to an output buffer: a kernel on another stream
    writing that buffer before the draws finish would corrupt the inputs."""
    import torch
    cur = torch.cuda.current_stream()
    for st in streams:
        st.wait_stream(cur)


def time_bandwidth(binding, inp, steps, warmup, stream, config=None):
    """Set up K back-to-back calls, each to be bracketed by CUDA events on
    `stream`; runs the warm-up calls."""
    import torch
    out = torch.empty_like(inp.prefix)
    newp = torch.empty_like(inp.prefix)
    call = lambda: binding.attnres_add_rmsnorm(inp.prefix, inp.add, inp.add2, inp.bank, inp.w,  # noqa: E731
                                               inp.gamma, inp.eps, out, newp, stream=stream, check=False,
                                               config=config)
    after_current(stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    return call, ev, t_all0, t_all1, out, newp


def _decode_shape_times(binding, M, N, configs, seed, reps=200, replays=20):
    """Microseconds per call at (M, N), H=7168, both addends, for each named
    launch configuration (None = the library's choice), from CUDA-graph
    replays of back-to-back calls on one stream:
      warm: `reps` calls on the same buffers (inputs L2-resident);
      cold: calls cycling through distinct buffer sets whose total exceeds
            2.5x the L2 size, so every call reads its inputs from HBM.
    Each figure is the median over `replays` replays of graph time / calls."""
    import torch
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size or (128 << 20)
    s = torch.cuda.Stream()
    per_set = algorithmic_bytes(M, N, H)
    nsets = max(2, min(4096, -(-int(2.5 * l2) // per_set)))
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    rnd = lambda *shape: torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
    P, A, A2 = rnd(nsets, M, H), rnd(nsets, M, H), rnd(nsets, M, H)
    B = rnd(nsets, N, M, H)
    w = (rnd(H).float() / H ** 0.5).to(torch.bfloat16)
    gam = (1 + 0.1 * rnd(H).float()).to(torch.bfloat16)
    O = torch.empty_like(P)
    NP = torch.empty_like(P)

    def timed(graph, calls):
        out = []
        for _ in range(replays):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                graph.replay()
                e1.record(s)
            e1.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3 / calls)
        return round(statistics.median(out), 3)

    res = {}
    after_current(s)
    for name, cfg in configs.items():
        def call(i, cfg=cfg):
            binding.attnres_add_rmsnorm(P[i], A[i], A2[i], B[i], w, gam, 1e-6, O[i], NP[i],
                                        stream=s, check=False, config=cfg)
        with torch.cuda.stream(s):
            for i in range(min(nsets, 8)):
                call(i)
        torch.cuda.synchronize()
        gw = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gw, stream=s):
            for _ in range(reps):
                call(0)
        gc = torch.cuda.CUDAGraph()
        ncold = max(reps, nsets)
        with torch.cuda.graph(gc, stream=s):
            for k in range(ncold):
                call(k % nsets)
        with torch.cuda.stream(s):
            gw.replay()
            gc.replay()
        torch.cuda.synchronize()
        res[name] = {"warm_us": timed(gw, reps), "cold_us": timed(gc, ncold), "cold_sets": nsets,
                     "plan": binding.attnres_plan(M, N, H) if cfg is None else cfg.as_dict()}
        del gw, gc
    del P, A, A2, B, O, NP
    torch.cuda.synchronize()
    return res


def decode_latencies(binding, wl):
    """The decode window (M <= 32 tokens), automatic launch configuration:
    warm and cold microseconds per call (see _decode_shape_times)."""
    res = {}
    for M in (1, 8, 16, 32):
        for N in (1, 3, 6, 12):
            r = _decode_shape_times(binding, M, N, {"auto": None}, seed=900 + M * 16 + N)["auto"]
            res[f"M{M}_N{N}"] = {"warm_us": r["warm_us"], "cold_us": r["cold_us"],
                                 "cold_sets": r["cold_sets"], "variant": r["plan"]["variant"],
                                 "cluster": r["plan"]["cluster"]}
    return res


def single_cta_vs_cluster(binding):
    """The one-CTA-per-token variant (variant 1, the pages' single-CTA kernel
    for small N, TensorRT-LLM PR #20546 section "Op") against the automatic
    choice (a cluster of CTAs per token) where the single CTA is meant to
    serve: M in {1, 8}, N in {1..4}, warm and cold microseconds per call."""
    res = {}
    for M in (1, 8):
        for N in (1, 2, 3, 4):
            r = _decode_shape_times(binding, M, N, {"auto": None,
                                                    "single_cta": binding.make_config("cta")},
                                    seed=300 + M * 16 + N)
            res[f"M{M}_N{N}"] = {k: {"warm_us": v["warm_us"], "cold_us": v["cold_us"],
                                     "variant": v["plan"]["variant"], "cluster": v["plan"]["cluster"]}
                                 for k, v in r.items()}
    return res


def pattern_ceiling(binding, inp, nbytes, peak, steps=10, warmup=3):
    """GB/s of attnres_access_pattern on the bandwidth workload: the fused
    op's loads, stores, grid and L2 prefetch without its arithmetic (CUDA
    events around each launch on its stream, average)."""
    import torch
    s = torch.cuda.Stream()
    out, newp = torch.empty_like(inp.prefix), torch.empty_like(inp.prefix)

    def call():
        binding.attnres_access_pattern(inp.prefix, inp.add, inp.add2, inp.bank, out, newp, stream=s)
    after_current(s)
    with torch.cuda.stream(s):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(s):
        for a, b in ev:
            a.record(s)
            call()
            b.record(s)
    torch.cuda.synchronize()
    avg = sum(a.elapsed_time(b) for a, b in ev) / steps / 1e3
    nb = nbytes - 4 * H          # no w, gamma
    del out, newp
    return {"gbs": round(nb / avg / 1e9, 1), "avg_launch_us": round(avg * 1e6, 2),
            "frac_of_peak": round(nb / avg / 1e9 / peak, 4),
            "what": "attnres_access_pattern: same loads, stores, grid and L2 prefetch, no arithmetic"}


def _graph_us(build_calls, s, replays=20):
    """Capture build_calls() (which enqueues `n` calls on stream s and returns
    n) in a CUDA graph; median microseconds per call over `replays`."""
    import torch
    after_current(s)
    with torch.cuda.stream(s):
        build_calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        n = build_calls()
    ts = []
    for _ in range(replays + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n)
    del g
    return round(statistics.median(ts[1:]), 3)


def comparators(binding, reps=200):
    """The pages' microbenchmark form (TensorRT-LLM PR #20546, "Performance"):
    the fused op (both addends) against the attention-residual + RMSNorm alone
    and the standalone single-kernel addition it replaces, in microseconds per
    call, warm (same buffers) and cold (buffer sets > 2.5x L2)."""
    import torch
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size or (128 << 20)
    s = torch.cuda.Stream()
    res = {}
    for M in (1, 8, 16, 32):
        for N in (3, 12):
            per = algorithmic_bytes(M, N, H)
            nsets = max(2, min(4096, -(-int(2.5 * l2) // per)))
            g = torch.Generator(device="cuda")
            g.manual_seed(77 + M + N)
            rnd = lambda *sh: torch.randn(sh, generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
            P, A, A2, B = rnd(nsets, M, H), rnd(nsets, M, H), rnd(nsets, M, H), rnd(nsets, N, M, H)
            w = (rnd(H).float() / H ** 0.5).to(torch.bfloat16)
            gam = (1 + 0.1 * rnd(H).float()).to(torch.bfloat16)
            O, NP = torch.empty_like(P), torch.empty_like(P)
            ops = {
                "fused": lambda i: binding.attnres_add_rmsnorm(P[i], A[i], A2[i], B[i], w, gam, 1e-6,
                                                               O[i], NP[i], stream=s, check=False),
                "alone": lambda i: binding.attnres_rmsnorm(P[i], B[i], w, gam, 1e-6, O[i], stream=s),
                "tail_add": lambda i: binding.attnres_tail_add(P[i], A[i], A2[i], NP[i], stream=s),
            }
            row = {}
            for name, op in ops.items():
                def warm(op=op):
                    for _ in range(reps):
                        op(0)
                    return reps

                def cold(op=op):
                    n = max(reps, nsets)
                    for k in range(n):
                        op(k % nsets)
                    return n
                row[name] = {"warm_us": _graph_us(warm, s), "cold_us": _graph_us(cold, s)}
            row["delta_fused_minus_alone_us"] = {
                k: round(row["fused"][k] - row["alone"][k], 3) for k in ("warm_us", "cold_us")}
            res[f"M{M}_N{N}"] = row
            del P, A, A2, B, O, NP
    torch.cuda.synchronize()
    return res


def _domain_row(binding, wl, N, dtype, peak, seed, steps=5, warmup=3):
    """GB/s per call at M = 8192 tokens (inputs larger than L2; CUDA events
    around each call) and warm decode microseconds per call at M = 1 and 32
    (CUDA-graph replays), both addends, for N snapshots of `dtype` tensors."""
    import torch
    s = torch.cuda.Stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    rnd = lambda *sh: torch.randn(sh, generator=g, device="cuda").to(dtype)  # noqa: E731
    P, A, A2, B = rnd(M_BW, H), rnd(M_BW, H), rnd(M_BW, H), rnd(N, M_BW, H)
    w = (torch.randn(H, generator=g, device="cuda") / H ** 0.5).to(dtype)
    gam = (1 + 0.1 * torch.randn(H, generator=g, device="cuda")).to(dtype)
    out, newp = torch.empty_like(P), torch.empty_like(P)

    def call():
        binding.attnres_add_rmsnorm(P, A, A2, B, w, gam, 1e-6, out, newp, stream=s, check=False)
    after_current(s)
    with torch.cuda.stream(s):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(s):
        for a, b in ev:
            a.record(s)
            call()
            b.record(s)
    torch.cuda.synchronize()
    avg = sum(a.elapsed_time(b) for a, b in ev) / steps / 1e3
    nb = algorithmic_bytes(M_BW, N, H)
    row = {"M8192_gbs": round(nb / avg / 1e9, 1), "M8192_us": round(avg * 1e6, 2),
           "M8192_frac": round(nb / avg / 1e9 / peak, 4),
           "plan_M8192": binding.attnres_plan(M_BW, N, H)}
    del P, A, A2, B, out, newp
    torch.cuda.empty_cache()
    for M in (1, 32):
        d = wl.make_inputs(M, N, H, seed=seed + M, device="cuda", dtype=dtype)
        o, npf = torch.empty_like(d.prefix), torch.empty_like(d.prefix)

        def calls(d=d, o=o, npf=npf, reps=100):
            for _ in range(reps):
                binding.attnres_add_rmsnorm(d.prefix, d.add, d.add2, d.bank, d.w, d.gamma, d.eps,
                                            o, npf, stream=s, check=False)
            return reps
        row[f"M{M}_warm_us"] = _graph_us(calls, s)
    torch.cuda.synchronize()
    return row


def deep_banks(binding, wl, peak):
    """Banks deeper than the PR's fused path takes (TensorRT-LLM PR #20546,
    section "Op": N > 12 falls back there), fused here: N = 16, 24 and 31."""
    import torch
    return {f"N{N}": _domain_row(binding, wl, N, torch.bfloat16, peak, 60 + N) for N in (16, 24, 31)}


def fp16_tensors(binding, wl, peak):
    """The op on FP16 tensors (the PR's fused window is BF16), N = 12."""
    import torch
    return {"N12": _domain_row(binding, wl, 12, torch.float16, peak, 90)}


def chain_benchmark(binding, wl, layers=25):
    """The 25-layer decoder chain with deferred MoE tails as one CUDA graph:
    fused = one call per layer with both addends; eager = the standalone
    fold kernel, then the attention-residual + RMSNorm alone on the new
    prefix.  The bank grows 1 -> 12 (a layer that appends writes its new
    prefix straight into the next bank slot).  Microseconds per layer."""
    import torch
    s = torch.cuda.Stream()
    res = {}
    for M in (1, 8, 32):
        emb, p0, L = wl.chain_inputs(M=M, H=H, layers=layers)
        bank = torch.empty((12, M, H), dtype=torch.bfloat16, device="cuda")
        bank[0] = emb.to("cuda")
        P0 = p0.to("cuda")
        ping = [torch.empty_like(P0), torch.empty_like(P0)]
        out = torch.empty_like(P0)
        dev = [(x.w.to("cuda"), x.gamma.to("cuda"), x.routed.to("cuda"), x.shared.to("cuda")) for x in L]

        def chain(fused):
            P, n = P0, 1
            for li, (w, g, r, sh) in enumerate(dev):
                dst = bank[n] if wl.chain_appends_after(li) else ping[li % 2]
                if fused:
                    binding.attnres_add_rmsnorm(P, r, sh, bank[:n], w, g, wl.EPS, out, dst,
                                                stream=s, check=False)
                else:
                    binding.attnres_tail_add(P, r, sh, dst, stream=s)
                    binding.attnres_rmsnorm(dst, bank[:n], w, g, wl.EPS, out, stream=s)
                P = dst
                if wl.chain_appends_after(li):
                    n += 1
            return layers
        f = _graph_us(lambda: chain(True), s)
        e = _graph_us(lambda: chain(False), s)
        res[f"M{M}"] = {"fused_us_per_layer": f, "eager_us_per_layer": e,
                        "saving_us_per_layer": round(e - f, 3)}
    return res


def run_e2e(binding, inp, out, newp, stream, args, nbytes, barrier, max_ranks, ws):
    """The same metric through the public API with pinned host buffers: every
    step copies its inputs host->device, calls the op, and copies both outputs
    back, all inside the timed region.  Steps are pipelined the way a
    streaming caller would run them: uploads on one copy stream, the op on
    the compute stream, downloads on another, with two device buffer sets so
    that step k+1's upload overlaps step k's download."""
    import torch
    keys = ("prefix", "add", "add2", "bank", "w", "gamma")
    host = {k: getattr(inp, k).cpu().pin_memory() for k in keys}
    dev = [{k: torch.empty_like(getattr(inp, k)) for k in keys} for _ in range(2)]
    outs = [(torch.empty_like(out), torch.empty_like(newp)) for _ in range(2)]
    host_outs = [(torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                  torch.empty(out.shape, dtype=out.dtype, pin_memory=True)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = 2 * out.numel() * out.element_size()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    after_current(up, stream, down)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded = [ev(), ev()]
    computed = [ev(), ev()]
    downloaded = [ev(), ev()]
    used = [False, False]

    def step(k):
        b = k % 2
        with torch.cuda.stream(up):
            if used[b]:
                up.wait_event(computed[b])       # the op of step k-2 has read buffer set b
            for key in keys:
                dev[b][key].copy_(host[key], non_blocking=True)
            uploaded[b].record(up)
        with torch.cuda.stream(stream):
            stream.wait_event(uploaded[b])
            if used[b]:
                stream.wait_event(downloaded[b])  # step k-2's outputs are on the host
            d = dev[b]
            binding.attnres_add_rmsnorm(d["prefix"], d["add"], d["add2"], d["bank"], d["w"],
                                        d["gamma"], inp.eps, outs[b][0], outs[b][1], stream=stream)
            computed[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            host_outs[b][0].copy_(outs[b][0], non_blocking=True)
            host_outs[b][1].copy_(outs[b][1], non_blocking=True)
            downloaded[b].record(down)
        used[b] = True

    for k in range(max(1, args.warmup)):
        step(k)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for k in range(args.steps):
        step(k)
    down.wait_event(downloaded[(args.steps - 1) % 2])
    e1.record(down)
    barrier()
    e2e_s = max_ranks(e0.elapsed_time(e1) / 1e3)
    e2e_value = weak_scaling_value(nbytes, ws, args.steps, e2e_s)

    # The same calls on the pinned host buffers themselves: the kernel reads
    # the inputs and writes both outputs across the host link (the GPU
    # reaches pinned host memory directly), no copy in between.  The bulk L2
    # prefetch is left off for host addresses, and the split shape (every
    # row in registers) is used: the streaming shape's shared-memory rows
    # (cp.async) read host memory more slowly (GB300, M = 8192, N = 12: 214
    # against 186 GB/s, the same bits as on device buffers either way).
    zc_cfg = binding.make_config("cluster", prefetch=-1)

    def zc_call(b):
        binding.attnres_add_rmsnorm(host["prefix"], host["add"], host["add2"], host["bank"],
                                    host["w"], host["gamma"], inp.eps, host_outs[b][0],
                                    host_outs[b][1], stream=stream, check=False, config=zc_cfg)
    with torch.cuda.stream(stream):
        for k in range(max(1, args.warmup)):
            zc_call(k % 2)
    torch.cuda.synchronize()
    barrier()
    z0, z1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    z0.record(stream)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            zc_call(k % 2)
    z1.record(stream)
    z1.synchronize()
    barrier()
    zc_s = max_ranks(z0.elapsed_time(z1) / 1e3)
    zero_copy = {"value": round(weak_scaling_value(nbytes, ws, args.steps, zc_s), 2), "unit": UNIT,
                 "ms_per_step": round(zc_s / args.steps * 1e3, 3),
                 "what": "the op on the pinned host buffers themselves (inputs read and outputs "
                         "written across the host link by the kernel, no copies), split shape, "
                         "L2 prefetch off"}
    del dev, host, outs, host_outs
    return {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s / args.steps * 1e3, 3),
            "pipelined": "uploads, op and downloads on three streams, two buffer sets",
            "zero_copy": zero_copy}


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from kimi_k3_attention_gb300 import binding
    from kimi_k3_attention_gb300 import workloads as wl
    from kimi_k3_attention_gb300.build import LIB, build
    if not os.path.exists(LIB):
        build()
    binding.load()

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_ranks(x):
        return max_over_ranks(x, "cuda")

    # ---- the bandwidth workload, resident in HBM
    M, N = args.tokens, args.snapshots
    default_workload = M == M_BW and N == N_BW and not args.fp16
    inp = wl.bandwidth_inputs(device="cuda", seed=rank_seed(rank), M=M, N=N,
                              dtype=torch.float16 if args.fp16 else torch.bfloat16)
    stream = torch.cuda.Stream()
    config = None
    if args.variant != "auto" or args.cluster or args.stages:
        config = binding.make_config(args.variant, cluster=args.cluster, stages=args.stages)
    call, ev, t0, t1, out, newp = time_bandwidth(binding, inp, args.steps, args.warmup, stream, config)
    nbytes = algorithmic_bytes(M, N, H)

    # soak: the same calls back to back so that the clock samples see steady load
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ts = time.perf_counter()
        while time.perf_counter() - ts < args.soak_seconds:
            for _ in range(20):
                call()
            stream.synchronize()
    barrier()
    t0.record(stream)
    with torch.cuda.stream(stream):
        for a, b in ev:
            a.record(stream)
            call()
            b.record(stream)
    t1.record(stream)
    barrier()
    clocks = sampler.stop()
    total_s = t0.elapsed_time(t1) / 1e3
    launch_s = [a.elapsed_time(b) / 1e3 for a, b in ev]
    total_s = max_ranks(total_s)
    avg_launch = max_ranks(sum(launch_s) / len(launch_s))
    value = weak_scaling_value(nbytes, ws, args.steps, total_s)

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(binding, inp, out, newp, stream, args, nbytes, barrier, max_ranks, ws)

    decode = None
    comp = None
    chain = None
    deep = None
    fp16 = None
    cpu_base = None
    single = None
    ceiling = None
    if default_workload and config is None:
        ceiling = pattern_ceiling(binding, inp, nbytes, peaks()[0])
        # the fused kernel's GB/s per launch as a fraction of the pattern's
        ceiling["fused_over_pattern"] = round(nbytes / avg_launch / 1e9 / ceiling["gbs"], 4)
    if rank == 0 and not args.no_decode:
        decode = decode_latencies(binding, wl)
        single = single_cta_vs_cluster(binding)
        comp = comparators(binding)
        chain = chain_benchmark(binding, wl)
        deep = deep_banks(binding, wl, peaks()[0])
        fp16 = fp16_tensors(binding, wl, peaks()[0])
    if rank == 0 and not args.no_cpu_baseline and default_workload:
        # the oracle on the first tokens of this same workload; the GPU's
        # outputs for those tokens are checked against it on the way
        import numpy as np
        from oracle import check_out
        os.environ.setdefault("OMP_NUM_THREADS", "1")
        n_sample = 4096
        cpu_inp = wl.Inputs(inp.prefix[:n_sample].cpu(), inp.add[:n_sample].cpu(),
                            inp.add2[:n_sample].cpu(), inp.bank[:, :n_sample].cpu().contiguous(),
                            inp.w.cpu(), inp.gamma.cpu(), inp.eps)
        gbs, done, el, results = oracle_throughput(cpu_inp, args.cpu_seconds)

        def u(t):
            return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        g_np, g_out = u(newp[:done]), u(out[:done])
        parity = True
        for toks, (rnp, rout, rb) in results:
            parity &= bool((g_np[toks] == rnp).all()) and check_out(g_out[toks], rout, rb)["ok"]
        model, ncpu = cpu_info()
        cpu_base = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                    "sample": f"first {done} of the 8192 tokens, {el:.1f} s",
                    "cpu": model, "host_cpus": ncpu, "gpu_outputs_match_on_sample": parity,
                    "per_config": oracle_per_config()}

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    peak, peak_kind = peaks()
    achieved = nbytes / avg_launch / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "fp16" if args.fp16 else "bf16",
        "data": f"synthetic (seeded N(0,1) {'FP16' if args.fp16 else 'BF16'} tensors)",
        "config": {"workload": WORKLOAD.replace("M=8192", f"M={M}").replace("N=12", f"N={N}")
                   .replace("BF16", "FP16" if args.fp16 else "BF16"), "M": M, "N": N, "H": H, "add2": True,
                   "bytes_per_call": nbytes,
                   "l2": f"inputs ({nbytes / 1e9:.2f} GB) larger than L2, no flush" if nbytes > 2.5 * 129e6
                   else "inputs smaller than 2.5x L2 (profiling size)",
                   "plan": binding.attnres_plan(M, N, H) if config is None else config.as_dict(),
                   "parallelism": f"dp{ws} (each rank its own 8192 tokens)"},
        "us_per_call": round(total_s / args.steps * 1e6, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"of {peak_kind}",
                     "traffic": profiled_traffic() if default_workload else None,
                     "algorithmic_bytes": nbytes,
                     "avg_launch_us": round(avg_launch * 1e6, 2)},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "pattern_ceiling": ceiling,
        "decode_us_per_call": decode,
        "single_cta_vs_cluster_us": single,
        "fused_vs_alone_and_tail_add_us": comp,
        "chain_25_layers": chain,
        "deep_banks": deep,
        "fp16_tensors": fp16,
        "cpu_baseline": cpu_base,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_dry(args):
    """The multi-rank host logic alone: process group (gloo), barriers around
    K timed host steps (rank r sleeps (r + 1) ms, so the slowest rank is
    known), max over ranks, one line from rank 0.  No GPU, no kernel."""
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1:
        dist.init_process_group("gloo")

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        time.sleep(0.001 * (rank + 1))
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time.sleep(0.001 * (rank + 1))
    el = time.perf_counter() - t0
    barrier()
    total_s = max_over_ranks(el, "cpu")
    if rank == 0:
        nbytes = algorithmic_bytes(M_BW, N_BW, H)
        print(json.dumps({"metric": METRIC, "dry_run": True, "n_gpus": ws, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 4),
                          "value": round(weak_scaling_value(nbytes, ws, args.steps, total_s), 4),
                          "unit": UNIT, "scaling": "weak",
                          "note": "host logic only (gloo ranks sleeping, no GPU): not a measurement"}),
              flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=None,
                    help="GPUs (ranks) of this node; default 1, or WORLD_SIZE under torchrun")
    ap.add_argument("--dry-run", action="store_true",
                    help="host-side multi-rank logic only (gloo, no GPU); not a measurement")
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-decode", action="store_true", help="skip the M<=32 latency table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--soak-seconds", type=float, default=1.5,
                    help="back-to-back calls before the timed region, under the clock sampler")
    ap.add_argument("--tokens", type=int, default=M_BW,
                    help="tokens of the bandwidth workload (smaller only for profiling runs)")
    ap.add_argument("--snapshots", type=int, default=N_BW,
                    help="bank snapshots N of the bandwidth workload (other values only for profiling)")
    ap.add_argument("--fp16", action="store_true",
                    help="FP16 tensors instead of BF16 (profiling)")
    ap.add_argument("--variant", default="auto", choices=("auto", "cta", "cluster", "cluster2", "stream", "pipe"),
                    help="pin the launch variant of the bandwidth workload (profiling)")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    env_ws = os.environ.get("WORLD_SIZE")
    if env_ws is None:
        if args.gpus is not None and args.gpus > 1:
            # not under a launcher: start the ranks here, one per GPU
            return launch_ranks(argv, args.gpus)
    elif args.gpus is not None and args.gpus != int(env_ws):
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={env_ws}\n")
        return 2
    if args.dry_run:
        return run_dry(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
