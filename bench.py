"""Benchmark: KDA prefill forward tokens/s on one GB300 (or N replicas).

Workload: fixed length B=1, T=8192, H=32, dk=dv=128, bf16 q/k/v, fp32 g/beta/h0
(the Student-t / deep-gate recipe of tests/gen.py, fresh salt per run).  A step is
one kda_fwd over the whole batch: schedule, per-chunk factors, state recurrence.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` = tokens/s over all ranks with inputs resident in
HBM; `e2e` = the same metric through the public binding with pinned host buffers,
every step's host-to-device inputs and device-to-host outputs inside the timed
region (steps pipelined over two buffer sets and three streams, as a serving loop
would run them); `roofline` = the dominant kernel's algorithmic bytes per launch
over its CUDA-event duration, against the measured HBM copy bandwidth.  The
per-step input (337 MB) and factor workspace (438 MB) exceed the 129 MB L2, so no L2
flush is inserted between steps.  `--impl reference` times the fp64 CPU oracle on this
host's cores on the same workload (a bounded number of heads per step).
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from tests import gen  # noqa: E402

METRIC = "KDA fwd tokens/s at H=32,d=128,8192 tok; % tensor-pipe/HBM roofline"
WORKLOADS = {
    "cfg2": "fixed-length B=1 T=8192 H=32 dk=dv=128 bf16 q/k/v, fp32 g/beta/h0 (Student-t mixture, g=-softplus(N(-1,2)) clamped)",
    "cfg3": "varlen 8192 tokens in 8 sequences (uniform split, one of length 1), H=32, dk=dv=128, bf16",
    "cfg4": "varlen skewed 8192 tokens in 32 sequences (one ~5000), H=32, d=128, extreme-value probes",
}
KERNEL_NAMES = {"fused": ["schedule", "fused"],
                "split": ["schedule", "factors", "state_recurrence", "state_recurrence_128"],
                # few long chains: the segmented recurrence (pass A, scan, pass C), with
                # the tiled state kernel before it when the schedule decides on the device
                "split-seg": ["schedule", "factors", "segments_a", "segments_scan", "segments_c"],
                "split-seg-decide": ["schedule", "factors", "state_recurrence", "segments_a",
                                     "segments_scan", "segments_c"]}
STATE_KERNELS = ("state_recurrence", "state_recurrence_128", "segments_a", "segments_c")


def make_workload(name: str, seed: int, salt: int):
    """cfg2 (default), cfg3, cfg4, a throughput-sweep row cfg5-{fixed|varlen}-H{H}-{total},
    or long-B{B}-H{H}-{T} (fixed length, few long chains)."""
    if name == "cfg2":
        return gen.make_cfg2(seed=seed, salt=salt), WORKLOADS[name]
    if name == "cfg2-gbf16":
        x = gen.make_cfg2(seed=seed, salt=salt)
        x.g = x.g.to(torch.bfloat16)
        return x, WORKLOADS["cfg2"].replace("fp32 g/beta/h0", "bf16 g, fp32 beta/h0")
    if name == "cfg2-d64":
        x = gen.make_cfg2(seed=seed, salt=salt, d=64)
        return x, WORKLOADS["cfg2"].replace("dk=dv=128", "dk=dv=64")
    if name == "cfg3":
        return gen.make_cfg3(seed=seed, salt=salt), WORKLOADS[name]
    if name == "cfg4":
        return gen.make_cfg4(seed=seed, salt=salt), WORKLOADS[name]
    if name.startswith("cfg5-"):
        _, kind, hs, total = name.split("-")
        H_, total_ = int(hs[1:]), int(total)
        x = gen.make_cfg5(H_, total_, kind == "varlen", seed=seed, salt=salt, drawn_heads=2)
        desc = (f"throughput sweep: {kind} {total_} tokens, H={H_}, dk=dv=128, bf16 "
                f"({'B=' + str(total_ // 8192) + ' x 8192' if kind == 'fixed' else str(x.num_seqs) + ' sequences'}; "
                "heads 0-1 drawn from the recipe, the others token-rolled copies of them)")
        return x, desc
    if name.startswith("long-"):
        _, bs, hs, ts = name.split("-")
        B_, H_, T_ = int(bs[1:]), int(hs[1:]), int(ts)
        desc = (f"few long chains: fixed-length B={B_} T={T_} H={H_} dk=dv=128 bf16 q/k/v, "
                "fp32 g/beta/h0 (the cfg2 recipe)")
        return gen.make_cfg2(seed=seed, salt=salt, T=T_, H=H_, B=B_), desc
    raise ValueError(f"unknown workload {name}")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def _algorithmic_bytes(kernel: str, tokens: int, heads: int, dk: int, dv: int, nseq: int,
                       g_bytes: int = 4):
    """Algorithmic HBM bytes one launch of `kernel` must move (bf16 q/k/v/o, fp32 or bf16 g,
    fp32 beta/states)."""
    th = tokens * heads
    if kernel == "factors":       # reads q, k, v, g, beta
        return th * (2 * dk * 2 + dv * 2 + dk * g_bytes + 4)
    if kernel in STATE_KERNELS:   # writes o; reads h0, writes hT (a segment pass: charged the whole)
        return th * dv * 2 + 2 * nseq * heads * dk * dv * 4
    if kernel == "fused":         # the whole path: both of the above
        return _path_bytes(tokens, heads, dk, dv, nseq, g_bytes)
    return 0


def _path_bytes(tokens, heads, dk, dv, nseq, g_bytes=4):
    return tokens * heads * (2 * dk * 2 + 2 * dv * 2 + dk * g_bytes + 4) + 2 * nseq * heads * dk * dv * 4


class ClockSampler:
    """nvidia-smi samples while the timed region runs (median SM clock, throttle reasons)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def whole_job_rate(local_ms_per_step: float, units_per_rank: int, world: int, device=None):
    """Replicas: every rank times its own steps; the job takes as long as the slowest
    rank (max over ranks), and processes world x units_per_rank units per step.
    Returns (ms per step, units per second for the whole job)."""
    t = torch.tensor([local_ms_per_step], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms = float(t.item())
    return ms, world * units_per_rank / (ms * 1e-3)


def _traffic_for(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was captured on this
    workload and the kernel's source is unchanged since (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    ent = j.get(kernel)
    if not ent or ent.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "gated_delta_rule_25_gb300", "csrc", ent["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return ent["bytes_per_launch"] if h == ent["sha"] else None


def _oracle_sample(x, heads: int, nthreads: int = 0):
    import oracle
    t = x.tensors()
    for key in ("q", "k", "v", "g", "beta"):
        t[key] = t[key][:, :, :heads].contiguous()
    if t["h0"] is not None:
        t["h0"] = t["h0"][:, :heads].contiguous()
    t0 = time.perf_counter()
    oracle.kda_recurrence_fp64(**t, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(x, budget_s: float = 12.0):
    """The fp64 oracle, as it stands, on this host's cores: whole heads of the same
    workload until ~budget_s of work; tokens/s scaled to all H heads."""
    import oracle
    H = x.H
    cores = oracle.max_threads()
    heads = min(H, max(1, cores))
    dt = _oracle_sample(x, heads)
    reps = 1
    total = dt
    while total < budget_s and reps < 8:
        total += _oracle_sample(x, heads)
        reps += 1
    per_run = total / reps
    tok_s = (x.tokens * heads / H) / per_run
    return {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{heads} of {H} heads x {x.tokens} tokens, {reps} runs, fp64 C recurrence; "
                      "tokens/s scaled to all heads"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    x, desc = make_workload(args.workload, 0, gen.fresh_salt())
    H = x.H
    cores = oracle.max_threads()
    heads = min(H, max(1, cores))
    for _ in range(args.warmup):
        _oracle_sample(x, max(1, heads // 4))
    times = [_oracle_sample(x, heads) for _ in range(args.steps)]
    per = sum(times) / len(times)
    tok_s = (x.tokens * heads / H) / per
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3 * H / heads, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "tokens_per_step": x.tokens},
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: {heads} of {H} heads x {x.tokens} tokens "
                                       "(fp64 token recurrence); tokens/s scaled to all heads"},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DECODE_METRIC = "KDA decode tokens/s (one token per sequence per step); % HBM roofline"


def _decode_bytes(N, H, dk, dv):
    """Algorithmic HBM bytes of one decode step: the state read and written (fp32), the
    token's bf16 q, k, v, fp32 g, beta, and the bf16 output."""
    return N * H * (2 * dk * dv * 4 + 2 * dk * 2 + dk * 4 + 2 * dv * 2 + 4)


def run_decode(args):
    """Workload decode-N{N}-H{H}: one kda_decode step over N sequences x H heads,
    dk = dv = 128, bf16 q/k/v, fp32 g/beta, cfg2-style values, states ~ N(0, 0.1)
    updated in place (the state stays resident, as in serving)."""
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as kda
    _, ns, hs = args.workload.split("-")
    N, H, D = int(ns[1:]), int(hs[1:]), 128
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    salt = gen.fresh_salt()
    x = gen.make_lengths([1] * N, seed=0, salt=salt, H=H, d=D, name="decode")
    t = {n: getattr(x, n)[0].to(dev) for n in ("q", "k", "v", "g", "beta")}
    state = x.h0.to(dev)
    o = torch.empty((N, H, D), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, x.scale, out_state=state, o=o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    value = N / (ms * 1e-3)
    hbm, _, peak_src = _peaks()
    alg = _decode_bytes(N, H, D, D)
    achieved = alg / (ms * 1e-3) / 1e9

    # parity after timing: one step from a fresh state against the fp64 oracle (2 heads)
    import oracle
    from tests.metrics import rel_rmse
    x2 = gen.make_lengths([1] * N, seed=1, salt=salt + 7919, H=H, d=D, name="decode")
    for n in ("q", "k", "v", "g", "beta"):
        t[n].copy_(getattr(x2, n)[0].to(dev))
    state.copy_(x2.h0.to(dev))
    step()
    torch.cuda.synchronize(dev)
    hsel = [0, H // 2 + 1]
    tt = x2.tensors()
    for key in ("q", "k", "v", "g", "beta"):
        tt[key] = tt[key][:, :, hsel].contiguous()
    tt["h0"] = tt["h0"][:, hsel].contiguous()
    o_ref, h_ref = oracle.kda_recurrence_fp64(**tt)
    parity = {"heads": hsel, "o_rel_rmse": rel_rmse(o.cpu()[None][:, :, hsel], o_ref),
              "state_rel_rmse": rel_rmse(state.cpu()[:, hsel], h_ref), "salt": x2.salt}

    # end to end: the token's inputs from pinned host memory, the output back; states stay
    host_in = {n: getattr(x, n)[0].pin_memory() for n in ("q", "k", "v", "g", "beta")}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = o_host.numel() * o_host.element_size()

    def e2e_step():
        for n, v in host_in.items():
            t[n].copy_(v, non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_value = N / (e0.elapsed_time(e1) / args.steps * 1e-3)

    cpu = None
    if not args.no_cpu_baseline:
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 5.0:
            oracle.kda_recurrence_fp64(**x.tensors())
            reps += 1
        per = (time.perf_counter() - t0) / reps
        cpu = {"value": N / per, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"the whole step ({N} sequences x {H} heads), {reps} runs, fp64 C recurrence"}
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"decode step: N={N} sequences x H={H} heads, dk=dv=128, bf16 q/k/v, "
                               "fp32 states updated in place",
                   "name": args.workload, "tokens_per_step": N,
                   "l2": f"no flush: {N * H * D * D * 4 / 1e6:.0f} MB of state read and written per step vs the 129 MB L2",
                   "salt": salt},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "kernel": "decode", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": _traffic_for("decode", args.workload),
                     "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.steps},
        "parity": parity,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def measure_backward(kda, x, dev, steps: int, warmup: int, parity: bool, salt: int) -> dict:
    """Times kda_bwd (the gradients of sum(o do) + sum(h_T dh_T)) on x with random do
    and dh_T (CUDA events on the launching stream, inputs resident) and, with
    `parity`, checks two heads' gradients against the fp64 autograd oracle."""
    xd = x.to(dev)
    rng = np.random.default_rng(salt)
    do = torch.from_numpy(rng.standard_normal(tuple(x.v.shape)).astype(np.float32)).to(x.v.dtype)
    dhT = torch.from_numpy(rng.standard_normal((x.num_seqs, x.H, x.dk, x.dv)).astype(np.float32))
    do_d, dhT_d = do.to(dev), dhT.to(dev)
    ws = torch.empty(int(kda.load_library().kda_bwd_workspace_size(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs))
                     + 256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return kda.bwd(**xd.tensors(), do=do_d, dhT=dhT_d, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        out = step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    par = None
    if parity:
        from oracle.backward import kda_backward_fp64
        from tests.metrics import rel_rmse
        hs = sorted({0, min(1, x.H - 1)})
        t = x.tensors()
        for key in ("q", "k", "v", "g", "beta"):
            t[key] = t[key][:, :, hs].contiguous()
        if t["h0"] is not None:
            t["h0"] = t["h0"][:, hs].contiguous()
        ref = kda_backward_fp64(**t, do=do[:, :, hs].double(), dhT=dhT[:, hs].double())
        par = {"heads": hs}
        for name, a, r in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), out, ref):
            a = a.cpu()
            a = a[:, hs] if name == "dh0" else a[:, :, hs]
            par[name + "_rel_rmse"] = rel_rmse(a, r)
    return {"metric": "KDA backward tokens/s (gradients of o and h_T for q, k, v, g, beta, h0)",
            "value": x.tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "warmup": warmup, "dtype": "f32", "kernels_per_step": 3, "parity": par}


def run_backward(args):
    """--backward: the backward pass on the workload instead of the forward."""
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as kda
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    salt = gen.fresh_salt()
    x, desc = make_workload(args.workload, 0, salt)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.2)
    res = measure_backward(kda, x, dev, args.steps, args.warmup, not args.no_parity, salt)
    clk = clocks.stop()
    line = dict(res, n_gpus=1, higher_is_better=True, data="synthetic",
                config={"workload": desc, "name": args.workload, "tokens_per_step": x.tokens,
                        "heads": x.H, "dk": x.dk, "dv": x.dv, "salt": salt},
                gpu_launches=3 * args.steps, clocks=clk)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (kda_bwd) on the workload instead of the forward")
    ap.add_argument("--no-parity", action="store_true", help="--backward: skip the oracle check")
    ap.add_argument("--no-backward", action="store_true",
                    help="forward runs: skip the backward pass's measurement in the JSON line")
    ap.add_argument("--pipeline", default="auto", choices=["auto", "fused", "split", "split-whole"],
                    help="auto (default): the library's choice for the sizes; fused: factor "
                         "production and state chains in one kernel; split: a factor kernel, "
                         "then the state kernels (few long chains cut into segments where "
                         "predicted faster); split-whole: split, chains never cut")
    ap.add_argument("--workload", default="cfg2",
                    help="cfg2 (the headline workload), cfg2-gbf16 (bf16 gate), cfg2-d64 (dk = dv = 64), cfg3, cfg4, "
                         "cfg5-{fixed|varlen}-H{16|32|64}-{total}, long-B{B}-H{H}-{T} "
                         "(few long fixed-length chains), "
                         "decode-N{sequences}-H{heads}")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    if args.backward:
        return run_backward(args)
    if args.workload.startswith("decode-"):
        run_decode(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    if world > 1 and rank != 0:
        torch.distributed.barrier()      # rank 0 builds first; the others then find it built
    __graft_entry__.build()
    if world > 1 and rank == 0:
        torch.distributed.barrier()
    import gated_delta_rule_25_gb300 as kda
    kda.set_pipeline(args.pipeline)

    salt = gen.fresh_salt() + rank
    x, desc = make_workload(args.workload, 0, salt)
    xd = x.to(dev)
    nseq = x.num_seqs
    B, T, H, D = x.B, x.T, x.H, x.dk
    o = torch.empty_like(xd.v)
    hT = torch.empty_like(xd.h0)
    ws = torch.empty(kda.workspace_size(B, T, H, D, D, nseq) + 256, dtype=torch.uint8, device=dev)
    nl = kda.launch_count(B, T, H, D, D, nseq)
    fused = kda.uses_fused(B, T, H, D, D, nseq)
    pipeline = "fused" if fused else ("split-whole" if args.pipeline == "split-whole" else "split")
    names = KERNEL_NAMES["fused" if fused else "split" if nl < 5 else
                         ("split-seg" if nl == 5 else "split-seg-decide")]
    stream = torch.cuda.current_stream(dev)

    def step(events=None):
        kda.fwd(**xd.tensors(), o=o, hT=hT, workspace=ws, events=events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # per-launch boundary events for every timed step (kernel timing on the launching stream)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_kernel = [0.0] * nl
    for row in evs:
        for j in range(nl):
            per_kernel[j] += row[j].elapsed_time(row[j + 1])
    per_kernel = [t / args.steps for t in per_kernel]

    ms_step, value = whole_job_rate(elapsed_ms / args.steps, x.tokens, world, dev)

    # parity after timing, on fresh inputs through the same buffers (sampled heads)
    x2, _ = make_workload(args.workload, 1, salt + 7919)
    if x.cu_seqlens is not None:  # same layout, fresh values
        x2.cu_seqlens = x.cu_seqlens
        x2.h0 = x2.h0[: x.num_seqs]
    for name in ("q", "k", "v", "g", "beta", "h0"):
        getattr(xd, name).copy_(getattr(x2, name).to(dev))
    step()
    torch.cuda.synchronize(dev)
    parity = None
    if rank == 0:
        import oracle
        from tests.metrics import rel_rmse
        hs = sorted({0, min(x2.H - 1, x2.H // 2 + 1)})
        t = x2.tensors()
        for key in ("q", "k", "v", "g", "beta"):
            t[key] = t[key][:, :, hs].contiguous()
        t["h0"] = t["h0"][:, hs].contiguous()
        o_ref, h_ref = oracle.kda_recurrence_fp64(**t)
        parity = {"heads": hs, "o_rel_rmse": rel_rmse(o.cpu()[:, :, hs], o_ref),
                  "hT_rel_rmse": rel_rmse(hT.cpu()[:, hs], h_ref), "salt": x2.salt}

    # end to end through the public binding: every step copies its inputs in from
    # pinned host memory and its outputs back.  Steps are pipelined the way a serving
    # loop would run them: two input/output buffer sets, copies in on one stream,
    # the forward on the compute stream, copies out on a third, ordered by events.
    host_in = {n: getattr(x, n).pin_memory() for n in ("q", "k", "v", "g", "beta", "h0")}
    o_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    h_host = [torch.empty(hT.shape, dtype=hT.dtype).pin_memory() for _ in range(2)]
    dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host_in.items()} for _ in range(2)]
    dev_out = [(o, hT), (torch.empty_like(o), torch.empty_like(hT))]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = o_host[0].numel() * o_host[0].element_size() + h_host[0].numel() * h_host[0].element_size()
    e2e_steps = max(3, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[b])          # the forward of step i-2 has read buffer b
            for n, t in host_in.items():
                dev_in[b][n].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])             # step i-2's outputs have left buffer b
        ob, hb = dev_out[b]
        kda.fwd(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"], dev_in[b]["beta"],
                dev_in[b]["h0"], xd.cu_seqlens, x.scale, o=ob, hT=hb, workspace=ws)
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            o_host[b].copy_(ob, non_blocking=True)
            h_host[b].copy_(hb, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    e1.record(s_out)                             # after the last step's outputs are on the host
    torch.cuda.synchronize(dev)
    _, e2e_value = whole_job_rate(e0.elapsed_time(e1) / e2e_steps, x.tokens, world, dev)
    # the pipelined outputs are the forward's: the last step's o against the timed run's
    e2e_ok = bool(torch.equal(o_host[(e2e_steps - 1) & 1].to(dev), dev_out[(e2e_steps - 1) & 1][0]))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    hbm, bf16_tf, peak_src = _peaks()
    in_mb = sum(t.numel() * t.element_size() for t in (x.q, x.k, x.v, x.g, x.beta)) / 1e6
    ws_mb = ws.numel() / 1e6
    dom = int(np.argmax(per_kernel))
    dom_name = names[dom] if dom < len(names) else f"kernel{dom}"
    gb = x.g.element_size()
    alg = _algorithmic_bytes(dom_name, x.tokens, H, D, D, nseq, gb)
    achieved = alg / (per_kernel[dom] * 1e-3) / 1e9
    path_gbs = _path_bytes(x.tokens, H, D, D, nseq, gb) / (ms_step * 1e-3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x)
    # the backward pass on the same inputs (f3; a few steps, two heads against the
    # autograd oracle), for workloads of up to 16,384 tokens
    bwd = None
    if world == 1 and not args.no_backward and x.tokens <= 16384:
        bwd = measure_backward(kda, x, dev, 3, 1, True, salt)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "name": args.workload, "tokens_per_step": x.tokens,
                   "heads": H, "dk": D, "dv": D,
                   "l2": f"no flush: {in_mb:.0f} MB of inputs and {ws_mb:.0f} MB of factors per step vs the 129 MB L2",
                   "salt": salt, "pipeline": pipeline},
        "gpu_launches": nl * args.steps,
        "kernels_ms": {names[j] if j < len(names) else f"kernel{j}": per_kernel[j]
                       for j in range(nl)},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": _traffic_for(dom_name, args.workload),
                     "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"},
        "path_roofline": {"bytes_per_step": _path_bytes(x.tokens, H, D, D, nseq, gb),
                          "achieved_gbs": path_gbs, "frac": path_gbs / hbm},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelined": "two buffer sets; copies in, forward and copies out on three streams",
                "outputs_match": e2e_ok},
        "parity": parity,
        "cpu_baseline": cpu,
        "backward": bwd,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
