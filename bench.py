"""Benchmark of the verify-and-sample step on GB300.

One step = one spec_verify_linear call (all rows of the linear hot path fused
in one launch: row statistics, acceptance tests, first rejection, extra token,
emission) over one batch of the draft-target workload: B=64 sequences, K=4
draft tokens, V=128256, bf16 logits, T=0.7 (147,750,912 bytes of logits).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is verified sequences per second over
all ranks with inputs resident in HBM (CUDA events, max over ranks); `e2e` is
the same metric through the public Python API with the logits copied from
pinned host memory and the results copied back inside the timed region.  The
inputs of consecutive steps rotate over four copies (591 MB > the 129 MB L2),
so no step finds its logits in L2.  Under torchrun every rank verifies its
own independent batch (no collective on the data path; weak scaling).

--impl reference times the float64 CPU oracle on this machine's host cores on the
same workload (rank 0 only).

--workload NAME (one GPU) times another configuration instead, one JSON line
each: the kernel alone, calls replayed from a CUDA graph over rotating input
copies, with the oracle timed beside it on a bounded sample.  NAME is one of
small, small_greedy, mtp_greedy, mtp_sample, medusa_tree, medusa_tree_sample,
stress, draft_sampler, draft_sampler_greedy (one draft row per sequence of the
draft-target workload: the draft side's next token), medusa_tree_mask (the
tree attention mask of the 64-node tree), or all.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = 2
TEMPERATURE = 0.7
ROTATE = 4
METRIC = "verified seqs/s and logits GB/s (fraction of GB300 HBM peak) on 1 GPU"
KERNEL_PROFILE = os.path.join(ROOT, "profiles", "spec_verify_linear_draft_target.md")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="untimed same-kernel loop before the timed region, so clock samples see the load")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample length")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="draft_target",
                    help="draft_target (the headline), or another configuration: " + ", ".join(EXTRA) + ", all")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def workload_config(w, bytes_per_step):
    return {"workload": "draft_target linear verify: B=%d K=%d V=%d bf16 logits, T=%g" % (w.B, w.K, w.V, TEMPERATURE),
            "B": w.B, "K": w.K, "V": w.V, "logits_dtype": "bf16", "temperature": TEMPERATURE,
            "logits_bytes_per_step": bytes_per_step,
            "l2": "inputs rotate over %d copies (%.0f MB > 129 MB L2)" % (ROTATE, ROTATE * bytes_per_step / 1e6),
            "seed": w.seed}


def to_oracle(t):
    import numpy as np
    import torch
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def cpu_oracle_rate(host_inputs, B, seconds, max_reps=None):
    """Verified sequences per second of the float64 oracle on the host cores."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    oracle.threads(cores)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.verify_linear(*host_inputs, TEMPERATURE)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_reps and reps >= max_reps):
            break
    return B * reps / el, cores, reps, el


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def committed_traffic(src_hash):
    """dram bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    try:
        text = open(KERNEL_PROFILE).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != src_hash:
        return None
    return int(t.group(1))


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("spec_verify.cu", "verify_kernels.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "sampling_online_softmax_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ------------------------------------------------------------ reference arm
def max_over_ranks(value, device=None):
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, per_rank_units, steps, elapsed):
    """Units per second over all ranks: every rank processes its own batch each step."""
    return world * per_rank_units * steps / elapsed


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import torch
    from workloads import WORKLOADS, make_linear
    w = WORKLOADS[WORKLOAD]
    bytes_per_step = w.logits_bytes(TEMPERATURE)
    d = make_linear(WORKLOAD, TEMPERATURE, device="cpu")
    host = [to_oracle(d[k]) for k in ("target", "draft", "draft_tokens", "u_accept", "u_bonus")]
    import oracle
    cores = len(os.sched_getaffinity(0))
    oracle.threads(cores)
    for _ in range(args.warmup):
        oracle.verify_linear(*host, TEMPERATURE)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_linear(*host, TEMPERATURE)
    el = time.perf_counter() - t0
    value = w.B * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "gbps": bytes_per_step * args.steps / el / 1e9,
            "config": workload_config(w, bytes_per_step),
            "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": cores, "kind": "oracle",
                             "sample": "the full %d-sequence batch per step, %d steps" % (w.B, args.steps)},
            "e2e": {"value": value, "unit": "seqs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import ctypes

    import torch
    import torch.distributed as dist

    import sampling_online_softmax_gb300 as sv
    from workloads import WORKLOADS, make_linear

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    lib = sv.load_library()
    w = WORKLOADS[WORKLOAD]
    B, K, V = w.B, w.K, w.V
    bytes_per_step = w.logits_bytes(TEMPERATURE)

    d = make_linear(WORKLOAD, TEMPERATURE, device=dev, seed=w.seed + 7 * rank)
    targets = [d["target"]] + [d["target"].clone() for _ in range(ROTATE - 1)]
    drafts = [d["draft"]] + [d["draft"].clone() for _ in range(ROTATE - 1)]
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
               num_emitted=torch.empty(B, dtype=torch.int32, device=dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(sv.spec_workspace_bytes_linear(B, K, V, torch.bfloat16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    h = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p
    argsets = []
    for r in range(ROTATE):
        argsets.append((P(targets[r].data_ptr()), P(drafts[r].data_ptr()), sv.SPEC_BF16, B, K, V,
                        P(d["draft_tokens"].data_ptr()), P(d["u_accept"].data_ptr()), P(d["u_bonus"].data_ptr()),
                        ctypes.c_float(TEMPERATURE), P(out["accept_len"].data_ptr()),
                        P(out["out_tokens"].data_ptr()), P(out["num_emitted"].data_ptr()), None,
                        P(status.data_ptr()), P(ws.data_ptr()), ctypes.c_size_t(ws.numel()), h))
    call = lib.spec_verify_linear

    def step(k):
        st = call(*argsets[k % ROTATE])
        if st != 0:
            raise RuntimeError("spec_verify_linear failed: %s" % lib.spec_last_error().decode())

    for k in range(max(args.warmup, 3)):
        step(k)
    torch.cuda.synchronize()
    # short calibration, then an untimed soak so clock samples see the load
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(50):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1) / 1e3 / 50
    clocks = ClockSampler(local_rank) if rank == 0 else None
    soak = int(args.soak_seconds / max(est, 1e-6))
    for k in range(soak):
        step(k)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(k)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if clocks:
        clocks.stop()
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, dev)
    assert int(status.item()) == 0, "device status %#x" % int(status.item())

    # end to end through the public API: pinned host logits in, results out
    host = {k: d[k].cpu().pin_memory() for k in ("target", "draft", "draft_tokens", "u_accept", "u_bonus")}
    dev_in = {k: torch.empty_like(d[k]) for k in host}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    e2e_steps = max(5, min(args.steps, 100))

    def e2e_step():
        for k, v in host.items():
            dev_in[k].copy_(v, non_blocking=True)
        r = sv.spec_verify_linear(dev_in["target"], dev_in["draft"], dev_in["draft_tokens"], dev_in["u_accept"],
                                  dev_in["u_bonus"], TEMPERATURE, out=dict(out), status=status, workspace=ws)
        for k, v in host_out.items():
            v.copy_(r[k], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_el = max_over_ranks(x0.elapsed_time(x1) / 1e3, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hin = [to_oracle(d[k]) for k in ("target", "draft", "draft_tokens", "u_accept", "u_bonus")]
        rate, cores, reps, el = cpu_oracle_rate(hin, B, args.cpu_seconds)
        cpu = {"value": rate, "unit": "seqs/s", "cores": cores, "kind": "oracle",
               "sample": "the same %d-sequence batch, %d repetitions in %.1f s" % (B, reps, el)}

    if rank == 0:
        step_s = elapsed / args.steps
        peak, peak_kind = measured_peak()
        gbps = bytes_per_step / step_s / 1e9
        traffic = committed_traffic(kernel_source_hash())
        line = {
            "metric": METRIC, "value": job_rate(world, B, args.steps, elapsed), "unit": "seqs/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_s,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "gbps_per_gpu": gbps,
            "config": workload_config(w, bytes_per_step),
            "roofline": {"bound": "hbm", "achieved": gbps, "peak": peak, "unit": "GB/s", "frac": gbps / peak,
                         "peak_kind": peak_kind, "traffic": traffic,
                         "kernel": "spec_verify_kernel<2, kLinearSample>"},
            "e2e": {"value": job_rate(world, B, e2e_steps, e2e_el), "unit": "seqs/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clocks.summary() if clocks else None,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------ other configurations
# name: (workload number, temperature, kind)
EXTRA = {
    "small": (1, 1.0, "linear"),
    "small_greedy": (1, 0.0, "linear"),
    "mtp_greedy": (3, 0.0, "linear"),
    "mtp_sample": (3, 1.0, "linear"),
    "medusa_tree": (4, 0.0, "tree"),
    "medusa_tree_sample": (4, 1.0, "tree_sample"),
    "stress": (5, 0.7, "linear"),
    "draft_sampler": (2, 0.7, "rows"),
    "draft_sampler_greedy": (2, 0.0, "rows"),
    "medusa_tree_mask": (4, 0.0, "mask"),
}


def _extra_inputs(name, dev):
    """Device inputs of one configuration (with a uniform per node for the sampled tree)."""
    import numpy as np
    import torch
    from workloads import WORKLOADS, make_linear, make_tree
    number, T, kind = EXTRA[name]
    w = WORKLOADS[number]
    if kind == "linear":
        return w, T, kind, make_linear(number, T, device=dev)
    if kind == "mask":
        return w, T, kind, dict(parents=make_tree(number, device=dev, B=1, V=64)["parents"])
    if kind == "rows":
        lin = make_linear(number, max(T, 0.7), device=dev)
        return w, T, kind, dict(rows=lin["draft"][:, 0].contiguous(), u=lin["u_bonus"])
    d = make_tree(number, device=dev)
    B, N = d["node_tokens"].shape
    if kind == "tree_sample":
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed + 17)
        d["u_nodes"] = torch.rand((B, N), generator=g, device=dev, dtype=torch.float32)
        # the node tokens of the greedy workload name argmaxes; here a child carries the node's draw instead
        x = d["target"].float().double() / T
        p = torch.exp(x - x.amax(-1, keepdim=True))
        c = torch.cumsum(p, -1)
        draws = torch.clamp((c <= d["u_nodes"].double()[..., None] * c[..., -1:]).sum(-1), max=w.V - 1).cpu().numpy()
        am = torch.argmax(d["target"].float(), dim=-1).cpu().numpy()
        tok = d["node_tokens"].cpu().numpy()
        par = d["parents"].cpu().numpy()
        for b in range(B):
            for c_ in range(1, N):
                if tok[b, c_] == am[b, par[c_]]:
                    tok[b, c_] = draws[b, par[c_]]
        d["node_tokens"] = torch.from_numpy(np.ascontiguousarray(tok)).to(dev)
    return w, T, kind, d


def run_extra(args, name):
    """One configuration, the kernel alone, replayed from a CUDA graph; plus the oracle beside it."""
    import torch

    import sampling_online_softmax_gb300 as sv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w, T, kind, d = _extra_inputs(name, dev)
    if kind == "mask":
        Nm = d["parents"].numel()
        bytes_per_step = 4 * Nm * ((Nm + 31) // 32 + 2)  # mask words written, parents read, depths written
    elif kind == "rows":
        bytes_per_step = d["rows"].numel() * d["rows"].element_size()
    else:
        bytes_per_step = w.logits_bytes(T)
    rotate = max(1, min(4, int(2 * 129e6 // bytes_per_step) + 1))       # more than L2 over the copies
    keys = {"linear": ("target", "draft"), "rows": ("rows",), "mask": ("parents",)}.get(kind, ("target",))
    copies = [d] + [dict(d, **{k: d[k].clone() for k in keys if d.get(k) is not None}) for _ in range(rotate - 1)]
    B = 1 if kind == "mask" else w.B     # the mask is one per tree, shared by the batch
    unit = "masks/s" if kind == "mask" else "seqs/s"
    stream = torch.cuda.Stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def make_call(c):
        if kind == "mask":
            Nm = c["parents"].numel()
            out = dict(mask=torch.empty((Nm, (Nm + 31) // 32), dtype=torch.int32, device=dev),
                       depth=torch.empty(Nm, dtype=torch.int32, device=dev))
            return lambda: sv.spec_tree_mask(c["parents"], status=status, out=out, stream=stream)
        if kind == "rows":
            out = dict(tokens=torch.empty(B, dtype=torch.int32, device=dev))
            ws = torch.zeros(sv.spec_workspace_bytes_rows(B, w.V, c["rows"].dtype), dtype=torch.uint8, device=dev)
            return lambda: sv.spec_sample_rows(c["rows"], c["u"] if T > 0 else None, T, out=out, status=status,
                                               workspace=ws, stream=stream)
        if kind == "linear":
            K = w.K
            out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                       out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                       num_emitted=torch.empty(B, dtype=torch.int32, device=dev))
            ws = torch.zeros(sv.spec_workspace_bytes_linear(B, K, w.V, c["target"].dtype), dtype=torch.uint8,
                             device=dev)
            return lambda: sv.spec_verify_linear(c["target"], c["draft"] if T > 0 else None, c["draft_tokens"],
                                                 c["u_accept"], c["u_bonus"], T, out=out, status=status, workspace=ws,
                                                 stream=stream)
        N = c["node_tokens"].shape[1]
        D = int(c["max_depth"])
        out = dict(path_nodes=torch.empty((B, D + 1), dtype=torch.int32, device=dev),
                   path_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, D + 1), dtype=torch.int32, device=dev))
        if kind == "tree":
            ws = torch.zeros(sv.spec_workspace_bytes_tree(B, N, w.V, c["target"].dtype), dtype=torch.uint8,
                             device=dev)
            return lambda: sv.spec_verify_tree(c["target"], c["parents"], c["node_tokens"], D, out=out,
                                               status=status, workspace=ws, stream=stream)
        ws = torch.zeros(sv.spec_workspace_bytes_tree_sample(B, N, w.V, c["target"].dtype), dtype=torch.uint8,
                         device=dev)
        return lambda: sv.spec_verify_tree_sample(c["target"], c["parents"], c["node_tokens"], c["u_nodes"], T, D,
                                                  out=out, status=status, workspace=ws, stream=stream)

    calls = [make_call(c) for c in copies]
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3) * rotate):  # first calls set the library's per-device state
            calls[k % rotate]()
    torch.cuda.synchronize()
    per_graph = 8 * rotate
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(per_graph):
            calls[k % rotate]()
    torch.cuda.synchronize()
    # a graph replays on the current stream: time it there
    with torch.cuda.stream(stream):
        est0, est1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        est0.record(stream)
        graph.replay()
        est1.record(stream)
        torch.cuda.synchronize()
        per_call = est0.elapsed_time(est1) / 1e3 / per_graph
        reps = max(2, int(min(2.0, args.steps * per_call) / (per_call * per_graph)))
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
    step_s = t0.elapsed_time(t1) / 1e3 / (reps * per_graph)
    assert step_s > 1e-6, "the graph replay timed no work"
    assert int(status.item()) == 0, "device status %#x" % int(status.item())
    peak, peak_kind = measured_peak()
    gbps = bytes_per_step / step_s / 1e9

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        cores = len(os.sched_getaffinity(0))
        oracle.threads(cores)
        h = {k: to_oracle(v) for k, v in d.items() if hasattr(v, "detach")}
        if kind == "mask":
            f = lambda: oracle.tree_mask(h["parents"])  # noqa
        elif kind == "rows":
            f = lambda: oracle.sample_rows(h["rows"], h["u"] if T > 0 else None, T)  # noqa
        elif kind == "linear":
            f = lambda: oracle.verify_linear(h["target"], h["draft"] if T > 0 else None, h["draft_tokens"],  # noqa
                                             h["u_accept"], h["u_bonus"], T)
        elif kind == "tree":
            f = lambda: oracle.verify_tree(h["target"], h["parents"], h["node_tokens"], int(d["max_depth"]))  # noqa
        else:
            f = lambda: oracle.verify_tree_sample(h["target"], h["parents"], h["node_tokens"], h["u_nodes"],  # noqa
                                                  T, int(d["max_depth"]))
        n, c0 = 0, time.perf_counter()
        while True:
            f()
            n += 1
            el = time.perf_counter() - c0
            if el >= min(args.cpu_seconds, 20.0):
                break
        cpu = {"value": B * n / el, "unit": unit, "cores": cores, "kind": "oracle",
               "sample": "the full %d-sequence batch, %d repetitions in %.1f s" % (B, n, el)}

    cfg = {"workload": name, "number": w.number, "kind": kind, "B": B, "K": 0 if kind == "rows" else w.K, "V": w.V,
           "logits_dtype": w.dtype, "temperature": T, "logits_bytes_per_step": bytes_per_step,
           "l2": "inputs rotate over %d copies (%.0f MB %s the 129 MB L2)"
                 % (rotate, rotate * bytes_per_step / 1e6, ">" if rotate * bytes_per_step > 129e6 else "<"),
           "seed": w.seed}
    if kind in ("tree", "tree_sample"):
        cfg["N"] = int(d["node_tokens"].shape[1])
    line = {"metric": METRIC, "value": B / step_s, "unit": unit, "n_gpus": 1, "ms_per_step": 1e3 * step_s,
            "higher_is_better": True, "timing": "kernel alone, %d calls per CUDA graph replay, %d replays"
            % (per_graph, reps), "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "achieved": gbps, "peak": peak, "unit": "GB/s", "frac": gbps / peak,
                         "peak_kind": peak_kind},
            "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.workload != "draft_target":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "--workload times the oracle beside our arm"}))
            return
        for name in (list(EXTRA) if args.workload == "all" else [args.workload]):
            run_extra(args, name)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
