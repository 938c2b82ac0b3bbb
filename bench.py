"""Benchmark of the verify-and-sample step on GB300.

Headline (the default run): one step = one spec_verify_linear call through the
C ABI -- row statistics, acceptance tests, first rejection, extra token and
emission, fused in one launch -- over one batch of the large-batch stress
workload: B=512 sequences, K=8 draft tokens, V=152064, bf16 logits, T=0.7
(2,647,130,112 bytes of logits, far more than the 129 MB L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is verified sequences per second over
all ranks with the inputs resident in HBM (CUDA events on the launching
stream, max over ranks).  `e2e` is the same metric through the public Python
API with every input copied from pinned host memory and every output copied
back inside the timed region.  Under torchrun every rank verifies its own
independent batch (no collective on the data path; weak scaling).

At N=1 the line also carries `per_config`: every other configuration (the
small linear workload at T=1 and greedy, the draft/target pair, MTP greedy and
T=1, the Medusa tree greedy and sampled, the draft-side row sampler, the tree
attention mask, the MTP token plug-in), each timed as the kernel alone
(calls replayed from a CUDA graph over rotating input copies) with its own
clock record, roofline fraction, float64 oracle timed beside it on all host
cores and on one, and the near-tie counts of a parity comparison of its
outputs with the oracle's (made outside the timed region).

--impl reference times the float64 CPU oracle on this machine's host cores on the
headline workload, a bounded sample of the batch per step (rank 0 only).

--workload NAME times one configuration alone (one JSON line each; NAME as in
`per_config`, or "all").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = 5                 # the stress workload: the largest configuration on one GPU
TEMPERATURE = 0.7
METRIC = "verified seqs/s and logits GB/s (fraction of GB300 HBM peak) on 1 GPU"
L2_BYTES = 129e6
PROFILES = os.path.join(ROOT, "profiles")
HEADLINE_KERNEL = "spec_verify_kernel<2, kLinearSample>"
HEADLINE_PROFILE = "spec_verify_kernel_linear_sample_stress.md"
REF_SAMPLE = 64              # sequences of the batch the reference arm verifies per step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="untimed same-kernel loop before each timed region, so clock samples see the load")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample length (headline)")
    ap.add_argument("--config-cpu-seconds", type=float, default=2.0,
                    help="CPU-baseline sample length per extra configuration (all cores, then one core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="the headline line without per_config")
    ap.add_argument("--workload", default="headline",
                    help="headline, or one configuration alone: " + ", ".join(list(CONFIGS) + list(ALONE)) + ", all")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --workload: the first N sequences only (a smaller case of the same kernel, for "
                         "profiler captures)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def headline_config(w, bytes_per_step):
    return {"workload": "stress linear verify: B=%d K=%d V=%d bf16 logits, T=%g" % (w.B, w.K, w.V, TEMPERATURE),
            "B": w.B, "K": w.K, "V": w.V, "logits_dtype": "bf16", "temperature": TEMPERATURE,
            "logits_bytes_per_step": bytes_per_step,
            "l2": "inputs of %.0f MB per step, larger than the 129 MB L2: no step finds its logits there"
                  % (bytes_per_step / 1e6),
            "seed": w.seed}


def to_oracle(t):
    import numpy as np
    import torch
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def host_cores():
    return len(os.sched_getaffinity(0))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms while running."""
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
            return self
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return self

    def summary(self):
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    """Median SM clock, max clock and the throttle reasons seen in nvidia-smi CSV lines."""
    sm, mx, reasons = [], None, set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for ln in lines:
        f = [x.strip() for x in ln.split(",")]
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
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ ncu summaries
def kernel_source_hash():
    """First 16 hex digits of SHA-256 over the kernel sources (sorted by name)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sampling_online_softmax_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(profile, src_hash):
    """dram bytes per launch from a committed ncu summary, if it was taken on the current sources."""
    try:
        text = open(os.path.join(PROFILES, profile)).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != src_hash:
        return None
    return int(t.group(1))


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------- multi-rank
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


# ------------------------------------------------------------ reference arm
def run_reference(args):
    """The float64 oracle on the host cores, on the headline workload: each step
    verifies a bounded sample (REF_SAMPLE sequences, rotating through the batch)."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import torch
    import oracle
    from workloads import WORKLOADS, make_linear
    w = WORKLOADS[HEADLINE]
    bytes_per_step = w.logits_bytes(TEMPERATURE)
    # the same seeded bytes our arm verifies (generated on the GPU when there is one, which is quicker)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = make_linear(HEADLINE, TEMPERATURE, device=gen_dev)
    host = {k: to_oracle(d[k]) for k in ("target", "draft", "draft_tokens", "u_accept", "u_bonus")}
    del d
    cores = host_cores()
    oracle.threads(cores)
    n = min(REF_SAMPLE, w.B)

    def step(k):
        b0 = (k * n) % w.B
        sl = slice(b0, b0 + n)
        oracle.verify_linear(host["target"][sl], host["draft"][sl], host["draft_tokens"][sl],
                             host["u_accept"][sl], host["u_bonus"][sl], TEMPERATURE)

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(k)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = "%d of the %d sequences per step (rotating through the batch), %d steps" % (n, w.B, args.steps)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "gbps": bytes_per_step * n / w.B * args.steps / el / 1e9,
            "config": headline_config(w, bytes_per_step),
            "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": cores, "kind": "oracle", "sample": sample},
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
    w = WORKLOADS[HEADLINE]
    B, K, V = w.B, w.K, w.V
    bytes_per_step = w.logits_bytes(TEMPERATURE)

    d = make_linear(HEADLINE, TEMPERATURE, device=dev, seed=w.seed + 7 * rank)
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
               num_emitted=torch.empty(B, dtype=torch.int32, device=dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(sv.spec_workspace_bytes_linear(B, K, V, torch.bfloat16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    P = ctypes.c_void_p
    argset = (P(d["target"].data_ptr()), P(d["draft"].data_ptr()), sv.SPEC_BF16, B, K, V,
              P(d["draft_tokens"].data_ptr()), P(d["u_accept"].data_ptr()), P(d["u_bonus"].data_ptr()),
              ctypes.c_float(TEMPERATURE), P(out["accept_len"].data_ptr()), P(out["out_tokens"].data_ptr()),
              P(out["num_emitted"].data_ptr()), None, P(status.data_ptr()), P(ws.data_ptr()),
              ctypes.c_size_t(ws.numel()), P(stream.cuda_stream))
    call = lib.spec_verify_linear

    def step():
        st = call(*argset)
        if st != 0:
            raise RuntimeError("spec_verify_linear failed: %s" % lib.spec_last_error().decode())

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    # short calibration, then an untimed soak so that clock samples see the load
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1) / 1e3 / 10
    clocks = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(int(args.soak_seconds / max(est, 1e-6))):
        step()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if clocks:
        clocks.stop()
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, dev)
    assert int(status.item()) == 0, "device status %#x" % int(status.item())

    # parity of the timed call's outputs with the oracle (outside the timed region, rank 0, N=1)
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        parity = linear_parity(d, {k: v for k, v in out.items()}, TEMPERATURE, status)

    # end to end through the public API: pinned host inputs in, results out
    host = {k: d[k].cpu().pin_memory() for k in ("target", "draft", "draft_tokens", "u_accept", "u_bonus")}
    dev_in = {k: torch.empty_like(d[k]) for k in host}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    e2e_steps = max(5, min(args.steps, 40))

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
    del host, dev_in

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cores = host_cores()
        oracle.threads(cores)
        n = min(REF_SAMPLE, B)
        hin = [to_oracle(d[k][:n]) for k in ("target", "draft", "draft_tokens", "u_accept", "u_bonus")]
        reps, c0 = 0, time.perf_counter()
        while True:
            oracle.verify_linear(*hin, TEMPERATURE)
            reps += 1
            el = time.perf_counter() - c0
            if el >= args.cpu_seconds:
                break
        cpu = {"value": n * reps / el, "unit": "seqs/s", "cores": cores, "kind": "oracle",
               "sample": "the first %d of the %d sequences, %d repetitions in %.1f s" % (n, B, reps, el)}

    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config:
        del d
        torch.cuda.empty_cache()
        per_config = {name: run_config(args, name, in_line=True) for name in CONFIGS}

    if rank == 0:
        step_s = elapsed / args.steps
        peak, peak_kind = measured_peak()
        gbps = bytes_per_step / step_s / 1e9
        line = {
            "metric": METRIC, "value": job_rate(world, B, args.steps, elapsed), "unit": "seqs/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_s,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "gbps_per_gpu": gbps,
            "config": headline_config(w, bytes_per_step),
            "roofline": {"bound": "hbm", "achieved": gbps, "peak": peak, "unit": "GB/s", "frac": gbps / peak,
                         "peak_kind": peak_kind, "frac_of_nominal_8000": gbps / 8000.0,
                         "traffic": committed_traffic(HEADLINE_PROFILE, kernel_source_hash()),
                         "kernel": HEADLINE_KERNEL},
            "e2e": {"value": job_rate(world, B, e2e_steps, e2e_el), "unit": "seqs/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clocks.summary() if clocks else None,
            "cpu_baseline": cpu,
            "parity": parity,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def linear_parity(d, out, T, status):
    """Near-tie counts of one call's outputs against the oracle (rank 0, outside any timed region)."""
    import oracle
    from oracle import compare
    oracle.threads(host_cores())
    g = {k: v.cpu().numpy() for k, v in out.items()}
    g["status"] = status.cpu().numpy()
    o = oracle.verify_linear(to_oracle(d["target"]), to_oracle(d["draft"]) if T > 0 else None,
                             to_oracle(d["draft_tokens"]), to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]), T)
    rep = compare.compare_linear(g, o, to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]), T, check_probs=False)
    return parity_dict(rep)


def parity_dict(rep):
    return {"sequences": rep.sequences, "exact": rep.exact, "acceptance_near_ties": rep.accept_ties,
            "inverse_cdf_near_ties": rep.bonus_ties, "failures": len(rep.failures),
            "near_tie": "|u - p/q| < 1e-6 at the first differing position, or |u_b - C/W| < 1e-6 at the drawn "
                        "token's interval edge"}


# ------------------------------------------------------ other configurations
# name: (workload number, temperature, kind)
CONFIGS = {
    "small_T1": (1, 1.0, "linear"),
    "small_greedy": (1, 0.0, "linear"),
    "draft_target_T0.7": (2, 0.7, "linear"),
    "mtp_greedy": (3, 0.0, "linear"),
    "mtp_T1": (3, 1.0, "linear"),
    "medusa_tree_greedy": (4, 0.0, "tree"),
    "medusa_tree_sampled_T1": (4, 1.0, "tree_sample"),
    "draft_sampler_T0.7": (2, 0.7, "rows"),
    "draft_sampler_greedy": (2, 0.0, "rows"),
    "medusa_tree_mask": (4, 0.0, "mask"),
    "mtp_plug_T1": (3, 1.0, "plug"),
    "medusa_tree_build": (4, 0.0, "build"),
}
# configurations timed only when named with --workload (the headline's own workload, for captures)
ALONE = {
    "stress_T0.7": (5, 0.7, "linear"),
}
# committed ncu summaries (profiles/) behind each configuration's traffic figure
CONFIG_PROFILES = {
    "small_T1": "spec_verify_kernel_linear_sample_small.md",
    "small_greedy": "spec_verify_kernel_linear_greedy_small.md",
    "draft_target_T0.7": "spec_verify_kernel_linear_sample_draft_target.md",
    "mtp_greedy": "spec_verify_kernel_linear_greedy_mtp.md",
    "mtp_T1": "spec_verify_kernel_linear_sample_mtp.md",
    "medusa_tree_greedy": "spec_verify_kernel_tree_greedy_medusa.md",
    "medusa_tree_sampled_T1": "spec_verify_kernel_tree_sample_medusa.md",
    "draft_sampler_T0.7": "spec_verify_kernel_bonus_sample_draft_rows.md",
    "draft_sampler_greedy": "spec_verify_kernel_bonus_greedy_draft_rows.md",
    "medusa_tree_mask": "tree_mask_kernel_medusa.md",
    "mtp_plug_T1": "mtp_plug_kernel_mtp.md",
}
CONFIG_KERNELS = {
    "linear": "spec_verify_kernel<EB, kLinearSample or kLinearGreedy>",
    "tree": "spec_verify_kernel<4, kTreeGreedy>",
    "tree_sample": "spec_verify_kernel<4, kTreeSample>",
    "rows": "spec_verify_kernel<2, kBonusSample or kBonusGreedy>",
    "mask": "tree_mask_kernel",
    "plug": "mtp_plug_kernel",
    "build": "spec_build_sparse_tree (host)",
}


def config_inputs(name, dev, batch=0):
    """Device inputs of one configuration (with a uniform per node for the sampled tree);
    batch > 0 keeps the first `batch` sequences of a linear configuration."""
    import dataclasses

    import numpy as np
    import torch
    from workloads import WORKLOADS, make_linear, make_tree
    number, T, kind = {**CONFIGS, **ALONE}[name]
    w = WORKLOADS[number]
    if kind == "linear":
        if batch:
            w = dataclasses.replace(w, B=min(batch, w.B))
            return w, T, kind, make_linear(number, T, device=dev, B=w.B)
        return w, T, kind, make_linear(number, T, device=dev)
    if kind == "mask":
        return w, T, kind, dict(parents=make_tree(number, device=dev, B=1, V=64)["parents"])
    if kind == "plug":
        # a T=1 verify of the MTP workload supplies the plug-in's inputs (made once, not timed)
        import sampling_online_softmax_gb300 as sv
        lin = make_linear(number, T, device=dev)
        r = sv.spec_verify_linear(lin["target"], lin["draft"], lin["draft_tokens"], lin["u_accept"], lin["u_bonus"], T)
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed + 29)
        start = torch.randint(0, w.V, (w.B, 1), generator=g, device=dev, dtype=torch.int32)
        torch.cuda.synchronize()
        return w, T, kind, dict(in_tokens=torch.cat([start, lin["draft_tokens"]], dim=1).contiguous(),
                                out_tokens=r["out_tokens"], num_emitted=r["num_emitted"],
                                seq_lens=torch.randint(1, 4000, (w.B,), generator=g, device=dev, dtype=torch.int32))
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


def config_bytes(w, T, kind, d):
    if kind == "mask":
        n = d["parents"].numel()
        return 4 * n * ((n + 31) // 32 + 2)  # mask words written, parents read, depths written
    if kind == "rows":
        return d["rows"].numel() * d["rows"].element_size()
    if kind == "plug":
        B, W = d["in_tokens"].shape
        return 4 * B * (3 * W + 3)  # in, out_tokens, num_emitted, lengths read; next tokens, lengths written
    return w.logits_bytes(T)


def make_call(sv, kind, w, T, c, dev, stream, status):
    """A closure that launches one call of this configuration on `stream`, and its outputs."""
    import torch
    B = w.B
    if kind == "plug":
        out = torch.empty_like(c["in_tokens"])
        return (lambda: sv.spec_mtp_plug(c["in_tokens"], c["out_tokens"], c["num_emitted"], 0, c["seq_lens"],
                                         out=out, status=status, stream=stream)), dict(next_tokens=out)
    if kind == "mask":
        n = c["parents"].numel()
        out = dict(mask=torch.empty((n, (n + 31) // 32), dtype=torch.int32, device=dev),
                   depth=torch.empty(n, dtype=torch.int32, device=dev))
        return (lambda: sv.spec_tree_mask(c["parents"], status=status, out=out, stream=stream)), out
    if kind == "rows":
        out = dict(tokens=torch.empty(B, dtype=torch.int32, device=dev))
        ws = torch.zeros(sv.spec_workspace_bytes_rows(B, w.V, c["rows"].dtype), dtype=torch.uint8, device=dev)
        return (lambda: sv.spec_sample_rows(c["rows"], c["u"] if T > 0 else None, T, out=out, status=status,
                                            workspace=ws, stream=stream)), out
    if kind == "linear":
        K = w.K
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                   num_emitted=torch.empty(B, dtype=torch.int32, device=dev))
        ws = torch.zeros(sv.spec_workspace_bytes_linear(B, K, w.V, c["target"].dtype), dtype=torch.uint8, device=dev)
        return (lambda: sv.spec_verify_linear(c["target"], c["draft"] if T > 0 else None, c["draft_tokens"],
                                              c["u_accept"], c["u_bonus"], T, out=out, status=status, workspace=ws,
                                              stream=stream)), out
    N = c["node_tokens"].shape[1]
    D = int(c["max_depth"])
    out = dict(path_nodes=torch.empty((B, D + 1), dtype=torch.int32, device=dev),
               path_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty((B, D + 1), dtype=torch.int32, device=dev))
    if kind == "tree":
        ws = torch.zeros(sv.spec_workspace_bytes_tree(B, N, w.V, c["target"].dtype), dtype=torch.uint8, device=dev)
        return (lambda: sv.spec_verify_tree(c["target"], c["parents"], c["node_tokens"], D, out=out, status=status,
                                            workspace=ws, stream=stream)), out
    ws = torch.zeros(sv.spec_workspace_bytes_tree_sample(B, N, w.V, c["target"].dtype), dtype=torch.uint8, device=dev)
    return (lambda: sv.spec_verify_tree_sample(c["target"], c["parents"], c["node_tokens"], c["u_nodes"], T, D,
                                               out=out, status=status, workspace=ws, stream=stream)), out


def oracle_call(kind, T, h, d):
    """The oracle on host copies h of one configuration's inputs."""
    import oracle
    if kind == "plug":
        return lambda: oracle.mtp_plug(h["in_tokens"], h["out_tokens"], h["num_emitted"], 0, None)
    if kind == "mask":
        return lambda: oracle.tree_mask(h["parents"])
    if kind == "rows":
        return lambda: oracle.sample_rows(h["rows"], h["u"] if T > 0 else None, T)
    if kind == "linear":
        return lambda: oracle.verify_linear(h["target"], h["draft"] if T > 0 else None, h["draft_tokens"],
                                            h["u_accept"], h["u_bonus"], T)
    if kind == "tree":
        return lambda: oracle.verify_tree(h["target"], h["parents"], h["node_tokens"], int(d["max_depth"]))
    return lambda: oracle.verify_tree_sample(h["target"], h["parents"], h["node_tokens"], h["u_nodes"], T,
                                             int(d["max_depth"]))


def config_parity(kind, T, h, o, g):
    """Compare one call's outputs g with the oracle's o; near-tie counts."""
    import numpy as np
    from oracle import compare
    if kind == "linear":
        return parity_dict(compare.compare_linear(g, o, h["u_accept"], h["u_bonus"], T, check_probs=False))
    if kind == "tree":
        return parity_dict(compare.compare_tree(g, o))
    if kind == "tree_sample":
        return parity_dict(compare.compare_tree_sample(g, o, h["u_nodes"]))
    if kind == "rows":
        rep = compare.compare_rows(g["tokens"], o, h["u"] if T > 0 else None, T)
        return parity_dict(rep)
    if kind == "plug":
        eq = np.all(g["next_tokens"] == o["next_tokens"], axis=1)
        return {"sequences": int(len(eq)), "exact": int(eq.sum()), "failures": int((~eq).sum())}
    same = bool(np.array_equal(g["mask"].view(np.uint32), o["mask"]) and np.array_equal(g["depth"], o["depth"]))
    return {"rows": int(len(o["depth"])), "exact": same, "failures": 0 if same else 1}


def time_oracle(f, seconds, cores):
    import oracle
    oracle.threads(cores)
    n, c0 = 0, time.perf_counter()
    while True:
        f()
        n += 1
        el = time.perf_counter() - c0
        if el >= seconds:
            return n, el


def run_build_config(args, name, in_line=False):
    """The sparse-tree builder runs on the host: trees per second, the oracle's builder beside it,
    and node-for-node parity of the two trees."""
    import numpy as np

    import oracle
    import sampling_online_softmax_gb300 as sv
    from workloads import WORKLOADS, medusa_tree
    w = WORKLOADS[CONFIGS[name][0]]
    acc = np.array([[medusa_tree.synthetic_accuracy(k, i) for i in range(1, 9)] for k in range(1, w.K + 1)])
    n_nodes = w.N

    def timed(f, seconds):
        f()
        n, c0 = 0, time.perf_counter()
        while True:
            f()
            n += 1
            el = time.perf_counter() - c0
            if el >= seconds:
                return n / el

    rate = timed(lambda: sv.spec_build_sparse_tree(acc, n_nodes), 0.5)
    got = sv.spec_build_sparse_tree(acc, n_nodes)
    cpu = parity = None
    if not args.no_cpu_baseline:
        want = oracle.build_sparse_tree(acc, n_nodes)
        eq = all(np.array_equal(got[k], want[k]) for k in ("parents", "depth", "rank"))
        parity = {"nodes": int(len(want["parents"])), "exact": bool(eq), "failures": 0 if eq else 1,
                  "expected_len": want["expected_len"]}
        cpu = {"value": timed(lambda: oracle.build_sparse_tree(acc, n_nodes), args.config_cpu_seconds),
               "unit": "trees/s", "cores": 1, "kind": "oracle",
               "sample": "the %d-node tree of the %dx8 accuracy table, repeated" % (n_nodes, w.K)}
    entry = {"us_per_call": 1e6 / rate, "value": rate, "unit": "trees/s",
             "timing": "host code (the tree is built once per accuracy table, not per step), wall clock",
             "config": {"workload": name, "K": w.K, "S": 8, "n_nodes": n_nodes,
                        "accuracy": "a_k^(i) = 0.6 * 0.8^k * 0.5^i"},
             "roofline": None, "clocks": None, "cpu_baseline": cpu, "parity": parity}
    if not in_line:
        entry.update({"metric": "sparse candidate trees built per second (host)", "higher_is_better": True})
        print(json.dumps(entry), flush=True)
    return entry


def run_config(args, name, in_line=False):
    """One configuration, the kernel alone, replayed from a CUDA graph; clocks, roofline, oracle beside it."""
    import torch
    if {**CONFIGS, **ALONE}[name][2] == "build":
        return run_build_config(args, name, in_line)

    import sampling_online_softmax_gb300 as sv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w, T, kind, d = config_inputs(name, dev, getattr(args, "batch", 0))
    bytes_per_step = config_bytes(w, T, kind, d)
    rotate = max(1, min(4, int(2 * L2_BYTES // bytes_per_step) + 1))   # more than L2 over the copies
    keys = {"linear": ("target", "draft"), "rows": ("rows",), "mask": ("parents",),
            "plug": ("in_tokens", "out_tokens")}.get(kind, ("target",))
    copies = [d] + [dict(d, **{k: d[k].clone() for k in keys if d.get(k) is not None}) for _ in range(rotate - 1)]
    B = 1 if kind == "mask" else w.B     # the mask is one per tree, shared by the batch
    unit = "masks/s" if kind == "mask" else "seqs/s"
    stream = torch.cuda.Stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    calls = [make_call(sv, kind, w, T, c, dev, stream, status) for c in copies]
    # the copies and the zeroed workspaces were made on the default stream; the calls run on `stream`
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3) * rotate):  # first calls set the library's per-device state
            calls[k % rotate][0]()
    torch.cuda.synchronize()
    first_out = {k: v.cpu().numpy() for k, v in calls[(max(args.warmup, 3) * rotate - 1) % rotate][1].items()}
    per_graph = 8 * rotate
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(per_graph):
            calls[k % rotate][0]()
    torch.cuda.synchronize()
    # a graph replays on the current stream: time it there
    with torch.cuda.stream(stream):
        est0, est1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        est0.record(stream)
        graph.replay()
        est1.record(stream)
        torch.cuda.synchronize()
        per_call = est0.elapsed_time(est1) / 1e3 / per_graph
        per_replay = per_call * per_graph
        clocks = ClockSampler(0)
        for _ in range(int(args.soak_seconds / per_replay) + 1):
            graph.replay()
        torch.cuda.synchronize()
        reps = max(2, int(max(0.5, min(2.0, args.steps * per_call)) / per_replay))
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        clocks.stop()
    step_s = t0.elapsed_time(t1) / 1e3 / (reps * per_graph)
    assert step_s > 1e-6, "the graph replay timed no work"
    assert int(status.item()) == 0, "device status %#x" % int(status.item())
    peak, peak_kind = measured_peak()
    gbps = bytes_per_step / step_s / 1e9
    del graph, calls, copies
    torch.cuda.empty_cache()

    cpu = parity = None
    if not args.no_cpu_baseline:
        h = {k: to_oracle(v) for k, v in d.items() if hasattr(v, "detach")}
        f = oracle_call(kind, T, h, d)
        cores = host_cores()
        parity = config_parity(kind, T, h, f(), first_out)
        n, el = time_oracle(f, args.config_cpu_seconds, cores)
        cpu = {"value": B * n / el, "unit": unit, "cores": cores, "kind": "oracle",
               "sample": "the full %d-sequence batch, %d repetitions in %.1f s" % (B, n, el)}
        n1, el1 = time_oracle(f, args.config_cpu_seconds, 1)
        cpu["single_thread"] = {"value": B * n1 / el1, "unit": unit, "cores": 1,
                                "sample": "the full batch, %d repetitions in %.1f s" % (n1, el1)}
        import oracle
        oracle.threads(cores)

    cfg = {"workload": name, "number": w.number, "kind": kind, "B": B, "K": 0 if kind == "rows" else w.K,
           "V": w.V, "logits_dtype": w.dtype, "temperature": T, "logits_bytes_per_step": bytes_per_step,
           "l2": "inputs rotate over %d copies (%.0f MB %s the 129 MB L2)"
                 % (rotate, rotate * bytes_per_step / 1e6, ">" if rotate * bytes_per_step > L2_BYTES else "<"),
           "seed": w.seed}
    if kind in ("tree", "tree_sample"):
        cfg["N"] = int(d["node_tokens"].shape[1])
    prof = CONFIG_PROFILES.get(name) if not getattr(args, "batch", 0) else None
    entry = {"us_per_call": 1e6 * step_s, "value": B / step_s, "unit": unit,
             "timing": "kernel alone, %d calls per CUDA graph replay, %d replays" % (per_graph, reps),
             "config": cfg,
             "roofline": {"bound": "hbm", "achieved": gbps, "peak": peak, "unit": "GB/s", "frac": gbps / peak,
                          "peak_kind": peak_kind, "frac_of_nominal_8000": gbps / 8000.0,
                          "traffic": committed_traffic(prof, kernel_source_hash()) if prof else None,
                          "kernel": CONFIG_KERNELS[kind]},
             "clocks": clocks.summary(), "cpu_baseline": cpu, "parity": parity}
    if not in_line:
        entry.update({"metric": METRIC, "n_gpus": 1, "ms_per_step": 1e3 * step_s, "higher_is_better": True,
                      "data": "synthetic"})
        print(json.dumps(entry), flush=True)
    return entry


def main():
    args = parse()
    if args.workload != "headline":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "--workload times the oracle beside our arm"}))
            return
        names = list(CONFIGS) if args.workload == "all" else [args.workload]
        for name in names:
            if name not in CONFIGS and name not in ALONE:
                raise SystemExit("unknown workload %r" % name)
            run_config(args, name)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
