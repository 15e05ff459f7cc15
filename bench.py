"""Benchmark of the multi-LoRA decode hot path on GB300.

One step = one InvisibleLoRA decode cycle through one transformer block's
seven projections on the Llama-3-8B-shaped workload (64 requests, 16
resident rank-16 adapters with Zipf(1.1) popularity, 1 draft token per
request, vocabulary 128256).  Projections that read the same rows go through
one sliced layer call (q|k|v, gate|up), as a block computes them:

    plan (a1, on a second stream, beside the draft pass)
    draft pass:  4 layer calls (q|k|v, o, gate|up, down), M = 64 rows, LoRA off (a3)
    verify pass: 4 x (shrink a2 + GEMM a3 + fused expand a4), M = 128 rows
    accept / resample for 64 requests (a5, a6)

`value` is verified tokens (M = 128 per step, summed over ranks) per second
with every input resident in HBM, from CUDA events around K replays of the
step captured as one CUDA graph.  The W working set (436 MB per pass, read
twice per step) is larger than L2, so weights stream from HBM every launch.
`e2e` is the same metric through the Python C-ABI binding with pinned host
buffers: each step copies that step's activations and probabilities to the
device and reads every output back; the copy-in of the next step overlaps
the current step on a second stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica on its own requests
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

CFG = WL.LLAMA8B_R16
K_DRAFT = 1
METRIC = "multi-LoRA decode-step tokens/s (draft+verify layer x7 projections + accept)"
UNIT = "tokens/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# Algorithmic work
# ---------------------------------------------------------------------------


def layer_bytes_flops(M, K, N, active_ranks, verify, n_proj=1):
    """Algorithmic HBM bytes and flops of one layer call: W, x and y once; in
    verify mode each active adapter's A (once per projection slice) and B."""
    b = 2 * (N * K + M * K + M * N)
    f = 2 * M * N * K
    if verify:
        b += sum(2 * r * K * n_proj + 2 * N * r for r in active_ranks)
        f += 2 * M * int(np.mean(active_ranks) if active_ranks else 0) * (K * n_proj + N)
    return b, f


# DRAM traffic per launch of a kernel, from a committed ncu summary; valid
# only while the kernel's sources are the ones the counters were taken on.
TRAFFIC_SOURCES = {
    "gemm_sk_kernel": ("gemm_sk.cu", "common.cuh", "launch.h"),
    "gemm_kernel": ("gemm.cu", "common.cuh", "launch.h"),
}


def sources_hash(kernel):
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[kernel]:
        with open(os.path.join(ROOT, "speculative_lora_decoding_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel):
    """(bytes per launch, note) from profiles/<kernel>_traffic_llama8b.md, or
    (None, why) when there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic_llama8b.md")
    if not os.path.exists(path):
        return None, "no ncu traffic summary"
    fields = {}
    for line in open(path):
        if ":" in line and line.strip().startswith(("sources_sha256", "dram_bytes_per_launch")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("sources_sha256") != sources_hash(kernel):
        return None, "kernel changed since the ncu capture"
    return float(fields["dram_bytes_per_launch"]), f"ncu capture, {os.path.relpath(path, ROOT)}"


def accept_bytes(B, V, accepted, k):
    # the draw reads p_n (+ q_n when a draft was rejected); gathers are negligible
    return int(sum(4 * V * (2 if a < k else 1) for a in accepted)) + 8 * B * k


# ---------------------------------------------------------------------------
# Clock sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------


class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return out
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        out.update(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                   reasons=reasons, samples=len(rows))
        return out


# ---------------------------------------------------------------------------
# Workload on the device
# ---------------------------------------------------------------------------


def _bf16(torch, bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class DeviceWorkload:
    def __init__(self, torch, ml, device, seed):
        self.torch, self.ml = torch, ml
        cfg = CFG
        self.ranks = WL.adapter_ranks(cfg, seed)
        self.idx_d = WL.row_adapters(cfg, "draft", seed=seed)
        self.idx_v = WL.row_adapters(cfg, "verify", k=K_DRAFT, seed=seed)
        self.Md, self.Mv = len(self.idx_d), len(self.idx_v)
        # One entry per input group: the projections' W stacked along N, their
        # A stacks side by side, their B stacks along N, the shared rows x.
        self.proj = []
        for group in WL.input_groups(cfg):
            Ws, As, Bs = [], [], []
            for p in group:
                W, A, B, _ = WL.projection_weights(cfg, p, seed=seed)
                Ws.append(W)
                As.append(A)
                Bs.append(B)
            K = cfg.projections[group[0]][1]
            ends = [int(e) for e in np.cumsum([w.shape[0] for w in Ws])]
            N = ends[-1]
            name = "_".join(cfg.projections[p][0] for p in group)
            xd = WL.activations(cfg, group[0], "draft", seed=seed)
            xv = WL.activations(cfg, group[0], "verify", k=K_DRAFT, seed=seed)
            self.proj.append(dict(name=name, K=K, N=N, ends=ends, n_proj=len(group),
                                  W=_bf16(torch, np.concatenate(Ws, axis=0), device),
                                  A=_bf16(torch, np.stack(As), device),
                                  B=_bf16(torch, np.concatenate(Bs, axis=1), device),
                                  xd=_bf16(torch, xd, device), xv=_bf16(torch, xv, device), xd_h=xd, xv_h=xv,
                                  yd=torch.empty((self.Md, N), dtype=torch.bfloat16, device=device),
                                  yv=torch.empty((self.Mv, N), dtype=torch.bfloat16, device=device)))
        self.rank_of = torch.from_numpy(self.ranks).to(device)
        self.adx_d = torch.from_numpy(self.idx_d).to(device)
        self.adx_v = torch.from_numpy(self.idx_v).to(device)
        p, q, tok, u = WL.accept_inputs(cfg.vocab, cfg.n_requests, K_DRAFT, seed=seed)
        self.acc_h = (p, q, tok, u)
        self.p, self.q, self.tok, self.u = (torch.from_numpy(a).to(device) for a in (p, q, tok, u))
        self.out_tok = torch.empty((cfg.n_requests, K_DRAFT + 1), dtype=torch.int32, device=device)
        self.accepted = torch.empty((cfg.n_requests,), dtype=torch.int32, device=device)
        ws_bytes = max(ml.linear_sliced_workspace_bytes(self.Mv, P["N"], P["K"], cfg.n_adapters, len(P["ends"]))
                       for P in self.proj)
        ws_bytes = max(ws_bytes, ml.accept_workspace_bytes(cfg.n_requests, K_DRAFT, cfg.vocab))
        self.ws = ml.Workspace(ws_bytes, device=device)
        self.seg = None

    # individual ops of one step, in order
    def ops(self):
        ml, cfg = self.ml, CFG
        out = []

        def plan():
            self.seg, _ = ml.plan_segments(self.adx_v, self.rank_of, cfg.n_adapters, cfg.r_max, self.ws)
        out.append(("plan", plan))
        for P in self.proj:
            out.append((f"draft.{P['name']}", lambda P=P: ml.linear_sliced(
                P["xd"], P["W"], P["ends"], None, None, None, None, cfg.scale, ml.DRAFT | ml.PREFETCH_WEIGHTS,
                ws=self.ws, y=P["yd"])))
        for P in self.proj:
            out.append((f"verify.{P['name']}", lambda P=P: ml.linear_sliced(
                P["xv"], P["W"], P["ends"], P["A"], P["B"], self.rank_of, self.adx_v, cfg.scale,
                ml.VERIFY | ml.PREFETCH_WEIGHTS, ws=self.ws, y=P["yv"], seg_offsets_ptr=self.seg)))
        out.append(("accept", lambda: ml.verify_accept(self.p, self.q, self.tok, self.u, ws=self.ws,
                                                      out_tok=self.out_tok, accepted=self.accepted)))
        return out

    def step(self, side=None):
        """One step in stream order.  With `side` (a second stream) the plan,
        which needs only the adapter indices, runs on it concurrently with the
        draft pass, and the verify pass waits for it."""
        ops = self.ops()
        if side is None:
            for _, f in ops:
                f()
            return
        torch = self.torch
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            ops[0][1]()
        for name, f in ops[1:]:
            if name.startswith("verify.") and side is not None:
                main.wait_stream(side)
                side = None
            f()


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------


def oracle_sample_step(requests, seed=0, prepared=None):
    """Run the oracle over `requests` requests of the workload (all 7
    projections, draft and verify rows, then accept).  Returns (seconds,
    verify tokens)."""
    from oracle import accept as OA
    from oracle import layer as OL
    cfg = CFG
    if prepared is None:
        prepared = prepare_oracle(seed)
    ranks, idx_d, idx_v, proj, acc = prepared
    rows_d = np.arange(requests)
    rows_v = np.arange(requests * (K_DRAFT + 1))
    t0 = time.perf_counter()
    for (W, A, B, xd, xv) in proj:
        OL.mlora_linear(xd[rows_d], W, None, None, None, None, cfg.scale, OL.DRAFT)
        OL.mlora_linear(xv[rows_v], W, A, B, ranks, idx_v[rows_v], cfg.scale, OL.VERIFY)
    p, q, tok, u = acc
    OA.verify_accept(p[:requests], q[:requests], tok[:requests], u[:requests])
    return time.perf_counter() - t0, len(rows_v)


def prepare_oracle(seed=0):
    cfg = CFG
    f = WL.bf16_to_f64
    ranks = WL.adapter_ranks(cfg, seed)
    idx_d = WL.row_adapters(cfg, "draft", seed=seed)
    idx_v = WL.row_adapters(cfg, "verify", k=K_DRAFT, seed=seed)
    proj = []
    for p in range(len(cfg.projections)):
        W, A, B, _ = WL.projection_weights(cfg, p, seed=seed)
        proj.append((f(W), f(A), f(B), f(WL.activations(cfg, p, "draft", seed=seed)),
                     f(WL.activations(cfg, p, "verify", k=K_DRAFT, seed=seed))))
    acc = WL.accept_inputs(cfg.vocab, 8, K_DRAFT, seed=seed)
    return ranks, idx_d, idx_v, proj, acc


# ---------------------------------------------------------------------------
# Ranks (one process per GPU, replicas only)
# ---------------------------------------------------------------------------


def rank_env():
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(torch, value, world, device):
    """The slowest rank's value: every rank times the same number of steps on
    its own requests, so the job's time per step is the maximum."""
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens per second: every rank's tokens over the slowest time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# Reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------


def run_reference(args):
    _, rank, _ = rank_env()
    if rank != 0:
        return 0
    prepared = prepare_oracle(0)
    req = 1
    for _ in range(args.warmup):
        oracle_sample_step(req, prepared=prepared)
    times, toks = [], 0
    for _ in range(args.steps):
        t, n = oracle_sample_step(req, prepared=prepared)
        times.append(t)
        toks += n
    total = sum(times)
    value = toks / total
    cores = cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": CFG.name + f"/k={K_DRAFT}/vocab={CFG.vocab}", "requests_per_step": req},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{req} request per step: 7 projections draft+verify rows + accept, float64 numpy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    import speculative_lora_decoding_gb300 as ml
    if not os.path.exists(ml.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    if not ml.device_supported():
        raise RuntimeError("this benchmark needs a compute capability 10.3 GPU")

    wl = DeviceWorkload(torch, ml, device, seed=rank)
    stream = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            wl.step(side)
    stream.synchronize()
    if wl.ws.status() != 0:
        raise RuntimeError("device status bits raised during warm-up")

    # Whole step as one CUDA graph.
    graph = torch.cuda.CUDAGraph()
    n0 = ml.launch_count()
    with torch.cuda.graph(graph, stream=stream):
        wl.step(side)
    launches_per_step = ml.launch_count() - n0
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms = max_over_ranks(torch, ms, world, device)
    ms_per_step = ms / args.steps
    value = job_throughput(wl.Mv, world, ms_per_step)
    if wl.ws.status() != 0:
        raise RuntimeError("device status bits raised during the timed region")

    op_ms, timing_kind = per_op_durations(torch, wl, stream, args)

    # Algorithmic work.
    hbm_gbs, bf16_tf, peak_kind = _peaks()
    active = sorted(set(int(a) for a in wl.idx_v if a >= 0))
    active_ranks = [int(wl.ranks[a]) for a in active]
    draft_b = draft_t = verify_b = verify_t = 0.0
    draft_f = verify_f = 0.0
    per_kernel = {}  # GEMM kernel -> draft bytes, draft ms, draft launches, ms over both passes
    for P in wl.proj:
        b, f = layer_bytes_flops(wl.Md, P["K"], P["N"], [], False)
        draft_b += b
        draft_f += f
        draft_t += op_ms[f"draft.{P['name']}"]
        kd = ml.gemm_kernel_name(wl.Md, P["N"], P["K"], CFG.n_adapters, CFG.r_max, ml.DRAFT)
        e = per_kernel.setdefault(kd, {"bytes": 0.0, "ms": 0.0, "launches": 0, "ops": [], "both_ms": 0.0})
        e["bytes"] += b
        e["ms"] += op_ms[f"draft.{P['name']}"]
        e["launches"] += 1
        e["ops"].append(P["name"])
        e["both_ms"] += op_ms[f"draft.{P['name']}"]
        b, f = layer_bytes_flops(wl.Mv, P["K"], P["N"], active_ranks, True, P["n_proj"])
        verify_b += b
        verify_f += f
        verify_t += op_ms[f"verify.{P['name']}"]
        kv = ml.gemm_kernel_name(wl.Mv, P["N"], P["K"], CFG.n_adapters, CFG.r_max, ml.VERIFY)
        per_kernel.setdefault(kv, {"bytes": 0.0, "ms": 0.0, "launches": 0, "ops": [], "both_ms": 0.0})
        per_kernel[kv]["both_ms"] += op_ms[f"verify.{P['name']}"]
    acc_host = wl.accepted.cpu().numpy()
    acc_b = accept_bytes(CFG.n_requests, CFG.vocab, acc_host, K_DRAFT)
    # The dominant kernel: the GEMM kernel with the most time over both
    # passes; its roofline from its draft-pass launches, where a layer call is
    # that one kernel (a verify call also runs the shrink).
    dom = max((k for k in per_kernel if per_kernel[k]["launches"]), key=lambda k: per_kernel[k]["both_ms"])
    d = per_kernel[dom]
    achieved = d["bytes"] / (d["ms"] * 1e-3) / 1e9
    traffic, traffic_note = profiled_traffic(dom)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                "traffic": traffic,
                "kernel": f"{dom} (draft pass: {', '.join(d['ops'])}; M={wl.Md})",
                "peak_kind": f"{peak_kind} hbm_gbs",
                "algorithmic_bytes_per_launch": d["bytes"] / d["launches"],
                "avg_launch_us": 1e3 * d["ms"] / d["launches"],
                "traffic_source": traffic_note,
                "other_kernels": {k: {"draft_GBps": v["bytes"] / (v["ms"] * 1e-3) / 1e9 if v["ms"] else None,
                                      "draft_ops": v["ops"], "ms_both_passes": v["both_ms"]}
                                  for k, v in per_kernel.items() if k != dom}}
    modes = {
        "draft_layer": {"us": 1e3 * draft_t, "tokens_per_s": wl.Md / (draft_t * 1e-3),
                        "GBps": draft_b / (draft_t * 1e-3) / 1e9, "frac_hbm": draft_b / (draft_t * 1e-3) / 1e9 / hbm_gbs},
        "verify_layer": {"us": 1e3 * verify_t, "tokens_per_s": wl.Mv / (verify_t * 1e-3),
                         "GBps": verify_b / (verify_t * 1e-3) / 1e9,
                         "frac_hbm": verify_b / (verify_t * 1e-3) / 1e9 / hbm_gbs,
                         "TFLOPs": verify_f / (verify_t * 1e-3) / 1e12},
        "accept": {"us": 1e3 * op_ms["accept"], "rows_per_s": CFG.n_requests / (op_ms["accept"] * 1e-3),
                   "GBps": acc_b / (op_ms["accept"] * 1e-3) / 1e9,
                   "mean_accepted": float(acc_host.mean())},
        "plan_us": 1e3 * op_ms["plan"],
        "per_op_timing": timing_kind,
        "per_op_us": {k: 1e3 * v for k, v in op_ms.items()},
    }

    # End to end through the binding with pinned host buffers.
    e2e = run_e2e(torch, ml, wl, stream, side, args, world)
    try:
        tensor = tensor_probe(torch, ml, device, stream, bf16_tf, peak_kind)
    except Exception as exc:  # the probe is context; it does not void the step measurement
        tensor = {"failed": str(exc)}

    cpu = None
    if rank == 0 and world == 1:
        try:
            prepared = prepare_oracle(0)
            oracle_sample_step(1, prepared=prepared)
            secs, toks, nrep = 0.0, 0, 0
            while secs < 10.0 and nrep < 50:
                t, n = oracle_sample_step(8, prepared=prepared)
                secs += t
                toks += n
                nrep += 1
            cpu = {"value": toks / secs, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"{nrep} x 8 requests (16 verify + 8 draft rows) through 7 projections + accept, "
                             "float64 numpy, BLAS default threads"}
        except Exception as exc:  # a baseline that fails does not void the GPU number
            cpu = {"value": None, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": f"failed: {exc}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": CFG.name + f"/k={K_DRAFT}/vocab={CFG.vocab}", "requests": CFG.n_requests,
                       "draft_rows": wl.Md, "verify_rows": wl.Mv,
                       "projections": [p[0] for p in CFG.projections],
                       "layer_calls": [p["name"] for p in wl.proj],
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: 436 MB of W streamed per pass, two passes per step",
                       "graph": "one CUDA graph per step; the plan runs on a second stream beside the draft pass"},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline,
            "modes": modes,
            "e2e": e2e,
            "tensor_bound_verify": tensor,
            "cpu_baseline": cpu,
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def per_op_durations(torch, wl, stream, args):
    """Median duration of every op of the step, from CUDA events on the
    launching stream.  Preferred: one step graph with an event node between
    consecutive ops (external events), replayed and read back step by step.
    Fallback: each op in its own graph, replayed back to back."""
    ops = wl.ops()
    reps = max(10, min(args.steps, 200))
    try:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(ops) + 1)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            evs[0].record(stream)
            for i, (_, fn) in enumerate(ops):
                fn()
                evs[i + 1].record(stream)
        torch.cuda.synchronize()
        samples = [[] for _ in ops]
        for _ in range(reps):
            g.replay()
            torch.cuda.synchronize()
            for i in range(len(ops)):
                samples[i].append(evs[i].elapsed_time(evs[i + 1]))
        return {name: float(np.median(samples[i])) for i, (name, _) in enumerate(ops)}, "events inside the step graph"
    except Exception:
        pass
    op_graphs = []
    for name, fn in ops:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        op_graphs.append((name, g))
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(op_graphs) + 1)] for _ in range(reps)]
    with torch.cuda.stream(stream):
        for r in range(reps):
            evs[r][0].record(stream)
            for i, (_, g) in enumerate(op_graphs):
                g.replay()
                evs[r][i + 1].record(stream)
    torch.cuda.synchronize()
    return ({name: float(np.median([evs[r][i].elapsed_time(evs[r][i + 1]) for r in range(reps)]))
             for i, (name, _) in enumerate(op_graphs)}, "one graph per op")


def tensor_probe(torch, ml, device, stream, bf16_tf, peak_kind):
    """The verify base GEMM where the tensor cores bound it: the fused gate|up
    call of the 32B-shaped block with k = 4 drafts (128 requests x 5 = 640
    rows, 64 rank-16 adapters, ids uniform), random weights on the device,
    timed over 20 replays of a captured graph with CUDA events: once without
    the adapters (the base GEMM alone) and once as the full verify call."""
    cfg = WL.QWEN32B_R16
    dims = {name: (k_in, n_out) for name, k_in, n_out in cfg.projections}
    K = dims["gate"][0]
    N = dims["gate"][1] + dims["up"][1]
    M, n_ad, r = cfg.rows("verify", 4), cfg.n_adapters, cfg.r_max
    g = torch.Generator(device=device)
    g.manual_seed(5)
    W = (torch.randn(N, K, device=device, generator=g) * 0.02).bfloat16()
    x = torch.randn(M, K, device=device, generator=g).bfloat16()
    A = (torch.randn(2, n_ad, r, K, device=device, generator=g) * 0.02).bfloat16()
    B = (torch.randn(n_ad, N, r, device=device, generator=g) * 0.25).bfloat16()
    rank_of = torch.full((n_ad,), r, dtype=torch.int32, device=device)
    idx = torch.randint(0, n_ad, (M,), dtype=torch.int32, device=device, generator=g)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
    ends = [dims["gate"][1], N]
    ws = ml.Workspace(ml.linear_sliced_workspace_bytes(M, N, K, n_ad, 2), device=device)

    def timed(call):
        reps = 20
        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                call()
            graph.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    us_base = timed(lambda: ml.linear_sliced(x, W, ends, None, None, None, None, 1.0, ml.DRAFT, ws=ws, y=y))
    us_ver = timed(lambda: ml.linear_sliced(x, W, ends, A, B, rank_of, idx, cfg.scale, ml.VERIFY, ws=ws, y=y))
    if ws.status() != 0:
        raise RuntimeError("device status bits raised in the tensor-bound probe")
    base = 2.0 * M * N * K
    lora = 2.0 * M * r * (2 * K + N)  # shrink + expand
    tf_base = base / (us_base * 1e-6) / 1e12
    tf_ver = (base + lora) / (us_ver * 1e-6) / 1e12
    out = {"call": f"gate|up, 32B shapes, k=4: M={M} N={N} K={K}, {n_ad} rank-{r} adapters",
           "kernel": ml.gemm_kernel_name(M, N, K, n_ad, r, ml.VERIFY), "peak_TFLOPs": bf16_tf,
           "peak_kind": f"{peak_kind} bf16_tflops_sustained",
           "base_gemm": {"us_per_call": us_base, "TFLOPs": tf_base, "frac": tf_base / bf16_tf},
           "verify_call": {"us_per_call": us_ver, "TFLOPs": tf_ver, "frac": tf_ver / bf16_tf,
                           "expand": "CUDA-core bucket walk (the tensor-core expand's masked operand covers at most 256 rows)"}}
    del W, x, A, B, y, ws
    torch.cuda.empty_cache()
    return out


def run_e2e(torch, ml, wl, stream, side, args, world):
    """Host buffers in, host buffers out, through the public binding.  Every
    step copies its activations, adapter indices and probabilities from
    pinned host memory and reads every output back.  The copy-in of step s+1
    runs on a second stream while step s computes (two device input sets,
    each with its own captured graph of the same binding calls); the
    read-back follows each step on the compute stream."""
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_x = [(pin(P["xd_h"].view(np.int16)), pin(P["xv_h"].view(np.int16))) for P in wl.proj]
    p, q, tok, u = wl.acc_h
    h_acc = [pin(p), pin(q), pin(tok), pin(u)]
    h_idx = pin(wl.idx_v)
    h_yd = [torch.empty(tuple(P["yd"].shape), dtype=torch.int16).pin_memory() for P in wl.proj]
    h_yv = [torch.empty(tuple(P["yv"].shape), dtype=torch.int16).pin_memory() for P in wl.proj]
    h_out = torch.empty(tuple(wl.out_tok.shape), dtype=torch.int32).pin_memory()
    h_acc_out = torch.empty(tuple(wl.accepted.shape), dtype=torch.int32).pin_memory()
    h2d = sum(a.numel() * a.element_size() for pair in h_x for a in pair) + sum(
        a.numel() * a.element_size() for a in h_acc) + h_idx.numel() * 4
    d2h = sum(a.numel() * 2 for a in h_yd + h_yv) + h_out.numel() * 4 + h_acc_out.numel() * 4

    # Two sets of device inputs: the workload's own tensors and a copy.
    def current():
        return {"x": [(P["xd"], P["xv"]) for P in wl.proj], "idx": wl.adx_v, "acc": [wl.p, wl.q, wl.tok, wl.u]}

    def use(st):
        for P, (xd, xv) in zip(wl.proj, st["x"]):
            P["xd"], P["xv"] = xd, xv
        wl.adx_v = st["idx"]
        wl.p, wl.q, wl.tok, wl.u = st["acc"]

    set0 = current()
    set1 = {"x": [(torch.empty_like(xd), torch.empty_like(xv)) for xd, xv in set0["x"]],
            "idx": torch.empty_like(set0["idx"]), "acc": [torch.empty_like(a) for a in set0["acc"]]}
    sets = (set0, set1)

    def copy_in(st):
        for (xd, xv), (hd, hv) in zip(st["x"], h_x):
            xd.view(torch.int16).copy_(hd, non_blocking=True)
            xv.view(torch.int16).copy_(hv, non_blocking=True)
        st["idx"].copy_(h_idx, non_blocking=True)
        for d, h in zip(st["acc"], h_acc):
            d.copy_(h, non_blocking=True)

    def read_back():
        for P, hd, hv in zip(wl.proj, h_yd, h_yv):
            hd.copy_(P["yd"].view(torch.int16), non_blocking=True)
            hv.copy_(P["yv"].view(torch.int16), non_blocking=True)
        h_out.copy_(wl.out_tok, non_blocking=True)
        h_acc_out.copy_(wl.accepted, non_blocking=True)

    graphs = []
    with torch.cuda.stream(stream):
        for st in sets:
            use(st)
            copy_in(st)
            wl.step(side)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                wl.step(side)
            graphs.append(g)
    use(set0)
    copy = torch.cuda.Stream(device=wl.p.device)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    free = [torch.cuda.Event(), torch.cuda.Event()]

    def run(n):
        copy.wait_stream(stream)
        with torch.cuda.stream(copy):
            copy_in(sets[0])
            ready[0].record(copy)
        for s in range(n):
            cur, nxt = s % 2, (s + 1) % 2
            if s + 1 < n:
                if s >= 1:
                    copy.wait_event(free[nxt])  # step s-1 has read that set
                with torch.cuda.stream(copy):
                    copy_in(sets[nxt])
                    ready[nxt].record(copy)
            stream.wait_event(ready[cur])
            graphs[cur].replay()
            free[cur].record(stream)
            read_back()

    steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        run(3)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(steps)
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if wl.ws.status() != 0:
        raise RuntimeError("device status bits raised during the end-to-end run")
    ms = max_over_ranks(torch, ms, world, wl.p.device)
    return {"value": job_throughput(wl.Mv, world, ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "steps": steps,
            "overlap": "copy-in of step s+1 on a second stream during step s; read-back after each step"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
