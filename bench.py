"""Benchmark of the multi-LoRA speculative decode hot path on GB300.

One step = one InvisibleLoRA decode cycle of one transformer block's seven
projections ("InvisibleLoRA: Fast Multi-LoRA Serving Without Per-Token LoRA
Decoding", abstract): k LoRA-off draft passes, one LoRA-on pass that
verifies the committed token and the k drafts of every request, and the
accept / resample step.  Projections that read the same rows go through one
sliced layer call (q|k|v, gate|up), as a block computes them:

    plan (a1, on a second stream, beside the draft passes)
    k draft passes: 4 layer calls each (q|k|v, o, gate|up, down), one row per request, LoRA off (a3)
    verify pass:    4 x (row gather + shrink a2 + GEMM a3 with the fused expand a4), (k+1) rows per request
    accept / resample for every request (a5, a6)

The headline is the largest single-GPU workload: the 32B-class shapes, 128
requests, 64 rank-16 adapters with uniform popularity and k = 4 drafts (640
verify rows).  `value` is verified tokens (rows of the LoRA-on pass, summed
over ranks) per second with every input resident in HBM, from CUDA events
around K replays of the step captured as one CUDA graph; the W working set
(1 GB per pass) is far larger than L2, so weights stream from HBM every pass.
`e2e` is the same metric through the Python C-ABI binding with pinned host
buffers: each step copies that step's activations, adapter indices and
probabilities to the device and reads every output back.

The same JSON line carries, under "configs", the other layer workloads (the
tiny 512x512 layer, the Llama-3-8B-shaped block with 16 rank-16 adapters and
with 128 heterogeneous-rank adapters, the 32B block at k = 1 and 2) and,
under "accept_sweep", the accept step alone at batch 256, vocabulary 128256,
k = 1..4, each with its roofline fraction and the float64 oracle timed on the
host cores beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--extra all|none] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica on its own requests
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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

# Layer workloads: (layer config, draft length k).
LAYER_RUNS = {
    "tiny": (WL.TINY, 1),
    "llama8b-r16": (WL.LLAMA8B_R16, 1),
    "llama8b-het": (WL.LLAMA8B_HET, 1),
    "32b-k1": (WL.QWEN32B_R16, 1),
    "32b-k2": (WL.QWEN32B_R16, 2),
    "32b-k4": (WL.QWEN32B_R16, 4),
}
HEADLINE = "32b-k4"
ACCEPT_SWEEP_K = (1, 2, 3, 4)
ACCEPT_CALLS = 8  # accept calls per graph in the sweep's back-to-back timing
METRIC = "multi-LoRA decode-step verified tokens/s (k draft passes + 1 verify pass of one block's 7 projections + accept)"
UNIT = "tokens/s"
L2_BYTES = 126 * 1024 * 1024


def _peaks():
    """(HBM GB/s, bf16 burst TF/s, bf16 sustained TF/s, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


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
    "gemm_sk_kernel": ("gemm_sk.cu", "expand.cuh", "common.cuh"),
    "gemm_kernel": ("gemm.cu", "expand.cuh", "common.cuh"),
    "accept_blocks_kernel": ("accept.cu", "common.cuh"),
}


def sources_hash(kernel):
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[kernel]:
        with open(os.path.join(ROOT, "speculative_lora_decoding_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel, workload):
    """(bytes per launch, note) from profiles/<kernel>_traffic_<workload>.md,
    or (None, why) when there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic_{workload}.md")
    if not os.path.exists(path):
        return None, "no ncu traffic summary for this kernel and workload"
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
# Synthetic inputs on the device (the recipe of `workloads`, drawn with
# torch's generator on the device so that the 32B-shaped block is ready in
# seconds; the float64 oracle baseline reads host copies of these tensors)
# ---------------------------------------------------------------------------


def _gen(torch, device, seed, *key):
    g = torch.Generator(device=device)
    g.manual_seed(int(hashlib.sha256(repr((seed,) + key).encode()).hexdigest()[:15], 16))
    return g


def _normal_bf16(torch, shape, std, g, device):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def accept_inputs_device(torch, V, B, k, device, seed=0, sigma=WL.ACCEPT_SIGMA, target_std=2.0):
    """p [B, k+1, V], q [B, k, V] fp32 (float64 softmax of target logits
    N(0, target_std^2) and of the same logits + N(0, sigma^2)), draft tokens
    [B, k] drawn from q, uniforms [B, k+1] in [0, 1)."""
    g = _gen(torch, device, seed, "accept", V, B, k)
    p = torch.empty((B, k + 1, V), dtype=torch.float32, device=device)
    q = torch.empty((B, k, V), dtype=torch.float32, device=device)
    step = max(1, (1 << 27) // ((2 * k + 1) * V))  # bound the float64 temporaries
    for b0 in range(0, B, step):
        b1 = min(B, b0 + step)
        z = torch.randn((b1 - b0, k + 1, V), generator=g, device=device, dtype=torch.float64) * target_std
        p[b0:b1] = torch.softmax(z, dim=-1).float()
        zq = z[:, :k] + torch.randn((b1 - b0, k, V), generator=g, device=device, dtype=torch.float64) * sigma
        q[b0:b1] = torch.softmax(zq, dim=-1).float()
        del z, zq
    tok = torch.multinomial(q.reshape(B * k, V), 1, generator=g).reshape(B, k).to(torch.int32).contiguous()
    u = torch.rand((B, k + 1), generator=g, device=device, dtype=torch.float32)
    return p, q, tok, u


def accept_logits_device(torch, V, B, k, device, seed=0, sigma=WL.ACCEPT_SIGMA, target_std=2.0):
    """Logits for the softmax row: z_p [B, k+1, V] ~ N(0, target_std^2) and
    z_q [B, k, V] = z_p[:, :k] + N(0, sigma^2) in fp32; draft tokens drawn from
    softmax(z_q); uniforms [B, k+1] in [0, 1)."""
    g = _gen(torch, device, seed, "logits", V, B, k)
    zp = torch.randn((B, k + 1, V), generator=g, device=device, dtype=torch.float32) * target_std
    zq = zp[:, :k] + torch.randn((B, k, V), generator=g, device=device, dtype=torch.float32) * sigma
    tok = torch.multinomial(torch.softmax(zq.reshape(B * k, V).double(), -1).float(), 1, generator=g)
    tok = tok.reshape(B, k).to(torch.int32).contiguous()
    u = torch.rand((B, k + 1), generator=g, device=device, dtype=torch.float32)
    return zp.contiguous(), zq.contiguous(), tok, u


class StepWorkload:
    """Device tensors of one decode-step workload: per input group (q|k|v, o,
    gate|up, down) the stacked W, A and B, one activation block per draft
    pass and one for the verify pass; adapter indices; accept inputs."""

    def __init__(self, torch, ml, device, name, seed):
        self.torch, self.ml, self.name = torch, ml, name
        cfg, k = LAYER_RUNS[name]
        self.cfg, self.k = cfg, k
        self.ranks = WL.adapter_ranks(cfg, seed)
        self.idx_d = WL.row_adapters(cfg, "draft", seed=seed)
        self.idx_v = WL.row_adapters(cfg, "verify", k=k, seed=seed)
        self.Md, self.Mv = len(self.idx_d), len(self.idx_v)
        self.proj = []
        rk = torch.from_numpy(self.ranks.astype(np.int64)).to(device)
        r_max = cfg.r_max
        for group in WL.input_groups(cfg):
            Ws, As, Bs = [], [], []
            K = cfg.projections[group[0]][1]
            for p in group:
                _, Kp, N = cfg.projections[p]
                g = _gen(torch, device, seed, "W", p)
                Ws.append(_normal_bf16(torch, (N, Kp), 1.0 / math.sqrt(Kp), g, device))
                A = _normal_bf16(torch, (cfg.n_adapters, r_max, Kp), 1.0 / math.sqrt(Kp), _gen(torch, device, seed, "A", p),
                                 device)
                A *= (torch.arange(r_max, device=device)[None, :] < rk[:, None]).to(torch.bfloat16)[:, :, None]
                Bm = torch.randn((cfg.n_adapters, N, r_max), generator=_gen(torch, device, seed, "B", p), device=device)
                Bm = Bm / torch.sqrt(torch.clamp(rk, min=1).float())[:, None, None]
                Bm = (Bm * (torch.arange(r_max, device=device)[None, None, :] < rk[:, None, None])).to(torch.bfloat16)
                As.append(A)
                Bs.append(Bm)
            ends = [int(e) for e in np.cumsum([w.shape[0] for w in Ws])]
            N = ends[-1]
            gname = "_".join(cfg.projections[p][0] for p in group)
            xd = [_normal_bf16(torch, (self.Md, K), 1.0, _gen(torch, device, seed, "xd", group[0], d), device)
                  for d in range(k)]
            xv = _normal_bf16(torch, (self.Mv, K), 1.0, _gen(torch, device, seed, "xv", group[0]), device)
            self.proj.append(dict(name=gname, K=K, N=N, ends=ends, n_proj=len(group), W=torch.cat(Ws, 0).contiguous(),
                                  A=torch.stack(As).contiguous(), B=torch.cat(Bs, 1).contiguous(), xd=xd, xv=xv,
                                  yd=torch.empty((self.Md, N), dtype=torch.bfloat16, device=device),
                                  yv=torch.empty((self.Mv, N), dtype=torch.bfloat16, device=device),
                                  yb=torch.empty((self.Mv, N), dtype=torch.bfloat16, device=device)))
            del Ws, As, Bs
        self.rank_of = torch.from_numpy(self.ranks).to(device)
        self.adx_v = torch.from_numpy(self.idx_v).to(device)
        self.adx_d = torch.from_numpy(self.idx_d).to(device)
        B = cfg.n_requests
        self.p, self.q, self.tok, self.u = accept_inputs_device(torch, cfg.vocab, B, k, device, seed=seed)
        self.out_tok = torch.empty((B, k + 1), dtype=torch.int32, device=device)
        self.accepted = torch.empty((B,), dtype=torch.int32, device=device)
        ws_bytes = max(ml.linear_sliced_workspace_bytes(self.Mv, P["N"], P["K"], cfg.n_adapters, len(P["ends"]))
                       for P in self.proj)
        ws_bytes = max(ws_bytes, ml.accept_workspace_bytes(B, k, cfg.vocab))
        self.ws = ml.Workspace(ws_bytes, device=device)
        # The draft passes run beside the plan (second stream): a workspace of their own.
        self.ws_draft = ml.Workspace(max(ml.linear_sliced_workspace_bytes(self.Md, P["N"], P["K"], 0, len(P["ends"]))
                                         for P in self.proj), device=device)
        self.ws_plain = ml.Workspace(max(ml.linear_sliced_workspace_bytes(self.Md, P["N"], P["K"], cfg.n_adapters,
                                                                          len(P["ends"])) for P in self.proj),
                                     device=device)
        self.seg_plain = None
        torch.cuda.synchronize(device) if device.type == "cuda" else None
        self.seg = None
        self.w_bytes_per_pass = sum(2 * P["N"] * P["K"] for P in self.proj)
        self.fp8 = False
        self.ws_fp8 = None

    def enable_fp8(self):
        """Draft passes on E4M3 copies of W (quantized once, per output row)."""
        ml = self.ml
        for P in self.proj:
            if "W8" not in P:
                P["W8"], P["sw"] = ml.quantize_rows_fp8(P["W"])
        if self.ws_fp8 is None:
            self.ws_fp8 = ml.Workspace(max(ml.linear_fp8_workspace_bytes(self.Md, P["N"], P["K"]) for P in self.proj),
                                       device=self.p.device)
        self.fp8 = True

    @property
    def workload(self):
        return f"{self.cfg.name}/k={self.k}/vocab={self.cfg.vocab}"

    def ops(self, with_base=False):
        """The step's ops in stream order (name, kind, group, callable);
        with_base adds, after the step, a draft-mode call of each group at the
        verify rows (the base GEMM alone at that shape, for comparison)."""
        ml, cfg = self.ml, self.cfg
        out = []

        def plan():
            self.seg, _ = ml.plan_segments(self.adx_v, self.rank_of, cfg.n_adapters, cfg.r_max, self.ws)
        out.append(("plan", "plan", None, plan))
        for d in range(self.k):
            for P in self.proj:
                if self.fp8:
                    out.append((f"draft{d}.{P['name']}", "draft", P, lambda P=P, d=d: ml.linear_fp8(
                        P["xd"][d], P["W8"], P["sw"], ml.PREFETCH_WEIGHTS, ws=self.ws_fp8, y=P["yd"])))
                    continue
                out.append((f"draft{d}.{P['name']}", "draft", P, lambda P=P, d=d: ml.linear_sliced(
                    P["xd"][d], P["W"], P["ends"], None, None, None, None, cfg.scale, ml.DRAFT | ml.PREFETCH_WEIGHTS,
                    ws=self.ws_draft, y=P["yd"])))
        for P in self.proj:
            out.append((f"verify.{P['name']}", "verify", P, lambda P=P: ml.linear_sliced(
                P["xv"], P["W"], P["ends"], P["A"], P["B"], self.rank_of, self.adx_v, cfg.scale,
                ml.VERIFY | ml.PREFETCH_WEIGHTS, ws=self.ws, y=P["yv"], seg_offsets_ptr=self.seg)))
        out.append(("accept", "accept", None, lambda: ml.verify_accept(
            self.p, self.q, self.tok, self.u, ws=self.ws, out_tok=self.out_tok, accepted=self.accepted)))
        if with_base:
            for P in self.proj:
                out.append((f"base.{P['name']}", "base", P, lambda P=P: ml.linear_sliced(
                    P["xv"], P["W"], P["ends"], None, None, None, None, cfg.scale, ml.DRAFT | ml.PREFETCH_WEIGHTS,
                    ws=self.ws, y=P["yb"])))
            # Plain multi-LoRA decoding: one LoRA-on pass over one row per request.
            def plain_plan():
                self.seg_plain, _ = ml.plan_segments(self.adx_d, self.rank_of, cfg.n_adapters, cfg.r_max,
                                                     self.ws_plain)
            out.append(("plain.plan", "plain", None, plain_plan))
            for P in self.proj:
                out.append((f"plain.{P['name']}", "plain", P, lambda P=P: ml.linear_sliced(
                    P["xd"][0], P["W"], P["ends"], P["A"], P["B"], self.rank_of, self.adx_d, cfg.scale,
                    ml.VERIFY | ml.PREFETCH_WEIGHTS, ws=self.ws_plain, y=P["yd"], seg_offsets_ptr=self.seg_plain)))
        return out

    def step(self, side=None):
        """One step in stream order.  With `side` (a second stream) the plan,
        which needs only the adapter indices, runs on it concurrently with the
        draft passes, and the verify pass waits for it."""
        ops = self.ops()
        if side is None:
            for _, _, _, f in ops:
                f()
            return
        torch = self.torch
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            ops[0][3]()
        for _, kind, _, f in ops[1:]:
            if kind == "verify" and side is not None:
                main.wait_stream(side)
                side = None
            f()


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------


def _f64(torch, t):
    return t.float().cpu().numpy().astype(np.float64)


def oracle_sample(torch, wl, requests):
    """Host float64 copies of what the oracle needs for `requests` requests
    of the workload: every group's full W, the A and B of the adapters those
    requests use (relabelled 0..), their rows, and their accept inputs."""
    cfg, k = wl.cfg, wl.k
    req = np.arange(requests)
    ads = sorted({int(a) for a in wl.idx_d[req] if a >= 0})
    remap = {a: i for i, a in enumerate(ads)}
    sub = lambda arr: np.array([remap.get(int(a), -1) for a in arr], dtype=np.int32)  # noqa: E731
    rows_v = np.concatenate([np.arange(r * (k + 1), (r + 1) * (k + 1)) for r in req])
    sel = torch.tensor(ads if ads else [0], dtype=torch.long, device=wl.p.device)
    groups = []
    for P in wl.proj:
        ends = [0] + P["ends"]
        W = _f64(torch, P["W"])
        A = _f64(torch, P["A"][:, sel]) if ads else None
        B = _f64(torch, P["B"][sel]) if ads else None
        per_slice = [(W[ends[s]:ends[s + 1]], A[s] if ads else None, B[:, ends[s]:ends[s + 1]] if ads else None)
                     for s in range(len(P["ends"]))]
        xd = [_f64(torch, P["xd"][d][req]) for d in range(k)]
        xv = _f64(torch, P["xv"][torch.from_numpy(rows_v).to(wl.p.device)])
        groups.append((per_slice, xd, xv))
    ranks = wl.ranks[ads] if ads else np.zeros(1, np.int32)
    acc = tuple(t[:requests].cpu().numpy() for t in (wl.p, wl.q, wl.tok, wl.u))
    return dict(groups=groups, ranks=ranks, idx_v=sub(wl.idx_v[rows_v]), acc=acc, rows_v=len(rows_v),
                scale=cfg.scale)


def oracle_step(sample):
    """The oracle over the sample: k draft passes and the verify pass of every
    projection, then the accept step.  Returns (seconds, verified tokens)."""
    from oracle import accept as OA
    from oracle import layer as OL
    t0 = time.perf_counter()
    for per_slice, xd, xv in sample["groups"]:
        for W, A, B in per_slice:
            for x in xd:
                OL.mlora_linear(x, W, None, None, None, None, sample["scale"], OL.DRAFT)
            if A is not None:
                OL.mlora_linear(xv, W, A, B, sample["ranks"], sample["idx_v"], sample["scale"], OL.VERIFY)
            else:
                OL.mlora_linear(xv, W, None, None, None, None, sample["scale"], OL.DRAFT)
    OA.verify_accept(*sample["acc"])
    return time.perf_counter() - t0, sample["rows_v"]


def time_oracle(torch, wl, seconds, requests=1):
    sample = oracle_sample(torch, wl, requests)
    oracle_step(sample)  # first call: BLAS start-up
    secs, toks, nrep = 0.0, 0, 0
    while secs < seconds and nrep < 50:
        t, n = oracle_step(sample)
        secs += t
        toks += n
        nrep += 1
    return {"value": toks / secs, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{nrep} x {requests} request(s) ({wl.k} draft rows + {wl.k + 1} verify rows each) through the "
                      f"7 projections + accept, float64 numpy on the host cores, BLAS default threads"}


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
    import torch
    name = getattr(args, "config", None) or HEADLINE
    wl = StepWorkload(torch, _NoLib(), torch.device("cpu"), name, seed=0)
    sample = oracle_sample(torch, wl, 1)
    for _ in range(args.warmup):
        oracle_step(sample)
    times, toks = [], 0
    for _ in range(args.steps):
        t, n = oracle_step(sample)
        times.append(t)
        toks += n
    total = sum(times)
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.workload, "requests_per_step": 1},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"1 request per step ({wl.k} draft rows + {wl.k + 1} verify rows through the 7 "
                                   "projections + accept), float64 numpy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


class _NoLib:
    """Stands in for the library when the reference arm builds the workload
    on the CPU: only the workspace sizing is asked, and no workspace is made."""

    def linear_sliced_workspace_bytes(self, *a):
        return 0

    def accept_workspace_bytes(self, *a):
        return 0

    def Workspace(self, *a, **k):
        return None

    def __getattr__(self, name):
        raise RuntimeError(f"the reference arm does not call the library ({name})")


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def graph_of(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_replays(torch, graph, stream, reps, flush=None):
    """ms per replay.  Without `flush`: events around `reps` back-to-back
    replays.  With it: the flush (a write larger than L2) runs before every
    replay and only the replays are timed (one event pair each)."""
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush()
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in evs]))


def time_ops_graph(torch, ops, stream, reps, flush=None):
    """ms for the ops in stream order, from replays of one graph of them (the
    launches overlap at their boundaries as they do inside the step)."""
    g = graph_of(torch, lambda: [op[3]() for op in ops], stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    return time_replays(torch, g, stream, reps, flush)


def per_op_durations(torch, ops, stream, reps):
    """Median duration of every op, from CUDA events on the launching stream
    between consecutive ops inside one captured graph (external events),
    replayed and read back one replay at a time."""
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(ops) + 1)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        evs[0].record(stream)
        for i, op in enumerate(ops):
            op[3]()
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    samples = [[] for _ in ops]
    for _ in range(reps):
        g.replay()
        torch.cuda.synchronize()
        for i in range(len(ops)):
            samples[i].append(evs[i].elapsed_time(evs[i + 1]))
    return {op[0]: float(np.median(samples[i])) for i, op in enumerate(ops)}


def measure_layer(torch, ml, wl, stream, side, steps, peaks, flush):
    """Step time, per-op breakdown, roofline figures of one workload."""
    hbm_gbs, bf16_burst, bf16_sus, peak_kind = peaks
    with torch.cuda.stream(stream):
        for _ in range(3):
            wl.step(side)
    stream.synchronize()
    if wl.ws.status() != 0 or wl.ws_draft.status() != 0:
        raise RuntimeError(f"{wl.name}: device status bits raised during warm-up")
    n0 = ml.launch_count()
    graph = graph_of(torch, lambda: wl.step(side), stream)
    launches = ml.launch_count() - n0
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    use_flush = wl.w_bytes_per_pass < 2 * L2_BYTES
    ms_step = time_replays(torch, graph, stream, steps, flush if use_flush else None)
    if wl.ws.status() != 0 or wl.ws_draft.status() != 0:
        raise RuntimeError(f"{wl.name}: device status bits raised during the timed region")
    op_ms = per_op_durations(torch, wl.ops(with_base=True), stream, max(10, min(steps, 100)))
    # The k draft passes alone, from their own graph.
    ms_draft = time_ops_graph(torch, [op for op in wl.ops() if op[1] == "draft"], stream, max(10, min(steps, 100)),
                              flush if use_flush else None)

    cfg, k = wl.cfg, wl.k
    active = sorted(set(int(a) for a in wl.idx_v if a >= 0))
    active_ranks = [int(wl.ranks[a]) for a in active]
    draft_b = draft_t = verify_b = verify_t = verify_f = 0.0
    kernels = {}  # GEMM kernel -> {bytes, flops, ms, launches, ops, kind}
    calls = {}
    for P in wl.proj:
        bd, fd = layer_bytes_flops(wl.Md, P["K"], P["N"], [], False)
        kd = ml.gemm_kernel_name(wl.Md, P["N"], P["K"], cfg.n_adapters, cfg.r_max, ml.DRAFT)
        td = sum(op_ms[f"draft{d}.{P['name']}"] for d in range(k))
        draft_b += k * bd
        draft_t += td
        e = kernels.setdefault(kd, {"draft_bytes": 0.0, "draft_ms": 0.0, "draft_launches": 0, "draft_ops": [],
                                    "verify_flops": 0.0, "verify_ms": 0.0, "verify_ops": []})
        e["draft_bytes"] += k * bd
        e["draft_ms"] += td
        e["draft_launches"] += k
        e["draft_ops"].append(P["name"])
        bv, fv = layer_bytes_flops(wl.Mv, P["K"], P["N"], active_ranks, True, P["n_proj"])
        tv = op_ms[f"verify.{P['name']}"]
        tb = op_ms[f"base.{P['name']}"]
        verify_b += bv
        verify_f += fv
        verify_t += tv
        kv = ml.gemm_kernel_name(wl.Mv, P["N"], P["K"], cfg.n_adapters, cfg.r_max, ml.VERIFY)
        e = kernels.setdefault(kv, {"draft_bytes": 0.0, "draft_ms": 0.0, "draft_launches": 0, "draft_ops": [],
                                    "verify_flops": 0.0, "verify_ms": 0.0, "verify_ops": []})
        e["verify_flops"] += fv
        e["verify_ms"] += tv
        e["verify_ops"].append(P["name"])
        base_f = 2.0 * wl.Mv * P["N"] * P["K"]
        calls[P["name"]] = {
            "M_verify": wl.Mv, "N": P["N"], "K": P["K"], "verify_kernel": kv, "draft_kernel": kd,
            "verify_us": 1e3 * tv, "verify_TFLOPs": fv / (tv * 1e-3) / 1e12,
            "base_at_verify_rows_us": 1e3 * tb, "base_TFLOPs": base_f / (tb * 1e-3) / 1e12,
            "verify_over_base": tv / tb, "draft_us_per_pass": 1e3 * td / k,
            "draft_GBps": k * bd / (td * 1e-3) / 1e9}
    acc_host = wl.accepted.cpu().numpy()
    acc_b = accept_bytes(cfg.n_requests, cfg.vocab, acc_host, k)
    t_acc = op_ms["accept"]
    # The dominant kernel: the GEMM kernel with the most time over the step.
    dom = max(kernels, key=lambda n: kernels[n]["draft_ms"] + kernels[n]["verify_ms"])
    d = kernels[dom]
    if d["draft_launches"]:
        # Every draft launch on this kernel: its time is the draft passes'
        # graph time; otherwise the per-op times of its launches.
        all_draft = d["draft_launches"] == k * len(wl.proj)
        d_ms = ms_draft if all_draft else d["draft_ms"]
        achieved = d["draft_bytes"] / (d_ms * 1e-3) / 1e9
        traffic, note = profiled_traffic(dom, wl.name)
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                "traffic": traffic, "kernel": f"{dom} (draft passes: {', '.join(d['draft_ops'])}; M={wl.Md})",
                "peak_kind": f"{peak_kind} hbm_gbs",
                "algorithmic_bytes_per_launch": d["draft_bytes"] / d["draft_launches"],
                "avg_launch_us": 1e3 * d_ms / d["draft_launches"], "traffic_source": note,
                "timing": ("events around replays of a graph of the k draft passes (all of this kernel's draft "
                           "launches), divided by its launches" if all_draft else
                           "events between the ops inside one step graph, summed over this kernel's draft launches")}
    else:
        achieved = d["verify_flops"] / (d["verify_ms"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_sus, "unit": "TFLOP/s", "frac": achieved / bf16_sus,
                "traffic": None, "kernel": f"{dom} (verify pass: {', '.join(d['verify_ops'])}; M={wl.Mv})",
                "peak_kind": f"{peak_kind} bf16_tflops_sustained"}
    others = {}
    for n, e in kernels.items():
        if n == dom:
            continue
        o = {}
        if e["draft_ms"]:
            o["draft_GBps"] = e["draft_bytes"] / (e["draft_ms"] * 1e-3) / 1e9
            o["draft_frac_hbm"] = o["draft_GBps"] / hbm_gbs
        if e["verify_ms"]:
            o["verify_TFLOPs"] = e["verify_flops"] / (e["verify_ms"] * 1e-3) / 1e12
            o["verify_frac_bf16_sustained"] = o["verify_TFLOPs"] / bf16_sus
        o["ops"] = {"draft": e["draft_ops"], "verify": e["verify_ops"]}
        others[n] = o
    roof["other_kernels"] = others
    modes = {
        "draft_pass": {"passes": k, "us_per_pass": 1e3 * ms_draft / k, "tokens_per_s": wl.Md * k / (ms_draft * 1e-3),
                       "GBps": draft_b / (ms_draft * 1e-3) / 1e9,
                       "frac_hbm": draft_b / (ms_draft * 1e-3) / 1e9 / hbm_gbs,
                       "us_per_pass_per_op_events": 1e3 * draft_t / k,
                       "timing": "events around replays of a graph of the k draft passes"},
        "verify_pass": {"us": 1e3 * verify_t, "tokens_per_s": wl.Mv / (verify_t * 1e-3),
                        "GBps": verify_b / (verify_t * 1e-3) / 1e9, "frac_hbm": verify_b / (verify_t * 1e-3) / 1e9 / hbm_gbs,
                        "TFLOPs": verify_f / (verify_t * 1e-3) / 1e12,
                        "frac_bf16_sustained": verify_f / (verify_t * 1e-3) / 1e12 / bf16_sus},
        "accept": {"us": 1e3 * t_acc, "requests": cfg.n_requests, "rows_per_s": cfg.n_requests / (t_acc * 1e-3),
                   "GBps": acc_b / (t_acc * 1e-3) / 1e9, "frac_hbm": acc_b / (t_acc * 1e-3) / 1e9 / hbm_gbs,
                   "mean_accepted": float(acc_host.mean())},
        "plain_lora_on_pass": {"us": 1e3 * sum(op_ms[f"plain.{P['name']}"] for P in wl.proj) + 1e3 * op_ms["plain.plan"],
                               "rows": wl.Md,
                               "note": "plain multi-LoRA decoding: one LoRA-on pass over one row per request (plan + 4 calls)"},
        "plan_us": 1e3 * op_ms["plan"],
        "per_op_timing": "events between the ops inside one step graph (breaks the launch overlap at each boundary)",
        "per_op_us": {n: 1e3 * v for n, v in op_ms.items()},
        "calls": calls,
    }
    return {"ms_per_step": ms_step, "tokens_per_s": wl.Mv / (ms_step * 1e-3), "launches_per_step": launches,
            "roofline": roof, "modes": modes,
            "l2": ("L2 flushed before each timed step (W smaller than 2x L2)" if use_flush else
                   f"inputs larger than L2: {wl.w_bytes_per_pass / 1e6:.0f} MB of W streamed per pass, "
                   f"{k + 1} passes per step")}


def measure_accept_sweep(torch, ml, device, stream, reps, peaks, flush, oracle_seconds):
    """The accept step alone at batch 256, vocabulary 128256, k = 1..4:
    back-to-back calls alternating between two input sets, each larger than
    L2 (so no call finds the previous one's rows in L2), from CUDA events
    around replays of a graph of ACCEPT_CALLS calls; and one call alone after
    an L2 flush (launch latency included) for reference."""
    from oracle import accept as OA
    hbm_gbs = peaks[0]
    cfg = WL.ACCEPT_SWEEP
    out = {"workload": f"{cfg.name}: B={cfg.batch} V={cfg.vocab} k=1..4, target logits N(0, 2^2), draft logits + "
                       f"N(0, {WL.ACCEPT_SIGMA}^2)",
           "l2": "inputs larger than L2: two input sets of p and q (394-1182 MB each) alternate between back-to-back "
                 "calls; 'us_single' is one call after an L2 flush", "k": {}}
    for k in ACCEPT_SWEEP_K:
        sets = []
        for seed in (17, 18):
            p, q, tok, u = accept_inputs_device(torch, cfg.vocab, cfg.batch, k, device, seed=seed)
            sets.append(dict(p=p, q=q, tok=tok, u=u, out_tok=torch.empty((cfg.batch, k + 1), dtype=torch.int32,
                                                                         device=device),
                             accepted=torch.empty((cfg.batch,), dtype=torch.int32, device=device)))
        ws = ml.Workspace(ml.accept_workspace_bytes(cfg.batch, k, cfg.vocab), device=device)

        def call(i):
            st = sets[i % 2]
            ml.verify_accept(st["p"], st["q"], st["tok"], st["u"], ws=ws, out_tok=st["out_tok"],
                             accepted=st["accepted"])
        with torch.cuda.stream(stream):
            for i in range(4):
                call(i)
        stream.synchronize()
        g1 = graph_of(torch, lambda: call(0), stream)
        ms_single = time_replays(torch, g1, stream, reps, flush)
        gn = graph_of(torch, lambda: [call(i) for i in range(ACCEPT_CALLS)], stream)
        with torch.cuda.stream(stream):
            gn.replay()
        ms = time_replays(torch, gn, stream, max(3, reps // 4)) / ACCEPT_CALLS
        if ws.status() != 0:
            raise RuntimeError("device status bits raised in the accept sweep")
        accs = [st["accepted"].cpu().numpy() for st in sets]
        b = 0.5 * sum(accept_bytes(cfg.batch, cfg.vocab, a, k) for a in accs)
        st = sets[0]
        host = tuple(t[:4].cpu().numpy() for t in (st["p"], st["q"], st["tok"], st["u"]))
        OA.verify_accept(*host)
        secs, rows = 0.0, 0
        while secs < oracle_seconds:
            t0 = time.perf_counter()
            OA.verify_accept(*host)
            secs += time.perf_counter() - t0
            rows += 4
        out["k"][str(k)] = {"us": 1e3 * ms, "us_single": 1e3 * ms_single, "rows_per_s": cfg.batch / (ms * 1e-3),
                            "GBps": b / (ms * 1e-3) / 1e9, "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_gbs,
                            "algorithmic_bytes": int(b), "mean_accepted": float(np.mean([a.mean() for a in accs])),
                            "oracle": {"rows_per_s": rows / secs, "cores": cpu_cores(),
                                       "sample": f"{rows} requests, float64/integer numpy"}}
        del sets, ws, g1, gn
        torch.cuda.empty_cache()
    return out


def measure_softmax_row(torch, ml, wl, device, stream, reps, peaks, flush):
    """The steps beside the accept step at the workload's sizes: the draft
    draw from LoRA-off logits (one per draft pass) and the accept step on
    logits (softmax fused), each from CUDA events around graph replays with
    L2 flushed before each."""
    hbm_gbs = peaks[0]
    cfg, k = wl.cfg, wl.k
    B, V = cfg.n_requests, cfg.vocab
    zp, zq, tok, u = accept_logits_device(torch, V, B, k, device, seed=23)
    ws_s = ml.Workspace(int(ml.library().mlora_draft_sample_workspace_bytes(B, V)), device=device)
    ws_a = ml.Workspace(ml.accept_workspace_bytes(B, k, V), device=device)
    zq0 = zq[:, 0].contiguous()
    u0 = u[:, 0].contiguous()
    t_s = torch.empty((B,), dtype=torch.int32, device=device)
    out_tok = torch.empty((B, k + 1), dtype=torch.int32, device=device)
    accepted = torch.empty((B,), dtype=torch.int32, device=device)
    sample = lambda: ml.draft_sample(zq0, u0, ws=ws_s, tok=t_s, want_q=False)  # noqa: E731
    acc = lambda: ml.verify_accept_logits(zp, zq, tok, u, ws=ws_a, out_tok=out_tok, accepted=accepted)  # noqa: E731
    res = {}
    for name, fn in (("draft_sample", sample), ("accept_logits", acc)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = graph_of(torch, fn, stream)
        res[name] = time_replays(torch, g, stream, reps, flush)
    if ws_s.status() != 0 or ws_a.status() != 0:
        raise RuntimeError("device status bits raised in the softmax-row measurement")
    acc_h = accepted.cpu().numpy()
    rej = int((acc_h < k).sum())
    # Bytes the design reads: the draw reads its logit row twice (statistics,
    # then weights); the accept reads every target and draft row once for the
    # statistics, then the scanned row (p_n, and q_n on a rejection).
    b_sample = 2 * 4 * V * B
    b_acc = (2 * k + 1) * 4 * V * B + 4 * V * (B + rej)
    return {
        "sizes": f"B={B} V={V} k={k}",
        "draft_sample": {"us": 1e3 * res["draft_sample"], "rows_per_s": B / (res["draft_sample"] * 1e-3),
                         "GBps": b_sample / (res["draft_sample"] * 1e-3) / 1e9,
                         "frac_hbm": b_sample / (res["draft_sample"] * 1e-3) / 1e9 / hbm_gbs,
                         "bytes": b_sample, "per_draft_pass": True},
        "accept_logits": {"us": 1e3 * res["accept_logits"], "rows_per_s": B / (res["accept_logits"] * 1e-3),
                          "GBps": b_acc / (res["accept_logits"] * 1e-3) / 1e9,
                          "frac_hbm": b_acc / (res["accept_logits"] * 1e-3) / 1e9 / hbm_gbs, "bytes": b_acc,
                          "mean_accepted": float(acc_h.mean())},
        "l2": "L2 flushed before each timed call",
    }


def measure_fp8_draft(torch, ml, wl, stream, side, steps, peaks, flush, bf16_step_ms, bf16_draft_us):
    """The same decode step with the draft passes on E4M3 weights: step time,
    draft-pass time and bytes (W codes + x + its codes + y), and the quality
    of each draft projection against its bf16 output (relative error)."""
    hbm_gbs = peaks[0]
    wl.enable_fp8()
    try:
        with torch.cuda.stream(stream):
            for _ in range(3):
                wl.step(side)
        stream.synchronize()
        graph = graph_of(torch, lambda: wl.step(side), stream)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        ms = time_replays(torch, graph, stream, steps)
        t_draft = time_ops_graph(torch, [op for op in wl.ops() if op[1] == "draft"], stream, max(10, min(steps, 50)))
        if wl.ws_fp8.status() != 0 or wl.ws.status() != 0:
            raise RuntimeError("device status bits raised in the FP8 draft measurement")
        k = wl.k
        nbytes = k * sum(P["N"] * P["K"] + 4 * wl.Md * P["K"] + 2 * wl.Md * P["N"] for P in wl.proj)
        quality = {}
        for P in wl.proj:
            y8 = ml.linear_fp8(P["xd"][0], P["W8"], P["sw"], ws=wl.ws_fp8).float()
            y16 = ml.linear_sliced(P["xd"][0], P["W"], P["ends"], None, None, None, None, 1.0, ml.DRAFT,
                                   ws=wl.ws_draft).float()
            quality[P["name"]] = float(torch.linalg.norm(y8 - y16) / torch.linalg.norm(y16))
        torch.cuda.synchronize()
    finally:
        wl.fp8 = False
    return {"ms_per_step": ms, "tokens_per_s": wl.Mv / (ms * 1e-3), "speedup_vs_bf16_step": bf16_step_ms / ms,
            "draft_pass": {"us_per_pass": 1e3 * t_draft / k, "GBps": nbytes / (t_draft * 1e-3) / 1e9,
                           "frac_hbm": nbytes / (t_draft * 1e-3) / 1e9 / hbm_gbs,
                           "speedup_vs_bf16_pass": bf16_draft_us / (1e3 * t_draft / k),
                           "bytes_per_pass": nbytes / k},
            "quality_rel_error_vs_bf16": quality,
            "note": "draft passes on E4M3 W (per-row scales) and per-token E4M3 activations; verify pass and "
                    "accept unchanged (bf16), so emitted tokens keep the target distribution"}


KV_HEAD_DIM = 128  # head size of the 32B- and 8B-class shapes (q 5120 = 40 x 128, k/v 1024 = 8 x 128)


def measure_kv_cache(torch, ml, wl, device, stream, reps, peaks, flush):
    """The hybrid KV cache at the workload's sizes: one draft step's K/V rows
    (one per request), the verify pass's (k + 1 per request) and the commit,
    from the fused q|k|v output into a paged cache of 16-token blocks; CUDA
    events around graph replays with L2 flushed before each.  The oracle's
    copy of the same rows is timed beside it."""
    import numpy as np
    from oracle import kvcache as OK
    hbm_gbs = peaks[0]
    cfg, k = wl.cfg, wl.k
    P = wl.proj[0]
    if P["n_proj"] != 3:
        return {"skipped": "the workload has no fused q|k|v projection"}
    ends = [int(e) for e in P["ends"]]
    Nq, Nkv = ends[0], ends[1] - ends[0]
    D = KV_HEAD_DIM if Nkv % KV_HEAD_DIM == 0 else Nkv
    H = Nkv // D
    B, bs, max_blocks = cfg.n_requests, 16, 64
    num_blocks = B * max_blocks
    g = torch.Generator(device=device)
    g.manual_seed(31)
    bt = torch.randperm(num_blocks, generator=g, device=device).to(torch.int32).view(B, max_blocks)
    seq0 = torch.randint(0, max_blocks * bs - 2 * k - 2, (B,), generator=g, device=device, dtype=torch.int32)
    seq = seq0.clone()
    kc = torch.zeros((num_blocks, bs, H, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    yd = torch.randn((wl.Md, P["N"]), generator=g, device=device).to(torch.bfloat16)
    yv = torch.randn((wl.Mv, P["N"]), generator=g, device=device).to(torch.bfloat16)
    acc = torch.randint(0, k + 1, (B,), generator=g, device=device, dtype=torch.int32)
    ws = ml.Workspace(ml.kv_workspace_bytes(), device=device)
    calls = {
        "draft_step": lambda: ml.kv_write(yd, Nq, Nq + Nkv, H, D, bt, seq, 1, 0, kc, vc, ws=ws),
        "verify_pass": lambda: ml.kv_write(yv, Nq, Nq + Nkv, H, D, bt, seq, k + 1, 0, kc, vc, ws=ws),
    }
    res = {}
    for name, fn in calls.items():
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        gr = graph_of(torch, fn, stream)
        ms = time_replays(torch, gr, stream, reps, flush)
        rows = wl.Md if name == "draft_step" else wl.Mv
        nbytes = rows * 2 * H * D * 2 * 2  # K and V rows read from y and written to the cache
        res[name] = {"rows": rows, "us": 1e3 * ms, "GBps": nbytes / (ms * 1e-3) / 1e9,
                     "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_gbs, "bytes": nbytes}
    with torch.cuda.stream(stream):
        ml.kv_commit(acc, seq, stream=stream)
    stream.synchronize()
    if not torch.equal(seq, seq0 + acc + 1) or ws.status() != 0:
        raise RuntimeError("KV cache measurement: commit or status check failed")
    # the oracle on the verify pass's rows (host, numpy)
    yh = yv.view(torch.int16).cpu().numpy().view(np.uint16)
    bth, sh = bt.cpu().numpy(), seq0.cpu().numpy()
    kh = np.zeros((num_blocks, bs, H, D), np.uint16)
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < 2.0:
        OK.kv_write(yh, Nq, Nq + Nkv, H, D, bth, sh, k + 1, 0, kh, kh)
        n += 1
    secs = time.perf_counter() - t0
    return {"sizes": f"B={B} k={k} H={H} D={D} block_size={bs}", **res,
            "oracle": {"rows_per_s": n * wl.Mv / secs, "cores": 1, "sample": f"{n} verify passes, numpy"},
            "note": "a copy of a few MB: launch latency bounds it, not HBM",
            "l2": "L2 flushed before each timed call"}


def run_e2e(torch, ml, wl, stream, side, steps, world):
    """Host buffers in, host buffers out, through the public binding.  Every
    step copies its activations, adapter indices and probabilities from
    pinned host memory and reads every output back.  The copy-in of step s+1
    runs on a second stream while step s computes (two device input sets,
    each with its own captured graph of the same binding calls); the
    read-back follows each step on the compute stream."""
    def pin_like(t):
        return torch.empty(tuple(t.shape), dtype=t.dtype).pin_memory()

    def inputs_of():
        return [x for P in wl.proj for x in P["xd"]] + [P["xv"] for P in wl.proj] + [wl.adx_v, wl.p, wl.q, wl.tok, wl.u]

    def set_inputs(lst):
        i = 0
        for P in wl.proj:
            P["xd"] = lst[i:i + wl.k]
            i += wl.k
        for P in wl.proj:
            P["xv"] = lst[i]
            i += 1
        wl.adx_v, wl.p, wl.q, wl.tok, wl.u = lst[i:i + 5]

    set0 = inputs_of()
    host_in = [pin_like(t) for t in set0]
    for h, t in zip(host_in, set0):
        h.copy_(t)
    set1 = [torch.empty_like(t) for t in set0]
    sets = (set0, set1)
    outs = [P["yd"] for P in wl.proj] + [P["yv"] for P in wl.proj] + [wl.out_tok, wl.accepted]
    host_out = [pin_like(t) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def copy_in(st):
        for d, h in zip(st, host_in):
            d.copy_(h, non_blocking=True)

    def read_back():
        for h, d in zip(host_out, outs):
            h.copy_(d, non_blocking=True)

    graphs = []
    with torch.cuda.stream(stream):
        for st in sets:
            set_inputs(st)
            copy_in(st)
            wl.step(side)
            stream.synchronize()
            graphs.append(graph_of(torch, lambda: wl.step(side), stream))
    set_inputs(set0)
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
    ml.set_shrink_path({"auto": ml.SHRINK_AUTO, "warp": ml.SHRINK_WARP, "tensor": ml.SHRINK_TENSOR}[args.shrink])

    peaks = _peaks()
    stream = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device)
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    flush = lambda: flush_buf.fill_(1.0)  # noqa: E731

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- headline workload
    wl = StepWorkload(torch, ml, device, args.config, seed=rank)
    head = measure_layer(torch, ml, wl, stream, side, min(args.steps, 200), peaks, flush)
    # the timed headline run: K replays, clocks sampled meanwhile
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            wl.step(side)
    stream.synchronize()
    graph = graph_of(torch, lambda: wl.step(side), stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ms = time_replays(torch, graph, stream, args.steps)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    if wl.ws.status() != 0:
        raise RuntimeError("device status bits raised during the timed region")
    ms = max_over_ranks(torch, ms, world, device)
    value = job_throughput(wl.Mv, world, ms)
    e2e = run_e2e(torch, ml, wl, stream, side, max(3, min(args.steps, 50)), world)
    try:
        softmax_row = measure_softmax_row(torch, ml, wl, device, stream, 30, peaks, flush)
    except Exception as exc:
        softmax_row = {"failed": f"{type(exc).__name__}: {exc}"}
    try:
        kv_cache = measure_kv_cache(torch, ml, wl, device, stream, 30, peaks, flush)
    except Exception as exc:
        kv_cache = {"failed": f"{type(exc).__name__}: {exc}"}
    try:
        fp8_draft = measure_fp8_draft(torch, ml, wl, stream, side, min(args.steps, 100), peaks, flush, ms,
                                      head["modes"]["draft_pass"]["us_per_pass"])
    except Exception as exc:
        fp8_draft = {"failed": f"{type(exc).__name__}: {exc}"}
    alpha_hat = ml.estimate_acceptance(wl.accepted.cpu().numpy(), wl.k)
    cpu = None
    if rank == 0 and world == 1:
        try:
            cpu = time_oracle(torch, wl, 10.0)
        except Exception as exc:  # a baseline that fails does not void the GPU number
            cpu = {"value": None, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": f"failed: {exc}"}
    head_workload, head_cfg = wl.workload, wl.cfg
    head_rows = (wl.Md, wl.Mv, [P["name"] for P in wl.proj], wl.k)
    del wl, graph
    torch.cuda.empty_cache()

    # ---- the other workloads (rank 0 of a single-GPU run reports them)
    extra, sweep = {}, None
    if args.extra == "all" and world == 1:
        for name in LAYER_RUNS:
            if name == args.config:
                continue
            try:
                w2 = StepWorkload(torch, ml, device, name, seed=0)
                r = measure_layer(torch, ml, w2, stream, side, max(20, min(args.steps, 100)), peaks, flush)
                r["workload"] = w2.workload
                r["cpu_baseline"] = time_oracle(torch, w2, 3.0, requests=min(4, w2.cfg.n_requests))
                extra[name] = r
                del w2
            except Exception as exc:
                extra[name] = {"failed": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()
        try:
            sweep = measure_accept_sweep(torch, ml, device, stream, 30, peaks, flush, 2.0)
        except Exception as exc:
            sweep = {"failed": f"{type(exc).__name__}: {exc}"}

    # The run-time draft gate on the measured cycle times: a cycle with k
    # drafts costs the measured step plus k draft draws; plain decoding costs
    # one LoRA-on pass over one row per request plus one draw.
    gate = None
    try:
        t_draw = softmax_row["draft_sample"]["us"] if "draft_sample" in softmax_row else 0.0
        t_plain = head["modes"]["plain_lora_on_pass"]["us"] + t_draw
        cycles = {head_rows[3]: 1e3 * ms + head_rows[3] * t_draw}
        for name, r in extra.items():
            if "failed" not in r and LAYER_RUNS[name][0] is head_cfg:
                kk = LAYER_RUNS[name][1]
                cycles[kk] = 1e3 * r["ms_per_step"] + kk * t_draw
        full = {kk: cycles[kk] for kk in sorted(cycles)}
        kmax = max(full)
        if all(kk in full for kk in range(1, kmax + 1)):
            kk, gain = ml.draft_gate(full, t_plain, alpha_hat)
        else:
            # only some draft lengths measured: the gate over those, by its formula
            rates = {kk: ml.library().mlora_expected_tokens(alpha_hat, kk) / t for kk, t in full.items()}
            best = max(rates, key=rates.get)
            kk, gain = (best, rates[best] * t_plain) if rates[best] > 1.0 / t_plain else (0, 1.0)
        gate = {"alpha_estimate": alpha_hat, "t_plain_us": t_plain, "t_cycle_us": full, "k": kk,
                "tokens_per_plain_step_time": gain,
                "expected_tokens": {str(j): ml.library().mlora_expected_tokens(alpha_hat, j) for j in full},
                "note": "k = 0 would skip drafting; gain = emitted tokens per request in the time of one plain step"}
    except Exception as exc:
        gate = {"failed": f"{type(exc).__name__}: {exc}"}

    if rank == 0:
        Md, Mv, calls, k = head_rows
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": head_workload, "requests": head_cfg.n_requests, "draft_len": k,
                       "draft_rows_per_pass": Md, "verify_rows": Mv,
                       "projections": [p[0] for p in head_cfg.projections], "layer_calls": calls,
                       "parallelism": f"replicas x{world}", "l2": head["l2"], "shrink": args.shrink,
                       "graph": "one CUDA graph per step; the plan runs on a second stream beside the draft passes"},
            "gpu_launches": head["launches_per_step"] * args.steps,
            "roofline": head["roofline"],
            "modes": head["modes"],
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "configs": extra,
            "accept_sweep": sweep,
            "softmax_and_draft_draw": softmax_row,
            "kv_cache": kv_cache,
            "fp8_draft": fp8_draft,
            "draft_gate": gate,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=HEADLINE, choices=sorted(LAYER_RUNS))
    ap.add_argument("--extra", default="all", choices=["all", "none"])
    ap.add_argument("--only", default=None, choices=["accept"],
                    help="run only the accept sweep (batch 256, vocabulary 128256, k = 1..4) and print its results")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--shrink", default="auto", choices=["auto", "warp", "tensor"],
                    help="which kernel writes the verify pass's low-rank operand (default: the library's choice)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.only == "accept":
        return run_accept_only(args)
    return run_gpu(args)


def run_accept_only(args):
    """The accept sweep alone (for profiling the accept kernels): one JSON
    line with the sweep's results, not a bench line."""
    import torch
    import speculative_lora_decoding_gb300 as ml
    if not os.path.exists(ml.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream(device)
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    sweep = measure_accept_sweep(torch, ml, device, stream, max(3, min(args.steps, 30)), _peaks(),
                                 lambda: flush_buf.fill_(1.0), 0.5)
    print(json.dumps({"accept_sweep": sweep}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
