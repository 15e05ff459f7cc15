"""Seeded synthetic inputs for the multi-LoRA layer and the accept/resample step.

This module only draws random numbers and rounds them to the storage types the
kernels read (bf16 bit patterns, fp32, int32).  It holds none of the method's
arithmetic: no GEMM, no low-rank update, no accept test and no residual sample.
Both the float64 oracle and the CUDA path take their inputs from here, so the
two see bit-identical data.

Workload shapes follow the multi-LoRA serving setting of the InvisibleLoRA
abstract ("InvisibleLoRA: Fast Multi-LoRA Serving Without Per-Token LoRA
Decoding", abstract) and the LoRA layer "output = W·x + scale · B(A·x)" of
"Multi-LoRA Serving in Practice" (section "Core Principle: Shared Base Model,
Per-Request Adapter Selection").  Models are stood in for by their projection
shapes only; all weights are random.

Random streams: every component draws from its own PCG64 stream keyed by
(seed, component id, projection index, mode), so a test that needs only one
projection does not have to draw the others first.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# ----------------------------------------------------------------------------
# bf16 storage rounding (input quantisation, not part of the method)
# ----------------------------------------------------------------------------


def bf16_bits(a) -> np.ndarray:
    """Round float values to bf16 (round to nearest, ties to even); uint16 bits."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = u.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Workload definitions
# ----------------------------------------------------------------------------

# (name, K = in features, N = out features)
PROJ_TINY = (("proj", 512, 512),)
PROJ_8B = (
    ("q", 4096, 4096),
    ("k", 4096, 1024),
    ("v", 4096, 1024),
    ("o", 4096, 4096),
    ("gate", 4096, 14336),
    ("up", 4096, 14336),
    ("down", 14336, 4096),
)
PROJ_32B = (
    ("q", 5120, 5120),
    ("k", 5120, 1024),
    ("v", 5120, 1024),
    ("o", 5120, 5120),
    ("gate", 5120, 27648),
    ("up", 5120, 27648),
    ("down", 27648, 5120),
)

LLAMA3_VOCAB = 128256

# Draft-logit noise that puts the mean closed-form acceptance sum_v min(p, q)
# near 0.945, the middle of the 92-97% median acceptance band of the
# InvisibleLoRA abstract.  Target logits are N(0, 2^2).  The value comes from
# tests/golden/calibrate_sigma.py (bisection over the float64 acceptance rate).
ACCEPT_SIGMA = 0.1378


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    projections: tuple
    n_requests: int
    n_adapters: int
    ranks: tuple            # one value: every adapter; several: drawn uniformly
    popularity: str         # "uniform" | "zipf"
    zipf_s: float
    draft_lengths: tuple    # k values; verify rows per request = k + 1
    scale: float
    vocab: int = LLAMA3_VOCAB

    @property
    def r_max(self) -> int:
        return max(self.ranks)

    def rows(self, mode: str, k: int | None = None) -> int:
        if mode == "draft":
            return self.n_requests
        k = self.draft_lengths[0] if k is None else k
        return self.n_requests * (k + 1)


TINY = LayerConfig("tiny-512", PROJ_TINY, 8, 4, (8,), "uniform", 0.0, (1,), 16.0 / 8.0, vocab=1000)
LLAMA8B_R16 = LayerConfig("llama3-8b-shapes/64req/16ad-r16/zipf1.1", PROJ_8B, 64, 16, (16,), "zipf", 1.1, (1,), 2.0)
LLAMA8B_HET = LayerConfig("llama3-8b-shapes/256req/128ad-r8..64/zipf1.1", PROJ_8B, 256, 128, (8, 16, 32, 64), "zipf", 1.1, (1,), 2.0)
QWEN32B_R16 = LayerConfig("32b-shapes/128req/64ad-r16/uniform", PROJ_32B, 128, 64, (16,), "uniform", 0.0, (1, 2, 4), 2.0)

LAYER_CONFIGS = {c.name: c for c in (TINY, LLAMA8B_R16, LLAMA8B_HET, QWEN32B_R16)}


@dataclasses.dataclass(frozen=True)
class AcceptConfig:
    name: str
    vocab: int
    batch: int
    draft_lengths: tuple
    target_std: float = 2.0
    sigma: float = ACCEPT_SIGMA


ACCEPT_SWEEP = AcceptConfig("accept-v128256-b256", LLAMA3_VOCAB, 256, (1, 2, 3, 4))
ACCEPT_TINY = AcceptConfig("accept-v1000-b8", 1000, 8, (1,))

# ----------------------------------------------------------------------------
# Random streams
# ----------------------------------------------------------------------------

_STREAM = {"W": 1, "A": 2, "B": 3, "rank": 4, "idx": 5, "x": 6,
           "z": 7, "noise": 8, "draft_u": 9, "u": 10}
_MODE = {"draft": 0, "verify": 1}


def rng(seed: int, component: str, *extra: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAM[component], *extra])))


def _normal_bf16(g: np.random.Generator, shape, std: float) -> np.ndarray:
    z = g.standard_normal(shape, dtype=np.float32)
    z *= np.float32(std)
    return bf16_bits(z)


# ----------------------------------------------------------------------------
# Layer inputs
# ----------------------------------------------------------------------------


def adapter_ranks(cfg: LayerConfig, seed: int = 0) -> np.ndarray:
    """Rank of each resident adapter (int32 [n_adapters])."""
    if len(cfg.ranks) == 1:
        return np.full(cfg.n_adapters, cfg.ranks[0], dtype=np.int32)
    g = rng(seed, "rank")
    return np.asarray(cfg.ranks, dtype=np.int32)[g.integers(0, len(cfg.ranks), cfg.n_adapters)]


def request_adapters(cfg: LayerConfig, seed: int = 0) -> np.ndarray:
    """Adapter id of each request (int32 [n_requests]).

    "zipf": truncated Zipf over the resident adapters, P(i) proportional to
    i^-s for i = 1..n_adapters, id = i - 1.  "uniform": ids uniform.
    """
    g = rng(seed, "idx")
    n = cfg.n_adapters
    if cfg.popularity == "uniform":
        return g.integers(0, n, cfg.n_requests).astype(np.int32)
    w = np.arange(1, n + 1, dtype=np.float64) ** (-cfg.zipf_s)
    w /= w.sum()
    return g.choice(n, size=cfg.n_requests, p=w).astype(np.int32)


def row_adapters(cfg: LayerConfig, mode: str, k: int | None = None, seed: int = 0) -> np.ndarray:
    """Adapter index per token row.  Verify rows are request-major:
    row = request * (k + 1) + t, t = 0 the committed token, t >= 1 drafts."""
    req = request_adapters(cfg, seed)
    if mode == "draft":
        return req
    k = cfg.draft_lengths[0] if k is None else k
    return np.repeat(req, k + 1).astype(np.int32)


def projection_weights(cfg: LayerConfig, p: int, seed: int = 0, r_max: int | None = None):
    """bf16 bits of W [N, K], A_stack [n_ad, r_max, K], B_stack [n_ad, N, r_max].

    W ~ N(0, 1/K), A ~ N(0, 1/K), B ~ N(0, 1/r) (the tiny workload's recipe,
    applied to every workload).  Entries of A past row rank_of[a] and of B past
    column rank_of[a] are padding, filled with zeros here.
    """
    _, K, N = cfg.projections[p]
    r_max = cfg.r_max if r_max is None else r_max
    ranks = adapter_ranks(cfg, seed)
    W = _normal_bf16(rng(seed, "W", p), (N, K), 1.0 / math.sqrt(K))
    A = np.zeros((cfg.n_adapters, r_max, K), dtype=np.uint16)
    B = np.zeros((cfg.n_adapters, N, r_max), dtype=np.uint16)
    ga, gb = rng(seed, "A", p), rng(seed, "B", p)
    for a in range(cfg.n_adapters):
        r = int(ranks[a])
        A[a, :r, :] = _normal_bf16(ga, (r, K), 1.0 / math.sqrt(K))
        B[a, :, :r] = _normal_bf16(gb, (N, r), 1.0 / math.sqrt(r))
    return W, A, B, ranks


# Projections of one transformer block that read the same input rows: q, k
# and v read the normalised hidden state, gate and up the normalised output of
# attention; o and down each read their own.
_SHARED_INPUT = (("q", "k", "v"), ("gate", "up"))


def input_groups(cfg: LayerConfig) -> list:
    """Projection indices grouped by the input rows they read, in order:
    [(0, 1, 2), (3,), (4, 5), (6,)] for the 8B and 32B shapes."""
    names = [n for n, _, _ in cfg.projections]
    groups, seen = [], set()
    for i, n in enumerate(names):
        if i in seen:
            continue
        g = (i,)
        for shared in _SHARED_INPUT:
            if n == shared[0] and all(x in names for x in shared):
                g = tuple(names.index(x) for x in shared)
        seen.update(g)
        groups.append(g)
    return groups


def activations(cfg: LayerConfig, p: int, mode: str, k: int | None = None, seed: int = 0) -> np.ndarray:
    """bf16 bits of x [M, K], entries N(0, 1).  Projections of one input group
    (see input_groups) get the same rows."""
    _, K, _ = cfg.projections[p]
    M = cfg.rows(mode, k)
    kk = cfg.draft_lengths[0] if k is None else k
    first = next(g[0] for g in input_groups(cfg) if p in g)
    return _normal_bf16(rng(seed, "x", first, _MODE[mode], kk), (M, K), 1.0)


# ----------------------------------------------------------------------------
# Accept/resample inputs
# ----------------------------------------------------------------------------


def _softmax_f32(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def accept_inputs(V: int, B: int, k: int, sigma: float = ACCEPT_SIGMA, target_std: float = 2.0,
                  seed: int = 0):
    """Target probabilities p [B, k+1, V], draft probabilities q [B, k, V]
    (float64 softmax rounded to fp32), draft tokens [B, k] drawn from q, and
    uniforms [B, k+1] in [0, 1) as fp32.

    Target logits ~ N(0, target_std^2); draft logits = target logits of the
    same position + N(0, sigma^2).  Draft tokens are drawn from the fp32 q
    with a float64 cumulative sum and their own uniform stream.
    """
    gz, gn, gd, gu = rng(seed, "z", V, k), rng(seed, "noise", V, k), rng(seed, "draft_u", V, k), rng(seed, "u", V, k)
    p = np.empty((B, k + 1, V), dtype=np.float32)
    q = np.empty((B, k, V), dtype=np.float32)
    tok = np.empty((B, k), dtype=np.int32)
    for b in range(B):
        z = gz.standard_normal((k + 1, V)) * target_std
        p[b] = _softmax_f32(z)
        q[b] = _softmax_f32(z[:k] + gn.standard_normal((k, V)) * sigma)
        for i in range(k):
            c = np.cumsum(q[b, i].astype(np.float64))
            t = int(np.searchsorted(c, gd.random() * c[-1], side="right"))
            tok[b, i] = min(t, V - 1)
    u = gu.random((B, k + 1), dtype=np.float32)
    return p, q, tok, u


def accept_logits(V: int, B: int, k: int, sigma: float = ACCEPT_SIGMA, target_std: float = 2.0, seed: int = 0):
    """Logits for the accept step and the draft draw: target logits z_p
    [B, k+1, V] ~ N(0, target_std^2), draft logits z_q [B, k, V] = z_p[:, :k] +
    N(0, sigma^2), both rounded to fp32; draft tokens [B, k] drawn from the fp32
    probabilities of z_q (float64 softmax, float64 cumulative sum, their own
    uniform stream); uniforms [B, k+1] in [0, 1) as fp32."""
    gz, gn, gd, gu = (rng(seed, c, V, k, 1) for c in ("z", "noise", "draft_u", "u"))
    zp = (gz.standard_normal((B, k + 1, V)) * target_std).astype(np.float32)
    zq = (zp[:, :k].astype(np.float64) + gn.standard_normal((B, k, V)) * sigma).astype(np.float32)
    tok = np.empty((B, k), dtype=np.int32)
    for b in range(B):
        q = _softmax_f32(zq[b].astype(np.float64))
        for i in range(k):
            c = np.cumsum(q[i].astype(np.float64))
            tok[b, i] = min(int(np.searchsorted(c, gd.random() * c[-1], side="right")), V - 1)
    u = gu.random((B, k + 1), dtype=np.float32)
    return zp, zq, tok, u
