"""GPU parity of the accept / resample step (a5-a6): out_tok and accepted must
equal the oracle's bit for bit on identical fp32 inputs and uniforms."""
import json
import os

import numpy as np
import pytest
import torch

import workloads as WL
from oracle import accept as OA
from tests.gpu_util import dev, needs_gpu

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gpu(ml, p, q, tok, u, ws=None):
    out, acc = ml.verify_accept(dev(p), dev(q), dev(tok), dev(u), ws=ws)
    return out.cpu().numpy(), acc.cpu().numpy()


def _check(ml, p, q, tok, u):
    B, k1, V = p.shape
    ws = ml.Workspace(ml.accept_workspace_bytes(B, k1 - 1, V))
    out, acc = _gpu(ml, p, q, tok, u, ws)
    out_r, acc_r, st_r = OA.verify_accept(p, q, tok, u)
    assert np.array_equal(acc, acc_r)
    assert np.array_equal(out, out_r)
    assert ws.status() == st_r
    return acc


def test_hand_worked_examples():
    ml = needs_gpu()
    g = json.load(open(os.path.join(GOLDEN, "accept_hand_example.json")))
    for c in g["cases"]:
        p = np.asarray(c["p"], np.float32)
        q = np.asarray(c["q"], np.float32)
        tok = np.asarray(c["draft_tok"], np.int32)
        u = np.asarray(c["u"], np.float32)
        ws = ml.Workspace(ml.accept_workspace_bytes(*tok.shape, p.shape[-1]))
        out, acc = _gpu(ml, p, q, tok, u, ws)
        assert out.tolist() == c["out_tok"] and acc.tolist() == c["accepted"], c["why"]
        assert ws.status() == c.get("status", 0), c["why"]


def test_tiny_workload():
    ml = needs_gpu()
    cfg = WL.ACCEPT_TINY
    p, q, tok, u = WL.accept_inputs(cfg.vocab, cfg.batch, 1, seed=0)
    _check(ml, p, q, tok, u)


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_full_sweep_bit_exact(k):
    ml = needs_gpu()
    cfg = WL.ACCEPT_SWEEP
    p, q, tok, u = WL.accept_inputs(cfg.vocab, cfg.batch, k, seed=0)
    acc = _check(ml, p, q, tok, u)
    assert 0 < acc.mean() <= k


@pytest.mark.parametrize("B,k,V", [(1, 1, 1), (3, 2, 5), (7, 1, 1001), (64, 1, 128256), (2, 3, 32000), (5, 16, 4099),
                                   (37, 16, 4100), (19, 5, 8200), (45, 3, 12292)])
def test_ragged_sizes(B, k, V):
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(V, B, k, sigma=0.5, seed=B + k)
    _check(ml, p, q, tok, u)


def test_forced_rejections_and_bonus():
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(50000, 32, 2, seed=4)
    u[:16, 0] = np.float32(0.999999)   # mostly rejects at 0
    u[16:, :2] = np.float32(0.0)       # always keeps both drafts -> bonus from p_2
    acc = _check(ml, p, q, tok, u)
    assert (acc[16:] == 2).all()


def test_q_equal_p_accepts_all():
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(4096, 16, 3, seed=5)
    q = p[:, :3].copy()
    acc = _check(ml, p, q, tok, u)
    assert (acc == 3).all()


def test_invalid_inputs_match_oracle_status():
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(4096, 8, 2, seed=6)
    tok[0, 0] = 4096          # out of range
    tok[1, 1] = -3
    p[2, 0, 17] = np.nan      # inside a row that is read when request 2 rejects at 0
    u[2, 0] = np.float32(0.999999)
    u[3, 2] = np.float32(1.5)
    p[4, :, :] = 0.0          # zero mass
    q[4, :, :] = 0.0
    u[5, :2] = np.float32(0.0)  # request 5 keeps both drafts: its bonus row holds a value above 1
    p[5, 2, 33] = np.float32(1.5)
    u[6, :2] = np.float32(0.0)  # request 6: a negative zero in its bonus row (valid, no status bit)
    p[6, 2, 7] = np.float32(-0.0)
    _check(ml, p, q, tok, u)


def _offset_copy(a):
    """The same values in a device buffer whose start is 4 bytes past a
    16-byte boundary (rows of aligned float4 are then unavailable)."""
    flat = torch.empty(a.size + 1, dtype=torch.float32, device="cuda")
    view = flat[1:].view(a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    assert view.data_ptr() % 16 == 4
    return view


def test_streaming_and_per_chunk_forms_agree():
    """Aligned rows take the streaming form, rows starting off a 16-byte
    boundary the per-chunk form; both must give the oracle's tokens."""
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(12288, 40, 2, seed=8)
    u[::3, 0] = np.float32(0.999999)   # rejections at position 0 in every third request
    out_r, acc_r, st_r = OA.verify_accept(p, q, tok, u)
    for mk in (dev, _offset_copy):
        ws = ml.Workspace(ml.accept_workspace_bytes(40, 2, 12288))
        out, acc = ml.verify_accept(mk(p), mk(q), dev(tok), dev(u), ws=ws)
        assert np.array_equal(acc.cpu().numpy(), acc_r) and np.array_equal(out.cpu().numpy(), out_r)
        assert ws.status() == st_r


def test_streaming_form_many_units_per_cta():
    """Two chunks per request (the second 8 entries long) and 20000 units:
    more than 128 units per SM, so the streaming form launches more CTAs
    than SMs, each owning up to 128 units of as many requests."""
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(4104, 10000, 1, sigma=0.5, seed=9)
    _check(ml, p, q, tok, u)


def test_mixed_rejections_full_vocabulary():
    """A 128256-entry vocabulary with about half the requests rejected: the
    streaming form's CTAs mix bonus and residual rows, and the speculative
    bonus chunks of rejected requests are dropped."""
    ml = needs_gpu()
    p, q, tok, u = WL.accept_inputs(128256, 80, 2, sigma=0.5, seed=10)
    u[::2, 1] = np.float32(0.999999)
    acc = _check(ml, p, q, tok, u)
    assert (acc < 2).sum() >= 30
