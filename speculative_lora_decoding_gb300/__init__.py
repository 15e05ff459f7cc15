"""Multi-LoRA decode hot path for GB300 (sm_103a): Python binding.

A thin ctypes binding of the C ABI declared in ``include/mlora.h``.  It only
marshals torch tensors into pointers and sizes and passes the current CUDA
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU or PyTorch fallback: if ``libmlora.so`` is missing or the
device is not compute capability 10.3, the calls raise.

    linear(x, W, A_stack, B_stack, rank_of, adapter_idx, scale, mode)   steps a1-a4
    linear_sliced(x, W, slice_end, A_stack, B_stack, ...)               the same, projections sharing x
    verify_accept(p, q, draft_tok, uniforms)                             steps a5-a6
    verify_accept_logits(z_p, z_q, draft_tok, uniforms)                  the same on logits (softmax fused)
    softmax(z), draft_sample(z_q, uniforms)                              logits -> probabilities; draft draw
    kv_write(y, ...), kv_commit(accepted, seq_len)                       hybrid KV cache (paged)
    quantize_rows_fp8(W), linear_fp8(x, W8, w_scale)                     draft pass on E4M3 weights
    plan_segments(...), shrink(...)                                      steps a1, a2 alone

The layer is y = W x (draft, LoRA off) or y = W x + scale * B_a (A_a x)
(verify, LoRA on), per token row ("Multi-LoRA Serving in Practice", section
"Core Principle: Shared Base Model, Per-Request Adapter Selection"; the modes
are the InvisibleLoRA abstract's LoRA-off draft and LoRA-on verify passes).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

DRAFT = 0
VERIFY = 1
PREFETCH_WEIGHTS = 0x100  # mode flag: W is constant; may be streamed before the preceding kernel ends
SHRINK_AUTO, SHRINK_WARP, SHRINK_TENSOR = 0, 1, 2  # which kernel writes the verify pass's low-rank operand

# Limits of mlora_linear_noalloc (its scratch is a fixed array in the library).
NOALLOC_MAX_ROWS = 1024
NOALLOC_MAX_ADAPTERS = 256

DEV_BAD_ADAPTER = 1 << 0
DEV_BAD_RANK = 1 << 1
DEV_BAD_PROB = 1 << 2
DEV_BAD_TOKEN = 1 << 3
DEV_ZERO_MASS = 1 << 4
DEV_TIMEOUT = 1 << 5
DEV_BAD_PLAN = 1 << 6
DEV_BAD_SLOT = 1 << 7

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmlora.so")
HEADER_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mlora.h")

_c_size = ctypes.c_size_t
_c_int = ctypes.c_int
_c_ptr = ctypes.c_void_p
_c_float = ctypes.c_float

_SIGNATURES = {
    "mlora_linear_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "mlora_linear_sliced_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "mlora_accept_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "mlora_workspace_init": (_c_int, [_c_ptr, _c_size, _c_ptr]),
    "mlora_read_device_status": (_c_int, [_c_ptr, ctypes.POINTER(ctypes.c_uint32), _c_int, _c_ptr]),
    "mlora_plan_segments": (_c_int, [_c_ptr, _c_int, _c_ptr, _c_int, _c_int, _c_ptr, _c_size,
                                     ctypes.POINTER(_c_ptr), ctypes.POINTER(_c_ptr), _c_ptr]),
    "mlora_shrink": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_size,
                              _c_ptr]),
    "mlora_linear": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int, _c_ptr,
                              _c_ptr, _c_ptr, _c_float, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "mlora_linear_sliced": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_int, _c_int, ctypes.POINTER(ctypes.c_int32),
                                     _c_ptr, _c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_float, _c_int, _c_ptr,
                                     _c_ptr, _c_size, _c_ptr]),
    "mlora_verify_accept": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_ptr, _c_ptr,
                                     _c_ptr, _c_size, _c_ptr]),
    "mlora_linear_noalloc": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int,
                                      _c_ptr, _c_ptr, _c_float, _c_int, _c_ptr, _c_ptr]),
    "mlora_linear_gemm_kernel": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "mlora_debug_set_flag_wait_ns": (None, [ctypes.c_uint32]),
    "mlora_debug_q40_mismatches": (_c_int, [ctypes.c_uint32, ctypes.c_uint32, _c_ptr, _c_ptr]),
    "mlora_debug_exp_max_rel_error": (_c_int, [ctypes.c_uint32, ctypes.c_uint32, _c_ptr, _c_ptr]),
    "mlora_set_shrink_path": (_c_int, [_c_int]),
    "mlora_verify_accept_logits": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_ptr, _c_ptr,
                                            _c_ptr, _c_size, _c_ptr]),
    "mlora_softmax_workspace_bytes": (_c_size, [_c_int, _c_int]),
    "mlora_softmax": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "mlora_draft_sample_workspace_bytes": (_c_size, [_c_int, _c_int]),
    "mlora_draft_sample": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "mlora_expected_tokens": (ctypes.c_double, [ctypes.c_double, _c_int]),
    "mlora_draft_gate": (_c_int, [ctypes.POINTER(ctypes.c_double), _c_int, ctypes.c_double, ctypes.c_double,
                                  ctypes.POINTER(ctypes.c_double)]),
    "mlora_estimate_acceptance": (ctypes.c_double, [ctypes.POINTER(ctypes.c_int32), _c_int, _c_int]),
    "mlora_quantize_rows_fp8": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr]),
    "mlora_linear_fp8_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "mlora_linear_fp8": (_c_int, [_c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int, _c_ptr, _c_size,
                                  _c_ptr]),
    "mlora_kv_workspace_bytes": (_c_size, []),
    "mlora_kv_write": (_c_int, [_c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_int, _c_int,
                                _c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_int, _c_int, _c_ptr, _c_size, _c_ptr]),
    "mlora_kv_commit": (_c_int, [_c_ptr, _c_int, _c_ptr, _c_ptr]),
    "mlora_status_string": (ctypes.c_char_p, [_c_int]),
    "mlora_device_supported": (_c_int, []),
    "mlora_launch_count": (ctypes.c_uint64, []),
}

_lib = None


class MLoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _load().mlora_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


def header_symbols(path: str = HEADER_PATH) -> list:
    """Names of the entry points include/mlora.h declares."""
    text = open(path).read()
    return re.findall(r"MLORA_API\s+[\w\s\*]*?\b(mlora_\w+)\s*\(", text)


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() (needs nvcc, targets sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def _check(status: int, where: str):
    if status != 0:
        raise MLoraError(status, where)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, dim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions")
    return t.data_ptr()


def device_supported() -> bool:
    return bool(_load().mlora_device_supported())


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(_load().mlora_launch_count())


def gemm_kernel_name(M: int, N: int, K: int, n_adapters: int, r_max: int, mode: int) -> str:
    """The GEMM kernel a layer call of this shape runs: "gemm_kernel" (cluster
    split-K) or "gemm_sk_kernel" (persistent stream-K)."""
    k = int(_load().mlora_linear_gemm_kernel(M, N, K, n_adapters, r_max, int(mode)))
    if k < 0:
        raise ValueError("sizes or mode outside the supported ranges")
    return ("gemm_kernel", "gemm_sk_kernel")[k]


def set_shrink_path(path: int) -> None:
    """Which kernel writes the verify pass's low-rank operand in later layer
    calls: SHRINK_AUTO (the library's choice), SHRINK_WARP or SHRINK_TENSOR."""
    _check(_load().mlora_set_shrink_path(int(path)), "mlora_set_shrink_path")


def linear_workspace_bytes(M: int, N: int, K: int, n_adapters: int) -> int:
    return int(_load().mlora_linear_workspace_bytes(M, N, K, n_adapters))


def linear_sliced_workspace_bytes(M: int, N: int, K: int, n_adapters: int, n_slices: int) -> int:
    return int(_load().mlora_linear_sliced_workspace_bytes(M, N, K, n_adapters, n_slices))


def accept_workspace_bytes(B: int, k: int, V: int) -> int:
    return int(_load().mlora_accept_workspace_bytes(B, k, V))


class Workspace:
    """A device buffer for the library's scratch, status word and counters."""

    def __init__(self, nbytes: int, device=None, stream=None):
        if nbytes <= 0:
            raise ValueError("workspace size must be positive (sizes outside the supported range give 0)")
        self.nbytes = int(nbytes)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _check(_load().mlora_workspace_init(self.buf.data_ptr(), self.nbytes, _stream(stream)), "workspace_init")
        # The zeroing is asynchronous on `stream`; calls may come on any stream.
        (torch.cuda.current_stream(self.buf.device) if stream is None else stream).synchronize()

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self, clear: bool = True, stream=None) -> int:
        """Device status bits (synchronises the stream)."""
        bits = ctypes.c_uint32(0)
        st = _load().mlora_read_device_status(self.ptr, ctypes.byref(bits), 1 if clear else 0, _stream(stream))
        if st not in (0, 5, 6):
            raise MLoraError(st, "read_device_status")
        return int(bits.value)

    def view_int32(self, ptr: int, count: int) -> torch.Tensor:
        """int32 view of `count` words of this workspace starting at device pointer `ptr`."""
        off = int(ptr) - self.ptr
        if off < 0 or off + 4 * count > self.nbytes or off % 4:
            raise ValueError("pointer is not inside this workspace")
        return self.buf[off:off + 4 * count].view(torch.int32)


def plan_segments(adapter_idx: torch.Tensor, rank_of: torch.Tensor, n_adapters: int, r_max: int, ws: Workspace,
                  stream=None):
    """Step a1.  Returns (seg_offsets_ptr, perm_ptr): device pointers into `ws`."""
    M = adapter_idx.numel()
    seg = _c_ptr(0)
    perm = _c_ptr(0)
    st = _load().mlora_plan_segments(_need(adapter_idx, "adapter_idx", torch.int32, 1), M,
                                     _need(rank_of, "rank_of", torch.int32, 1), n_adapters, r_max, ws.ptr, ws.nbytes,
                                     ctypes.byref(seg), ctypes.byref(perm), _stream(stream))
    _check(st, "plan_segments")
    return seg.value, perm.value


def shrink(x: torch.Tensor, A_stack: torch.Tensor, seg_offsets_ptr: int, ws: Workspace, T: torch.Tensor = None,
           stream=None) -> torch.Tensor:
    """Step a2: T[m, j] = A_a[j, :] . x[m, :] for j < rank, fp32 [M, r_max]."""
    M, K = x.shape
    n_ad, r_max, K2 = A_stack.shape
    if K2 != K:
        raise ValueError("A_stack and x disagree on K")
    if T is None:
        T = torch.empty((M, r_max), dtype=torch.float32, device=x.device)
    st = _load().mlora_shrink(_need(x, "x", torch.bfloat16, 2), M, K, _need(A_stack, "A_stack", torch.bfloat16, 3),
                              n_ad, r_max, seg_offsets_ptr, _need(T, "T", torch.float32, 2), ws.ptr, ws.nbytes,
                              _stream(stream))
    _check(st, "shrink")
    return T


def linear(x: torch.Tensor, W: torch.Tensor, A_stack, B_stack, rank_of, adapter_idx, scale: float, mode: int,
           ws: Workspace = None, y: torch.Tensor = None, seg_offsets_ptr: int = None, stream=None) -> torch.Tensor:
    """Steps a1-a4: y = W x (+ scale * B_a (A_a x) in verify mode), bf16 [M, N]."""
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("W and x disagree on K")
    verify = (mode & ~PREFETCH_WEIGHTS) == VERIFY
    n_ad, r_max = 0, 0
    a_ptr = b_ptr = r_ptr = i_ptr = None
    if verify:
        n_ad, r_max, K3 = A_stack.shape
        if K3 != K or tuple(B_stack.shape) != (n_ad, N, r_max):
            raise ValueError("A_stack [n_ad, r_max, K] / B_stack [n_ad, N, r_max] shapes disagree")
        a_ptr = _need(A_stack, "A_stack", torch.bfloat16, 3)
        b_ptr = _need(B_stack, "B_stack", torch.bfloat16, 3)
        r_ptr = _need(rank_of, "rank_of", torch.int32, 1)
        i_ptr = _need(adapter_idx, "adapter_idx", torch.int32, 1)
        if adapter_idx.numel() != M or rank_of.numel() != n_ad:
            raise ValueError("adapter_idx must have M entries and rank_of n_adapters entries")
    if ws is None:
        ws = Workspace(linear_workspace_bytes(M, N, K, max(n_ad, 1)), device=x.device, stream=stream)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = _load().mlora_linear(_need(x, "x", torch.bfloat16, 2), M, K, _need(W, "W", torch.bfloat16, 2), N, a_ptr,
                              b_ptr, n_ad, r_max, r_ptr, i_ptr, seg_offsets_ptr, float(scale), int(mode),
                              _need(y, "y", torch.bfloat16, 2), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "linear")
    return y


def linear_sliced(x: torch.Tensor, W: torch.Tensor, slice_end, A_stack, B_stack, rank_of, adapter_idx,
                  scale: float, mode: int, ws: Workspace = None, y: torch.Tensor = None, seg_offsets_ptr: int = None,
                  stream=None) -> torch.Tensor:
    """mlora_linear_sliced: projections that read the same rows x in one call.

    W [N, K] stacks the projections along N; `slice_end` (host ints) gives
    each slice's end row; A_stack is [n_slices, n_ad, r_max, K] and B_stack
    [n_ad, N, r_max].  Returns y [M, N] (bf16)."""
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("W and x disagree on K")
    ends = [int(e) for e in slice_end]
    S = len(ends)
    verify = (mode & ~PREFETCH_WEIGHTS) == VERIFY
    n_ad, r_max = 0, 0
    a_ptr = b_ptr = r_ptr = i_ptr = None
    if verify:
        S2, n_ad, r_max, K3 = A_stack.shape
        if S2 != S or K3 != K or tuple(B_stack.shape) != (n_ad, N, r_max):
            raise ValueError("A_stack [S, n_ad, r_max, K] / B_stack [n_ad, N, r_max] shapes disagree")
        a_ptr = _need(A_stack, "A_stack", torch.bfloat16, 4)
        b_ptr = _need(B_stack, "B_stack", torch.bfloat16, 3)
        r_ptr = _need(rank_of, "rank_of", torch.int32, 1)
        i_ptr = _need(adapter_idx, "adapter_idx", torch.int32, 1)
        if adapter_idx.numel() != M or rank_of.numel() != n_ad:
            raise ValueError("adapter_idx must have M entries and rank_of n_adapters entries")
    if ws is None:
        ws = Workspace(linear_sliced_workspace_bytes(M, N, K, max(n_ad, 1), S), device=x.device, stream=stream)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ends_c = (ctypes.c_int32 * max(S, 1))(*ends)
    st = _load().mlora_linear_sliced(_need(x, "x", torch.bfloat16, 2), M, K, _need(W, "W", torch.bfloat16, 2), N, S,
                                     ends_c, a_ptr, b_ptr, n_ad, r_max, r_ptr, i_ptr, seg_offsets_ptr, float(scale),
                                     int(mode), _need(y, "y", torch.bfloat16, 2), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "linear_sliced")
    return y


def verify_accept(p: torch.Tensor, q: torch.Tensor, draft_tok: torch.Tensor, uniforms: torch.Tensor,
                  ws: Workspace = None, out_tok: torch.Tensor = None, accepted: torch.Tensor = None, stream=None):
    """Steps a5-a6.  Returns (out_tok int32 [B, k+1], accepted int32 [B])."""
    B, k1, V = p.shape
    k = k1 - 1
    if tuple(q.shape) != (B, k, V) or tuple(draft_tok.shape) != (B, k) or tuple(uniforms.shape) != (B, k1):
        raise ValueError("p [B,k+1,V], q [B,k,V], draft_tok [B,k], uniforms [B,k+1] shapes disagree")
    if ws is None:
        ws = Workspace(accept_workspace_bytes(B, k, V), device=p.device, stream=stream)
    if out_tok is None:
        out_tok = torch.empty((B, k1), dtype=torch.int32, device=p.device)
    if accepted is None:
        accepted = torch.empty((B,), dtype=torch.int32, device=p.device)
    st = _load().mlora_verify_accept(_need(p, "p", torch.float32, 3), _need(q, "q", torch.float32, 3),
                                     _need(draft_tok, "draft_tok", torch.int32, 2),
                                     _need(uniforms, "uniforms", torch.float32, 2), B, k, V,
                                     _need(out_tok, "out_tok", torch.int32, 2),
                                     _need(accepted, "accepted", torch.int32, 1), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "verify_accept")
    return out_tok, accepted


def verify_accept_logits(z_target: torch.Tensor, z_draft: torch.Tensor, draft_tok: torch.Tensor,
                         uniforms: torch.Tensor, ws: Workspace = None, out_tok: torch.Tensor = None,
                         accepted: torch.Tensor = None, stream=None):
    """Steps a5-a6 on logits (softmax fused).  Returns (out_tok, accepted)."""
    B, k1, V = z_target.shape
    k = k1 - 1
    if tuple(z_draft.shape) != (B, k, V) or tuple(draft_tok.shape) != (B, k) or tuple(uniforms.shape) != (B, k1):
        raise ValueError("z_target [B,k+1,V], z_draft [B,k,V], draft_tok [B,k], uniforms [B,k+1] shapes disagree")
    if ws is None:
        ws = Workspace(accept_workspace_bytes(B, k, V), device=z_target.device, stream=stream)
    if out_tok is None:
        out_tok = torch.empty((B, k1), dtype=torch.int32, device=z_target.device)
    if accepted is None:
        accepted = torch.empty((B,), dtype=torch.int32, device=z_target.device)
    st = _load().mlora_verify_accept_logits(_need(z_target, "z_target", torch.float32, 3),
                                            _need(z_draft, "z_draft", torch.float32, 3),
                                            _need(draft_tok, "draft_tok", torch.int32, 2),
                                            _need(uniforms, "uniforms", torch.float32, 2), B, k, V,
                                            _need(out_tok, "out_tok", torch.int32, 2),
                                            _need(accepted, "accepted", torch.int32, 1), ws.ptr, ws.nbytes,
                                            _stream(stream))
    _check(st, "verify_accept_logits")
    return out_tok, accepted


def softmax(z: torch.Tensor, ws: Workspace = None, p: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Row softmax of fp32 logits [..., V] (the library's one definition of a probability)."""
    V = z.shape[-1]
    rows = z.numel() // V
    if ws is None:
        ws = Workspace(int(_load().mlora_softmax_workspace_bytes(rows, V)), device=z.device, stream=stream)
    if p is None:
        p = torch.empty_like(z)
    st = _load().mlora_softmax(_need(z, "z", torch.float32), rows, V, _need(p, "p", torch.float32), ws.ptr, ws.nbytes,
                               _stream(stream))
    _check(st, "softmax")
    return p


def draft_sample(z_draft: torch.Tensor, uniforms: torch.Tensor, ws: Workspace = None, tok: torch.Tensor = None,
                 q: torch.Tensor = None, want_q: bool = True, stream=None):
    """Draft tokens from LoRA-off logits [B, V]: returns (tok int32 [B], q fp32 [B, V] or None)."""
    B, V = z_draft.shape
    if tuple(uniforms.shape) != (B,):
        raise ValueError("uniforms must have B entries")
    if ws is None:
        ws = Workspace(int(_load().mlora_draft_sample_workspace_bytes(B, V)), device=z_draft.device, stream=stream)
    if tok is None:
        tok = torch.empty((B,), dtype=torch.int32, device=z_draft.device)
    if q is None and want_q:
        q = torch.empty_like(z_draft)
    st = _load().mlora_draft_sample(_need(z_draft, "z_draft", torch.float32, 2), B, V,
                                    _need(uniforms, "uniforms", torch.float32, 1), _need(tok, "tok", torch.int32, 1),
                                    _need(q, "q", torch.float32, 2) if q is not None else None, ws.ptr, ws.nbytes,
                                    _stream(stream))
    _check(st, "draft_sample")
    return tok, q


def quantize_rows_fp8(src: torch.Tensor, q: torch.Tensor = None, scale: torch.Tensor = None, stream=None):
    """E4M3 codes (uint8 [R, K]) and fp32 row scales [R] of bf16 rows [R, K]."""
    R, K = src.shape
    if q is None:
        q = torch.empty((R, K), dtype=torch.uint8, device=src.device)
    if scale is None:
        scale = torch.empty((R,), dtype=torch.float32, device=src.device)
    st = _load().mlora_quantize_rows_fp8(_need(src, "src", torch.bfloat16, 2), R, K, _need(q, "q", torch.uint8, 2),
                                         _need(scale, "scale", torch.float32, 1), _stream(stream))
    _check(st, "quantize_rows_fp8")
    return q, scale


def linear_fp8_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_load().mlora_linear_fp8_workspace_bytes(M, N, K))


def linear_fp8(x: torch.Tensor, W8: torch.Tensor, w_scale: torch.Tensor, flags: int = 0, ws: Workspace = None,
               y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Draft (LoRA-off) layer on E4M3 weights from quantize_rows_fp8: bf16 [M, N]."""
    M, K = x.shape
    N, K2 = W8.shape
    if K2 != K or w_scale.numel() != N:
        raise ValueError("W8 [N, K] / w_scale [N] disagree with x [M, K]")
    if ws is None:
        ws = Workspace(linear_fp8_workspace_bytes(M, N, K), device=x.device, stream=stream)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = _load().mlora_linear_fp8(_need(x, "x", torch.bfloat16, 2), M, K, _need(W8, "W8", torch.uint8, 2),
                                  _need(w_scale, "w_scale", torch.float32, 1), N, _need(y, "y", torch.bfloat16, 2),
                                  int(flags), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "linear_fp8")
    return y


def kv_workspace_bytes() -> int:
    return int(_load().mlora_kv_workspace_bytes())


def kv_write(y: torch.Tensor, k_col: int, v_col: int, H: int, D: int, block_table: torch.Tensor,
             seq_len: torch.Tensor, rows_per_req: int, t0: int, k_cache: torch.Tensor, v_cache: torch.Tensor,
             ws: Workspace = None, stream=None):
    """Hybrid KV cache: the K and V rows of one pass (y bf16 [M, ld], the fused
    q|k|v output) into the paged caches k_cache, v_cache bf16
    [num_blocks, block_size, H, D].  Row m is request m // rows_per_req at step
    m % rows_per_req and goes to position seq_len[b] + t0 + step."""
    M, ld = y.shape
    B, max_blocks = block_table.shape
    num_blocks, block_size = k_cache.shape[0], k_cache.shape[1]
    if tuple(k_cache.shape) != (num_blocks, block_size, H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must both be [num_blocks, block_size, H, D]")
    if seq_len.numel() != B:
        raise ValueError("seq_len must have one entry per block-table row")
    if ws is None:
        ws = Workspace(kv_workspace_bytes(), device=y.device, stream=stream)
    st = _load().mlora_kv_write(_need(y, "y", torch.bfloat16, 2), M, ld, int(k_col), int(v_col), int(H), int(D),
                                _need(block_table, "block_table", torch.int32, 2), B, max_blocks,
                                _need(seq_len, "seq_len", torch.int32, 1), int(rows_per_req), int(t0),
                                _need(k_cache, "k_cache", torch.bfloat16, 4), _need(v_cache, "v_cache", torch.bfloat16, 4),
                                num_blocks, block_size, ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "kv_write")
    return k_cache, v_cache


def kv_commit(accepted: torch.Tensor, seq_len: torch.Tensor, stream=None) -> torch.Tensor:
    """seq_len[b] += accepted[b] + 1 for every used request slot (in place)."""
    B = seq_len.numel()
    if accepted.numel() != B:
        raise ValueError("accepted and seq_len must have the same length")
    st = _load().mlora_kv_commit(_need(accepted, "accepted", torch.int32, 1), B, _need(seq_len, "seq_len", torch.int32, 1),
                                 _stream(stream))
    _check(st, "kv_commit")
    return seq_len


def draft_gate(t_cycle: dict, t_plain: float, alpha: float):
    """The run-time draft gate: t_cycle {k: measured cycle time} for k = 1..k_max,
    t_plain the plain LoRA-on step time, alpha the acceptance rate.  Returns
    (k, gain) with k = 0 meaning "skip drafting"."""
    k_max = max(t_cycle)
    arr = (ctypes.c_double * (k_max + 1))(*([0.0] + [float(t_cycle.get(k, 0.0)) for k in range(1, k_max + 1)]))
    gain = ctypes.c_double(0.0)
    k = int(_load().mlora_draft_gate(arr, k_max, float(t_plain), float(alpha), ctypes.byref(gain)))
    if k < 0:
        raise ValueError("draft gate: invalid times or acceptance rate (every k in 1..k_max needs a positive time)")
    return k, gain.value


def estimate_acceptance(accepted, k: int) -> float:
    """Maximum-likelihood acceptance rate from kept-draft counts (host ints)."""
    a = [int(v) for v in accepted]
    arr = (ctypes.c_int32 * max(len(a), 1))(*a)
    return float(_load().mlora_estimate_acceptance(arr, len(a), int(k)))


def linear_noalloc(x: torch.Tensor, W: torch.Tensor, A_stack, B_stack, rank_of, adapter_idx, scale: float, mode: int,
                   y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """mlora_linear_noalloc: the layer without a workspace, for callers that
    cannot allocate device memory (the library's own fixed scratch array is
    used instead; M <= NOALLOC_MAX_ROWS, n_adapters <= NOALLOC_MAX_ADAPTERS).
    The output buffer `y` is the caller's; pass it to avoid the allocation
    this wrapper would otherwise make for it."""
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("W and x disagree on K")
    verify = (mode & ~PREFETCH_WEIGHTS) == VERIFY
    n_ad, r_max = 0, 0
    a_ptr = b_ptr = r_ptr = i_ptr = None
    if verify:
        n_ad, r_max, K3 = A_stack.shape
        if K3 != K or tuple(B_stack.shape) != (n_ad, N, r_max):
            raise ValueError("A_stack [n_ad, r_max, K] / B_stack [n_ad, N, r_max] shapes disagree")
        a_ptr = _need(A_stack, "A_stack", torch.bfloat16, 3)
        b_ptr = _need(B_stack, "B_stack", torch.bfloat16, 3)
        r_ptr = _need(rank_of, "rank_of", torch.int32, 1)
        i_ptr = _need(adapter_idx, "adapter_idx", torch.int32, 1)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = _load().mlora_linear_noalloc(_need(x, "x", torch.bfloat16, 2), M, K, _need(W, "W", torch.bfloat16, 2), N,
                                      a_ptr, b_ptr, n_ad, r_max, r_ptr, i_ptr, float(scale), int(mode),
                                      _need(y, "y", torch.bfloat16, 2), _stream(stream))
    _check(st, "linear_noalloc")
    return y
