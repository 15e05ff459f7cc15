"""The C-ABI library loads and exports every entry point the header declares.
No compute call is made here (this runs without a GPU)."""
import ctypes
import os
import subprocess

import pytest

import speculative_lora_decoding_gb300 as ml


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ml.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return ml.library()


def test_header_declares_the_boundary():
    names = set(ml.header_symbols())
    for n in ("mlora_linear", "mlora_linear_sliced", "mlora_verify_accept", "mlora_plan_segments", "mlora_shrink",
              "mlora_linear_workspace_bytes", "mlora_accept_workspace_bytes", "mlora_workspace_init",
              "mlora_read_device_status", "mlora_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ml.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in ml.header_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_host_checks(lib):
    for s in range(8):
        assert lib.mlora_status_string(s)
    # null pointers are rejected before any CUDA call
    assert lib.mlora_linear(None, 4, 8, None, 8, None, None, 0, 0, None, None, None, 1.0, 0, None, None, 0, None) == 1
    assert lib.mlora_verify_accept(None, None, None, None, 1, 1, 4, None, None, None, 0, None) == 1
    # bad mode
    p = ctypes.c_void_p(16)
    assert lib.mlora_linear(p, 4, 8, p, 8, None, None, 0, 0, None, None, None, 1.0, 7, p, p, 1 << 20, None) == 1


def test_workspace_sizes(lib):
    a = lib.mlora_linear_workspace_bytes(128, 4096, 4096, 16)
    b = lib.mlora_linear_workspace_bytes(256, 4096, 4096, 16)
    c = lib.mlora_linear_workspace_bytes(512, 14336, 4096, 128)
    assert 0 < a < b and c > 0
    # one workspace sized for the largest K serves every projection of a step: the verify pass keeps the
    # token rows in adapter-sorted order (M x K bf16), so the size grows with K and not with N
    assert lib.mlora_linear_workspace_bytes(128, 1024, 4096, 16) == a
    assert lib.mlora_linear_workspace_bytes(128, 4096, 14336, 16) >= a + 128 * (14336 - 4096) * 2
    assert lib.mlora_linear_workspace_bytes(128, 4096, 4097, 16) == 0      # K % 8 != 0
    assert lib.mlora_linear_workspace_bytes(0, 4096, 4096, 16) == 0
    assert lib.mlora_accept_workspace_bytes(256, 4, 128256) > 0
    assert lib.mlora_accept_workspace_bytes(256, 0, 128256) == 0


def test_sliced_host_checks(lib):
    """Slice ends are checked on the host, before any CUDA call."""
    p = ctypes.c_void_p(256)
    SHAPE = 2

    def call(ends, N=640, mode=0):
        arr = (ctypes.c_int32 * max(len(ends), 1))(*ends)
        return lib.mlora_linear_sliced(p, 4, 8, p, N, len(ends), arr, None, None, 0, 0, None, None, None, 1.0, mode,
                                       p, p, 1 << 24, None)

    assert call([100, 640]) == SHAPE                 # an inner end that is not a multiple of 128
    assert call([256, 256, 640]) == SHAPE            # not increasing
    assert call([256, 512]) == SHAPE                 # last end != N
    assert call([128, 256, 384, 512, 640]) == SHAPE  # more than MLORA_MAX_SLICES
    assert call([]) == SHAPE
    assert lib.mlora_linear_sliced_workspace_bytes(128, 6144, 4096, 16, 3) > \
        lib.mlora_linear_sliced_workspace_bytes(128, 6144, 4096, 16, 1) == lib.mlora_linear_workspace_bytes(128, 6144, 4096, 16)
    assert lib.mlora_linear_sliced_workspace_bytes(128, 6144, 4096, 16, 5) == 0


def test_kv_host_checks(lib):
    """Sizes and pointers of the KV-cache calls are checked on the host, before any CUDA call."""
    p = ctypes.c_void_p(256)
    SHAPE, ARG, WS = 2, 1, 3
    big = 1 << 20

    def call(y=p, M=4, ld=48, k_col=16, v_col=32, H=2, D=8, B=2, max_blocks=4, rpr=2, t0=0, nb=8, bs=16, ws=p,
             wsb=big):
        return lib.mlora_kv_write(y, M, ld, k_col, v_col, H, D, p, B, max_blocks, p, rpr, t0, p, p, nb, bs, ws, wsb,
                                  None)

    assert call(M=5) == SHAPE                  # more rows than B * rows_per_req
    assert call(v_col=33) == SHAPE             # V columns past ld
    assert call(k_col=-1) == SHAPE
    assert call(H=0) == SHAPE
    assert call(t0=-1) == SHAPE
    assert call(bs=0) == SHAPE
    assert call(y=None) == ARG
    assert call(ws=None) == WS
    assert call(wsb=16) == WS
    assert lib.mlora_kv_workspace_bytes() > 0
    assert lib.mlora_kv_commit(None, 4, None, None) == ARG
    assert lib.mlora_kv_commit(p, 0, p, None) == SHAPE


def test_fp8_host_checks(lib):
    p = ctypes.c_void_p(256)
    SHAPE, ARG, WS = 2, 1, 3
    assert lib.mlora_linear_fp8_workspace_bytes(128, 5120, 5120) > 0
    assert lib.mlora_linear_fp8_workspace_bytes(257, 5120, 5120) == 0   # the stream-K kernel's 256 rows
    assert lib.mlora_linear_fp8_workspace_bytes(128, 5120, 5128) == 0   # K % 16 != 0
    assert lib.mlora_linear_fp8(p, 128, 5128, p, p, 64, p, 0, p, 1 << 30, None) == SHAPE
    assert lib.mlora_linear_fp8(None, 128, 512, p, p, 64, p, 0, p, 1 << 30, None) == ARG
    assert lib.mlora_linear_fp8(p, 128, 512, p, p, 64, p, 7, p, 1 << 30, None) == ARG   # unknown flag
    assert lib.mlora_linear_fp8(p, 128, 512, p, p, 64, p, 0, None, 0, None) == WS
    assert lib.mlora_quantize_rows_fp8(p, 4, 24, p, p, None) == SHAPE
    assert lib.mlora_quantize_rows_fp8(None, 4, 32, p, p, None) == ARG


def test_q40_hook_host_checks(lib):
    """The Q(f) check hook refuses a null counter and a range past 2^32
    before any CUDA call; an empty range does nothing."""
    dummy = ctypes.c_void_p(16)  # never dereferenced: these calls return before any launch
    assert lib.mlora_debug_q40_mismatches(0, 1, None, None) == 1                 # MLORA_ERR_ARG
    assert lib.mlora_debug_q40_mismatches(2, 0xFFFFFFFF, dummy, None) == 1       # past 2^32
    assert lib.mlora_debug_q40_mismatches(0xFFFFFFFF, 2, dummy, None) == 1
    assert lib.mlora_debug_q40_mismatches(5, 0, dummy, None) == 0                # MLORA_OK, nothing launched


def test_exp_hook_host_checks(lib):
    """The e^d check hook refuses a null result pointer and a range past 2^32
    before any CUDA call; an empty range does nothing."""
    dummy = ctypes.c_void_p(16)  # never dereferenced: these calls return before any launch
    assert lib.mlora_debug_exp_max_rel_error(0, 1, None, None) == 1              # MLORA_ERR_ARG
    assert lib.mlora_debug_exp_max_rel_error(2, 0xFFFFFFFF, dummy, None) == 1    # past 2^32
    assert lib.mlora_debug_exp_max_rel_error(7, 0, dummy, None) == 0             # MLORA_OK, nothing launched
