"""Helpers shared by the GPU tests: move generator output (numpy bf16 bit
patterns, fp32, int32) onto the device as torch tensors.  Plumbing only."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def needs_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_lora_decoding_gb300 as ml
    if not ml.device_supported():
        pytest.fail("device is not compute capability 10.3; the library targets sm_103a only")
    return ml
