"""Helpers shared by the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

# Tolerances stated for the layer: BF16 outputs max-abs <= 2e-2 and
# relative L2 <= 5e-3; NVFP4 relative L2 <= 1e-2.
MAX_ABS = 2e-2
REL_L2 = 5e-3
REL_L2_NVFP4 = 1e-2


def bf16_vals(bits):
    a = np.ascontiguousarray(bits).view(np.int16)
    return torch.from_numpy(a.copy()).view(torch.bfloat16).to(torch.float64).numpy()


def dev_bf16_vals(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(gpu_bf16: torch.Tensor, oracle_bits: np.ndarray, rel_l2=REL_L2, max_abs=MAX_ABS, what=""):
    g = dev_bf16_vals(gpu_bf16).reshape(-1)
    o = bf16_vals(oracle_bits).reshape(-1)
    assert g.shape == o.shape, what
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    diff = np.abs(g - o)
    rel = np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30)
    assert diff.max() <= max_abs and rel <= rel_l2, f"{what}: max_abs={diff.max():.3e} rel_l2={rel:.3e}"
    return diff.max(), rel


def to_np_bits(t: torch.Tensor):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
