"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

# Attention outputs and lse: max abs error against the fp64 oracle (bf16 K/V,
# fp32 q, fp32 accumulate and output, values ~ N(0, 1)).
ATTN_ATOL = 2e-3


def dev(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to("cuda")


def max_abs_err(gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu.detach().double().cpu().numpy()
    if g.shape != ref.shape:
        raise AssertionError(f"shape {g.shape} != {ref.shape}")
    both_inf = np.isneginf(g) & np.isneginf(ref)
    diff = np.abs(np.where(both_inf, 0.0, g) - np.where(both_inf, 0.0, ref))
    return float("nan") if np.isnan(diff).any() else float(diff.max(initial=0.0))


def assert_attn_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "", atol: float = ATTN_ATOL):
    err = max_abs_err(gpu, ref)
    assert err <= atol, f"{what}: max abs error {err:.3e} > {atol:.1e}"
    return err


def bits(t: torch.Tensor) -> torch.Tensor:
    """Integer view of a tensor's bit patterns (bit-exact comparisons, NaN-safe)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def assert_bits_equal(a: torch.Tensor, b: torch.Tensor, what: str = ""):
    ba, bb = bits(a), bits(b)
    if not torch.equal(ba, bb):
        n = int((ba != bb).sum())
        raise AssertionError(f"{what}: {n} elements differ bit-wise")
