"""Test helpers: host <-> device marshalling and the GEMM acceptance bound.

GEMM acceptance (element by element against the oracle fed the same fp8 codes):
    ||gpu - ref||_F / ||ref||_F <= 5e-3   and   |gpu - ref| <= 1e-2 * |ref| + 1e-3 * rms(ref).
The bf16 store alone costs at most 2^-9 |ref| (about 1.95e-3 |ref|), inside the bound; the rest
is fp32 accumulation order against the oracle's fp64.
"""
import numpy as np
import torch

REL_FRO = 5e-3
REL_ELT = 1e-2
ABS_RMS = 1e-3


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_dev_fp16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.float16)


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def gemm_check(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    """Assert the acceptance bound; returns (rel Frobenius, worst element ratio)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), what + ": non-finite output"
    diff = gpu - ref
    den = float(np.sqrt(np.sum(ref * ref)))
    rel = float(np.sqrt(np.sum(diff * diff))) / max(den, 1e-300)
    rms = den / np.sqrt(max(ref.size, 1))
    bound = REL_ELT * np.abs(ref) + ABS_RMS * rms
    worst = float(np.max(np.abs(diff) / np.maximum(bound, 1e-300))) if ref.size else 0.0
    assert rel <= REL_FRO, f"{what}: rel Frobenius {rel:.3e} > {REL_FRO}"
    assert worst <= 1.0, f"{what}: element bound exceeded (worst ratio {worst:.3f})"
    return rel, worst
