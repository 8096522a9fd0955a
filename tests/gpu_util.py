"""Helpers shared by the GPU tests: device copies of BF16 bit patterns and the
GEMM tolerance (elementwise |y - y_ref| <= 1e-2 (|y_ref| + 1e-2 rms(y_ref)),
relative Frobenius error <= 2e-3, against the fp64 oracle over the original
BF16 weights; where rounding the exact result to BF16 already costs more than
2e-3, as on some small outputs, that rounding error (+5 %) is the bound)."""
import numpy as np
import torch

from lossless_bit_weight_encode_gb300 import build as libbuild

ELEM_TOL = 1e-2
RMS_FLOOR = 1e-2
FRO_TOL = 2e-3


def ensure_built():
    libbuild.build()


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_tolerance(y_bits: np.ndarray, ref: np.ndarray, what: str = "") -> tuple[float, float]:
    y = bits_to_f64(y_bits)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(y - ref)
    bound = ELEM_TOL * (np.abs(ref) + RMS_FLOOR * rms)
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} elements outside tolerance; worst at "
        f"{np.unravel_index(int(np.argmax(err - bound)), err.shape)}")
    fro = float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))
    # BF16 output alone can cost more than 2e-3 on small outputs (its relative
    # rounding error reaches 2^-8): the bound is then the error of the
    # correctly rounded reference itself, which no BF16 result can beat
    ref_bf16 = (np.ascontiguousarray(ref, dtype=np.float32).view(np.uint32) + 0x7FFF
                + ((np.ascontiguousarray(ref, dtype=np.float32).view(np.uint32) >> 16) & 1)) >> 16 << 16
    floor = float(np.linalg.norm(ref_bf16.view(np.float32).astype(np.float64) - ref) /
                  max(np.linalg.norm(ref), 1e-300))
    assert fro <= max(FRO_TOL, 1.05 * floor), f"{what}: relative Frobenius error {fro:.3e} (rounding floor {floor:.3e})"
    return float((err / np.maximum(bound, 1e-300)).max()), fro
