"""Helpers shared by the GPU parity tests: moving seeded inputs to the device and the tolerance check.

Attention tolerance (BF16 output against the FP64 oracle over the same dequantized values), per
output vector o = out[row, head, :]:
    max_d |o - ref| <= 1e-2 * max(1, max_d mag)      ("1e-2 max-abs", in units of the vector's scale)
where mag = sum_j p_j |v_j| / sum_j p_j is the attention-weighted magnitude of the summed terms (the
oracle computes it; mag >= |ref|), and over the whole output ||o - ref||_2 <= 1e-2 ||ref||_2.
A bare absolute 1e-2 cannot hold once |ref| >= ~2: rounding the output to BF16 already costs up to
2^-9 |ref|, the workloads with x1e3 rows reach |ref| ~ 1e5, and an element that cancels to a small value
still carries the rounding of its large terms (FP32 logits of size ~1e4, 8-11 bit probabilities) --
hence the scale of the terms, not of the result.
"""
from __future__ import annotations

import numpy as np
import torch

ATOL = 1e-2
REL_L2 = 1e-2


def bits_to_cuda_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def cuda_bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def check_attention(out: torch.Tensor, ref: np.ndarray, what: str = "", mag: np.ndarray = None) -> dict:
    o = bf16_to_f64(out) if isinstance(out, torch.Tensor) else out
    assert o.shape == ref.shape, (o.shape, ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref)
    m = np.abs(ref) if mag is None else np.maximum(np.abs(ref), mag)
    scale = np.maximum(1.0, m.max(axis=-1, keepdims=True)) if ref.size else ref
    bound = ATOL * scale
    bad = err > bound
    rel_l2 = float(np.linalg.norm(o - ref) / max(np.linalg.norm(ref), 1e-300))
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "max_abs_over_max_ref": float(err.max() / max(np.abs(ref).max(), 1e-300)) if err.size else 0.0,
             "rel_l2": rel_l2}
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance; worst at " \
                          f"{np.unravel_index(np.argmax(err - bound), err.shape)} stats={stats}"
    assert rel_l2 <= REL_L2, f"{what}: relative L2 {rel_l2} > {REL_L2}"
    return stats


def pool_to_host(pool):
    """GPU KVPool -> numpy arrays (codes, scales) for bit comparisons."""
    return (pool.k_codes.cpu().numpy(), pool.v_codes.cpu().numpy(), pool.k_scales.cpu().numpy(),
            pool.v_scales.cpu().numpy())
