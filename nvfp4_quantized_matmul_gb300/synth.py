"""Seeded synthetic inputs for the NVFP4 planes, activations and routing.

This module holds only random draws and storage conversions; none of the
NVFP4 arithmetic (decode, scaling, matmul) lives here, so the CUDA path and
the CPU oracle can both consume its output without sharing any of the method.

Value recipes (all drawn from ``numpy.random.Generator(PCG64(seed))``):

* packed E2M1 weight planes: uniform random 32-bit words, i.e. eight uniform
  4-bit codes per word (both signed zeros included);
* E4M3 block scales: magnitudes ``2**U(log2 lo, log2 hi)`` rounded to E4M3 by
  ``torch.float8_e4m3fn`` (round-to-nearest-even), stored as raw bytes;
* global scales: ``U(0.5, 2) * 448 * 6`` as float32;
* activations: ``N(0, 1)`` rounded to the activation dtype;
* ModelOpt triplets: uniform bytes (two codes per byte), E4M3 scales and a
  float32 ``weight_scale_2`` drawn from ``U(1e-4, 1e-2)``;
* MoE routing: top-k distinct experts per token drawn with probability
  proportional to ``(e + 1) ** -a`` (Zipf-like), rows stably sorted by expert.
"""
from __future__ import annotations

import numpy as np
import torch

_TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def packed_weight(g: np.random.Generator, *shape_nk: int) -> np.ndarray:
    """Uniform E2M1 codes packed eight per uint32: shape ``[..., N, K/8]``."""
    *lead, k = shape_nk
    assert k % 8 == 0
    return g.integers(0, 2**32, size=(*lead, k // 8), dtype=np.uint64).astype(np.uint32)


def e4m3_bytes(values: np.ndarray) -> np.ndarray:
    """Round float values to E4M3 bytes with torch's float8_e4m3fn cast."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def log_uniform_scales(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    """E4M3 scale bytes with log-uniform magnitudes in ``[lo, hi]``."""
    mag = np.exp2(g.uniform(np.log2(lo), np.log2(hi), size=shape))
    return e4m3_bytes(mag)


def global_scales(g: np.random.Generator, n: int) -> np.ndarray:
    """``n`` float32 global scales in ``[0.5, 2] * 448 * 6``."""
    return (g.uniform(0.5, 2.0, size=n) * 2688.0).astype(np.float32)


def activations(g: np.random.Generator, shape, dtype: str) -> torch.Tensor:
    """Standard-normal activations rounded to ``dtype`` (a CPU tensor)."""
    x = torch.from_numpy(g.standard_normal(size=shape).astype(np.float32))
    return x.to(_TORCH_DTYPES[dtype])


def modelopt_triplet(g: np.random.Generator, n: int, k: int,
                     scale_lo: float = 2.0**-6, scale_hi: float = 4.0):
    """A ModelOpt NVFP4 triplet: (weight u8 [N,K/2], weight_scale u8 [N,K/16], ws2 f32)."""
    assert k % 16 == 0
    weight = g.integers(0, 256, size=(n, k // 2), dtype=np.uint16).astype(np.uint8)
    weight_scale = log_uniform_scales(g, (n, k // 16), scale_lo, scale_hi)
    ws2 = np.float32(g.uniform(1e-4, 1e-2))
    return weight, weight_scale, ws2


def zipf_routing(g: np.random.Generator, tokens: int, experts: int, top_k: int,
                 a: float = 1.1, sort: bool = True):
    """Top-k distinct experts per token with p(e) proportional to (e+1)^-a.

    Returns ``(lhs, rhs)`` uint32 arrays of length ``tokens * top_k``: ``lhs``
    is the token (activation row) and ``rhs`` the expert. With ``sort`` the
    rows are stably sorted by expert, as a sorted MoE prefill sees them.
    """
    p = (np.arange(experts, dtype=np.float64) + 1.0) ** -a
    p /= p.sum()
    rhs = np.empty((tokens, top_k), dtype=np.int64)
    for t in range(tokens):
        rhs[t] = g.choice(experts, size=top_k, replace=False, p=p)
    lhs = np.repeat(np.arange(tokens, dtype=np.int64), top_k)
    rhs = rhs.reshape(-1)
    if sort:
        order = np.argsort(rhs, kind="stable")
        lhs, rhs = lhs[order], rhs[order]
    return lhs.astype(np.uint32), rhs.astype(np.uint32)


def zipf_experts(g: np.random.Generator, rows: int, experts: int, a: float = 1.1) -> np.ndarray:
    """One expert per row (unsorted decode routing), p(e) proportional to (e+1)^-a."""
    p = (np.arange(experts, dtype=np.float64) + 1.0) ** -a
    p /= p.sum()
    return g.choice(experts, size=rows, p=p).astype(np.uint32)


def device_modelopt_triplet(seed: int, n: int, k: int, device, lo: float = 2.0**-6, hi: float = 4.0):
    """The ModelOpt triplet of :func:`modelopt_triplet`, drawn on the device
    (for planes too large to draw on the host quickly): weight bytes uniform
    over 0..255 and weight_scale the E4M3 (round to nearest even) of
    2**U(log2 lo, log2 hi), from a torch generator seeded with `seed`;
    weight_scale_2 U(1e-4, 1e-2) from rng(seed)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    weight = torch.randint(0, 256, (n, k // 2), dtype=torch.uint8, device=device, generator=gen)
    e = torch.rand((n, k // 16), device=device, generator=gen) * (np.log2(hi) - np.log2(lo)) + np.log2(lo)
    scale = torch.exp2(e).to(torch.float8_e4m3fn).view(torch.uint8)
    ws2 = np.float32(rng(seed).uniform(1e-4, 1e-2))
    return weight, scale, ws2
