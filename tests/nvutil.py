"""Shared helpers for the GPU parity tests (inputs from synth, references from the oracle)."""
import numpy as np
import torch

from nvfp4_quantized_matmul_gb300 import synth
from oracle import nvfp4_oracle as O

# Error bound on max|y - ref| / max|ref| per activation dtype (f32 / f16 / bf16).
TOL = {"f32": 1e-5, "f16": 1e-3, "bf16": 8e-3}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
SENTINEL = {"f32": float("nan"), "f16": -7.0, "bf16": -7.0}


def dev():
    return torch.device("cuda:0")


def u32_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(dev())


def u8_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev())


def f32_to_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.atleast_1d(a), dtype=np.float32)).to(dev())


def guarded_empty(shape, dtype, guard=64, fill=-7.0):
    """An output tensor with guard bands on both sides, all set to a sentinel.

    Returns (view, backing, guard). The view starts 256 bytes into the backing
    buffer so alignment is preserved.
    """
    n = int(np.prod(shape))
    backing = torch.full((n + 2 * guard,), fill, dtype=dtype, device=dev())
    view = backing[guard:guard + n].view(*shape)
    return view, backing, guard


def guards_intact(backing, guard, fill=-7.0):
    head = backing[:guard].float().cpu()
    tail = backing[-guard:].float().cpu()
    f = torch.tensor(fill)
    if np.isnan(fill):
        return bool(torch.isnan(head).all() and torch.isnan(tail).all())
    return bool((head == f).all() and (tail == f).all())


def weights(seed, *shape_nk, lo=2.0**-6, hi=4.0):
    g = synth.rng(seed)
    w = synth.packed_weight(g, *shape_nk)
    s = synth.log_uniform_scales(g, (*shape_nk[:-1], shape_nk[-1] // 16), lo, hi)
    return w, s


def rel_err(y: torch.Tensor, ref: np.ndarray) -> float:
    return O.rel_to_max_error(y.double().cpu().numpy(), ref)
