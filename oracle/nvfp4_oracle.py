"""CPU oracle for the NVFP4 quantized-matmul path (test infrastructure only).

This module is the plain, slow definition the CUDA library is checked
against. Only the tests, the package's smoke check and the benchmark's CPU
baseline leg may import it; the library never does, and it shares no code with
the CUDA path. Floating-point arithmetic is done in float64 except where the
format fixes a narrower precision (float32 global-scale factor, the
dequantized output dtype).

Sources, cited by page title and section:

* "perf(nvfp4): direct-transcode ModelOpt triplets to MLX native" (mlxcel
  issue #693), Technical notes: eight E2M1 nibbles per uint32 word, the E2M1
  magnitude table (0, 0.5, 1, 1.5, 2, 3, 4, 6 with a sign bit), one E4M3 byte
  scale per 16 input columns, and the global-scale sidecar kept apart from the
  block scales. Implementation plan, step 3: the triplet transcode packs four
  source bytes into one little-endian uint32 and keeps the block scales and
  ``weight_scale_2``.
* mlxcel PR #2629 (ROCm native NVFP4), Summary: the global scale is applied as
  ``global_scale / (448 * 6)`` once per output; the dequantize kernel expands a
  plane exactly. Changes during review: the scale plane has shape
  ``w.shape[:-1] + [w.shape[-1] / 2]``; out-of-range expert indices give zero
  rows. Implementation Review Summary: the same factor is used by MLX's
  dequantize.

Readings where the pages leave a step open (each also listed in the design
notes): the nibble order is low nibble = lower column index; E4M3 bytes follow
the OCP E4M3FN definition including NaN at 0x7F/0xFF; the dequantized element
is ``cast(f32(f32(fp4 * e4m3) * f32(gs / 2688)))`` with round-to-nearest-even;
the transcode's global-scale sidecar is ``f32(ws2 * 2688)`` so that the
sidecar convention reproduces ``ws2``; an activation row index at or beyond
the activation batch yields a zero row, like an out-of-range expert.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(printed table, bit-definition vs library decode, closed-form packing,
exact-rational brute force, sidecar identity against the ModelOpt formula,
zero rows; the gated-MLP activations against their symmetry identities, the
exact erf GELU and the library sigmoid, and the gate/up halves through
one-hot products; the non-transposed product against an exact-rational
brute force indexed [input, output] and through identity activations; the
quantizer's encoders against a brute-force nearest search and hand-worked
ties, the quantizer through its round trip with dequantize and a worked
global-scale case, the quantizer's code choice against exact rational
arithmetic at, above and below every midpoint for block multipliers whose
reciprocal is inexact; the folded scales against the identity at ws2 = 1,
exact power-of-two shifts, saturation and underflow). The quantizer's and the
folded scales' rounding rules (nearest, ties to even, saturating) are this
module's reading, pinned to their own definitions: the pages name the
conventions, not the rounding. The equivalence of ModelOpt's on-disk nibble
order with the MLX order is taken from the page ("likely matches") and is
parity unpinned: no real checkpoint is available to confirm it.
"""
from __future__ import annotations

import numpy as np
import torch

# E2M1 magnitudes indexed by the low three bits of a code; bit 3 is the sign.
# (issue #693, Technical notes)
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)

# 448 is the largest finite E4M3 value and 6 the largest E2M1 value; the
# global scale is divided by their product (PR #2629, Summary).
GLOBAL_SCALE_DIVISOR = 448 * 6


def e2m1_value(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (float64; code 8 is -0.0)."""
    c = np.asarray(codes).astype(np.int64)
    mag = np.asarray(E2M1_MAGNITUDES, dtype=np.float64)[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e4m3_value(b) -> np.ndarray:
    """Value of each E4M3FN byte by its bit fields (float64).

    sign = bit 7, exponent = bits 6..3 (bias 7), mantissa = bits 2..0.
    Exponent 0 is subnormal (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN;
    there are no infinities.
    """
    b = np.asarray(b).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    sub = (m / 8.0) * 2.0**-6
    nrm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    mag = np.where(e == 0, sub, nrm)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def unpack_codes(w: np.ndarray) -> np.ndarray:
    """Expand packed words ``[..., K/8]`` into codes ``[..., K]``.

    Column ``8*j + i`` is nibble ``i`` of word ``j``, counting from the least
    significant nibble (little-endian, low nibble first).
    """
    w = np.asarray(w, dtype=np.uint32).astype(np.int64)
    shifts = 4 * np.arange(8, dtype=np.int64)
    codes = (w[..., :, None] >> shifts) & 0xF
    return codes.reshape(*w.shape[:-1], w.shape[-1] * 8)


def check_planes(w: np.ndarray, scales: np.ndarray) -> None:
    """Scale plane must be ``w.shape[:-1] + [w.shape[-1] / 2]`` (PR #2629, Changes during review)."""
    if w.shape[-1] % 2 or tuple(scales.shape) != tuple(w.shape[:-1]) + (w.shape[-1] // 2,):
        raise ValueError(f"scale plane {scales.shape} does not match weight plane {w.shape}")


def block_values(w: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp4 * e4m3 for every element, ``[..., N, K]`` float64 (exact)."""
    check_planes(w, scales)
    vals = e2m1_value(unpack_codes(w))
    s = e4m3_value(scales)
    return vals * np.repeat(s, 16, axis=-1)


def global_factor(gs) -> np.float32:
    """``f32(gs) / f32(2688)`` in IEEE float32 (round to nearest even); 1 without gs."""
    if gs is None:
        return np.float32(1.0)
    return np.float32(gs) / np.float32(GLOBAL_SCALE_DIVISOR)


_OUT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def dequantize(w, scales, gs=None, out_dtype: str = "f32") -> torch.Tensor:
    """Dequantized plane ``[E?, N, K]`` as a CPU tensor of ``out_dtype``.

    Element = cast_RNE(f32(f32(fp4 * e4m3) * factor)). The fp4 * e4m3 product
    is exact in float32 (at most six significant bits). ``gs`` is None, a
    scalar, or one value per expert when ``w`` has a leading expert axis.
    """
    prod = block_values(w, scales).astype(np.float32)  # exact
    if gs is not None:
        g = np.atleast_1d(np.asarray(gs, dtype=np.float32))
        fac = np.array([global_factor(v) for v in g], dtype=np.float32)
        if prod.ndim == 3:
            fac = fac.reshape(-1, 1, 1)
        elif fac.size == 1:
            fac = fac.reshape(())
        prod = (prod * fac).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(prod)).to(_OUT[out_dtype])


def qmm(x, w, scales, gs=None) -> np.ndarray:
    """QuantizedMatmul ``y = factor * (x @ (fp4 * e4m3).T)`` in float64.

    ``x`` is ``[M, K]`` (any float array; values taken exactly), ``w`` is
    ``[N, K/8]``. The global factor multiplies each output once, after the
    sum over K (PR #2629, Summary: applied once per output).
    """
    xd = np.asarray(x, dtype=np.float64)
    deq = block_values(w, scales)
    y = xd @ deq.T
    return y * np.float64(global_factor(gs))


def qmm_nontransposed(x, w, scales, gs=None) -> np.ndarray:
    """QuantizedMatmul with a non-transposed weight: ``w`` is ``[K, N/8]``,
    quantized along its last axis N (PR #2629, Changes during review: the
    multiple-of-16 rule applies to N when the weight is not transposed), and
    ``y = factor * (x @ (fp4 * e4m3))``, ``[M, N]`` in float64."""
    xd = np.asarray(x, dtype=np.float64)
    deq = block_values(w, scales)  # [K, N]
    y = xd @ deq
    return y * np.float64(global_factor(gs))


def qmm_nontransposed_entries(x, w, scales, gs, rows, cols) -> np.ndarray:
    """Selected outputs ``y[rows[i], cols[i]]`` of :func:`qmm_nontransposed`,
    one dot product each (output n reads word column n // 8 of every input)."""
    xd = np.asarray(x, dtype=np.float64)
    fac = np.float64(global_factor(gs))
    out = np.empty(len(rows), dtype=np.float64)
    for i, (m, n) in enumerate(zip(rows, cols)):
        g = int(n) // 16  # the 16-output block: two words, one scale byte per input
        deq = block_values(w[:, 2 * g:2 * g + 2], scales[:, g:g + 1])[:, int(n) - 16 * g]
        out[i] = float(np.dot(xd[m], deq)) * fac
    return out


def qmm_entries(x, w, scales, gs, rows, cols) -> np.ndarray:
    """Selected outputs ``y[rows[i], cols[i]]`` of :func:`qmm`, one dot product each."""
    xd = np.asarray(x, dtype=np.float64)
    fac = np.float64(global_factor(gs))
    out = np.empty(len(rows), dtype=np.float64)
    for i, (m, n) in enumerate(zip(rows, cols)):
        deq = block_values(w[n:n + 1], scales[n:n + 1])[0]
        out[i] = float(np.dot(xd[m], deq)) * fac
    return out


def gather_qmm(x, lhs, rhs, w, scales, gs=None) -> np.ndarray:
    """GatherQMM: row ``r`` is ``x[lhs[r]] @ deq(w[rhs[r]]).T * factor[rhs[r]]``.

    ``w`` is ``[E, N, K/8]``; ``lhs`` None means row ``r`` uses ``x[r]``.
    Indices are unsigned 32-bit; ``rhs[r] >= E`` or ``lhs[r] >= B`` gives an
    exact +0.0 row (PR #2629, Changes during review: out-of-range experts
    produce exact zeros).
    """
    xd = np.asarray(x, dtype=np.float64)
    B = xd.shape[0]
    E, N = w.shape[0], w.shape[1]
    rhs = np.asarray(rhs, dtype=np.uint32).astype(np.int64)
    R = rhs.shape[0]
    lhs = np.arange(R, dtype=np.int64) if lhs is None else np.asarray(lhs, dtype=np.uint32).astype(np.int64)
    y = np.zeros((R, N), dtype=np.float64)
    g = None if gs is None else np.asarray(gs, dtype=np.float32).reshape(-1)
    for e in np.unique(rhs[rhs < E]):
        sel = np.nonzero((rhs == e) & (lhs < B))[0]
        if sel.size == 0:
            continue
        deq = block_values(w[e], scales[e])
        y[sel] = (xd[lhs[sel]] @ deq.T) * np.float64(global_factor(None if g is None else g[e]))
    return y


def transcode(mo_weight, mo_weight_scale, weight_scale_2):
    """ModelOpt triplet -> (packed uint32 [N, K/8], E4M3 bytes [N, K/16], f32 gs).

    Four consecutive source bytes become one little-endian word; the block
    scales are kept byte for byte; the sidecar is ``f32(ws2) * f32(2688)`` so
    that the native factor ``gs / 2688`` stands for ``weight_scale_2``
    (issue #693, Implementation plan step 3 and Technical notes).
    """
    b = np.asarray(mo_weight, dtype=np.uint8)
    n, half_k = b.shape
    if half_k % 8:
        raise ValueError("K must be a multiple of 16")
    q = b.reshape(n, half_k // 4, 4).astype(np.uint32)
    words = q[..., 0] | (q[..., 1] << 8) | (q[..., 2] << 16) | (q[..., 3] << 24)
    scales = np.array(mo_weight_scale, dtype=np.uint8, copy=True)
    gs = np.float32(weight_scale_2) * np.float32(GLOBAL_SCALE_DIVISOR)
    return words.astype(np.uint32), scales, np.float32(gs)


def fold_scales(mo_weight_scale, weight_scale_2) -> np.ndarray:
    """The folded-scale alternative that issue #693 (Technical notes) rejects:
    weight_scale * weight_scale_2 folded into each E4M3 byte, with no
    sidecar. Byte = :func:`e4m3_encode` (f32(e4m3(b) * f32(ws2))): round to
    nearest, ties to even, saturating at 448; products below half the
    smallest subnormal become 0. Non-negative, finite scale bytes only."""
    b = np.asarray(mo_weight_scale, dtype=np.uint8)
    v = (e4m3_value(b).astype(np.float32) * np.float32(weight_scale_2)).astype(np.float32)
    return e4m3_encode(v)


def transcode_folded(mo_weight, mo_weight_scale, weight_scale_2):
    """ModelOpt triplet -> (packed uint32 [N, K/8], folded E4M3 bytes [N, K/16]):
    the words of :func:`transcode` and the scales of :func:`fold_scales`."""
    words, _, _ = transcode(mo_weight, mo_weight_scale, weight_scale_2)
    return words, fold_scales(mo_weight_scale, weight_scale_2)


def modelopt_values(mo_weight, mo_weight_scale, weight_scale_2) -> np.ndarray:
    """ModelOpt's own dequantization fp4 * e4m3(weight_scale) * weight_scale_2 (float64).

    Written from the byte layout (two codes per byte, low nibble = even
    column) rather than through the packed-word path.
    """
    b = np.asarray(mo_weight, dtype=np.uint8).astype(np.int64)
    codes = np.stack([b & 0xF, b >> 4], axis=-1).reshape(b.shape[0], -1)
    s = np.repeat(e4m3_value(mo_weight_scale), 16, axis=-1)
    return e2m1_value(codes) * s * np.float64(np.float32(weight_scale_2))


# Gated MLP (issue #705 "close native NVFP4 prefill gap", Hypothesis and
# Activation-path follow-up: the Gemma and Llama MLP paths apply a GeGLU
# activation to the fused gate/up projection and scale it by the global
# factor). Readings: the fused plane holds the gate rows first and the up rows
# after them (2 I rows for I outputs); the output is act(gate) * up, each half
# already multiplied by the global factor; GeGLU uses GELU's tanh form (as
# Gemma's MLP does); SiLU (x * sigmoid(x)) is the Llama-family activation.

def gelu_tanh(v) -> np.ndarray:
    """0.5 v (1 + tanh(sqrt(2 / pi) (v + 0.044715 v^3))), float64."""
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (v + 0.044715 * v ** 3)))


def silu(v) -> np.ndarray:
    """v / (1 + exp(-v)), float64."""
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


ACTIVATIONS = {"silu": silu, "gelu_tanh": gelu_tanh}


def qmm_glu(x, w, scales, gs=None, act="gelu_tanh") -> np.ndarray:
    """Fused gate/up projection with its activation: ``w`` is ``[2 I, K/8]``
    (gate rows, then up rows); ``y = act(g) * u`` with ``[g | u] = qmm(x, w)``,
    ``y`` of shape ``[M, I]`` in float64."""
    h = qmm(x, w, scales, gs)
    half = h.shape[1] // 2
    if 2 * half != h.shape[1]:
        raise ValueError("the fused plane needs an even number of rows")
    return ACTIVATIONS[act](h[:, :half]) * h[:, half:]


def pack_codes(codes) -> np.ndarray:
    """Pack codes ``[..., K]`` into words ``[..., K/8]``: column ``8*j + i``
    into nibble ``i`` of word ``j``, least significant nibble first (the
    inverse of :func:`unpack_codes`)."""
    c = np.asarray(codes).astype(np.uint64) & 0xF
    k = c.shape[-1]
    if k % 8:
        raise ValueError("the packed axis needs a multiple of 8 columns")
    c = c.reshape(*c.shape[:-1], k // 8, 8)
    words = np.zeros(c.shape[:-1], dtype=np.uint64)
    for i in range(8):
        words |= c[..., i] << np.uint64(4 * i)
    return words.astype(np.uint32)


def _round_to_grid(v, grid) -> np.ndarray:
    """Index of the grid entry nearest to each v >= 0 (``grid`` increasing,
    index i the code of entry i). A tie goes to the even index; v beyond the
    last entry gives the last (saturation). Exact: every comparison is
    against a midpoint of two grid entries, which float64 holds exactly."""
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(grid, dtype=np.float64)
    i = np.clip(np.searchsorted(g, v, side="right") - 1, 0, len(g) - 1)  # g[i] <= v < g[i + 1]
    j = np.minimum(i + 1, len(g) - 1)
    mid = (g[i] + g[j]) / 2.0
    up = (v > mid) | ((v == mid) & (j % 2 == 0) & (j != i))
    return np.where(up, j, i)


# The finite non-negative E4M3 values, byte b at index b (0x00 .. 0x7E).
def _e4m3_grid() -> np.ndarray:
    return e4m3_value(np.arange(0x7F))


def e4m3_encode(v) -> np.ndarray:
    """Byte of the E4M3FN value nearest to each v >= 0: round to nearest,
    ties to the even byte (the even mantissa), saturating at 448 (0x7E)."""
    return _round_to_grid(v, _e4m3_grid()).astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """Magnitude code (0..7) of the E2M1 value nearest to each v >= 0: ties to
    the even code, saturating at 6 (code 7)."""
    return _round_to_grid(v, E2M1_MAGNITUDES).astype(np.int64)


def e2m1_encode_quotient(a, d) -> np.ndarray:
    """Magnitude code (0..7) of the E2M1 value nearest to the exact quotient
    ``a / d`` (a >= 0, d > 0, both float32 values): ties to the even code,
    saturating at 6 (code 7).

    The quotient is never formed. For each midpoint m of two neighbouring
    grid values, ``a`` is compared with ``m * d`` in float64, where the product
    is exact (m has at most three significant bits, d at most 24), so every
    decision is the exact one; the code is the number of midpoints the
    quotient lies above, a quotient equal to a midpoint counting it only when
    the code above it is even.
    """
    a = np.asarray(a, dtype=np.float64)
    d = np.asarray(d, dtype=np.float64)
    code = np.zeros(np.broadcast(a, d).shape, dtype=np.int64)
    for i in range(len(E2M1_MAGNITUDES) - 1):
        m = (E2M1_MAGNITUDES[i] + E2M1_MAGNITUDES[i + 1]) / 2.0
        md = m * d
        code += (a > md) | ((a == md) & ((i + 1) % 2 == 0))
    return code


def quantize(x, gs=None):
    """Dense -> NVFP4 planes ``(w [..., K/8] uint32, scales [..., K/16] uint8)``.

    The encoding half of MLX's global-scale convention (PR #2629,
    Implementation Review Summary: fp_quantize encodes block scales times
    448 * 6 / global_scale), with the rounding and saturation the pages leave
    open read as follows, per 16-column block:

    * amax = max |x|; s = amax / 6, then s * (2688 / gs) when gs is given
      (each step an IEEE float32 operation, round to nearest even);
    * scale byte = :func:`e4m3_encode` (s);
    * d = float32(e4m3(byte) * (gs / 2688)), the multiplier the
      dequantization applies to the block;
    * code = the E2M1 value nearest to the exact |x| / d
      (:func:`e2m1_encode_quotient`), with the sign bit of x; +0 where the
      magnitude code is 0, and every code 0 where d == 0.
    """
    xf = np.asarray(x, dtype=np.float32)
    k = xf.shape[-1]
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    blocks = xf.reshape(*xf.shape[:-1], k // 16, 16)
    amax = np.max(np.abs(blocks), axis=-1)
    s = (amax / np.float32(6.0)).astype(np.float32)
    if gs is not None:
        inv = np.float32(np.float32(GLOBAL_SCALE_DIVISOR) / np.float32(gs))
        s = (s * inv).astype(np.float32)
    sbytes = e4m3_encode(s)
    d = (e4m3_value(sbytes).astype(np.float32) * global_factor(gs)).astype(np.float32)
    live = d[..., None] > 0
    mag = np.where(live, e2m1_encode_quotient(np.abs(blocks), np.where(live, d[..., None], 1.0)), 0)
    codes = np.where((blocks < 0) & (mag != 0), mag | 8, mag).reshape(xf.shape)
    return pack_codes(codes), sbytes


def rel_to_max_error(y, ref) -> float:
    """max|y - ref| / max|ref| (the pages' error-relative-to-max metric)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.max(np.abs(ref)) if ref.size else 0.0
    if denom == 0.0:
        return float(np.max(np.abs(y))) if y.size else 0.0
    return float(np.max(np.abs(y - ref)) / denom)
