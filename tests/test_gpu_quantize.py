"""GPU parity of the dense -> NVFP4 quantizer (``nvfp4_quantize``) against the
oracle's ``quantize``: packed words and scale bytes must match bit for bit.

The block scale is decided in IEEE float32 (amax / 6, times 2688 / gs; the
E4M3 byte nearest to that, ties to even, saturating) and each code is the
E2M1 value nearest to the exact |x| / d, d = e4m3 * gs / 2688 (ties to even,
saturating; +0 for a zero magnitude). The cases cover the three input dtypes,
with and without a global scale (per expert), zero blocks, values that tie
exactly on both grids, values one float32 step beside every midpoint for
multipliers whose reciprocal is inexact, saturation of both, the round trip
through dequantize, and planes with experts.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O
from nvfp4_quantized_matmul_gb300 import synth

from nvutil import TORCH, u32_to_dev, u8_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


def dense(seed, shape, dt):
    """Normal values with a per-row spread of magnitudes (2^-12 .. 2^12), a
    zero block and a block of tiny values per row."""
    g = synth.rng(seed)
    x = g.standard_normal(shape) * np.exp2(g.integers(-12, 13, size=shape[:-1] + (1,)))
    x[..., :16] = 0.0
    if shape[-1] >= 48:
        x[..., 32:48] *= 2.0**-30
    t = torch.from_numpy(x.astype(np.float32)).to(TORCH[dt])
    return t


def check(nv, x, gs):
    wq, sq = nv.quantize(x.cuda(), gs=None if gs is None else torch.from_numpy(gs).cuda())
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    xe = x.float().numpy()
    ge = None if gs is None else gs
    if x.dim() == 3:
        for e in range(x.shape[0]):
            w_ref, s_ref = O.quantize(xe[e], None if ge is None else ge[e])
            assert np.array_equal(sq[e].cpu().numpy(), s_ref), f"expert {e}: scale bytes"
            assert np.array_equal(wq[e].cpu().numpy().view(np.uint32), w_ref), f"expert {e}: codes"
    else:
        w_ref, s_ref = O.quantize(xe, None if ge is None else ge[0])
        assert np.array_equal(sq.cpu().numpy(), s_ref), "scale bytes"
        assert np.array_equal(wq.cpu().numpy().view(np.uint32), w_ref), "codes"


SHAPES = [(1, 16), (3, 64), (100, 272), (257, 1024), (64, 5376)]


@pytest.mark.parametrize("nk", SHAPES, ids=lambda v: "N%d_K%d" % v)
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("gs_kind", ["none", "amax", "arbitrary"])
def test_quantize_bit_exact(nv, nk, dt, gs_kind):
    N, K = nk
    x = dense(N + 3 * K, (N, K), dt)
    if gs_kind == "none":
        gs = None
    elif gs_kind == "amax":
        gs = np.array([max(np.abs(x.float().numpy()).max(), 1.0)], dtype=np.float32)  # gs must be positive
    else:
        gs = np.array([2688 * 0.37], dtype=np.float32)
    check(nv, x, gs)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_quantize_experts(nv, dt):
    x = dense(77, (3, 40, 512), dt)
    gs = np.abs(x.float().numpy()).reshape(3, -1).max(axis=1).astype(np.float32)
    check(nv, x, gs)
    check(nv, x, None)


def test_quantize_experts_partial_chunks(nv):
    """Experts whose block count is not a multiple of the bulk kernel's chunk
    (512 blocks): 5 experts of 37 x 2064 (4773 blocks each), and more experts
    (70) than one CTA per expert would give."""
    x = dense(93, (5, 37, 2064), "bf16")
    gs = np.abs(x.float().numpy()).reshape(5, -1).max(axis=1).astype(np.float32)
    check(nv, x, gs)
    x = dense(94, (70, 3, 64), "f16")
    check(nv, x, None)


def test_quantize_exact_ties(nv):
    """Codes at the midpoints of the E2M1 grid (d = 1) and block scales at the
    midpoints of the E4M3 grid: both roundings must go to the even code."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    row = [6.0] + mids + [-m for m in mids] + [0.0]
    x = np.array([row], dtype=np.float32)
    vals = O.e4m3_value(np.arange(0x38, 0x60))
    emids = (vals[:-1] + vals[1:]) / 2  # scales between 1 and 256
    xs = np.zeros((len(emids), 16), dtype=np.float32)
    xs[:, 0] = (6.0 * emids).astype(np.float32)  # amax / 6 is the midpoint exactly
    xs[:, 1] = -xs[:, 0] / 7
    for dt in ("f32", "bf16"):
        check(nv, torch.from_numpy(x).to(TORCH[dt]), None)
    check(nv, torch.from_numpy(xs), None)


def test_quantize_beside_midpoints(nv):
    """Blocks led by amax = 6 d whose other values sit at, one float32 step
    above and one below m * d for every midpoint m, for d = every fourth E4M3
    value (gs absent) and the same values times a global factor near 0.1:
    the quotients |x| / d land on or within two roundings of a midpoint,
    where the code taken from |x| * (1 / d) can differ from the nearest one."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for gs in (None, np.array([268.8], dtype=np.float32)):
        fac = np.float32(1.0) if gs is None else np.float32(np.float32(268.8) / np.float32(2688.0))
        rows = []
        for b in range(1, 0x7F, 4):
            d = np.float32(np.float32(O.e4m3_value(b)) * fac)
            amax = np.float32(6.0 * float(O.e4m3_value(b))) if gs is None else np.float32(6.0 * float(d))
            vals = []
            for m in mids:
                c = np.float32(m * float(d))
                vals += [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(0.0))]
            vals = [v for v in vals if v < amax][:21]
            vals += [np.float32(0.0)] * (21 - len(vals))
            rows.append([amax] + vals[:15] + [amax] + vals[15:] + [-v for v in vals[:9]])
        check(nv, torch.from_numpy(np.array(rows, dtype=np.float32)), gs)


def test_quantize_subnormal_multiplier(nv):
    """gs = 2688 * 2^-120 and blocks whose scale is the E4M3 subnormal 3 *
    2^-9: d = 3 * 2^-129 is a float32 subnormal, whose reciprocal overflows.
    Values at and one float32 step beside m * d for every midpoint m still
    take the nearest code."""
    gs = np.array([np.float32(2688.0 * 2.0**-120)], dtype=np.float32)
    d = np.float32(3 * 2.0**-129)
    amax = np.float32(6.0 * float(d))
    vals = []
    for m in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]:
        c = np.float32(m * float(d))
        vals += [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(0.0))]
    x = np.zeros((1, 48), dtype=np.float32)
    x[0, 0], x[0, 16], x[0, 32] = amax, amax, -amax
    x[0, 1:16] = vals[:15]
    x[0, 17:23] = vals[15:21]
    x[0, 33:48] = [-v for v in vals[:15]]
    w_ref, s_ref = O.quantize(x, gs[0])
    assert s_ref.tolist() == [[0x03, 0x03, 0x03]]
    check(nv, torch.from_numpy(x), gs)


def test_quantize_saturation(nv):
    x = np.zeros((2, 32), dtype=np.float32)
    x[0, :4] = [3000.0, -3000.0, 2.9, 100.0]   # scale saturates at 448, 3000 / 448 > 6
    x[1, 16:20] = [1e30, -1e-30, 5.0, -7.0]
    check(nv, torch.from_numpy(x), None)
    check(nv, torch.from_numpy(x), np.array([2688 * 1e-3], dtype=np.float32))


def test_quantize_dequantize_round_trip(nv):
    """A plane whose every block holds a +-6 comes back unchanged, through the
    library's own dequantize (bf16 output is exact for these products)."""
    g = synth.rng(88)
    N, K = 96, 512
    codes = g.integers(0, 16, size=(N, K))
    codes[codes == 8] = 0
    pos = g.integers(0, 16, size=(N, K // 16))
    for b in range(K // 16):
        codes[np.arange(N), 16 * b + pos[:, b]] = g.choice([7, 15], size=N)
    w = O.pack_codes(codes)
    s = synth.log_uniform_scales(g, (N, K // 16), 2.0**-8, 2.0**7)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    xd = nv.dequantize(dw, ds, None, torch.bfloat16)
    wq, sq = nv.quantize(xd)
    torch.cuda.synchronize()
    assert np.array_equal(sq.cpu().numpy(), s)
    assert np.array_equal(wq.cpu().numpy().view(np.uint32), w)


def test_quantize_full_size_plane(nv):
    """The gate/up plane [43008, 5376] in bf16 with gs = amax: compared with
    the oracle on a sample of rows."""
    N, K = 43008, 5376
    g = synth.rng(99)
    x = torch.from_numpy((g.standard_normal((N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    amax = float(x.abs().max())
    gs = torch.tensor([amax], dtype=torch.float32).cuda()
    wq, sq = nv.quantize(x.cuda(), gs=gs)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    rows = np.concatenate([synth.rng(100).integers(0, N, size=64), [0, N - 1]])
    w_ref, s_ref = O.quantize(x[rows].float().numpy(), np.float32(amax))
    assert np.array_equal(sq[rows].cpu().numpy(), s_ref)
    assert np.array_equal(wq[rows].cpu().numpy().view(np.uint32), w_ref)
