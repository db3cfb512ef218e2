"""GPU parity of the fused gate/up projection with its activation
(``nvfp4_qmm_glu``) against the oracle's ``qmm_glu``.

The plane holds the I gate rows and then the I up rows; both routes stack
128 gate rows on the matching 128 up rows in one tile and apply
act(gate) * up in the epilogue. The cases cover both activations, both
routes (forced and automatic), ragged I, several 16-row launches on the
decode route, K cut into groups, the global scale, back-to-back calls and the
fused gate/up plane of the decode step at full size on sampled outputs.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O
from nvfp4_quantized_matmul_gb300 import synth

from nvutil import TOL, TORCH, guarded_empty, guards_intact, rel_err, u32_to_dev, u8_to_dev, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


# (I, K): ragged I (not a multiple of 128, or of 8), one to 21 chunks of K
GLU_SHAPES = [(128, 256), (300, 2048), (1000, 768), (2688, 5376), (131, 512)]


@pytest.mark.parametrize("ik", GLU_SHAPES, ids=lambda v: "I%d_K%d" % v)
@pytest.mark.parametrize("M", [1, 5, 16, 17, 40])
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_glu_decode_route(nv, ik, M, act, dt):
    I, K = ik
    # small block scales keep act(gate) * up inside f16's range
    w, s = weights(I + K + M, 2 * I, K, lo=2.0**-8, hi=2.0**-3)
    g = synth.rng(3 * I + K + M)
    x = synth.activations(g, (M, K), dt).cuda()
    gs = np.float32(2688 * 0.9)
    ref = O.qmm_glu(x.cpu().double().numpy(), w, s, gs, act)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    for rep in range(2):  # the second call finds the decode workspace as the first left it
        y, backing, guard = guarded_empty((M, I), TORCH[dt], fill=-7.0)
        nv.qmm_glu(x, dw, ds, gs=float(gs), act=act, route="qmv", out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"call {rep}: rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)


# (M, I, K): one M half, both halves, ragged M and I, several k-blocks
TC_GLU = [(1, 128, 64), (130, 300, 96), (300, 1000, 512), (600, 2688, 256)]


@pytest.mark.parametrize("mik", TC_GLU, ids=lambda v: "M%d_I%d_K%d" % v)
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("with_gs", [False, True])
def test_glu_tensor_core_route(nv, mik, act, dt, with_gs):
    M, I, K = mik
    w, s = weights(M + I + K, 2 * I, K, lo=2.0**-6, hi=0.5)
    g = synth.rng(M * 3 + I + K)
    x = synth.activations(g, (M, K), dt)
    gs = np.float32(2688 * 0.37) if with_gs else None
    ref = O.qmm_glu(x.double().numpy(), w, s, gs, act)
    y, backing, guard = guarded_empty((M, I), TORCH[dt], fill=-7.0)
    nv.qmm_glu(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=None if gs is None else float(gs), act=act, route="tc",
               out=y)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert rel_err(y, ref) <= TOL[dt]
    assert guards_intact(backing, guard)


def test_glu_routes_agree_and_auto(nv):
    """Both routes compute the same sums; the automatic route matches them."""
    M, I, K = 48, 1024, 2048
    w, s = weights(11, 2 * I, K)
    x = synth.activations(synth.rng(12), (M, K), "bf16").cuda()
    args = (x, u32_to_dev(w), u8_to_dev(s))
    a = nv.qmm_glu(*args, act="silu", route="qmv").float()
    b = nv.qmm_glu(*args, act="silu", route="tc").float()
    c = nv.qmm_glu(*args, act="silu").float()
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    scale = b.abs().max().item()
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * scale
    assert (c - b).abs().max().item() <= 2 * 2.0**-8 * scale


@pytest.mark.parametrize("M,route", [(1, "qmv"), (16, "qmv"), (512, "tc")])
def test_glu_gate_up_plane_sampled(nv, M, route):
    """The decode step's fused gate/up plane [43008, 5376] (I = 21504) with
    GeGLU: sampled outputs against the oracle's per-entry dot products."""
    I, K = 21504, 5376
    g = synth.rng(4300 + M)
    w = synth.packed_weight(g, 2 * I, K)
    s = synth.log_uniform_scales(g, (2 * I, K // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, 1)[0]
    x = synth.activations(g, (M, K), "bf16")
    y = nv.qmm_glu(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=float(gs), act="gelu_tanh", route=route)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    assert np.isfinite(yc).all()
    pick = synth.rng(4400 + M)
    rows = pick.integers(0, M, size=400)
    cols = np.concatenate([pick.integers(0, I, size=390), np.arange(I - 10, I)])
    xd = x.double().numpy()
    gate = O.qmm_entries(xd, w, s, gs, rows, cols)
    up = O.qmm_entries(xd, w, s, gs, rows, cols + I)
    ref = O.gelu_tanh(gate) * up
    assert np.max(np.abs(yc[rows, cols] - ref)) <= TOL["bf16"] * np.max(np.abs(ref))
