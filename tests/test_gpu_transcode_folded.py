"""GPU parity of the folded-scale transcode (``nvfp4_transcode_folded``)
against the oracle's ``transcode_folded``: words and folded scale bytes bit
for bit.

The scale bytes become the E4M3 value nearest to e4m3(b) * ws2 (float32
product, ties to even, saturating at 448, small products to 0 or a
subnormal). The cases cover planes whose byte counts are not multiples of 16
(the scalar tails), weight_scale_2 values that keep, shift, saturate and
flush the scales, and a triplet in ModelOpt's convention (ws2 = amax / 2688,
block scales up to 448) made by the library's quantizer at full size.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O
from nvfp4_quantized_matmul_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


@pytest.mark.parametrize("nk", [(1, 16), (3, 48), (7, 160), (64, 2048), (300, 5376)], ids=lambda v: "N%d_K%d" % v)
@pytest.mark.parametrize("ws2", [1.0, 0.125, 1.9e-4, 7.5, 1e-7])
def test_transcode_folded_bit_exact(nv, nk, ws2):
    N, K = nk
    g = synth.rng(N + K)
    mo_w, mo_ws, _ = synth.modelopt_triplet(g, N, K, scale_lo=2.0**-9, scale_hi=448.0)
    w, s = nv.transcode_folded(torch.from_numpy(mo_w).cuda(), torch.from_numpy(mo_ws).cuda(), float(ws2))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    rw, rs = O.transcode_folded(mo_w, mo_ws, np.float32(ws2))
    assert np.array_equal(w.cpu().numpy().view(np.uint32), rw)
    assert np.array_equal(s.cpu().numpy(), rs)


def test_transcode_folded_modelopt_convention(nv):
    """A triplet as ModelOpt writes it, made by the quantizer from a dense
    gate/up plane [43008, 5376] with gs = amax (so ws2 = amax / 2688)."""
    N, K = 43008, 5376
    x = (torch.randn((N, K), device="cuda", generator=torch.Generator(device="cuda").manual_seed(5)) * 0.02).to(
        torch.bfloat16)
    gs = x.abs().max().float().reshape(1)
    wq, sq = nv.quantize(x, gs=gs)
    ws2 = gs / 2688.0
    mo_w = wq.view(torch.uint8).reshape(N, K // 2)  # the word plane is ModelOpt's byte stream
    w, s = nv.transcode_folded(mo_w, sq, ws2)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert torch.equal(w, wq)
    rs = O.fold_scales(sq.cpu().numpy(), np.float32(ws2.item()))
    assert np.array_equal(s.cpu().numpy(), rs)
