"""The allocation-free QuantizedMatmul entry point (nvfp4_qmm_noalloc).

It exists for callers that may not allocate device memory (a runtime with a
memory plan fixed at start-up, or code running during a strict-mode graph
capture); it keeps its scratch in a fixed array inside the library. Each case
calls it twice in a row through the C ABI and compares both results with the
regular nvfp4_qmm on the same inputs: the second call finds the array as the
first left it, so it also checks that the scratch is cleared. The file is
named to be collected last; it must pass alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from nvfp4_quantized_matmul_gb300 import synth

from nvutil import TOL, rel_err, u32_to_dev, u8_to_dev, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


@pytest.mark.parametrize("nkm", [(3000, 4096, 1), (5376, 21504, 4), (2304, 2560, 16), (257, 256, 9)],
                         ids=lambda v: "N%d_K%d_M%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_noalloc_matches_qmm_twice(nv, nkm, dt):
    N, K, M = nkm
    w, s = weights(N + K + M, N, K)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    x = synth.activations(synth.rng(N * 3 + M), (M, K), dt).cuda()
    gs = float(np.float32(2688 * 0.41))
    ref = nv.qmm(x, dw, ds, gs=gs).double().cpu().numpy()
    for call in range(2):
        y = nv.qmm_noalloc(x, dw, ds, gs=gs)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"call {call}: rel-to-max error {err:.3g} against nvfp4_qmm > {TOL[dt]}"


def test_noalloc_refuses_shapes_beyond_its_scratch(nv):
    K = 256
    x = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    w, s = weights(1, 65537, K)
    with pytest.raises(nv.binding.Nvfp4Error, match="ERR_LIMIT"):
        nv.qmm_noalloc(x, u32_to_dev(w), u8_to_dev(s))
    w, s = weights(2, 64, K)
    with pytest.raises(nv.binding.Nvfp4Error, match="ERR_LIMIT"):
        nv.qmm_noalloc(torch.zeros((17, K), dtype=torch.bfloat16, device="cuda"), u32_to_dev(w), u8_to_dev(s))
    w, s = weights(3, 64, 272)
    with pytest.raises(nv.binding.Nvfp4Error, match="ERR_SHAPE"):
        nv.qmm_noalloc(torch.zeros((1, 272), dtype=torch.bfloat16, device="cuda"), u32_to_dev(w), u8_to_dev(s))
