"""The allocation-free QuantizedMatmul entry point (nvfp4_qmm_noalloc).

Some callers cannot allocate device memory: a serving runtime that plans all
of its memory once at start-up, or code that runs while a CUDA graph is being
captured in the strict mode, where an allocation would break the capture.
nvfp4_qmm_noalloc serves them with its scratch in a fixed array inside the
library. Each case calls it twice in a row through the C ABI and checks both
results against the CPU oracle (every output of the small shapes, sampled
outputs of the large ones) and against the regular nvfp4_qmm. The second call
finds the array as the first one left it. The per-call clear itself guards
against leftovers of a call cut short by a bounded wait, which these tests do
not produce. The free device memory is checked to be unchanged across calls
made on a stream the library has never seen, where the regular entry point
would allocate its per-stream workspace. The file is named to be collected
last; it must pass alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from nvfp4_quantized_matmul_gb300 import synth
from oracle import nvfp4_oracle as O

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


def _reference(x, w, s, gs, n, full):
    """The oracle's outputs: every one (full) or a sample of rows and columns
    (every token row, the first and last weight rows, 256 random ones)."""
    xd = x.double().cpu().numpy()
    if full:
        return None, O.qmm(xd, w, s, gs)
    g = np.random.default_rng(n)
    cols = np.unique(np.concatenate([[0, n - 1], g.integers(0, n, size=256)]))
    rows = np.repeat(np.arange(xd.shape[0]), cols.size)
    cc = np.tile(cols, xd.shape[0])
    return (rows, cc), O.qmm_entries(xd, w, s, gs, rows, cc)


@pytest.mark.parametrize("nkm", [(3000, 4096, 1), (5376, 21504, 4), (2304, 2560, 16), (257, 256, 9)],
                         ids=lambda v: "N%d_K%d_M%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_noalloc_matches_oracle_twice(nv, nkm, dt):
    N, K, M = nkm
    w, s = weights(N + K + M, N, K)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    x = synth.activations(synth.rng(N * 3 + M), (M, K), dt).cuda()
    gs = np.float32(2688 * 0.41)
    gsd = torch.tensor([float(gs)], dtype=torch.float32, device="cuda")
    full = N * K <= 1 << 20
    pick, ref = _reference(x, w, s, gs, N, full)
    regular = nv.qmm(x, dw, ds, gs=gsd).double().cpu().numpy()
    for call in range(2):
        y = nv.qmm_noalloc(x, dw, ds, gs=gsd)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        yc = y.double().cpu().numpy()
        got = yc if pick is None else yc[pick]
        err = O.rel_to_max_error(got, ref)
        assert err <= TOL[dt], f"call {call}: rel-to-max error {err:.3g} against the oracle > {TOL[dt]}"
        err = rel_err(y, regular)
        assert err <= TOL[dt], f"call {call}: rel-to-max error {err:.3g} against nvfp4_qmm > {TOL[dt]}"


def test_noalloc_allocates_nothing(nv):
    """Calls on a stream the library has never seen leave the device's free
    memory as it was (inputs, output and global scale made beforehand; the
    first call on the device, which looks up the array's address and may load
    the kernel's module, made beforehand as well)."""
    N, K, M = 2304, 2560, 16
    w, s = weights(7, N, K)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    x = synth.activations(synth.rng(8), (M, K), "bf16").cuda()
    gsd = torch.tensor([2688.0 * 0.7], dtype=torch.float32, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nv.qmm_noalloc(x, dw, ds, gs=gsd, out=out)
    torch.cuda.synchronize()
    ref = out.clone()
    fresh = torch.cuda.Stream()
    free0, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(fresh):
        for _ in range(3):
            out.zero_()
            nv.qmm_noalloc(x, dw, ds, gs=gsd, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert nv.take_device_error() == 0
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    # split row tiles add their partial sums in arrival order, so repeated
    # calls agree to rounding, not bit for bit
    err = rel_err(out, ref.double().cpu().numpy())
    assert err <= TOL["bf16"], f"rel-to-max error {err:.3g} against the first call"


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
