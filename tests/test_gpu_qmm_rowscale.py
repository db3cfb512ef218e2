"""GPU parity of bf16 activations on the tensor-core routes, which run the f16
kernels: each activation row is first scaled by the power of two that brings
its largest finite magnitude into [2^14, 2^15) and rounded to f16, and the
row's sums are scaled back before the bf16 output is written.

The rows below stress that conversion: far above f16's range, far below it,
values above 65504 beside values below f16's subnormals in one row, an
infinity, an all-zero row, and ordinary rows; both tile schedules (whole
tiles and the stream-K split), the fused gate/up route, and a CUDA graph.
Each row is checked against its own largest reference output.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O
from nvfp4_quantized_matmul_gb300 import synth

from nvutil import TOL, u32_to_dev, u8_to_dev, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


def wide_rows(seed, M, K):
    g = synth.rng(seed)
    x = torch.from_numpy(g.standard_normal(size=(M, K)).astype(np.float32))
    x[0] *= 2.0**100                 # far above f16's range
    x[1] *= 2.0**-100                # far below it
    x[2, ::7] *= 1.0e5               # above 65504 ...
    x[2, 3::11] *= 1.0e-7            # ... beside values below f16's subnormals
    x[3, 17] = float("inf")
    x[4] = 0.0
    return x.to(torch.bfloat16)


def check_rows(y, ref, inf_rows=(3,)):
    yc = y.double().cpu().numpy()
    for m in range(ref.shape[0]):
        if m in inf_rows:
            assert np.array_equal(np.isfinite(yc[m]), np.isfinite(ref[m])), f"row {m}: non-finite outputs differ"
            continue
        scale = np.max(np.abs(ref[m]))
        if scale == 0:
            assert np.all(yc[m] == 0), f"row {m}: expected zeros"
            continue
        err = np.max(np.abs(yc[m] - ref[m])) / scale
        assert err <= TOL["bf16"], f"row {m}: rel-to-row-max error {err:.3g}"


@pytest.mark.parametrize("split", ["1", "0"], ids=["streamk", "whole_tiles"])
@pytest.mark.parametrize("with_gs", [False, True])
def test_bf16_rows_through_f16_kernel(nv, opt, split, with_gs):
    opt("tc_streamk", int(split))
    M, N, K = 300, 640, 1024
    w, s = weights(901, N, K)
    x = wide_rows(902, M, K)
    gs = np.float32(2688 * 0.37) if with_gs else None
    ref = O.qmm(x.double().numpy(), w, s, gs)
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=None if gs is None else float(gs), route="tc")
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert y.dtype == torch.bfloat16
    check_rows(y, ref)


def test_bf16_rows_through_f16_glu(nv):
    M, cols, K = 200, 384, 512
    w, s = weights(903, 2 * cols, K)
    x = wide_rows(904, M, K)
    # keep act(gate) * up inside bf16's range: rows of 2^10 and 2^-56
    x[0] *= 2.0**-90
    x[1] *= 2.0**44
    ref = O.qmm_glu(x.double().numpy(), w, s, None, act="silu")
    y = nv.qmm_glu(x.cuda(), u32_to_dev(w), u8_to_dev(s), act="silu", route="tc")
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    check_rows(y, ref, inf_rows=(3,))


def test_bf16_rows_graph_replay(nv):
    M, N, K = 130, 512, 768
    w, s = weights(905, N, K)
    x = wide_rows(906, M, K).cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        nv.qmm(x, dw, ds, route="tc", out=y)
    ref = O.qmm(x.cpu().double().numpy(), w, s, None)
    for _ in range(2):
        y.fill_(-7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        check_rows(y, ref)


@pytest.mark.parametrize("K", [512, 300], ids=["K512", "K300_padded"])
def test_bf16_rows_nontransposed_tc(nv, opt, K):
    """The non-transposed tensor-core route converts (and, for K % 8 != 0,
    pads) the rows in one pass."""
    opt("nt_decode", 0)
    M, N = 260, 384
    w, s = weights(907 + K, K, N)  # [K, N/8] words, [K, N/16] scales
    x = wide_rows(908, M, K)
    ref = O.qmm_nontransposed(x.double().numpy(), w, s, None)
    y = nv.qmm_nontransposed(x.cuda(), u32_to_dev(w), u8_to_dev(s))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    check_rows(y, ref)


def test_bf16_rows_sorted_gather_tc(nv, opt):
    """The sorted gather gathers and converts the rows in one pass; rows whose
    activation index is out of range stay +0."""
    opt("gather_tc", 1)
    E, N, K, T = 4, 256, 512, 40
    w, s = weights(909, E, N, K)
    x = wide_rows(910, T, K)
    lhs = np.arange(T, dtype=np.uint32)
    rhs = np.sort(synth.rng(911).integers(0, E, size=T).astype(np.uint32))
    lhs[7] = T + 3  # out of range: an exact +0 row
    ref = O.gather_qmm(x.double().numpy(), lhs, rhs, w, s, None)
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs), sorted_indices=True)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    assert np.all(yc[7] == 0.0) and not np.any(np.signbit(yc[7]))
    # output row r holds x row lhs[r]: the special rows keep their indices
    inf_rows = tuple(int(r) for r in np.nonzero(lhs == 3)[0])
    check_rows(y, ref, inf_rows=inf_rows)
