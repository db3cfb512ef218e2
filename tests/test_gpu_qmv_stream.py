"""GPU parity of the persistent decode route (dense QuantizedMatmul with 1 to
16 token rows, K a multiple of 256) against the CPU oracle.

The route splits the weight plane evenly over the SMs, so most 256-row tiles
are shared by two or more CTAs and finished through the library's workspace;
the cases below cover ragged N, K cut into several groups (large M times K),
back-to-back calls (the workspace must come back clean), several streams,
graph replay and the decode linears at full size (sampled outputs).
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


# (N, K): ragged row tiles, one to 84 chunks, K split in groups for larger M
STREAM_SHAPES = [(1000, 4096), (300, 21504), (4100, 768), (2304, 2560), (257, 256)]


@pytest.mark.parametrize("nk", STREAM_SHAPES, ids=lambda v: "N%d_K%d" % v)
@pytest.mark.parametrize("M", [1, 2, 4, 5, 8, 9, 16, 17, 40])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_stream_route_parity(nv, nk, M, dt):
    N, K = nk
    w, s = weights(N + 3 * K + M, N, K)
    g = synth.rng(N * 5 + K + M)
    x = synth.activations(g, (M, K), dt).cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    for gs in (None, np.float32(2688 * 0.73)):
        ref = O.qmm(x.cpu().double().numpy(), w, s, gs)
        for rep in range(2):  # the second call finds the workspace as the first left it
            y, backing, guard = guarded_empty((M, N), TORCH[dt], fill=-7.0)
            nv.qmm(x, dw, ds, gs=None if gs is None else float(gs), route="qmv", out=y)
            torch.cuda.synchronize()
            assert nv.take_device_error() == 0
            err = rel_err(y, ref)
            assert err <= TOL[dt], f"call {rep}: rel-to-max error {err:.3g} > {TOL[dt]}"
            assert guards_intact(backing, guard)


@pytest.mark.parametrize("M", [3, 16])
def test_stream_route_two_row_tiles_per_warp(nv, opt, M):
    """Two row tiles per consumer warp: eight consumer warps of 32 weight rows
    each."""
    opt("qmv_row_tiles", 2)
    N, K = 1000, 4096
    w, s = weights(5 + M, N, K)
    x = synth.activations(synth.rng(M), (M, K), "bf16").cuda()
    for rep in range(2):
        y = nv.qmm(x, u32_to_dev(w), u8_to_dev(s), route="qmv")
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        assert rel_err(y, O.qmm(x.cpu().double().numpy(), w, s, None)) <= TOL["bf16"]


def test_stream_route_alternating_shapes_and_streams(nv):
    """Calls of different shapes interleaved on two streams; each stream has
    its own workspace."""
    cases = []
    for i, (N, K, M) in enumerate([(1000, 4096, 3), (300, 21504, 16), (4100, 768, 1)]):
        w, s = weights(500 + i, N, K)
        x = synth.activations(synth.rng(600 + i), (M, K), "bf16").cuda()
        cases.append((x, u32_to_dev(w), u8_to_dev(s), O.qmm(x.cpu().double().numpy(), w, s, None)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        for j, (x, dw, ds, ref) in enumerate(cases):
            st = streams[(rep + j) % 2]
            with torch.cuda.stream(st):
                outs.append((nv.qmm(x, dw, ds, route="qmv"), ref))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    for y, ref in outs:
        assert rel_err(y, ref) <= TOL["bf16"]


@pytest.mark.parametrize("capture", ["warm_stream", "torch_side_stream"])
def test_stream_route_graph_replay(nv, capture):
    """Graph replay with launch overlap on. `warm_stream`: the capture runs on
    the stream that made the first call; `torch_side_stream`: torch captures on
    a stream of its own that has never made a call, so the workspace is
    created during the capture."""
    N, K, M = 2304, 2560, 4
    w, s = weights(77 if capture == "warm_stream" else 78, N, K)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    prev = nv.set_launch_overlap(True)
    try:
        gr = torch.cuda.CUDAGraph()
        if capture == "warm_stream":
            s0 = torch.cuda.Stream()
            with torch.cuda.stream(s0):
                x.copy_(synth.activations(synth.rng(1), (M, K), "bf16").cuda())
                nv.qmm(x, dw, ds, out=y)  # warm-up: plan and workspace before capture
                s0.synchronize()
                with torch.cuda.graph(gr, stream=s0):
                    nv.qmm(x, dw, ds, out=y)
        else:
            torch.cuda.synchronize()
            with torch.cuda.graph(gr):
                nv.qmm(x, dw, ds, out=y)
        for seed in (2, 3, 4):
            xs = synth.activations(synth.rng(seed), (M, K), "bf16")
            x.copy_(xs.cuda())
            torch.cuda.synchronize()
            gr.replay()
            torch.cuda.synchronize()
            assert nv.take_device_error() == 0
            assert rel_err(y, O.qmm(xs.double().numpy(), w, s, None)) <= TOL["bf16"], f"seed {seed}"
    finally:
        nv.set_launch_overlap(prev)


def test_stream_route_matches_tensor_core_route(nv):
    """The decode route and the tensor-core route compute the same sums."""
    N, K, M = 3000, 5376, 8
    w, s = weights(88, N, K)
    x = synth.activations(synth.rng(89), (M, K), "bf16").cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    a = nv.qmm(x, dw, ds, route="qmv").float()
    b = nv.qmm(x, dw, ds, route="tc").float()
    assert nv.take_device_error() == 0
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * b.abs().max().item()


# The three decode linears of the benchmark at full size: outputs are checked
# on a sample of entries, each computed by the oracle as one dot product.
DECODE_LINEARS = [(43008, 5376), (5376, 21504), (8192, 5376)]


@pytest.mark.parametrize("nk", DECODE_LINEARS, ids=lambda v: "N%d_K%d" % v)
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_stream_route_decode_linears_sampled(nv, nk, M):
    N, K = nk
    g = synth.rng(N + K)
    w = synth.packed_weight(g, N, K)
    s = synth.log_uniform_scales(g, (N, K // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, 1)[0]
    x = synth.activations(synth.rng(M), (M, K), "bf16")
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=float(gs))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    assert np.isfinite(yc).all()
    pick = synth.rng(N + M)
    rows = pick.integers(0, M, size=600)
    cols = np.concatenate([pick.integers(0, N, size=580), np.arange(N - 20, N)])  # include the ragged end
    ref = O.qmm_entries(x.double().numpy(), w, s, gs, rows, cols)
    got = yc[rows, cols]
    # per-entry bound: bf16 output rounding plus f32 accumulation, relative to the sample's max
    assert np.max(np.abs(got - ref)) <= TOL["bf16"] * np.max(np.abs(ref))
