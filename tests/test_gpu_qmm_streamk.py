"""GPU parity of the tensor-core prefill route's stream-K work split.

Output tiles are dealt whole to the persistent CTAs, one tile each, unless
they make fewer than two waves: then every tile's k-blocks are spread evenly
over all CTAs. A tile cut between CTAs is summed in a per-stream f32
workspace with atomics, and the CTA whose k-blocks complete it writes the
outputs and clears its workspace block. The cases below split every tile
(fewer tiles than SMs, and between one and two waves), use ragged M and N,
deal more than two waves whole, call twice in a row (the workspace must come
back clean), replay a CUDA graph, agree with whole-tile scheduling, and cover
the prefill shapes at full size on sampled outputs.
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


# (M, N, K): with 256x256 tiles on 152 SMs
#   (512, 2048, 2048)   16 tiles x 32 k-blocks: every tile split four ways
#   (300, 1000, 1536)   8 ragged tiles, each split three ways
#   (2048, 5376, 2048)  168 tiles: all stream-K, 1.1 tiles per CTA
#   (4096, 8192, 512)   512 tiles: more than two waves, dealt whole
SK_SHAPES = [(512, 2048, 2048), (300, 1000, 1536), (2048, 5376, 2048), (4096, 8192, 512)]


@pytest.mark.parametrize("mnk", SK_SHAPES, ids=lambda v: "M%d_N%d_K%d" % v)
@pytest.mark.parametrize("tile", ["256x256", "256x128", "128x256"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_stream_k_parity(nv, opt, mnk, tile, dt):
    opt("tc_tile", tile)
    M, N, K = mnk
    w, s = weights(M + 3 * N + K, N, K)
    g = synth.rng(M + 5 * N + K)
    x = synth.activations(g, (M, K), dt)
    gs = np.float32(2688 * 0.61)
    ref = O.qmm(x.double().numpy(), w, s, gs)
    dx, dw, ds = x.cuda(), u32_to_dev(w), u8_to_dev(s)
    for rep in range(2):  # the second call finds the workspace as the first left it
        y, backing, guard = guarded_empty((M, N), TORCH[dt], fill=-7.0)
        nv.qmm(dx, dw, ds, gs=float(gs), route="tc", out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"call {rep}: rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)


def test_stream_k_matches_round_robin(nv, opt):
    """Stream-K and whole-tile scheduling compute the same sums (only the
    order of the f32 additions of split tiles differs)."""
    M, N, K = 2048, 5376, 2048
    w, s = weights(12, N, K)
    x = synth.activations(synth.rng(13), (M, K), "bf16").cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    a = nv.qmm(x, dw, ds, route="tc").float()
    opt("tc_streamk", 0)
    b = nv.qmm(x, dw, ds, route="tc").float()
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * b.abs().max().item()


@pytest.mark.parametrize("warm", [False, True])
def test_stream_k_graph_replay(nv, warm):
    """Captured into a CUDA graph (the capture stream's workspace is made
    during the capture unless a call came first) and replayed."""
    M, N, K = 512, 2048, 2048
    w, s = weights(21, N, K)
    x = synth.activations(synth.rng(22), (M, K), "bf16").cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    if warm:
        nv.qmm(x, dw, ds, route="tc", out=y)
        torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        nv.qmm(x, dw, ds, route="tc", out=y)
    ref = O.qmm(x.cpu().double().numpy(), w, s, None)
    for _ in range(3):
        y.fill_(-7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        assert rel_err(y, ref) <= TOL["bf16"]


# the prefill shapes: M = 512 on [21504, 5376] (168 tiles) and M = 2048 on
# [5376, 21504] (168 tiles of 336 k-blocks)
@pytest.mark.parametrize("mnk", [(512, 21504, 5376), (2048, 5376, 21504)], ids=lambda v: "M%d_N%d_K%d" % v)
def test_stream_k_prefill_shapes_sampled(nv, mnk):
    M, N, K = mnk
    g = synth.rng(M + N)
    w = synth.packed_weight(g, N, K)
    s = synth.log_uniform_scales(g, (N, K // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, 1)[0]
    x = synth.activations(g, (M, K), "bf16")
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=float(gs), route="tc")
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    assert np.isfinite(yc).all()
    pick = synth.rng(N + 3)
    rows = np.concatenate([pick.integers(0, M, size=700), np.arange(M - 10, M)])
    cols = np.concatenate([pick.integers(0, N, size=700), np.arange(N - 10, N)])
    ref = O.qmm_entries(x.double().numpy(), w, s, gs, rows, cols)
    assert np.max(np.abs(yc[rows, cols] - ref)) <= TOL["bf16"] * np.max(np.abs(ref))
