"""GPU parity of QuantizedMatmul with a non-transposed weight
(``nvfp4_qmm_nontransposed``) against the oracle's ``qmm_nontransposed``.

The weight is [K, N/8] words quantized along N with [K, N/16] scale bytes and
y = x @ dequantize(w) * gs/2688. The tensor-core producer warps decode the
words and transpose them into K-major tiles. The cases cover the shape the
pages name (x [1, 17] against a [17, 32] weight), K not a multiple of 8 (the
activations are padded into a scratch buffer first) or of the 64-input
k-block, N ending inside a weight tile and inside a word pair, one and two
128-row halves, both dtypes, the global scale, back-to-back calls, a CUDA
graph replay and the prefill shape at full size on sampled outputs, with
the stream-K split of the k-blocks and with whole tiles; and the decode
route (up to eight token rows: one streaming pass through m16n8k16 MMAs,
partial sums in a float workspace) on its own shapes, with activations
beyond f16's range, against the tensor cores and in a graph.
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


# (M, K, N)
NT_SHAPES = [(1, 17, 32), (3, 64, 272), (130, 100, 512), (257, 300, 1008), (600, 2048, 2560), (16, 5376, 256),
             (129, 8, 16)]


@pytest.mark.parametrize("mkn", NT_SHAPES, ids=lambda v: "M%d_K%d_N%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("with_gs", [False, True])
@pytest.mark.parametrize("split", ["1", "0"], ids=["streamk", "whole_tiles"])
def test_nontransposed_parity(nv, opt, mkn, dt, with_gs, split):
    # the tensor-core route for every M here (the decode route has its own
    # tests below); below two waves of tiles the k-blocks are split over the
    # CTAs unless the stream-K option is off (whole tiles)
    opt("nt_decode", 0)
    opt("tc_streamk", int(split))
    M, K, N = mkn
    w, s = weights(M + 7 * K + N, K, N)  # [K, N/8] words, [K, N/16] scales
    g = synth.rng(3 * M + K + 5 * N)
    x = synth.activations(g, (M, K), dt)
    gs = np.float32(2688 * 0.43) if with_gs else None
    ref = O.qmm_nontransposed(x.double().numpy(), w, s, gs)
    dx, dw, ds = x.cuda(), u32_to_dev(w), u8_to_dev(s)
    for rep in range(2):  # the second call finds the padding buffer as the first left it
        y, backing, guard = guarded_empty((M, N), TORCH[dt], fill=-7.0)
        nv.qmm_nontransposed(dx, dw, ds, gs=None if gs is None else float(gs), out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"call {rep}: rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)


def test_nontransposed_one_hot_rows_exact(nv):
    """Identity activations return the dequantized plane: every output is one
    exact product fp4 * e4m3, so bf16 output must match bit for bit."""
    K, N = 40, 528
    w, s = weights(91, K, N, lo=2.0**-6, hi=2.0**3)
    x = torch.eye(K, dtype=torch.bfloat16)
    ref = O.qmm_nontransposed(x.double().numpy(), w, s, None)
    y = nv.qmm_nontransposed(x.cuda(), u32_to_dev(w), u8_to_dev(s))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert np.array_equal(y.double().cpu().numpy(), ref)


def test_nontransposed_growing_padding_buffer(nv):
    """Calls with K % 8 != 0 of growing size on one stream (the padding buffer
    is replaced while an earlier call may still read the old one)."""
    outs, refs = [], []
    for i, (M, K, N) in enumerate([(4, 9, 64), (300, 77, 256), (1000, 301, 512)]):
        w, s = weights(40 + i, K, N)
        x = synth.activations(synth.rng(50 + i), (M, K), "bf16")
        refs.append(O.qmm_nontransposed(x.double().numpy(), w, s, None))
        outs.append(nv.qmm_nontransposed(x.cuda(), u32_to_dev(w), u8_to_dev(s)))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    for y, ref in zip(outs, refs):
        assert rel_err(y, ref) <= TOL["bf16"]


@pytest.mark.parametrize("K", [100, 256])
def test_nontransposed_graph_replay(nv, K):
    M, N = 200, 768
    w, s = weights(61 + K, K, N)
    x = synth.activations(synth.rng(62), (M, K), "bf16").cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        nv.qmm_nontransposed(x, dw, ds, out=y)
    ref = O.qmm_nontransposed(x.cpu().double().numpy(), w, s, None)
    for _ in range(3):
        y.fill_(-7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        assert rel_err(y, ref) <= TOL["bf16"]


def test_nontransposed_zero_k_and_empty(nv):
    x = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    s = torch.empty((0, 4), dtype=torch.uint8, device="cuda")
    y = nv.qmm_nontransposed(x, w, s)
    torch.cuda.synchronize()
    assert y.shape == (5, 64) and bool((y == 0).all())


# (M, K, N) for the decode route (M <= 16, eight rows per pass): K inside one 16-input step, across
# steps with a ragged last one, not a multiple of 4 or 8; N ending inside a
# 256-output slab and inside a word pair; planes that take the copy ring
# (N % 128 == 0, K % 4 == 0) and planes that take plain loads
NT_DECODE = [(1, 17, 32), (2, 100, 272), (1, 128, 1008), (2, 300, 256), (1, 2048, 2560), (2, 5376, 4096),
             (1, 777, 528), (2, 21504, 512), (3, 1000, 1024), (5, 260, 384), (8, 513, 640), (7, 4096, 2048),
             (4, 64, 16), (6, 18, 2304), (9, 77, 640), (12, 1000, 1024), (16, 300, 256)]


@pytest.mark.parametrize("mkn", NT_DECODE, ids=lambda v: "M%d_K%d_N%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("with_gs", [False, True])
def test_nontransposed_decode_route(nv, mkn, dt, with_gs):
    M, K, N = mkn
    w, s = weights(5 * M + 3 * K + N, K, N)
    g = synth.rng(7 * M + K + 3 * N)
    x = synth.activations(g, (M, K), dt)
    gs = np.float32(2688 * 0.71) if with_gs else None
    ref = O.qmm_nontransposed(x.double().numpy(), w, s, gs)
    dx, dw, ds = x.cuda(), u32_to_dev(w), u8_to_dev(s)
    for rep in range(2):  # the second call finds the workspace as the first left it
        y, backing, guard = guarded_empty((M, N), TORCH[dt], fill=-7.0)
        nv.qmm_nontransposed(dx, dw, ds, gs=None if gs is None else float(gs), out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"call {rep}: rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)


@pytest.mark.parametrize("aligned", [True, False], ids=["ring", "plain"])
def test_nontransposed_decode_bf16_beyond_f16(nv, aligned):
    """bf16 activations that f16 cannot hold (above its range, or below its
    normal range with more bits than its subnormals keep) take the bf16 MMA
    for the steps that hold them; the other steps keep the f16 MMA. Each token
    row is checked against its own largest output."""
    M, N = 4, 512 if aligned else 528
    K = 1024 if aligned else 1022
    w, s = weights(211 + K, K, N)
    g = synth.rng(212)
    x = torch.from_numpy(g.standard_normal(size=(M, K)).astype(np.float32))
    x[0] *= 2.0**20            # every value overflows f16
    x[1] *= 2.0**-30           # every value below f16's subnormals
    x[2, 300:310] *= 2.0**18   # a few steps of row 2 overflow f16
    x[3, 700] = 2.0**-20 * (1 + 2.0**-7)  # one value f16 rounds
    x = x.to(torch.bfloat16)
    ref = O.qmm_nontransposed(x.double().numpy(), w, s, None)
    y = nv.qmm_nontransposed(x.cuda(), u32_to_dev(w), u8_to_dev(s))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    for m in range(M):
        scale = np.max(np.abs(ref[m]))
        assert scale > 0
        err = np.max(np.abs(yc[m] - ref[m])) / scale
        assert err <= TOL["bf16"], f"row {m}: rel-to-max error {err:.3g}"


def test_nontransposed_decode_routes_agree(nv, opt):
    """The streaming route and the tensor cores compute the same sums."""
    M, K, N = 2, 2048, 4096
    w, s = weights(123, K, N)
    x = synth.activations(synth.rng(124), (M, K), "bf16").cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    a = nv.qmm_nontransposed(x, dw, ds).float()
    opt("nt_decode", 0)
    b = nv.qmm_nontransposed(x, dw, ds).float()
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * b.abs().max().item()


def test_nontransposed_decode_graph_replay(nv):
    M, K, N = 2, 1000, 2048
    w, s = weights(131, K, N)
    x = synth.activations(synth.rng(132), (M, K), "bf16").cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    gs = torch.tensor([2688.0 * 0.5], dtype=torch.float32, device="cuda")  # made before the capture
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        nv.qmm_nontransposed(x, dw, ds, gs=gs, out=y)
    ref = O.qmm_nontransposed(x.cpu().double().numpy(), w, s, np.float32(2688.0 * 0.5))
    for _ in range(3):
        y.fill_(-7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        assert rel_err(y, ref) <= TOL["bf16"]


@pytest.mark.parametrize("M", [1, 8, 2048])
def test_nontransposed_prefill_shape_sampled(nv, M):
    """The MLP up shape with the weight stored non-transposed: [5376, 21504 / 8]
    words; sampled outputs against the oracle's per-entry dot products."""
    K, N = 5376, 21504
    g = synth.rng(7000 + M)
    w = synth.packed_weight(g, K, N)
    s = synth.log_uniform_scales(g, (K, N // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, 1)[0]
    x = synth.activations(g, (M, K), "bf16")
    y = nv.qmm_nontransposed(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=float(gs))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    assert np.isfinite(yc).all()
    pick = synth.rng(7100 + M)
    rows = np.concatenate([pick.integers(0, M, size=300), [M - 1]])
    cols = np.concatenate([pick.integers(0, N, size=300), [N - 1]])
    ref = O.qmm_nontransposed_entries(x.double().numpy(), w, s, gs, rows, cols)
    assert np.max(np.abs(yc[rows, cols] - ref)) <= TOL["bf16"] * np.max(np.abs(ref))
