"""GPU parity: every route of libnvfp4.so against the CPU oracle.

Bit-exact for transcode and dequantize; max|y - ref| / max|ref| within the
per-dtype bound for the matmul routes (1e-5 f32, 1e-3 f16, 8e-3 bf16).
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O
from nvfp4_quantized_matmul_gb300 import synth

from nvutil import TOL, TORCH, f32_to_dev, guarded_empty, guards_intact, rel_err, u32_to_dev, u8_to_dev, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.view(torch.int16).numpy()


def _assert_bit_exact(got: torch.Tensor, ref: torch.Tensor):
    g, r = got.cpu(), ref.cpu()
    gn, rn = torch.isnan(g.float()), torch.isnan(r.float())
    assert torch.equal(gn, rn), "NaN positions differ"
    gb, rb = _bits(g), _bits(r)
    keep = ~rn.numpy()
    bad = np.nonzero((gb != rb) & keep)
    assert bad[0].size == 0, f"{bad[0].size} elements differ, first at {tuple(b[0] for b in bad)}"


# ------------------------------------------------------------------ dequantize

@pytest.mark.parametrize("shape", [(1, 272, 256), (1, 1, 16), (3, 17, 48), (2, 64, 5376), (1, 5, 32)])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("with_gs", [False, True])
def test_dequantize_bit_exact(nv, shape, dt, with_gs):
    E, N, K = shape
    w, s = weights(100 + N + K, E, N, K)
    # exercise special scale bytes: NaN, signed zeros, negatives, subnormals, max
    flat = s.reshape(-1)
    specials = np.array([0x7F, 0xFF, 0x00, 0x80, 0x01, 0x81, 0x7E, 0xFE, 0x38, 0xB8], dtype=np.uint8)
    flat[: min(flat.size, specials.size)] = specials[: flat.size]
    gs = synth.global_scales(synth.rng(7), E) if with_gs else None
    if E == 1:  # a single linear: [N, K/8] planes and a scalar global scale
        w, s = w[0], s[0]
        gs = None if gs is None else gs[0]
    out = nv.dequantize(u32_to_dev(w), u8_to_dev(s), None if gs is None else f32_to_dev(gs), TORCH[dt])
    torch.cuda.synchronize()
    ref = O.dequantize(w, s, gs, dt)
    _assert_bit_exact(out, ref)


def test_dequantize_guard_bands(nv):
    N, K = 33, 48
    w, s = weights(5, N, K)
    out, backing, guard = guarded_empty((N, K), torch.bfloat16)
    nv.dequantize(u32_to_dev(w), u8_to_dev(s), None, torch.bfloat16, out=out)
    torch.cuda.synchronize()
    assert guards_intact(backing, guard)
    _assert_bit_exact(out, O.dequantize(w, s, None, "bf16"))


# ------------------------------------------------------------------ transcode

# (43008, 5376): the fused gate/up plane, about 26 copy chunks per SM (more
# than the bulk copy's ring of six); (3, 16) and (1, 48): planes shorter than
# a 16-byte unit at their end.
@pytest.mark.parametrize("nk", [(3, 16), (272, 256), (33, 5376), (1, 48), (43008, 5376)])
def test_transcode_bit_exact(nv, nk):
    N, K = nk
    g = synth.rng(N * 7 + K)
    mo_w, mo_ws, ws2 = synth.modelopt_triplet(g, N, K)
    w, s, gs = nv.transcode(u8_to_dev(mo_w), u8_to_dev(mo_ws), float(ws2))
    rw, rs, rg = O.transcode(mo_w, mo_ws, ws2)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), rw)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert gs.cpu().numpy().view(np.uint32)[0] == np.float32(rg).view(np.uint32)


def test_transcode_then_dequantize_matches_modelopt(nv):
    """Sidecar identity on the GPU: native dequantize of the transcoded planes
    reproduces ModelOpt's fp4 * e4m3(weight_scale) * weight_scale_2."""
    g = synth.rng(77)
    N, K = 64, 256
    mo_w, mo_ws, ws2 = synth.modelopt_triplet(g, N, K)
    w, s, gs = nv.transcode(u8_to_dev(mo_w), u8_to_dev(mo_ws), float(ws2))
    deq = nv.dequantize(w, s, gs, torch.float32).cpu().numpy().astype(np.float64)
    ref = O.modelopt_values(mo_w, mo_ws, ws2)
    ulp = np.spacing(np.abs(ref.astype(np.float32))).astype(np.float64)
    assert np.all(np.abs(deq - ref) <= 2 * ulp)
    rw, rs, rg = O.transcode(mo_w, mo_ws, ws2)
    _assert_bit_exact(torch.from_numpy(deq.astype(np.float32)), O.dequantize(rw, rs, rg, "f32"))


# ------------------------------------------------------------------ QuantizedMatmul

QMM_SHAPES = [(512, 256), (272, 48), (1, 16), (17, 5376), (96, 1040)]


@pytest.mark.parametrize("nk", QMM_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16, 33])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_qmm_qmv_route(nv, nk, M, dt):
    N, K = nk
    w, s = weights(N * 31 + K, N, K, lo=2.0**-4, hi=16.0)
    g = synth.rng(M * 1000 + N + K)
    x = synth.activations(g, (M, K), dt)
    for gs in (None, np.float32(2688 * 0.01)):
        y, backing, guard = guarded_empty((M, N), TORCH[dt], fill=-7.0)
        nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=None if gs is None else float(gs), route="qmv", out=y)
        torch.cuda.synchronize()
        ref = O.qmm(x.double().numpy(), w, s, gs)
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)


def test_qmm_unit_scales_one_hot(nv):
    """Unit scales and one-hot activations reproduce E2M1 table entries exactly."""
    N, K = 16, 32
    codes = (np.arange(N * K).reshape(N, K) % 16).astype(np.int64)
    w = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        w |= (codes[:, i::8].astype(np.uint32) << (4 * i))
    s = np.full((N, K // 16), 0x38, dtype=np.uint8)
    x = torch.eye(K, dtype=torch.bfloat16)
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), route="qmv").float().cpu().numpy()
    ref = O.qmm(x.double().numpy(), w, s)
    assert np.array_equal(y, ref)


def test_qmm_empty(nv):
    w, s = weights(1, 32, 64)
    y = nv.qmm(torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"), u32_to_dev(w), u8_to_dev(s))
    assert y.shape == (0, 32)


# ------------------------------------------------------------------ GatherQMM

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("with_gs", [False, True])
def test_gather_unsorted_decode_with_zero_rows(nv, dt, with_gs):
    E, N, K, B = 8, 96, 256, 10
    w, s = weights(9, E, N, K)
    g = synth.rng(91)
    gs = synth.global_scales(g, E) if with_gs else None
    x = synth.activations(g, (B, K), dt)
    rhs = np.concatenate([synth.zipf_experts(g, 20, E), np.array([E, E + 1, 2**31 - 1, 2**32 - 1, 3, 5], dtype=np.uint32)])
    lhs = np.concatenate([g.integers(0, B, size=20).astype(np.uint32), np.array([0, 1, 2, 3, B, 2**32 - 1], dtype=np.uint32)])
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs),
                      gs=None if gs is None else f32_to_dev(gs))
    torch.cuda.synchronize()
    ref = O.gather_qmm(x.double().numpy(), lhs, rhs, w, s, gs)
    yc = y.float().cpu().numpy()
    for r in range(20, 26):
        assert np.all(yc[r] == 0.0) and not np.any(np.signbit(yc[r])), f"row {r} must be +0.0"
    assert rel_err(y, ref) <= TOL[dt]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_gather_sorted_prefill(nv, dt):
    E, N, K, T, topk = 16, 64, 512, 40, 4
    w, s = weights(19, E, N, K)
    g = synth.rng(191)
    gs = synth.global_scales(g, E)
    x = synth.activations(g, (T, K), dt)
    lhs, rhs = synth.zipf_routing(g, T, E, topk)
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs), gs=f32_to_dev(gs),
                      sorted_indices=True)
    torch.cuda.synchronize()
    ref = O.gather_qmm(x.double().numpy(), lhs, rhs, w, s, gs)
    assert rel_err(y, ref) <= TOL[dt]


def test_gather_identity_lhs(nv):
    E, N, K = 4, 40, 64
    w, s = weights(29, E, N, K)
    g = synth.rng(292)
    x = synth.activations(g, (6, K), "bf16")
    rhs = np.array([3, 0, 0, 2, 9, 1], dtype=np.uint32)
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs))
    ref = O.gather_qmm(x.double().numpy(), None, rhs, w, s)
    assert rel_err(y, ref) <= TOL["bf16"]
    assert np.all(y[4].float().cpu().numpy() == 0.0)


# ------------------------------------------------------------------ tensor-core (tcgen05) route

# (4096, 8192, 64) gives every persistent CTA several tiles, so accumulator
# reuse and barrier phase wrap-around are exercised for each tile shape.
TC_SHAPES = [(1, 256, 64), (100, 272, 96), (128, 512, 256), (129, 40, 64), (300, 520, 320), (256, 256, 5376),
             (4096, 8192, 64)]


@pytest.mark.parametrize("tile", ["auto", "256x256", "256x128", "128x256"])
@pytest.mark.parametrize("mnk", TC_SHAPES, ids=lambda v: "M%d_N%d_K%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_qmm_tc_route(nv, mnk, dt, tile, opt):
    if tile != "auto":
        opt("tc_tile", tile)
    M, N, K = mnk
    w, s = weights(M + 7 * N + K, N, K, lo=2.0**-4, hi=16.0)
    g = synth.rng(M * 77 + N + K)
    x = synth.activations(g, (M, K), dt)
    for gs in (None, np.float32(2688 * 0.37)):
        y, backing, guard = guarded_empty((M, N), TORCH[dt], fill=-7.0)
        nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=None if gs is None else float(gs), route="tc", out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        ref = O.qmm(x.double().numpy(), w, s, gs)
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)


def test_qmm_tc_matches_qmv_route(nv):
    """Both routes compute the same sums: outputs agree to bf16 rounding."""
    M, N, K = 192, 384, 1024
    w, s = weights(3, N, K)
    x = synth.activations(synth.rng(33), (M, K), "bf16").cuda()
    a = nv.qmm(x, u32_to_dev(w), u8_to_dev(s), route="tc").float()
    b = nv.qmm(x, u32_to_dev(w), u8_to_dev(s), route="qmv").float()
    assert nv.take_device_error() == 0
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * b.abs().max().item()


@pytest.mark.parametrize("special", [1e-30, 1e5, -3e30, 2.0**-20])
def test_qmm_qmv_bf16_values_outside_f16(nv, special):
    """bf16 activations that f16 cannot hold exactly take the bf16 decode path;
    the result still matches the oracle (the f16 fast path is only taken when
    every staged activation converts exactly)."""
    M, N, K = 3, 272, 512
    w, s = weights(11, N, K)
    x = synth.activations(synth.rng(12), (M, K), "bf16")
    x[1, 5] = special
    x[2, 300] = special
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), route="qmv")
    ref = O.qmm(x.double().numpy(), w, s, None)
    assert rel_err(y, ref) <= TOL["bf16"]
    # rows without the special value are unaffected by it
    ref0 = O.qmm(x[:1].double().numpy(), w, s, None)
    assert rel_err(y[:1], ref0) <= TOL["bf16"]


@pytest.mark.parametrize("count", [1, 40, 200])
def test_qmm_qmv_tiny_activations_exact(nv, count):
    """Rows whose only nonzero activations are below f16's normal range.

    With up to 64 such values in a CTA's slice the f16 path adds their exact
    residuals (x - f16(x)) times the weights in f32; with more it stages bf16.
    Either way the output must match the oracle to output rounding; rounding x
    to f16 alone would be tens of percent off here.
    """
    M, N, K = 2, 384, 512
    w, s = weights(41, N, K)
    g = synth.rng(42 + count)
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    cols = g.choice(K, size=min(count, K), replace=False)
    mags = np.exp2(g.uniform(-40, -18, size=cols.size)) * g.choice([-1.0, 1.0], size=cols.size)
    x[0, torch.from_numpy(cols)] = torch.from_numpy(mags.astype(np.float32)).to(torch.bfloat16)
    x[1] = synth.activations(g, (1, K), "bf16")[0]
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), route="qmv")
    ref = O.qmm(x.double().numpy(), w, s, None)
    assert rel_err(y[:1], ref[:1]) <= TOL["bf16"], "tiny-only row"
    assert rel_err(y[1:], ref[1:]) <= TOL["bf16"], "normal row"


def test_gather_tiny_activations_exact(nv):
    E, N, K, B = 4, 128, 512, 6
    w, s = weights(43, E, N, K)
    g = synth.rng(44)
    x = synth.activations(g, (B, K), "bf16")
    x[2] = 0
    cols = g.choice(K, size=30, replace=False)
    x[2, torch.from_numpy(cols)] = torch.from_numpy(np.exp2(g.uniform(-35, -20, size=30)).astype(np.float32)).to(torch.bfloat16)
    rhs = np.array([1, 3, 1, 0, 2, 3, 1], dtype=np.uint32)
    lhs = np.array([2, 2, 0, 2, 5, 1, 2], dtype=np.uint32)
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs))
    ref = O.gather_qmm(x.double().numpy(), lhs, rhs, w, s)
    for r in range(len(rhs)):
        assert rel_err(y[r:r + 1], ref[r:r + 1]) <= TOL["bf16"], f"row {r}"


# ------------------------------------------------------------------ launch overlap (programmatic dependent launch)

@pytest.fixture
def overlap(nv):
    prev = nv.set_launch_overlap(True)
    yield
    nv.set_launch_overlap(prev)


@pytest.mark.parametrize("graph", [False, True])
def test_launch_overlap_chained_calls(nv, overlap, graph):
    """With launch overlap on, a call whose activations are the previous
    call's output still reads them only after that call has finished, and a
    call writing a buffer the previous call reads waits for that read."""
    K1, N1, N2 = 4096, 8192, 1536
    w1, s1 = weights(61, N1, K1)
    w2, s2 = weights(62, N2, N1)
    g = synth.rng(63)
    x0 = synth.activations(g, (4, K1), "bf16").cuda()
    dw1, ds1, dw2, ds2 = u32_to_dev(w1), u8_to_dev(s1), u32_to_dev(w2), u8_to_dev(s2)
    y1 = torch.empty((4, N1), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((4, N2), dtype=torch.bfloat16, device="cuda")

    def step():
        nv.qmm(x0, dw1, ds1, out=y1)  # long call
        nv.qmm(y1, dw2, ds2, out=y2)  # reads y1 (read after write)
        nv.qmm(x0, dw1, ds1, out=y1)  # rewrites y1 after the second call read it (write after read)

    torch.cuda.synchronize()
    if graph:
        step()  # warm up plans outside capture
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            step()
        y1.zero_()
        y2.zero_()
        gr.replay()
    else:
        step()
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    ref1 = O.qmm(x0.cpu().double().numpy(), w1, s1, None)
    assert rel_err(y1, ref1) <= TOL["bf16"]
    # the second call's reference takes the first call's (bf16) output as input
    ref2 = O.qmm(y1.cpu().double().numpy(), w2, s2, None)
    assert rel_err(y2, ref2) <= TOL["bf16"]


def test_launch_overlap_gather_indices_from_previous_kernel(nv, overlap):
    """Indices produced by the kernel just before the gather are read only
    after it has finished."""
    E, N, K, B, R = 32, 1536, 2048, 16, 64
    w, s = weights(71, E, N, K)
    g = synth.rng(72)
    x = synth.activations(g, (B, K), "bf16").cuda()
    base = torch.from_numpy(synth.zipf_experts(g, R, E).astype(np.int64)).cuda()
    lhs_src = torch.from_numpy(g.integers(0, B, size=R).astype(np.int64)).cuda()
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    rhs = torch.zeros(R, dtype=torch.int32, device="cuda")
    lhs = torch.zeros(R, dtype=torch.int32, device="cuda")
    for shift in range(1, 4):
        torch.cuda.synchronize()
        # elementwise kernels write the indices immediately before the gather
        rhs.copy_(((base + shift) % E).to(torch.int32))
        lhs.copy_(((lhs_src + shift) % B).to(torch.int32))
        y = nv.gather_qmm(x, dw, ds, rhs, lhs)
        torch.cuda.synchronize()
        ref = O.gather_qmm(x.cpu().double().numpy(), lhs.cpu().numpy().astype(np.uint32),
                           rhs.cpu().numpy().astype(np.uint32), w, s)
        assert rel_err(y, ref) <= TOL["bf16"], f"shift {shift}"


# ------------------------------------------------------------------ expert-batched tensor-core gather

# (E, N, K, tokens, top_k): ragged N and K with short segments; R = 16384 so
# every persistent CTA takes many tiles; 128 Zipf experts, some without rows.
GATHER_TC_CASES = [(16, 272, 96, 300, 4), (8, 1024, 64, 4096, 4), (128, 256, 256, 512, 8)]


@pytest.mark.parametrize("case", GATHER_TC_CASES, ids=lambda v: "E%d_N%d_K%d_T%d_k%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("tile", ["256x256", "128x256", "256x128"])
def test_gather_sorted_tc_route(nv, opt, case, dt, tile):
    """Every tile shape (the activation rows gathered into output order first,
    then plain 128-row boxes)."""
    opt("gather_tc", 1)
    opt("gather_tile", tile)
    E, N, K, T, topk = case
    w, s = weights(7 * E + N, E, N, K)
    g = synth.rng(E + N + K + T)
    gs = synth.global_scales(g, E)
    x = synth.activations(g, (T, K), dt)
    lhs, rhs = synth.zipf_routing(g, T, E, topk)
    lhs = lhs.copy()
    bad = g.choice(len(lhs), size=7, replace=False)
    lhs[bad[:6]] = T + np.arange(6, dtype=np.uint32)  # activation rows out of range inside segments
    lhs[bad[6]] = 2**32 - 1
    rhs = np.concatenate([rhs, np.array([E, E, E + 1, 2**32 - 1], dtype=np.uint32)])  # sorted last
    lhs = np.concatenate([lhs, np.array([0, 1, 2, 3], dtype=np.uint32)])
    R = len(rhs)
    y, backing, guard = guarded_empty((R, N), TORCH[dt], fill=-7.0)
    nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs), gs=f32_to_dev(gs),
                  sorted_indices=True, out=y)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    ref = O.gather_qmm(x.double().numpy(), lhs, rhs, w, s, gs)
    yc = y.float().cpu().numpy()
    zero = (rhs >= E) | (lhs >= T)
    assert np.all(yc[zero] == 0.0) and not np.any(np.signbit(yc[zero])), "out-of-range rows must be +0.0"
    assert rel_err(y, ref) <= TOL[dt]
    assert guards_intact(backing, guard)


def test_gather_sorted_tc_identity_lhs(nv, opt):
    """Without lhs, row r reads x[r]; rows at or past B are +0.0."""
    opt("gather_tc", 1)
    E, N, K, R = 32, 256, 128, 2048
    w, s = weights(81, E, N, K)
    g = synth.rng(82)
    B = R - 3
    x = synth.activations(g, (B, K), "bf16")
    rhs = np.sort(synth.zipf_experts(g, R, E))
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), sorted_indices=True)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    ref = O.gather_qmm(x.double().numpy(), None, rhs, w, s)
    assert rel_err(y, ref) <= TOL["bf16"]
    assert np.all(y[B:].float().cpu().numpy() == 0.0)


def test_gather_sorted_tc_matches_decode_route(nv, opt):
    """The expert-batched and the decode-shape gather compute the same sums."""
    E, N, K, T, topk = 64, 512, 512, 1024, 4
    w, s = weights(91, E, N, K)
    g = synth.rng(92)
    x = synth.activations(g, (T, K), "bf16").cuda()
    lhs, rhs = synth.zipf_routing(g, T, E, topk)
    args = (x, u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs))
    opt("gather_tc", 1)
    a = nv.gather_qmm(*args, sorted_indices=True).float()
    opt("gather_tc", 0)
    b = nv.gather_qmm(*args, sorted_indices=True).float()
    assert nv.take_device_error() == 0
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * b.abs().max().item()


def test_gather_sorted_tc_two_calls(nv, opt):
    """About 160 expert tiles of 16 k-blocks on 152 CTAs (a second, partial
    wave), an activation index out of range inside a segment; every row
    against the oracle, twice in a row (the row buffer is reused)."""
    opt("gather_tc", 1)
    E, N, K, T, topk = 16, 1024, 1024, 2048, 4
    w, s = weights(61, E, N, K)
    g = synth.rng(62)
    gs = synth.global_scales(g, E)
    x = synth.activations(g, (T, K), "bf16")
    lhs, rhs = synth.zipf_routing(g, T, E, topk)
    lhs = lhs.copy()
    lhs[5] = T  # an activation row out of range inside a segment
    ref = O.gather_qmm(x.double().numpy(), lhs, rhs, w, s, gs)
    args = (x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs))
    for rep in range(2):
        y, backing, guard = guarded_empty((len(rhs), N), torch.bfloat16, fill=-7.0)
        nv.gather_qmm(*args, gs=f32_to_dev(gs), sorted_indices=True, out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        assert rel_err(y, ref) <= TOL["bf16"], f"call {rep}"
        assert guards_intact(backing, guard)
        yc = y[5].float().cpu().numpy()
        assert np.all(yc == 0.0) and not np.any(np.signbit(yc))


def test_gather_sorted_tc_moe_prefill_full_size(nv):
    """The MoE gate/up prefill: 4096 tokens, top-8 Zipf(1.1) routing over 128
    experts, rows sorted by expert; sampled rows against the oracle."""
    E, N, K, T = 128, 1536, 2048, 4096
    g = synth.rng(4242)
    w = synth.packed_weight(g, E, N, K)
    s = synth.log_uniform_scales(g, (E, N, K // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, E)
    x = synth.activations(g, (T, K), "bf16")
    lhs, rhs = synth.zipf_routing(g, T, E, 8)
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs), gs=f32_to_dev(gs),
                      sorted_indices=True)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    # first and last rows of every expert segment plus a random sample
    starts = np.searchsorted(rhs, np.arange(E + 1))
    pick = np.unique(np.concatenate([starts[:-1], np.maximum(starts[1:] - 1, 0),
                                     g.choice(len(rhs), size=256, replace=False)]))
    pick = pick[pick < len(rhs)]
    ref = O.gather_qmm(x.double().numpy(), lhs[pick], rhs[pick], w, s, gs)
    assert rel_err(y[torch.from_numpy(pick).cuda()], ref) <= TOL["bf16"]


def test_gather_sorted_tc_moe_down_prefill_full_size(nv):
    """The MoE down prefill: the 32768 gate/up output rows (4096 tokens, top-8
    Zipf(1.1) over 128 experts, sorted by expert) taken in order (identity
    activation indices) through [128, 2048, 768]; sampled rows against the
    oracle."""
    E, N, K, T = 128, 2048, 768, 4096
    g = synth.rng(4343)
    w = synth.packed_weight(g, E, N, K)
    s = synth.log_uniform_scales(g, (E, N, K // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, E)
    _, rhs = synth.zipf_routing(g, T, E, 8)
    x = synth.activations(g, (rhs.size, K), "bf16")
    y = nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), None, gs=f32_to_dev(gs),
                      sorted_indices=True)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    starts = np.searchsorted(rhs, np.arange(E + 1))
    pick = np.unique(np.concatenate([starts[:-1], np.maximum(starts[1:] - 1, 0),
                                     g.choice(len(rhs), size=256, replace=False)]))
    pick = pick[pick < len(rhs)]
    ref = O.gather_qmm(x.double().numpy(), pick.astype(np.uint32), rhs[pick], w, s, gs)
    assert rel_err(y[torch.from_numpy(pick).cuda()], ref) <= TOL["bf16"]


# The prefill configuration at full size, through the automatic route (whole
# tensor-core tiles: 17.7 and 4.4 waves of 256 x 256 tiles on 152 SMs):
# M = 8192 and M = 2048 on [21504, 5376]; sampled outputs against the oracle.
@pytest.mark.parametrize("mnk", [(8192, 21504, 5376), (2048, 21504, 5376)], ids=lambda v: "M%d_N%d_K%d" % v)
def test_prefill_full_size_sampled(nv, mnk):
    M, N, K = mnk
    g = synth.rng(M + 2 * N)
    w = synth.packed_weight(g, N, K)
    s = synth.log_uniform_scales(g, (N, K // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, 1)[0]
    x = synth.activations(g, (M, K), "bf16")
    y = nv.qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), gs=float(gs))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    yc = y.double().cpu().numpy()
    assert np.isfinite(yc).all()
    pick = synth.rng(N + M + 3)
    rows = np.concatenate([pick.integers(0, M, size=700), np.arange(M - 10, M), np.zeros(10, dtype=np.int64)])
    cols = np.concatenate([pick.integers(0, N, size=700), np.arange(N - 10, N), np.arange(10)])
    ref = O.qmm_entries(x.double().numpy(), w, s, gs, rows, cols)
    assert np.max(np.abs(yc[rows, cols] - ref)) <= TOL["bf16"] * np.max(np.abs(ref))


def test_transcode_sixty_layers(nv):
    """The 60-layer transcode workload: every layer's three ModelOpt triplets
    ([43008, 5376], [5376, 21504], [8192, 5376]; 13.2 GB in all) resident on
    the device and transcoded in one pass; then, layer by layer, each native
    plane and sidecar compared bit for bit with the oracle's transcode of the
    same input bytes, and the first 64 rows of each plane dequantized (bf16)
    bit for bit against the oracle."""
    dev = torch.device("cuda")
    lin = [(43008, 5376), (5376, 21504), (8192, 5376)]
    layers = []
    for layer in range(60):
        trip = []
        for j, (n, k) in enumerate(lin):
            mo_w, mo_s, ws2 = synth.device_modelopt_triplet(5000 + 3 * layer + j, n, k, dev)
            out = (torch.empty((n, k // 8), dtype=torch.int32, device=dev),
                   torch.empty((n, k // 16), dtype=torch.uint8, device=dev),
                   torch.empty((1,), dtype=torch.float32, device=dev))
            trip.append((mo_w, mo_s, ws2, f32_to_dev(ws2), out))
        layers.append(trip)
    for trip in layers:
        for (mo_w, mo_s, _, ws2_d, out) in trip:
            nv.transcode(mo_w, mo_s, ws2_d, out=out)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    for layer, trip in enumerate(layers):
        for j, (mo_w, mo_s, ws2, _, out) in enumerate(trip):
            hw, hs = mo_w.cpu().numpy(), mo_s.cpu().numpy()
            rw, rs, rg = O.transcode(hw, hs, ws2)
            assert np.array_equal(out[0].cpu().numpy().view(np.uint32), rw), (layer, j)
            assert np.array_equal(out[1].cpu().numpy(), rs), (layer, j)
            assert out[2].cpu().numpy()[0] == rg, (layer, j)
            deq = nv.dequantize(out[0][:64], out[1][:64], out[2], torch.bfloat16)
            ref = O.dequantize(rw[:64], rs[:64], rg, "bf16")
            assert torch.equal(deq.cpu().view(torch.int16), ref.view(torch.int16)), (layer, j)
        layers[layer] = None  # frees the layer's device planes


def test_gather_tc_unsorted_promise_is_memory_safe(nv, opt):
    """Indices that break the sorted promise still write every row once and
    read nothing out of range (values are then unspecified)."""
    opt("gather_tc", 1)
    E, N, K, T = 8, 256, 64, 600
    w, s = weights(95, E, N, K)
    g = synth.rng(96)
    x = synth.activations(g, (T, K), "bf16")
    rhs = g.integers(0, E + 2, size=T).astype(np.uint32)  # unsorted, some out of range
    y, backing, guard = guarded_empty((T, N), torch.bfloat16, fill=-7.0)
    nv.gather_qmm(x.cuda(), u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), sorted_indices=True, out=y)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert guards_intact(backing, guard)
    assert torch.isfinite(y.float()).all()
    assert not (y.float() == -7.0).all(dim=1).any(), "a row was left unwritten"
