"""GPU parity of nvfp4_qmm_sequence: several decode-shape QuantizedMatmuls in
one persistent launch, each checked against the CPU oracle.

Cases: mixed shapes and token counts (1..16 rows, gs present or absent) in
both 16-bit dtypes, launched twice in a row; the 15 calls of the decode step
(gate/up [43008, 5376], down [5376, 21504], qkv [8192, 5376] at M = 1, 2, 4,
8, 16) at full size on sampled outputs; a dependent chain (each call's
activations are an earlier call's outputs, after_previous set) against the
oracle's chain with the outputs rounded to the activation dtype in between,
launched twice (the completion counters must be back at zero), with an
independent call between the links; agreement with single nvfp4_qmm calls;
replay in a CUDA graph; empty calls skipped.
"""
import numpy as np
import pytest
import torch

from nvfp4_quantized_matmul_gb300 import synth
from oracle import nvfp4_oracle as O

from nvutil import TOL, TORCH, rel_err, u32_to_dev, u8_to_dev, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


def reference(x, w, s, gs, seed):
    """Oracle outputs: all of them for small planes, else a sample (every
    token row against the first and last weight rows and 192 random ones).
    Returns (index or None, values)."""
    xd = x.double().cpu().numpy()
    n = w.shape[0]
    if n * w.shape[1] * 8 <= 1 << 21:
        return None, O.qmm(xd, w, s, gs)
    g = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([[0, n - 1], g.integers(0, n, size=192)]))
    rows = np.repeat(np.arange(xd.shape[0]), cols.size)
    cc = np.tile(cols, xd.shape[0])
    return (rows, cc), O.qmm_entries(xd, w, s, gs, rows, cc)


def compare(y, ref, dt, what):
    pick, vals = ref
    yc = y.double().cpu().numpy()
    got = yc if pick is None else yc[pick]
    err = O.rel_to_max_error(got, vals)
    assert err <= TOL[dt], f"{what}: rel-to-max error {err:.3g} > {TOL[dt]}"


def make_calls(shapes, dt, seed):
    calls, refs = [], []
    for i, (n, k, m, with_gs) in enumerate(shapes):
        w, s = weights(seed + 17 * i + n, n, k)
        x = synth.activations(synth.rng(seed + 31 * i + m), (m, k), dt).cuda()
        gs = np.float32(synth.global_scales(synth.rng(seed + i), 1)[0]) if with_gs else None
        gsd = None if gs is None else torch.tensor([float(gs)], dtype=torch.float32, device="cuda")
        calls.append((x, u32_to_dev(w), u8_to_dev(s), gsd, None, False))
        refs.append(reference(x, w, s, gs, seed + i))
    return calls, refs


MIXED = [(3000, 4096, 1, True), (2304, 2560, 16, False), (257, 256, 9, True), (5376, 21504, 4, True),
         (1024, 1024, 2, False), (4096, 2048, 8, True), (512, 5376, 3, True), (8192, 5376, 13, False)]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_sequence_mixed_shapes_twice(nv, dt):
    calls, refs = make_calls(MIXED, dt, 100)
    for launch in range(2):
        outs = nv.qmm_sequence(calls)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        for i, (y, ref) in enumerate(zip(outs, refs)):
            compare(y, ref, dt, f"launch {launch} call {i} {MIXED[i][:3]}")


def test_sequence_decode_step_full_size(nv):
    """The decode step's 15 calls at full size, bf16, per-linear gs."""
    lin = [(43008, 5376), (5376, 21504), (8192, 5376)]
    shapes = [(n, k, m, True) for m in (1, 2, 4, 8, 16) for (n, k) in lin]
    # one weight plane per linear, shared by the five token counts
    planes = {}
    calls, refs = [], []
    for i, (n, k, m, _) in enumerate(shapes):
        if (n, k) not in planes:
            w, s = weights(n + k, n, k)
            gs = np.float32(synth.global_scales(synth.rng(n), 1)[0])
            planes[(n, k)] = (w, s, gs, u32_to_dev(w), u8_to_dev(s),
                              torch.tensor([float(gs)], dtype=torch.float32, device="cuda"))
        w, s, gs, dw, ds, gsd = planes[(n, k)]
        x = synth.activations(synth.rng(7 * i + m), (m, k), "bf16").cuda()
        calls.append((x, dw, ds, gsd, None, False))
        refs.append(reference(x, w, s, gs, i))
    outs = nv.qmm_sequence(calls)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    for i, (y, ref) in enumerate(zip(outs, refs)):
        compare(y, ref, "bf16", f"call {i} {shapes[i][:3]}")


def oracle_chain(x, links, dt):
    """The chain's outputs by the oracle, each rounded to the activation
    dtype (RNE) before it feeds the next link, as the library stores it."""
    outs = []
    cur = x.double().cpu().numpy()
    for (w, s, gs) in links:
        y = O.qmm(cur, w, s, gs)
        yt = torch.from_numpy(y).to(TORCH[dt])
        outs.append(y)
        cur = yt.double().numpy()
    return outs


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("m", [1, 5, 16])
def test_sequence_dependent_chain(nv, dt, m):
    """x -> y1 -> y2 -> y3, each link reading the previous output
    (after_previous), with an independent call between the links, launched
    twice."""
    dims = [2048, 1536, 2816, 1024]  # K of link 1, then each link's N (= next K)
    links, dev_links = [], []
    for i in range(3):
        k, n = dims[i], dims[i + 1]
        w, s = weights(500 + i, n, k, lo=2.0**-9, hi=2.0**-5)
        gs = np.float32(2688.0 * (0.5 + 0.25 * i))
        links.append((w, s, gs))
        dev_links.append((u32_to_dev(w), u8_to_dev(s), torch.tensor([float(gs)], dtype=torch.float32, device="cuda")))
    x = synth.activations(synth.rng(600 + m), (m, dims[0]), dt).cuda()
    ind_w, ind_s = weights(700, 1280, 2048)
    ind_x = synth.activations(synth.rng(701), (m, 2048), dt).cuda()
    ref_links = oracle_chain(x, links, dt)
    ref_ind = O.qmm(ind_x.double().cpu().numpy(), ind_w, ind_s, None)
    ys = [torch.empty((m, dims[i + 1]), dtype=TORCH[dt], device="cuda") for i in range(3)]
    y_ind = torch.empty((m, 1280), dtype=TORCH[dt], device="cuda")
    di = (ind_x, u32_to_dev(ind_w), u8_to_dev(ind_s), None, y_ind, False)
    calls = [(x, *dev_links[0], ys[0], False), di,
             (ys[0], *dev_links[1], ys[1], True),
             (ys[1], *dev_links[2], ys[2], True)]
    for launch in range(2):
        for y in ys + [y_ind]:
            y.fill_(7.0)
        nv.qmm_sequence(calls)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        for i in range(3):
            err = O.rel_to_max_error(ys[i].double().cpu().numpy(), ref_links[i])
            assert err <= TOL[dt], f"launch {launch} link {i}: rel-to-max error {err:.3g}"
        assert rel_err(y_ind, ref_ind) <= TOL[dt]


def test_sequence_agrees_with_single_calls_and_replays_in_a_graph(nv):
    shapes = [(2304, 2560, 16, True), (3000, 4096, 1, False), (1024, 1024, 7, True)]
    calls, refs = make_calls(shapes, "bf16", 900)
    outs = [torch.empty((c[0].shape[0], c[1].shape[0]), dtype=torch.bfloat16, device="cuda") for c in calls]
    calls = [(x, w, s, gs, y, a) for (x, w, s, gs, _, a), y in zip(calls, outs)]
    singles = [nv.qmm(x, w, s, gs=gs) for (x, w, s, gs, _, _) in calls]
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        nv.qmm_sequence(calls)  # warm: plans and workspace outside the capture
        torch.cuda.synchronize()
        for y in outs:
            y.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            nv.qmm_sequence(calls)
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    for i, (y, ref, single) in enumerate(zip(outs, refs, singles)):
        compare(y, ref, "bf16", f"graph call {i}")
        assert rel_err(y, single.double().cpu().numpy()) <= TOL["bf16"]


def test_sequence_skips_empty_calls(nv):
    """A call with no token rows is skipped; the call after it (whose
    after_previous then has nothing to wait for) still runs."""
    calls, refs = make_calls([(512, 1024, 3, True)], "f16", 950)
    x, w, s, gs, _, _ = calls[0]
    y = torch.full((3, 512), 5.0, dtype=torch.float16, device="cuda")
    outs = nv.qmm_sequence([(x[:0], w, s, gs, None, False), (x, w, s, gs, y, True)])
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    assert outs[0].shape == (0, 512)
    compare(y, refs[0], "f16", "call after an empty one")
