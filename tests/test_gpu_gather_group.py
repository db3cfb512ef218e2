"""GPU parity of the expert-group decode route of GatherQMM against the oracle.

Unsorted GatherQMM calls with at most one row per SM (16-bit activations, K a
multiple of 256) run on the persistent decode kernel as expert groups: every
CTA groups the rows by expert index (eight to a group, in row order) and the
CTAs of a group split that expert's plane. The cases cover ragged N, one to
many chunks, several groups of one expert, rows without an expert (exact
+0.0), a call whose rows all lack one, back-to-back calls (the workspace must
come back clean), agreement with the per-row route, graph replay and the MoE
decode linears at full size.
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


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def f32_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def routing(g, R, E, B, kind):
    """Expert and activation indices for R rows (uint32), with a few rows
    that belong to no expert."""
    if kind == "zipf":
        rhs = synth.zipf_experts(g, R, E)
    elif kind == "one_expert":  # R rows of one expert: ceil(R / 8) groups of it
        rhs = np.full(R, E // 2, dtype=np.uint32)
    else:  # every row its own expert where E allows
        rhs = (np.arange(R, dtype=np.uint32) * 7) % np.uint32(E)
    lhs = g.integers(0, B, size=R).astype(np.uint32)
    if R >= 6:
        rhs[1], rhs[R // 2], rhs[-1] = E, E + 1, 2**32 - 1
        lhs[3] = B  # activation index out of range
    return rhs.astype(np.uint32), lhs


# (E, N, K): ragged row tiles, one to sixteen chunks
GROUP_SHAPES = [(8, 1000, 768), (16, 1536, 2048), (4, 300, 4096), (32, 256, 256)]


@pytest.mark.parametrize("enk", GROUP_SHAPES, ids=lambda v: "E%d_N%d_K%d" % v)
@pytest.mark.parametrize("R", [1, 7, 9, 66, "sms"])
@pytest.mark.parametrize("kind", ["zipf", "one_expert", "spread"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_group_route_parity(nv, enk, R, kind, dt):
    E, N, K = enk
    R = sms() if R == "sms" else R
    B = 40
    w, s = weights(E + N + K + R, E, N, K)
    g = synth.rng(7 * N + K + R)
    x = synth.activations(g, (B, K), dt).cuda()
    rhs, lhs = routing(g, R, E, B, kind)
    gs = synth.global_scales(g, E)
    dw, ds, drhs, dlhs = u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs)
    ref = O.gather_qmm(x.cpu().double().numpy(), lhs, rhs, w, s, gs)
    zero_rows = [r for r in range(R) if rhs[r] >= E or lhs[r] >= B]
    for rep in range(2):  # the second call finds the workspace as the first left it
        y, backing, guard = guarded_empty((R, N), TORCH[dt], fill=-7.0)
        nv.gather_qmm(x, dw, ds, drhs, dlhs, gs=f32_to_dev(gs), out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        err = rel_err(y, ref)
        assert err <= TOL[dt], f"call {rep}: rel-to-max error {err:.3g} > {TOL[dt]}"
        assert guards_intact(backing, guard)
        yc = y.float().cpu().numpy()
        for r in zero_rows:
            assert np.all(yc[r] == 0.0) and not np.any(np.signbit(yc[r])), f"row {r} must be +0.0"


def test_group_route_identity_lhs_no_gs(nv):
    E, N, K, R = 12, 520, 512, 30
    w, s = weights(5, E, N, K)
    g = synth.rng(55)
    x = synth.activations(g, (R, K), "bf16").cuda()
    rhs = synth.zipf_experts(g, R, E)
    rhs[4] = E
    y = nv.gather_qmm(x, u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs))
    torch.cuda.synchronize()
    ref = O.gather_qmm(x.cpu().double().numpy(), None, rhs, w, s)
    assert rel_err(y, ref) <= TOL["bf16"]
    assert np.all(y[4].float().cpu().numpy() == 0.0)


def test_group_route_no_valid_rows(nv):
    """Every row lacks an expert: no group, every output row +0.0."""
    E, N, K, R = 4, 256, 512, 10
    w, s = weights(6, E, N, K)
    x = synth.activations(synth.rng(66), (R, K), "f16").cuda()
    rhs = np.array([E, E + 1, 2**32 - 1] * 3 + [E], dtype=np.uint32)
    y = torch.full((R, N), -7.0, dtype=torch.float16, device="cuda")
    nv.gather_qmm(x, u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), out=y)
    torch.cuda.synchronize()
    yc = y.float().cpu().numpy()
    assert np.all(yc == 0.0) and not np.any(np.signbit(yc))


def test_group_route_matches_row_route(nv, opt):
    """The expert-group and the per-row decode kernels compute the same sums."""
    E, N, K, R, B = 32, 1536, 2048, 64, 64
    w, s = weights(8, E, N, K)
    g = synth.rng(88)
    x = synth.activations(g, (B, K), "bf16").cuda()
    rhs, lhs = routing(g, R, E, B, "zipf")
    gs = f32_to_dev(synth.global_scales(g, E))
    args = (x, u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs))
    a = nv.gather_qmm(*args, gs=gs).float()
    opt("gather_group", 0)
    b = nv.gather_qmm(*args, gs=gs).float()
    torch.cuda.synchronize()
    scale = b.abs().max().item()
    assert (a - b).abs().max().item() <= 8e-3 * scale


@pytest.mark.parametrize("warm", [False, True])
def test_group_route_graph_replay(nv, warm):
    """Captured into a CUDA graph (on torch's capture stream, whose workspace
    is made during the capture unless a call came first) and replayed."""
    E, N, K, R, B = 16, 1000, 768, 40, 40
    w, s = weights(9, E, N, K)
    g = synth.rng(99)
    x = synth.activations(g, (B, K), "bf16").cuda()
    rhs, lhs = routing(g, R, E, B, "zipf")
    dw, ds, drhs, dlhs = u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), u32_to_dev(lhs)
    y = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
    if warm:
        nv.gather_qmm(x, dw, ds, drhs, dlhs, out=y)
        torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        nv.gather_qmm(x, dw, ds, drhs, dlhs, out=y)
    ref = O.gather_qmm(x.cpu().double().numpy(), lhs, rhs, w, s)
    for _ in range(3):
        y.fill_(-7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        assert rel_err(y, ref) <= TOL["bf16"]


@pytest.mark.parametrize("name,n,k", [("gate_up", 1536, 2048), ("down", 2048, 768)])
def test_group_route_moe_decode_full_size(nv, name, n, k):
    """The MoE decode linears: 128 experts, 64 Zipf(1.1)-routed rows plus rows
    for experts E and E+1 (zeros)."""
    E = 128
    g = synth.rng(1234 + n)
    w = synth.packed_weight(g, E, n, k)
    s = synth.log_uniform_scales(g, (E, n, k // 16), 2.0**-6, 4.0)
    gs = synth.global_scales(g, E)
    rhs = np.concatenate([synth.zipf_experts(g, 64, E), np.array([E, E + 1], dtype=np.uint32)])
    x = synth.activations(g, (66, k), "bf16").cuda()
    y = nv.gather_qmm(x, u32_to_dev(w), u8_to_dev(s), u32_to_dev(rhs), gs=f32_to_dev(gs))
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    ref = O.gather_qmm(x.cpu().double().numpy(), None, rhs, w, s, gs)
    assert rel_err(y, ref) <= TOL["bf16"]
    yc = y.float().cpu().numpy()
    assert np.all(yc[64:] == 0.0) and not np.any(np.signbit(yc[64:]))
