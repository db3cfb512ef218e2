"""GPU parity of QuantizedMatmul with batched weights (``nvfp4_qmm_batched``)
against the oracle, batch by batch.

Decode-size calls with at most one row per SM run as one launch of the
expert-group decode route (row r of the flattened activations uses batch
r / M's plane); the others run one QuantizedMatmul per batch (decode or
tensor-core route). The cases cover both, ragged N, the per-batch global
scale and back-to-back calls.
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


def f32_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


# (batches, M, N, K): one group launch (32 and 3 rows), per-batch decode calls
# (160 rows: more than one per SM), per-batch tensor-core calls (M = 300)
CASES = [(8, 4, 1536, 2048), (3, 1, 1000, 768), (40, 4, 264, 256), (2, 300, 512, 512)]


@pytest.mark.parametrize("case", CASES, ids=lambda v: "B%d_M%d_N%d_K%d" % v)
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("with_gs", [False, True])
def test_batched_parity(nv, case, dt, with_gs):
    bt, M, N, K = case
    w, s = weights(bt + M + N + K, bt, N, K)
    g = synth.rng(bt * 7 + M + N + K)
    x = synth.activations(g, (bt * M, K), dt).reshape(bt, M, K)
    gs = synth.global_scales(g, bt) if with_gs else None
    ref = np.stack([O.qmm(x[b].double().numpy(), w[b], s[b], None if gs is None else gs[b]) for b in range(bt)])
    dx, dw, ds = x.cuda(), u32_to_dev(w), u8_to_dev(s)
    dgs = None if gs is None else f32_to_dev(gs)
    for rep in range(2):
        y, backing, guard = guarded_empty((bt, M, N), TORCH[dt], fill=-7.0)
        nv.qmm_batched(dx, dw, ds, gs=dgs, out=y)
        torch.cuda.synchronize()
        assert nv.take_device_error() == 0
        for b in range(bt):
            err = rel_err(y[b], ref[b])
            assert err <= TOL[dt], f"call {rep}, batch {b}: rel-to-max error {err:.3g}"
        assert guards_intact(backing, guard)


def test_batched_group_launch_matches_per_batch_calls(nv, opt):
    """The one-launch route and one call per batch compute the same sums."""
    bt, M, N, K = 16, 2, 2048, 768
    w, s = weights(5, bt, N, K)
    x = synth.activations(synth.rng(6), (bt * M, K), "bf16").reshape(bt, M, K).cuda()
    args = (x, u32_to_dev(w), u8_to_dev(s))
    a = nv.qmm_batched(*args).float()
    opt("gather_group", 0)
    b = nv.qmm_batched(*args).float()
    torch.cuda.synchronize()
    assert (a - b).abs().max().item() <= 2 * 2.0**-8 * b.abs().max().item()
