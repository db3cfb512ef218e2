"""The stall path of the decode kernel's bounded waits, made to run out on
purpose (no fault, no trap, no hang: every wait of the kernel has a limit).

With the test options set, consumer warp 0 of the first CTA withholds its
release of the first pipeline stage it reads, so that its producer's wait
for that stage, and the waits of the CTA's other roles after it, run out
after the shortened limit (1 ms). The call must come back within a bound,
nvfp4_take_device_error must report one of the decode kernel's wait codes,
and the next normal call on the same stream must match the oracle (the
error read clears the workspace the aborted call left behind).
"""
import time

import numpy as np
import pytest
import torch

from nvfp4_quantized_matmul_gb300 import synth
from oracle import nvfp4_oracle as O

from nvutil import TOL, u32_to_dev, u8_to_dev, weights

pytestmark = pytest.mark.gpu

# error codes of the decode kernel's bounded waits (csrc/nvfp4_qmv_stream.cu)
DECODE_WAIT_CODES = set(range(21, 28))


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge

    ge.build()
    import nvfp4_quantized_matmul_gb300 as pkg

    return pkg


def test_bounded_wait_runs_out_and_the_next_call_is_correct(nv, opt):
    # 32 row tiles x 64 chunks: each CTA streams more chunks than its ring
    # holds, so the producer comes back to the withheld stage
    N, K = 8192, 16384
    w, s = weights(31, N, K)
    dw, ds = u32_to_dev(w), u8_to_dev(s)
    x = synth.activations(synth.rng(32), (1, K), "bf16").cuda()
    gs = np.float32(2688 * 0.8)
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    opt("wait_limit_us", 1000)
    opt("test_withhold", 1)
    t0 = time.perf_counter()
    nv.qmm(x, dw, ds, gs=float(gs), route="qmv")
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    code = nv.take_device_error()
    assert code in DECODE_WAIT_CODES, f"device error {code}"
    assert elapsed < 1.0, f"the stalled call took {elapsed:.3f} s"
    opt("test_withhold", 0)
    opt("wait_limit_us", 0)
    y = nv.qmm(x, dw, ds, gs=float(gs), route="qmv")
    torch.cuda.synchronize()
    assert nv.take_device_error() == 0
    pick = synth.rng(33)
    cols = np.concatenate([pick.integers(0, N, size=300), [0, N - 1]])
    rows = np.zeros_like(cols)
    ref = O.qmm_entries(x.double().cpu().numpy(), w, s, gs, rows, cols)
    got = y.double().cpu().numpy()[rows, cols]
    assert np.max(np.abs(got - ref)) <= TOL["bf16"] * np.max(np.abs(ref))
