"""Pins for the CPU oracle: checks against the pages, closed forms and exact arithmetic.

Each ``pin_*`` function takes the oracle module so that ``test_planted_*``
can run it against a copy with a deliberate mistake and show that the pin
notices. All tests here are CPU-only.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.nvfp4_oracle as O
from nvfp4_quantized_matmul_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- independent decoders

def frac_e2m1(c: int) -> Fraction:
    """E2M1 from its bit layout: sign(1) exponent(2, bias 1) mantissa(1)."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -mag if s else mag


def frac_e4m3(b: int):
    """E4M3FN from its bit layout (None for NaN)."""
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return None
    mag = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -mag if s else mag


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack codes [.., K] into words [.., K/8], column 8j+i in nibble i (test's own packer)."""
    codes = np.asarray(codes, dtype=np.int64)
    k = codes.shape[-1]
    c = codes.reshape(*codes.shape[:-1], k // 8, 8)
    w = np.zeros(c.shape[:-1], dtype=np.int64)
    for i in range(8):
        w |= c[..., i] << (4 * i)
    return w.astype(np.uint32)


# ---------------------------------------------------------------- pins

def pin_e2m1_table(orc):
    table = {int(c): float(v) for c, v in _read_table("e2m1_table.txt")}
    got = orc.e2m1_value(np.arange(16))
    for c in range(16):
        assert got[c] == table[c], (c, got[c], table[c])
        # the sign of zero matters: code 8 is -0.0
        assert np.signbit(got[c]) == (c >= 8), c
        assert got[c] == float(frac_e2m1(c))


def pin_e4m3_all_bytes(orc):
    b = np.arange(256)
    got = orc.e4m3_value(b)
    lib = torch.from_numpy(b.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], lib[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(lib[~nan]))
    for v in range(256):
        f = frac_e4m3(v)
        assert (f is None) == np.isnan(got[v])
        if f is not None:
            assert got[v] == float(f)
    assert got[0x7E] == 448.0 and got[0x01] == 2.0**-9 and got[0x38] == 1.0


def pin_packing(orc):
    w = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert orc.unpack_codes(w).tolist() == [list(range(16))]
    g = synth.rng(11)
    codes = g.integers(0, 16, size=(3, 64))
    assert np.array_equal(orc.unpack_codes(pack_codes(codes)), codes)


def pin_block_scale_broadcast(orc):
    # every code 2 (= 1.0); scale of group j is 2^(j-2): value at column k is 2^(k//16 - 2)
    n, k = 2, 64
    w = pack_codes(np.full((n, k), 2))
    sbytes = synth.e4m3_bytes(np.array([[2.0 ** (j - 2) for j in range(k // 16)]] * n))
    v = orc.block_values(w, sbytes)
    expect = np.array([2.0 ** (c // 16 - 2) for c in range(k)])
    assert np.array_equal(v, np.broadcast_to(expect, (n, k)))


def _brute_force_qmm(x, codes, sbytes, gs):
    """Exact-rational y = factor * x @ (fp4 * e4m3).T, factor = RN_f32(gs/2688)."""
    m_, k = x.shape
    n = codes.shape[0]
    fac = Fraction(1) if gs is None else Fraction(float(np.float32(np.float32(gs) / np.float32(2688))))
    y = np.empty((m_, n), dtype=np.float64)
    for m in range(m_):
        for j in range(n):
            acc = Fraction(0)
            for c in range(k):
                acc += Fraction(float(x[m, c])) * frac_e2m1(int(codes[j, c])) * frac_e4m3(int(sbytes[j, c // 16]))
            y[m, j] = float(acc * fac)
    return y


def pin_brute_force_matmul(orc):
    g = synth.rng(5)
    for gs in (None, np.float32(26.88)):
        m, n, k = 3, 5, 48
        codes = g.integers(0, 16, size=(n, k))
        sbytes = synth.log_uniform_scales(g, (n, k // 16), 2.0**-4, 2.0**4)
        x = synth.activations(g, (m, k), "bf16").double().numpy()
        got = orc.qmm(x, pack_codes(codes), sbytes, gs)
        ref = _brute_force_qmm(x, codes, sbytes, gs)
        # float64 accumulation of at most 48 dyadic terms: well inside 1e-12 of max
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def pin_qmm_entries(orc):
    # the per-entry products used for sampled full-size checks equal the
    # exact-rational brute force at the same (row, column) pairs
    g = synth.rng(6)
    m, n, k = 4, 7, 64
    codes = g.integers(0, 16, size=(n, k))
    sbytes = synth.log_uniform_scales(g, (n, k // 16), 2.0**-4, 2.0**4)
    x = synth.activations(g, (m, k), "bf16").double().numpy()
    gs = np.float32(123.0)
    ref = _brute_force_qmm(x, codes, sbytes, gs)
    rows = np.array([0, 3, 2, 1, 3])
    cols = np.array([6, 0, 3, 5, 6])
    got = orc.qmm_entries(x, pack_codes(codes), sbytes, gs, rows, cols)
    assert np.max(np.abs(got - ref[rows, cols])) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def pin_one_hot(orc):
    # unit scales and one-hot activations pick out single table entries
    n, k = 16, 32
    codes = np.arange(n * k).reshape(n, k) % 16
    sbytes = np.full((n, k // 16), 0x38, dtype=np.uint8)
    for col in (0, 7, 8, 31):
        x = np.zeros((1, k))
        x[0, col] = 1.0
        y = orc.qmm(x, pack_codes(codes), sbytes, None)
        table = {int(c): float(v) for c, v in _read_table("e2m1_table.txt")}
        assert y[0].tolist() == [table[int(codes[j, col])] for j in range(n)]


def pin_global_factor(orc):
    divisor = int(_read_table("global_scale_convention.txt")[0][0])
    g = synth.rng(3)
    for gs in list(synth.global_scales(g, 200)) + [np.float32(2688.0), np.float32(26.88)]:
        f = orc.global_factor(gs)
        assert f.dtype == np.float32
        exact = Fraction(float(gs)) / divisor
        # round-to-nearest float32: error at most half an ulp of the result
        ulp = Fraction(float(np.spacing(np.float32(f))))
        assert abs(Fraction(float(f)) - exact) <= ulp / 2
    assert orc.global_factor(np.float32(2688.0)) == 1.0
    assert orc.global_factor(None) == 1.0


def _bf16_rne_bits(f32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest even, written with integer ops."""
    u = f32.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(f32)
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def pin_dequantize_rounding(orc):
    g = synth.rng(9)
    n, k = 8, 64
    w = synth.packed_weight(g, n, k)
    s = synth.log_uniform_scales(g, (n, k // 16), 2.0**-6, 4.0)
    exact = orc.block_values(w, s)
    # without gs the dequantize is exact in every dtype
    for dt in ("f32", "f16", "bf16"):
        d = orc.dequantize(w, s, None, dt).double().numpy()
        assert np.array_equal(d, exact)
        assert np.array_equal(np.signbit(d), np.signbit(exact))
    gs = np.float32(1234.5)
    fac = np.float32(gs) / np.float32(2688)
    f32 = (exact.astype(np.float32) * fac).astype(np.float32)
    assert np.array_equal(orc.dequantize(w, s, gs, "f32").numpy().view(np.uint32), f32.view(np.uint32))
    assert np.array_equal(orc.dequantize(w, s, gs, "f16").numpy().view(np.uint16),
                          f32.astype(np.float16).view(np.uint16))
    assert np.array_equal(orc.dequantize(w, s, gs, "bf16").view(torch.uint16).numpy(), _bf16_rne_bits(f32))


def pin_sidecar_identity(orc):
    """native-with-sidecar dequantize reproduces ModelOpt's fp4 * e4m3(ws) * ws2."""
    g = synth.rng(21)
    exact_hits = total = 0
    for _ in range(40):
        mo_w, mo_ws, ws2 = synth.modelopt_triplet(g, 4, 64)
        w, s, gs = orc.transcode(mo_w, mo_ws, ws2)
        native = orc.dequantize(w, s, gs, "f32").numpy()
        ref = orc.modelopt_values(mo_w, mo_ws, ws2)  # float64
        ref32 = ref.astype(np.float32)
        roundtrip = np.float32(gs) / np.float32(2688) == np.float32(ws2)
        total += 1
        if roundtrip:
            exact_hits += 1
            assert np.array_equal(native.view(np.uint32), ref32.view(np.uint32))
        else:
            ulp = np.spacing(np.abs(ref32)).astype(np.float64)
            assert np.all(np.abs(native.astype(np.float64) - ref) <= 2 * ulp + 0.0)
    assert exact_hits > 0


def pin_transcode_layout(orc):
    mo_w = np.array([[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]], dtype=np.uint8)
    mo_ws = np.array([[0x38]], dtype=np.uint8)
    w, s, gs = orc.transcode(mo_w, mo_ws, np.float32(0.01))
    assert w.dtype == np.uint32 and w.tolist() == [[0x76543210, 0xFEDCBA98]]
    assert s.tolist() == [[0x38]]
    assert gs == np.float32(np.float32(0.01) * np.float32(2688))
    # ModelOpt byte j holds columns 2j (low nibble) and 2j+1 (high nibble)
    assert orc.unpack_codes(w).tolist() == [list(range(16))]


def pin_gather_zero_rows(orc):
    g = synth.rng(4)
    E, N, K, B = 3, 16, 32, 4
    w = synth.packed_weight(g, E, N, K)
    s = synth.log_uniform_scales(g, (E, N, K // 16), 0.25, 4.0)
    gs = synth.global_scales(g, E)
    x = synth.activations(g, (B, K), "f32").double().numpy()
    rhs = np.array([0, 2, E, E + 1, 2**31 - 1, 2**32 - 1, 1, 1], dtype=np.uint32)
    lhs = np.array([3, 0, 1, 2, 0, 1, B, 2**32 - 1], dtype=np.uint32)
    y = orc.gather_qmm(x, lhs, rhs, w, s, gs)
    for r in (2, 3, 4, 5, 6, 7):
        assert np.all(y[r] == 0.0) and not np.any(np.signbit(y[r]))
    for r in (0, 1):
        e = int(rhs[r])
        ref = orc.qmm(x[lhs[r]:lhs[r] + 1], w[e], s[e], gs[e])[0]
        assert np.array_equal(y[r], ref)


def pin_plane_check(orc):
    w = np.zeros((4, 8), dtype=np.uint32)
    orc.check_planes(w, np.zeros((4, 4), dtype=np.uint8))
    for bad in ((4, 3), (4, 5), (3, 4), (4, 4, 1)):
        with pytest.raises(ValueError):
            orc.check_planes(w, np.zeros(bad, dtype=np.uint8))


def pin_error_metric(orc):
    assert orc.rel_to_max_error([1.0, 2.0], [1.0, 4.0]) == 0.5
    assert orc.rel_to_max_error([0.0], [0.0]) == 0.0


def pin_gelu_tanh(orc):
    import math
    v = np.linspace(-8.0, 8.0, 4001)
    g = orc.gelu_tanh(v)
    assert orc.gelu_tanh(0.0) == 0.0
    # 0.5 v (1 + tanh a) - 0.5 (-v) (1 + tanh(-a)) = v for the odd inner a(v)
    assert np.max(np.abs(g - orc.gelu_tanh(-v) - v)) <= 1e-12
    # the tanh form stays within 1e-3 of the exact x * Phi(x) everywhere
    exact = np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in v])
    assert np.max(np.abs(g - exact)) <= 1e-3
    assert abs(orc.gelu_tanh(20.0) - 20.0) <= 1e-12 and abs(orc.gelu_tanh(-20.0)) <= 1e-12


def pin_silu(orc):
    from scipy.special import expit
    v = np.linspace(-30.0, 30.0, 6001)
    s = orc.silu(v)
    assert orc.silu(0.0) == 0.0
    assert np.max(np.abs(s - orc.silu(-v) - v)) <= 1e-12
    assert np.max(np.abs(s - v * expit(v))) <= 1e-12 * (1.0 + np.abs(v)).max()


def pin_glu_halves(orc):
    # unit scales, one-hot x: the gate half and the up half of the fused plane
    # are single table entries, so each output is act(table[g]) * table[u]
    half, k = 8, 32
    codes = synth.rng(705).integers(0, 16, size=(2 * half, k))
    codes[0, :], codes[half, :] = 7, 2  # gate 6.0 and up 1.0 in row 0: swapping halves shows
    sbytes = np.full((2 * half, k // 16), 0x38, dtype=np.uint8)
    table = {int(c): float(v) for c, v in _read_table("e2m1_table.txt")}
    for act in ("silu", "gelu_tanh"):
        f = orc.ACTIVATIONS[act]
        for col in (0, 9, 31):
            x = np.zeros((1, k))
            x[0, col] = 1.0
            y = orc.qmm_glu(x, pack_codes(codes), sbytes, None, act)
            want = [float(f(table[int(codes[j, col])])) * table[int(codes[half + j, col])] for j in range(half)]
            assert y.shape == (1, half) and np.allclose(y[0], want, rtol=0, atol=1e-15)
    # the global factor scales both halves before the activation
    gs = np.float32(2688 * 2.0)
    x = np.zeros((1, k))
    x[0, 3] = 1.0
    y = orc.qmm_glu(x, pack_codes(codes), sbytes, gs, "silu")
    want = [float(orc.silu(2.0 * table[int(codes[j, 3])])) * 2.0 * table[int(codes[half + j, 3])] for j in range(half)]
    assert np.allclose(y[0], want, rtol=0, atol=1e-15)


def _brute_force_qmm_nt(x, codes, sbytes, gs):
    """Exact-rational y = factor * x @ (fp4 * e4m3) for a weight indexed
    [input k, output n], one scale byte per 16 outputs of an input."""
    m_, k = x.shape
    n = codes.shape[1]
    fac = Fraction(1) if gs is None else Fraction(float(np.float32(np.float32(gs) / np.float32(2688))))
    y = np.empty((m_, n), dtype=np.float64)
    for m in range(m_):
        for j in range(n):
            acc = Fraction(0)
            for c in range(k):
                acc += Fraction(float(x[m, c])) * frac_e2m1(int(codes[c, j])) * frac_e4m3(int(sbytes[c, j // 16]))
            y[m, j] = float(acc * fac)
    return y


def pin_nontransposed_brute_force(orc):
    # x [1, 17] against a [17, 32] weight (the shape PR #2629 names), a square
    # plane on which a transposed operand would not fail on shape, and a
    # partial last word column of a 16-output block
    g = synth.rng(8)
    for (m, k, n), gs in (((1, 17, 32), None), ((2, 32, 32), np.float32(26.88)), ((3, 5, 48), np.float32(4.0))):
        codes = g.integers(0, 16, size=(k, n))
        sbytes = synth.log_uniform_scales(g, (k, n // 16), 2.0**-4, 2.0**4)
        x = synth.activations(g, (m, k), "bf16").double().numpy()
        got = orc.qmm_nontransposed(x, pack_codes(codes), sbytes, gs)
        ref = _brute_force_qmm_nt(x, codes, sbytes, gs)
        assert got.shape == (m, n)
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
        ent = orc.qmm_nontransposed_entries(x, pack_codes(codes), sbytes, gs, [m - 1, 0], [n - 1, 17 % n])
        assert np.max(np.abs(ent - ref[[m - 1, 0], [n - 1, 17 % n]])) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def pin_nontransposed_identity(orc):
    # identity activations return the dequantized plane itself, row k = input k
    k = n = 32
    codes = np.arange(k * n).reshape(k, n) * 7 % 16
    sbytes = np.full((k, n // 16), 0x38, dtype=np.uint8)
    table = {int(c): float(v) for c, v in _read_table("e2m1_table.txt")}
    y = orc.qmm_nontransposed(np.eye(k), pack_codes(codes), sbytes, None)
    assert y.tolist() == [[table[int(codes[r, c])] for c in range(n)] for r in range(k)]


def pin_pack_codes(orc):
    # packing is the inverse of the pinned unpacking, and puts column 8j+i in nibble i
    g = synth.rng(21)
    w = synth.packed_weight(g, 5, 64)
    assert np.array_equal(orc.pack_codes(orc.unpack_codes(w)), w)
    assert orc.pack_codes(np.arange(8))[0] == 0x76543210


def pin_e2m1_encode(orc):
    # hand-worked from the grid 0, .5, 1, 1.5, 2, 3, 4, 6 (codes 0..7): a
    # midpoint goes to the even code, anything past 6 to 6
    cases = [(0.0, 0), (0.2499, 0), (0.25, 0), (0.2501, 1), (0.75, 2), (1.25, 2), (1.2501, 3), (1.75, 4),
             (2.5, 4), (2.5001, 5), (3.5, 6), (4.9999, 6), (5.0, 6), (5.0001, 7), (6.0, 7), (7.0, 7), (1e30, 7)]
    got = orc.e2m1_encode(np.array([v for v, _ in cases], dtype=np.float32))
    assert got.tolist() == [c for _, c in cases]
    # brute force: the code's value is at least as near as every other value
    v = synth.rng(22).uniform(0, 8, size=4000).astype(np.float32).astype(np.float64)
    code = orc.e2m1_encode(v)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    dist = np.abs(v[:, None] - grid[None, :])
    assert np.all(dist[np.arange(v.size), code] <= dist.min(axis=1))


def pin_e4m3_encode(orc):
    # identity on the 127 finite non-negative values (bytes 0x00..0x7E, by the
    # bit definition pinned above), ties to the even byte, saturation at 448
    vals = orc.e4m3_value(np.arange(0x7F))
    assert orc.e4m3_encode(vals).tolist() == list(range(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2
    assert orc.e4m3_encode(mids).tolist() == [b + (b & 1) for b in range(0x7E)]
    assert orc.e4m3_encode(np.array([448.0, 460.0, 1e9])).tolist() == [0x7E] * 3
    assert orc.e4m3_encode(np.array([2.0**-10, 2.0**-10 * 1.0001])).tolist() == [0, 1]


def _plane_with_a_six_per_block(g, n, k):
    codes = g.integers(0, 16, size=(n, k))
    codes[codes == 8] = 0  # -0 requantizes as +0
    pos = g.integers(0, 16, size=(n, k // 16))
    for b in range(k // 16):
        codes[np.arange(n), 16 * b + pos[:, b]] = g.choice([7, 15], size=n)
    return codes


def pin_quantize_round_trip(orc):
    # a plane whose every block holds a +-6 is its own quantization: amax = 6
    # e4m3, so the scale comes back exactly and every x / d is a grid value;
    # gs = 2688 * 2^k keeps both global factors exact
    g = synth.rng(23)
    codes = _plane_with_a_six_per_block(g, 6, 64)
    w = pack_codes(codes)
    s = synth.log_uniform_scales(g, (6, 4), 2.0**-8, 2.0**8)
    for gs in (None, np.float32(2688.0), np.float32(2688.0 * 8)):
        x = orc.block_values(w, s) * (1.0 if gs is None else float(gs) / 2688.0)
        w2, s2 = orc.quantize(x.astype(np.float32), gs)
        assert np.array_equal(w2, w) and np.array_equal(s2, s)


def pin_quantize_worked_cases(orc):
    # a block [6, 0, ...] with gs = 4 * 2688: s = 1 / 4 -> byte 0x28, d = 1,
    # code 7; a zero block: scale 0, codes 0; a negative value rounding to
    # zero: +0; beyond range: saturation at 448 and 6
    x = np.zeros((4, 16), dtype=np.float32)
    x[0, 0] = 6.0
    x[2, :2] = [-0.1, 600.0]
    x[3, :3] = [3000.0, -3000.0, 2.9]
    w, s = orc.quantize(x, np.float32(4 * 2688.0))
    assert s[0, 0] == 0x28 and w[0, 0] == 0x7 and w[0, 1] == 0
    assert s[1, 0] == 0 and w[1].tolist() == [0, 0]
    # row 2: amax 600 -> s = 100 / 4 = 25 -> byte of 24 (0x5C, ties 25 to 24),
    # d = 24 * 4 = 96; 600 / 96 = 6.25 -> 6; -0.1 / 96 -> +0
    assert s[2, 0] == 0x5C and w[2, 0] == 0x70
    # row 3 with no global scale: s = 500 -> 448 (0x7E); 3000 / 448 > 6 -> 6;
    # 2.9 / 448 -> 0
    w3, s3 = orc.quantize(x[3:], None)
    assert s3[0, 0] == 0x7E and w3[0, 0] == 0xF7


def _nearest_code_exact(a: float, d: float) -> int:
    """E2M1 magnitude code nearest to a / d in exact rational arithmetic, ties to the even code."""
    q = Fraction(a) / Fraction(d)
    best = None
    for c in range(8):
        dist = abs(q - frac_e2m1(c))
        if best is None or dist < best[0] or (dist == best[0] and c % 2 == 0):
            best = (dist, c)
    return best[1]


def _unpack(w: np.ndarray) -> np.ndarray:
    w = np.asarray(w, dtype=np.int64)
    return np.stack([(w >> (4 * i)) & 0xF for i in range(8)], axis=-1).reshape(*w.shape[:-1], -1)


def pin_quantize_midpoints(orc):
    # Blocks whose multiplier d has an inexact reciprocal: gs absent (d is the
    # E4M3 scale itself) and gs = 268.8 (a global factor near 0.1). A row holds
    # two blocks, each led by its amax (6 d, so the scale byte is b), then the
    # values at, just above and just below m * d for every midpoint m of the
    # E2M1 grid, and the negatives of some. Every code must be the one exact
    # rational arithmetic gives for |x| / d, a tie going to the even code.
    grid = [frac_e2m1(c) for c in range(8)]
    mids = [(grid[i] + grid[i + 1]) / 2 for i in range(7)]
    for gs in (None, np.float32(268.8)):
        fac = np.float32(1.0) if gs is None else np.float32(np.float32(gs) / np.float32(2688.0))
        rows, ds, bs = [], [], []
        for b in list(range(1, 8)) + list(range(0x08, 0x7F, 3)):
            d = np.float32(np.float32(float(frac_e4m3(b))) * fac)
            amax = np.float32(6.0 * float(frac_e4m3(b))) if gs is None else np.float32(6.0 * float(d))
            vals = []
            for m in mids:
                c = np.float32(float(m) * float(d))
                vals += [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(0.0))]
            vals = [v for v in vals if v < amax][:21]
            vals += [np.float32(0.0)] * (21 - len(vals))
            row = [amax] + vals[:15] + [amax] + vals[15:] + [-v for v in vals[:9]]
            rows.append(row)
            ds.append(d)
            bs.append(b)
        x = np.array(rows, dtype=np.float32)
        w, s = orc.quantize(x, gs)
        assert s.tolist() == [[b, b] for b in bs]
        got = _unpack(w)
        for r, d in enumerate(ds):
            for k in range(32):
                a = float(x[r, k])
                mag = _nearest_code_exact(abs(a), float(d))
                want = mag | 8 if a < 0 and mag else mag
                assert got[r, k] == want, (gs, bs[r], k, a, float(d), int(got[r, k]), want)


def pin_fold_scales(orc):
    # ws2 = 1 leaves every finite non-negative byte as it is; ws2 = 2^k shifts
    # the normal values' exponent field by k while they stay normal and finite;
    # beyond 448 saturates; below half the smallest subnormal (2^-10) is 0
    b = np.arange(0x7F, dtype=np.uint8)
    assert orc.fold_scales(b, np.float32(1.0)).tolist() == list(range(0x7F))
    normal = np.arange(0x08, 0x70, dtype=np.uint8)  # exponent fields 1..13
    assert orc.fold_scales(normal, np.float32(2.0)).tolist() == [int(v) + 8 for v in normal]
    assert orc.fold_scales(normal[8:], np.float32(0.5)).tolist() == [int(v) - 8 for v in normal[8:]]
    assert orc.fold_scales(np.array([0x7E, 0x70]), np.float32(4.0)).tolist() == [0x7E, 0x7E]  # 448 * 4, 256 * 4
    # 0x38 is 1.0: 1.0 * 2^-10 ties to 0, a little more rounds up to the smallest subnormal
    assert orc.fold_scales(np.array([0x38, 0x38]), np.float32(2.0**-10)).tolist() == [0, 0]
    assert orc.fold_scales(np.array([0x39]), np.float32(2.0**-10)).tolist() == [1]
    # the words are those of the sidecar transcode
    g = synth.rng(31)
    mo_w, mo_ws, ws2 = synth.modelopt_triplet(g, 4, 64)
    w, s = orc.transcode_folded(mo_w, mo_ws, ws2)
    assert np.array_equal(w, orc.transcode(mo_w, mo_ws, ws2)[0])
    assert np.array_equal(s, orc.fold_scales(mo_ws, ws2))


PINS = [pin_e2m1_table, pin_e4m3_all_bytes, pin_packing, pin_block_scale_broadcast,
        pin_brute_force_matmul, pin_qmm_entries, pin_one_hot, pin_global_factor, pin_dequantize_rounding,
        pin_sidecar_identity, pin_transcode_layout, pin_gather_zero_rows, pin_plane_check,
        pin_error_metric, pin_gelu_tanh, pin_silu, pin_glu_halves, pin_nontransposed_brute_force,
        pin_nontransposed_identity, pin_pack_codes, pin_e2m1_encode, pin_e4m3_encode, pin_quantize_round_trip,
        pin_quantize_worked_cases, pin_quantize_midpoints, pin_fold_scales]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(O)


# ---------------------------------------------------------------- planted mistakes

def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    return O


def test_planted_wrong_table_entry(monkeypatch):
    monkeypatch.setattr(O, "E2M1_MAGNITUDES", (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0))
    with pytest.raises(AssertionError):
        pin_e2m1_table(O)


def test_planted_high_nibble_first(monkeypatch):
    orig = O.unpack_codes

    def swapped(w):
        c = orig(w)
        return c.reshape(*c.shape[:-1], -1, 8)[..., ::-1].reshape(c.shape)
    _planted(monkeypatch, "unpack_codes", swapped)
    with pytest.raises(AssertionError):
        pin_packing(O)


def test_planted_e4m3_bias(monkeypatch):
    orig = O.e4m3_value
    _planted(monkeypatch, "e4m3_value", lambda b: orig(b) * 2.0)
    with pytest.raises(AssertionError):
        pin_e4m3_all_bytes(O)


def test_planted_transposed_operand(monkeypatch):
    orig = O.block_values

    def transposed(w, s):
        v = orig(w, s)
        return v[::-1]  # rows in the wrong order
    _planted(monkeypatch, "block_values", transposed)
    with pytest.raises(AssertionError):
        pin_brute_force_matmul(O)


def test_planted_factor_inverted(monkeypatch):
    _planted(monkeypatch, "global_factor",
             lambda gs: np.float32(1.0) if gs is None else np.float32(2688) / np.float32(gs))
    with pytest.raises(AssertionError):
        pin_global_factor(O)


def test_planted_gather_ignores_bounds(monkeypatch):
    def unbounded(x, lhs, rhs, w, scales, gs=None):
        rhs = np.minimum(np.asarray(rhs, dtype=np.int64), w.shape[0] - 1)
        lhs = np.minimum(np.asarray(lhs, dtype=np.int64), np.asarray(x).shape[0] - 1)
        rows = [O.qmm(np.asarray(x)[l:l + 1], w[e], scales[e], None if gs is None else gs[e])[0]
                for l, e in zip(lhs, rhs)]
        return np.stack(rows)
    _planted(monkeypatch, "gather_qmm", unbounded)
    with pytest.raises(AssertionError):
        pin_gather_zero_rows(O)


def test_planted_scale_per_8_columns(monkeypatch):
    orig_repeat = np.repeat

    def block_values(w, scales):
        O.check_planes(w, scales)
        vals = O.e2m1_value(O.unpack_codes(w))
        s = O.e4m3_value(scales)
        s = orig_repeat(s, 8, axis=-1)
        s = np.concatenate([s, s], axis=-1)
        return vals * s
    _planted(monkeypatch, "block_values", block_values)
    with pytest.raises(AssertionError):
        pin_block_scale_broadcast(O)


def test_planted_sidecar_without_2688(monkeypatch):
    orig = O.transcode

    def bad(mo_w, mo_ws, ws2):
        w, s, _ = orig(mo_w, mo_ws, ws2)
        return w, s, np.float32(ws2)
    _planted(monkeypatch, "transcode", bad)
    with pytest.raises(AssertionError):
        pin_sidecar_identity(O)


def test_planted_glu_halves_swapped(monkeypatch):
    orig = O.qmm

    def swapped(x, w, scales, gs=None):
        h = orig(x, w, scales, gs)
        half = h.shape[1] // 2
        return np.concatenate([h[:, half:], h[:, :half]], axis=1)
    _planted(monkeypatch, "qmm", swapped)
    with pytest.raises(AssertionError):
        pin_glu_halves(O)


def test_planted_gelu_without_cubic(monkeypatch):
    def wrong(v):
        v = np.asarray(v, dtype=np.float64)
        return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * v))
    monkeypatch.setattr(O, "gelu_tanh", wrong)
    with pytest.raises(AssertionError):
        pin_gelu_tanh(O)


def test_planted_nontransposed_as_transposed(monkeypatch):
    def transposed(x, w, scales, gs=None):
        return np.asarray(x, dtype=np.float64) @ O.block_values(w, scales).T * np.float64(O.global_factor(gs))
    _planted(monkeypatch, "qmm_nontransposed", transposed)
    with pytest.raises(AssertionError):
        pin_nontransposed_identity(O)
    with pytest.raises((AssertionError, ValueError)):
        pin_nontransposed_brute_force(O)


def test_planted_nontransposed_scale_row_shifted(monkeypatch):
    # each input's outputs scaled by the previous input's scale bytes
    orig = O.qmm_nontransposed
    _planted(monkeypatch, "qmm_nontransposed", lambda x, w, s, gs=None: orig(x, w, np.roll(s, 1, axis=0), gs))
    with pytest.raises(AssertionError):
        pin_nontransposed_brute_force(O)


def test_planted_e2m1_ties_away_from_zero(monkeypatch):
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    mids = (grid[:-1] + grid[1:]) / 2
    _planted(monkeypatch, "e2m1_encode", lambda v: np.searchsorted(mids, np.asarray(v, dtype=np.float64), side="right"))
    with pytest.raises(AssertionError):
        pin_e2m1_encode(O)


def test_planted_quantize_without_global_scale(monkeypatch):
    orig = O.quantize
    _planted(monkeypatch, "quantize", lambda x, gs=None: orig(x, None))
    with pytest.raises(AssertionError):
        pin_quantize_worked_cases(O)


def test_planted_quantize_scale_off_by_constant(monkeypatch):
    # every block scale 1.5 times too large (as if amax were divided by 4
    # instead of 6)
    orig = O.quantize
    _planted(monkeypatch, "quantize", lambda x, gs=None: orig(np.asarray(x, dtype=np.float32) * np.float32(1.5), gs))
    with pytest.raises(AssertionError):
        pin_quantize_round_trip(O)


def test_planted_fold_without_ws2(monkeypatch):
    orig = O.fold_scales
    _planted(monkeypatch, "fold_scales", lambda b, ws2: orig(b, np.float32(1.0)))
    with pytest.raises(AssertionError):
        pin_fold_scales(O)


def test_planted_quantize_by_reciprocal(monkeypatch):
    # the code taken from the float32 product |x| * float32(1 / d), which
    # rounds twice: it picks the other code beside some midpoints
    def by_reciprocal(a, d):
        r = (np.float32(1.0) / np.asarray(d, dtype=np.float32)).astype(np.float32)
        return O.e2m1_encode((np.asarray(a, dtype=np.float32) * r).astype(np.float32))
    monkeypatch.setattr(O, "e2m1_encode_quotient", by_reciprocal)
    with pytest.raises(AssertionError):
        pin_quantize_midpoints(O)
