"""Host-side tests of libnvfp4.so (no GPU): it loads, exports what the header
declares, and refuses malformed calls before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__ as ge

    ge.build()
    from nvfp4_quantized_matmul_gb300 import binding

    return binding


def declared_functions():
    with open(os.path.join(ROOT, "include", "nvfp4.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(nv):
    names = declared_functions()
    assert "nvfp4_qmm" in names and "nvfp4_gather_qmm" in names
    lib = nv.library()
    for name in names:
        assert hasattr(lib, name), name
        assert name in nv.SIGNATURES, f"binding lacks {name}"


def test_version(nv):
    assert b"sm_103a" in nv.library().nvfp4_version()


# Fake, never-dereferenced device addresses: validation rejects before launch.
A = 0x10000  # 16-byte aligned
U = 0x10004  # 4-byte aligned only


def qmm_call(nv, **kw):
    args = dict(x=A, xdt=2, M=4, K=256, w=A, w_len=512 * 32, s=A, s_len=512 * 16, gs=None, gs_len=0, N=512,
                y=A, route=0)
    args.update(kw)
    lib = nv.library()
    return lib.nvfp4_qmm_routed(args["x"], args["xdt"], args["M"], args["K"], args["w"], args["w_len"], args["s"],
                                args["s_len"], args["gs"], args["gs_len"], args["N"], args["y"], args["route"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=24, w_len=512 * 3, s_len=512), "ERR_SHAPE"),          # K % 16 != 0
    (dict(s_len=512 * 16 - 1), "ERR_PLANE"),                      # short scale plane
    (dict(s_len=512 * 16 + 16), "ERR_PLANE"),                     # oversized scale plane
    (dict(w_len=512 * 32 + 1), "ERR_PLANE"),
    (dict(gs=A, gs_len=2), "ERR_GSCALE"),                         # qmm takes one global scale
    (dict(gs=None, gs_len=1), "ERR_GSCALE"),                      # length without a pointer
    (dict(xdt=7), "ERR_DTYPE"),
    (dict(route=9), "ERR_DTYPE"),
    (dict(x=U), "ERR_ALIGN"),
    (dict(w=U), "ERR_ALIGN"),
    (dict(y=None), "ERR_NULL"),
    (dict(w=None), "ERR_NULL"),
    (dict(M=-1), "ERR_SHAPE"),
    (dict(N=-1, w_len=0, s_len=0), "ERR_SHAPE"),
    (dict(N=2**62, w_len=0, s_len=0), "ERR_SHAPE"),               # overflow
])
def test_qmm_refusals(nv, kw, status):
    st = qmm_call(nv, **kw)
    assert nv.STATUS[st] == status, (st, nv.library().nvfp4_last_error())
    assert nv.library().nvfp4_last_error()


def glu_call(nv, **kw):
    args = dict(x=A, xdt=2, M=4, K=256, w=A, w_len=2 * 256 * 32, s=A, s_len=2 * 256 * 16, gs=None, gs_len=0,
                I=256, act=2, y=A, route=0)
    args.update(kw)
    return nv.library().nvfp4_qmm_glu(args["x"], args["xdt"], args["M"], args["K"], args["w"], args["w_len"],
                                      args["s"], args["s_len"], args["gs"], args["gs_len"], args["I"], args["act"],
                                      args["y"], args["route"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(xdt=0), "ERR_DTYPE"),                                   # f32 activations
    (dict(act=0), "ERR_DTYPE"),
    (dict(act=3), "ERR_DTYPE"),
    (dict(route=5), "ERR_DTYPE"),
    (dict(w_len=256 * 32), "ERR_PLANE"),                          # plane of I rows, not 2 I
    (dict(s_len=2 * 256 * 16 - 1), "ERR_PLANE"),
    (dict(gs=A, gs_len=2), "ERR_GSCALE"),
    (dict(I=-1), "ERR_SHAPE"),
    (dict(K=24, w_len=2 * 256 * 3, s_len=2 * 256), "ERR_SHAPE"),  # K % 16 != 0
    (dict(K=48, w_len=2 * 256 * 6, s_len=2 * 256 * 3, route=1), "ERR_SHAPE"),  # decode route needs K % 256
    (dict(K=48, w_len=2 * 256 * 6, s_len=2 * 256 * 3, route=2), "ERR_SHAPE"),  # tensor cores need K % 32
    (dict(y=U), "ERR_ALIGN"),
    (dict(y=None), "ERR_NULL"),
])
def test_qmm_glu_refusals(nv, kw, status):
    st = glu_call(nv, **kw)
    assert nv.STATUS[st] == status, (st, nv.library().nvfp4_last_error())


def test_qmm_batched_refusals(nv):
    lib = nv.library()
    ST = nv.STATUS
    # 3 batches of [64, 256]: planes of 3 * 64 * 32 words and 3 * 64 * 16 bytes
    call = lambda **kw: lib.nvfp4_qmm_batched(
        A, kw.get("xdt", 2), 3, 4, 256, A, kw.get("w_len", 3 * 64 * 32), A, kw.get("s_len", 3 * 64 * 16),
        kw.get("gs", None), kw.get("gs_len", 0), 64, kw.get("y", A), None)
    assert ST[call(w_len=2 * 64 * 32)] == "ERR_PLANE"
    assert ST[call(s_len=3 * 64 * 16 + 1)] == "ERR_PLANE"
    assert ST[call(gs=A, gs_len=1)] == "ERR_GSCALE"       # one scale per batch
    assert ST[call(xdt=5)] == "ERR_DTYPE"
    assert ST[call(y=U)] == "ERR_ALIGN"
    assert lib.nvfp4_qmm_batched(A, 2, 0, 4, 256, A, 0, A, 0, None, 0, 64, A, None) == 0  # no batches


def test_qmm_nontransposed_refusals(nv):
    lib = nv.library()
    ST = nv.STATUS
    # x [4, 17] against a [17, 32] weight: 17 * 4 words, 17 * 2 scale bytes
    def call(**kw):
        a = dict(x=A, xdt=2, M=4, K=17, w=A, w_len=17 * 4, s=A, s_len=17 * 2, gs=None, gs_len=0, N=32, y=A)
        a.update(kw)
        return ST[lib.nvfp4_qmm_nontransposed(a["x"], a["xdt"], a["M"], a["K"], a["w"], a["w_len"], a["s"],
                                              a["s_len"], a["gs"], a["gs_len"], a["N"], a["y"], None)]
    assert call(N=24, w_len=17 * 3, s_len=17) == "ERR_SHAPE"   # the quantized axis N % 16 != 0
    assert call(xdt=0) == "ERR_DTYPE"                          # f32 activations
    assert call(w_len=17 * 4 - 1) == "ERR_PLANE"
    assert call(s_len=32 * 2) == "ERR_PLANE"                   # a plane laid out [N, K/16]
    assert call(gs=A, gs_len=2) == "ERR_GSCALE"
    assert call(y=U) == "ERR_ALIGN"
    assert call(x=None) == "ERR_NULL"
    assert call(M=-1) == "ERR_SHAPE"
    assert call(M=0) == "OK"
    assert call(N=0, w_len=0, s_len=0) == "OK"


def test_quantize_refusals(nv):
    lib = nv.library()
    ST = nv.STATUS
    # x [2, 8, 64] -> w [2, 8, 8] words, scales [2, 8, 4]
    def call(**kw):
        a = dict(x=A, xdt=2, E=2, N=8, K=64, gs=None, gs_len=0, w=A, w_len=2 * 8 * 8, s=A, s_len=2 * 8 * 4)
        a.update(kw)
        return ST[lib.nvfp4_quantize(a["x"], a["xdt"], a["E"], a["N"], a["K"], a["gs"], a["gs_len"], a["w"],
                                     a["w_len"], a["s"], a["s_len"], None)]
    assert call(K=40, w_len=2 * 8 * 5, s_len=2 * 8 * 2) == "ERR_SHAPE"  # K % 16
    assert call(w_len=2 * 8 * 8 - 1) == "ERR_PLANE"
    assert call(s_len=2 * 8 * 4 + 8) == "ERR_PLANE"
    assert call(gs=A, gs_len=1) == "ERR_GSCALE"                         # one per expert
    assert call(xdt=4) == "ERR_DTYPE"
    assert call(x=U) == "ERR_ALIGN"
    assert call(x=None) == "ERR_NULL"
    assert call(w=U) == "ERR_ALIGN"
    assert call(N=0, w_len=0, s_len=0) == "OK"


def test_transcode_folded_refusals(nv):
    lib = nv.library()
    ST = nv.STATUS
    N, K = 8, 64
    call = lambda **kw: ST[lib.nvfp4_transcode_folded(A, kw.get("wl", N * K // 2), A, kw.get("sl", N * K // 16),
                                                      kw.get("ws2", A), N, kw.get("K", K), kw.get("wo", A), A, None)]
    assert call(K=40, wl=N * 20, sl=N * 2) == "ERR_SHAPE"
    assert call(wl=N * K // 2 + 16) == "ERR_PLANE"
    assert call(sl=N * K // 16 - 1) == "ERR_PLANE"
    assert call(ws2=None) == "ERR_NULL"
    assert call(wo=U) == "ERR_ALIGN"


def test_qmm_glu_empty_returns_ok(nv):
    assert glu_call(nv, M=0) == 0
    assert glu_call(nv, I=0, w_len=0, s_len=0) == 0


def test_empty_outputs_return_ok_without_launch(nv):
    assert qmm_call(nv, M=0) == 0
    assert qmm_call(nv, N=0, w_len=0, s_len=0) == 0
    lib = nv.library()
    st = lib.nvfp4_gather_qmm(A, 2, 4, 256, None, A, 0, 0, A, 3 * 64 * 32, A, 3 * 64 * 16, None, 0, 3, 64, A, None)
    assert st == 0
    st = lib.nvfp4_dequantize(A, 0, A, 0, None, 0, 1, 0, 256, 2, A, None)
    assert st == 0


def test_gather_refusals(nv):
    lib = nv.library()
    E, N, K = 3, 64, 256

    def call(**kw):
        a = dict(x=A, xdt=2, B=4, K=K, lhs=None, rhs=A, R=5, w=A, w_len=E * N * K // 8, s=A, s_len=E * N * K // 16,
                 gs=None, gs_len=0, E=E, N=N, y=A)
        a.update(kw)
        return nv.STATUS[lib.nvfp4_gather_qmm(a["x"], a["xdt"], a["B"], a["K"], a["lhs"], a["rhs"], a["R"], 0, a["w"],
                                              a["w_len"], a["s"], a["s_len"], a["gs"], a["gs_len"], a["E"], a["N"],
                                              a["y"], None)]

    assert call(gs=A, gs_len=E - 1) == "ERR_GSCALE"  # one global scale per expert
    assert call(gs=A, gs_len=1) == "ERR_GSCALE"
    assert call(s_len=E * N * K // 16 - N * K // 16) == "ERR_PLANE"  # missing expert in scales
    assert call(rhs=None) == "ERR_NULL"
    assert call(rhs=A + 2) == "ERR_ALIGN"
    assert call(B=-1) == "ERR_SHAPE"


def test_transcode_and_dequantize_refusals(nv):
    lib = nv.library()
    N, K = 8, 64
    st = lib.nvfp4_transcode(A, N * K // 2 - 1, A, N * K // 16, A, N, K, A, A, A, None)
    assert nv.STATUS[st] == "ERR_PLANE"
    st = lib.nvfp4_transcode(A, N * K // 2, A, N * K // 16, None, N, K, A, A, A, None)
    assert nv.STATUS[st] == "ERR_NULL"
    st = lib.nvfp4_transcode(A, N * 8, A, N, A, N, 17, A, A, A, None)
    assert nv.STATUS[st] == "ERR_SHAPE"
    st = lib.nvfp4_dequantize(A, N * K // 8, A, N * K // 16 + 4, None, 0, 1, N, K, 0, A, None)
    assert nv.STATUS[st] == "ERR_PLANE"
    st = lib.nvfp4_dequantize(A, N * K // 8, A, N * K // 16, A, 2, 1, N, K, 0, A, None)
    assert nv.STATUS[st] == "ERR_GSCALE"
    st = lib.nvfp4_dequantize(A, N * K // 8, A, N * K // 16, None, 0, 1, N, K, 3, A, None)
    assert nv.STATUS[st] == "ERR_DTYPE"


def test_crossover_env_override(nv, monkeypatch):
    monkeypatch.setenv("NVFP4_QMM_CROSSOVER", "96")
    assert nv.library().nvfp4_qmm_crossover(2, 21504, 5376) == 96


def test_crossover_model(nv, monkeypatch, opt):
    """The default crossover follows the route sweep on GB300: gate/up and
    down switch to the tensor cores at 48 token rows (two 16-row decode
    launches still beat them at 32), qkv at 32; f32 never. Without the
    stream-K split the tensor-core route is slower at small M and down (21
    weight tiles for 152 SMs) switches only at 112."""
    monkeypatch.delenv("NVFP4_QMM_CROSSOVER", raising=False)
    lib = nv.library()
    assert lib.nvfp4_qmm_crossover(2, 43008, 5376) == 48
    assert lib.nvfp4_qmm_crossover(2, 8192, 5376) == 32
    assert lib.nvfp4_qmm_crossover(2, 5376, 21504) == 48
    opt("tc_streamk", 0)
    assert lib.nvfp4_qmm_crossover(2, 43008, 5376) == 48
    assert lib.nvfp4_qmm_crossover(2, 8192, 5376) == 48
    assert lib.nvfp4_qmm_crossover(2, 5376, 21504) == 112
    opt("tc_streamk", 1)
    assert lib.nvfp4_qmm_crossover(1, 43008, 5376) == 48
    assert lib.nvfp4_qmm_crossover(0, 43008, 5376) > 2**62
    for n, k in ((256, 256), (1 << 20, 64), (64, 1 << 20)):
        assert 16 <= lib.nvfp4_qmm_crossover(2, n, k) <= 128


def test_binding_rejects_cpu_tensors(nv):
    import torch

    x = torch.zeros(2, 32, dtype=torch.bfloat16)
    w = torch.zeros(4, 4, dtype=torch.int32)
    s = torch.zeros(4, 2, dtype=torch.uint8)
    with pytest.raises(ValueError):
        nv.qmm(x, w, s)


def seq_calls(nv, n, **kw):
    """n calls of [512, 256] at M = 4 with fake aligned addresses; kw
    overrides fields of call 1 (or of the only call)."""
    arr = (nv.QmmCall * n)()
    for i in range(n):
        c = dict(x=A, M=4, K=256, N=512, w=A, w_len=512 * 32, scales=A, scales_len=512 * 16, gs=None, gs_len=0,
                 y=A, after_previous=0, reserved=0)
        if i == min(1, n - 1):
            c.update(kw)
        arr[i] = nv.QmmCall(**c)
    return arr


@pytest.mark.parametrize("kw,status", [
    (dict(M=17), "ERR_LIMIT"),                                    # more than 16 token rows
    (dict(K=272, w_len=512 * 34, scales_len=512 * 17), "ERR_SHAPE"),  # K % 256 != 0
    (dict(w_len=512 * 32 - 1), "ERR_PLANE"),
    (dict(scales_len=512 * 16 + 1), "ERR_PLANE"),
    (dict(gs=A, gs_len=2), "ERR_GSCALE"),
    (dict(x=U), "ERR_ALIGN"),
    (dict(y=None), "ERR_NULL"),
    (dict(M=-1), "ERR_SHAPE"),
])
def test_qmm_sequence_refusals(nv, kw, status):
    lib = nv.library()
    arr = seq_calls(nv, 3, **kw)
    st = lib.nvfp4_qmm_sequence(ctypes.addressof(arr), 3, 2, None)
    assert nv.STATUS[st] == status, (st, lib.nvfp4_last_error())
    assert b"call 1" in lib.nvfp4_last_error()


def test_qmm_sequence_refusals_of_the_whole(nv):
    lib = nv.library()
    arr = seq_calls(nv, 33)
    assert nv.STATUS[lib.nvfp4_qmm_sequence(ctypes.addressof(arr), 33, 2, None)] == "ERR_LIMIT"
    assert nv.STATUS[lib.nvfp4_qmm_sequence(ctypes.addressof(arr), -1, 2, None)] == "ERR_LIMIT"
    assert nv.STATUS[lib.nvfp4_qmm_sequence(ctypes.addressof(arr), 2, 0, None)] == "ERR_DTYPE"  # f32
    assert nv.STATUS[lib.nvfp4_qmm_sequence(None, 2, 2, None)] == "ERR_NULL"
    # nothing to run: no calls, or only empty outputs (M = 0 or N = 0)
    assert lib.nvfp4_qmm_sequence(None, 0, 2, None) == 0
    empty = seq_calls(nv, 2, M=0)
    empty[0] = nv.QmmCall(A, 4, 256, 0, A, 0, A, 0, None, 0, A, 0, 0)
    assert lib.nvfp4_qmm_sequence(ctypes.addressof(empty), 2, 2, None) == 0


def test_options_set_get_and_refusals(nv, opt):
    lib = nv.library()
    assert nv.get_option("tc_streamk") == 1 and nv.get_option("gather_tc") == -1
    opt("tc_tile", "256x128")
    assert nv.get_option("tc_tile") == 2
    assert nv.STATUS[lib.nvfp4_set_option(1, 4)] == "ERR_LIMIT"      # tile code out of range
    assert nv.get_option("tc_tile") == 2                              # unchanged
    assert nv.STATUS[lib.nvfp4_set_option(6, -2)] == "ERR_LIMIT"
    assert nv.STATUS[lib.nvfp4_set_option(0, 0)] == "ERR_DTYPE"       # unknown option
    assert nv.STATUS[lib.nvfp4_set_option(99, 0)] == "ERR_DTYPE"
    assert lib.nvfp4_get_option(99) == -2**31
