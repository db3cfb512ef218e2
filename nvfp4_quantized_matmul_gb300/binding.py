"""ctypes binding over libnvfp4.so: argument marshalling only.

Every function here checks that the tensors live on the GPU, passes their
device pointers, element counts and the current CUDA stream to the C ABI
(``include/nvfp4.h``) and raises ``Nvfp4Error`` with the library's message on
a non-OK status. All arithmetic runs in the library's CUDA kernels; there is
no CPU fallback. If the library has not been built the import fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnvfp4.so")

STATUS = ("OK", "ERR_NULL", "ERR_SHAPE", "ERR_PLANE", "ERR_DTYPE", "ERR_ALIGN", "ERR_GSCALE",
          "ERR_LIMIT", "ERR_CUDA")
DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
ROUTE_CODE = {"auto": 0, "qmv": 1, "tc": 2}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int

class QmmCall(ctypes.Structure):
    """nvfp4_qmm_call (include/nvfp4.h)."""

    _fields_ = [("x", _P), ("M", _I64), ("K", _I64), ("N", _I64), ("w", _P), ("w_len", _I64), ("scales", _P),
                ("scales_len", _I64), ("gs", _P), ("gs_len", _I64), ("y", _P), ("after_previous", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


# name -> (restype, argtypes); mirrors include/nvfp4.h
SIGNATURES = {
    "nvfp4_transcode": (_INT, [_P, _I64, _P, _I64, _P, _I64, _I64, _P, _P, _P, _P]),
    "nvfp4_dequantize": (_INT, [_P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _INT, _P, _P]),
    "nvfp4_qmm": (_INT, [_P, _INT, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _P]),
    "nvfp4_qmm_routed": (_INT, [_P, _INT, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _INT, _P]),
    "nvfp4_qmm_crossover": (_I64, [_INT, _I64, _I64]),
    "nvfp4_qmm_noalloc": (_INT, [_P, _INT, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _P]),
    "nvfp4_qmm_sequence": (_INT, [_P, ctypes.c_int32, _INT, _P]),
    "nvfp4_qmm_glu": (_INT, [_P, _INT, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _INT, _P, _INT, _P]),
    "nvfp4_qmm_batched": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _P]),
    "nvfp4_qmm_nontransposed": (_INT, [_P, _INT, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _P]),
    "nvfp4_quantize": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P]),
    "nvfp4_transcode_folded": (_INT, [_P, _I64, _P, _I64, _P, _I64, _I64, _P, _P, _P]),
    "nvfp4_gather_qmm": (_INT, [_P, _INT, _I64, _I64, _P, _P, _I64, _INT, _P, _I64, _P, _I64, _P, _I64,
                                _I64, _I64, _P, _P]),
    "nvfp4_last_error": (ctypes.c_char_p, []),
    "nvfp4_version": (ctypes.c_char_p, []),
    "nvfp4_take_device_error": (ctypes.c_int32, []),
    "nvfp4_set_launch_overlap": (_INT, [_INT]),
    "nvfp4_set_option": (_INT, [_INT, ctypes.c_int32]),
    "nvfp4_get_option": (ctypes.c_int32, [_INT]),
    "nvfp4_shutdown": (None, []),
}


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        name = STATUS[status] if 0 <= status < len(STATUS) else str(status)
        super().__init__(f"NVFP4_{name}: {message}")
        self.status = status
        self.name = name


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library():
    """The loaded ctypes library (for direct C-ABI calls)."""
    return _lib


def check(status: int) -> None:
    if status != 0:
        raise Nvfp4Error(status, _lib.nvfp4_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _n(t):
    return 0 if t is None else t.numel()


def _cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("nvfp4 ops take CUDA tensors (the library has no CPU path)")
            if not t.is_contiguous():
                raise ValueError("nvfp4 ops take contiguous tensors")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t):
    """The current CUDA stream of t's device, as a raw handle (the cheap
    accessor when this torch has it: building a Stream object per call costs
    several microseconds)."""
    if _raw_stream is not None:
        return _raw_stream(t.device.index)
    return torch.cuda.current_stream(t.device).cuda_stream


def _gs_tensor(gs, device):
    if gs is None:
        return None
    if not torch.is_tensor(gs):
        gs = torch.tensor([float(gs)], dtype=torch.float32, device=device)
    if gs.dtype != torch.float32:
        raise ValueError("gs must be float32")
    return gs if gs.dim() == 1 else gs.reshape(-1)


def transcode(mo_weight, mo_weight_scale, weight_scale_2, out=None):
    """ModelOpt triplet -> (w uint32 [N,K/8] as int32 storage, scales uint8 [N,K/16], gs float32 [1])."""
    _cuda(mo_weight, mo_weight_scale)
    n, half_k = mo_weight.shape
    k = half_k * 2
    ws2 = _gs_tensor(weight_scale_2, mo_weight.device)
    if out is None:
        w = torch.empty((n, k // 8), dtype=torch.int32, device=mo_weight.device)
        s = torch.empty((n, k // 16), dtype=torch.uint8, device=mo_weight.device)
        gs = torch.empty((1,), dtype=torch.float32, device=mo_weight.device)
    else:
        w, s, gs = out
    check(_lib.nvfp4_transcode(_ptr(mo_weight), mo_weight.numel(), _ptr(mo_weight_scale), mo_weight_scale.numel(),
                               _ptr(ws2), n, k, _ptr(w), _ptr(s), _ptr(gs), _stream(mo_weight)))
    return w, s, gs


def transcode_folded(mo_weight, mo_weight_scale, weight_scale_2, out=None):
    """ModelOpt triplet -> (w uint32 [N,K/8] as int32 storage, folded E4M3
    scales uint8 [N,K/16]); no sidecar (dequantize with gs=None)."""
    _cuda(mo_weight, mo_weight_scale)
    n, half_k = mo_weight.shape
    k = half_k * 2
    ws2 = _gs_tensor(weight_scale_2, mo_weight.device)
    if out is None:
        w = torch.empty((n, k // 8), dtype=torch.int32, device=mo_weight.device)
        s = torch.empty((n, k // 16), dtype=torch.uint8, device=mo_weight.device)
    else:
        w, s = out
    check(_lib.nvfp4_transcode_folded(_ptr(mo_weight), mo_weight.numel(), _ptr(mo_weight_scale),
                                      mo_weight_scale.numel(), _ptr(ws2), n, k, _ptr(w), _ptr(s), _stream(mo_weight)))
    return w, s


def dequantize(w, scales, gs=None, out_dtype=torch.bfloat16, out=None):
    """Exact dequantize of ``w`` [E?, N, K/8] -> [E?, N, K] of ``out_dtype``."""
    _cuda(w, scales)
    lead = tuple(w.shape[:-1])
    k = w.shape[-1] * 8
    e = lead[0] if len(lead) == 2 else 1
    n = lead[-1]
    gs = _gs_tensor(gs, w.device)
    if out is None:
        out = torch.empty((*lead, k), dtype=out_dtype, device=w.device)
    check(_lib.nvfp4_dequantize(_ptr(w), w.numel(), _ptr(scales), scales.numel(), _ptr(gs), _n(gs), e, n, k,
                                DTYPE_CODE[out.dtype], _ptr(out), _stream(w)))
    return out


def qmm(x, w, scales, gs=None, route="auto", out=None):
    """QuantizedMatmul: ``x`` [M, K] @ dequantize(w [N, K/8]).T -> [M, N] in x's dtype."""
    _cuda(x, w, scales)
    m, k = x.shape
    n = w.shape[0]
    gs = _gs_tensor(gs, x.device)
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    check(_lib.nvfp4_qmm_routed(_ptr(x), DTYPE_CODE[x.dtype], m, k, _ptr(w), w.numel(), _ptr(scales),
                                scales.numel(), _ptr(gs), _n(gs), n, _ptr(out), ROUTE_CODE[route], _stream(x)))
    return out


def qmm_batched(x, w, scales, gs=None, out=None):
    """QuantizedMatmul with batched weights: ``x`` [B, M, K], ``w`` [B, N, K/8],
    ``scales`` [B, N, K/16], ``gs`` None or [B] -> [B, M, N] in x's dtype."""
    _cuda(x, w, scales)
    bt, m, k = x.shape
    n = w.shape[1]
    gs = _gs_tensor(gs, x.device)
    if out is None:
        out = torch.empty((bt, m, n), dtype=x.dtype, device=x.device)
    check(_lib.nvfp4_qmm_batched(_ptr(x), DTYPE_CODE[x.dtype], bt, m, k, _ptr(w), w.numel(), _ptr(scales),
                                 scales.numel(), _ptr(gs), _n(gs), n, _ptr(out), _stream(x)))
    return out


def quantize(x, gs=None, out=None):
    """Dense ``x`` [E?, N, K] (f32, f16 or bf16) -> ``(w [E?, N, K/8] int32,
    scales [E?, N, K/16] uint8)``; ``gs`` None, a float or a device tensor with
    one value per expert (block scales encoded times 2688 / gs)."""
    _cuda(x)
    if x.dim() not in (2, 3):
        raise ValueError("x must be [N, K] or [E, N, K]")
    e = x.shape[0] if x.dim() == 3 else 1
    n, k = x.shape[-2], x.shape[-1]
    gs = _gs_tensor(gs, x.device)
    if out is None:
        lead = tuple(x.shape[:-1])
        out = (torch.empty(lead + (k // 8,), dtype=torch.int32, device=x.device),
               torch.empty(lead + (k // 16,), dtype=torch.uint8, device=x.device))
    w, s = out
    check(_lib.nvfp4_quantize(_ptr(x), DTYPE_CODE[x.dtype], e, n, k, _ptr(gs), _n(gs), _ptr(w), w.numel(), _ptr(s),
                              s.numel(), _stream(x)))
    return w, s


def qmm_nontransposed(x, w, scales, gs=None, out=None):
    """QuantizedMatmul with a non-transposed weight: ``w`` [K, N/8] quantized
    along N, ``scales`` [K, N/16]; returns x @ dequantize(w) * gs/2688, [M, N]
    in x's dtype."""
    _cuda(x, w, scales)
    m, k = x.shape
    n = w.shape[1] * 8
    gs = _gs_tensor(gs, x.device)
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    check(_lib.nvfp4_qmm_nontransposed(_ptr(x), DTYPE_CODE[x.dtype], m, k, _ptr(w), w.numel(), _ptr(scales),
                                       scales.numel(), _ptr(gs), _n(gs), n, _ptr(out), _stream(x)))
    return out


ACT_CODE = {"silu": 1, "gelu_tanh": 2}


def qmm_glu(x, w, scales, gs=None, act="gelu_tanh", route="auto", out=None):
    """Fused gate/up with its activation: ``w`` is [2 I, K/8] (gate rows, then
    up rows); returns act(gate) * up, [M, I] in x's dtype."""
    _cuda(x, w, scales)
    m, k = x.shape
    n2 = w.shape[0]
    if n2 % 2:
        raise ValueError("the fused plane needs an even number of rows")
    i = n2 // 2
    gs = _gs_tensor(gs, x.device)
    if out is None:
        out = torch.empty((m, i), dtype=x.dtype, device=x.device)
    check(_lib.nvfp4_qmm_glu(_ptr(x), DTYPE_CODE[x.dtype], m, k, _ptr(w), w.numel(), _ptr(scales), scales.numel(),
                             _ptr(gs), _n(gs), i, ACT_CODE[act], _ptr(out), ROUTE_CODE[route], _stream(x)))
    return out


def qmm_noalloc(x, w, scales, gs=None, out=None):
    """nvfp4_qmm without any device allocation by the library (fixed scratch
    inside it; 16-bit x, M <= 16, K % 256 == 0, N <= 65536). Calls that could
    overlap on the GPU must be ordered: they share that scratch."""
    _cuda(x, w, scales)
    m, k = x.shape
    n = w.shape[0]
    gs = _gs_tensor(gs, x.device)
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    check(_lib.nvfp4_qmm_noalloc(_ptr(x), DTYPE_CODE[x.dtype], m, k, _ptr(w), w.numel(), _ptr(scales),
                                 scales.numel(), _ptr(gs), _n(gs), n, _ptr(out), _stream(x)))
    return out


def qmm_sequence(calls, stream_of=None):
    """Several decode-shape QuantizedMatmuls in one launch, in order.

    ``calls`` holds tuples ``(x, w, scales, gs, out, after_previous)``: x [M, K]
    (f16 or bf16, the same dtype for all), w [N, K/8], scales [N, K/16], gs
    None or a float32 tensor of one element, out [M, N] of x's dtype (or None
    to allocate it), and after_previous: read x only after every earlier call
    has finished (x is an earlier call's output). Returns the outputs."""
    n = len(calls)
    arr = (QmmCall * max(n, 1))()
    outs, keep = [], []
    dtype = None
    for i, (x, w, scales, gs, out, after) in enumerate(calls):
        _cuda(x, w, scales)
        m, k = x.shape
        nrow = w.shape[0]
        gs = _gs_tensor(gs, x.device)
        if out is None:
            out = torch.empty((m, nrow), dtype=x.dtype, device=x.device)
        _cuda(out)
        dtype = x.dtype if dtype is None else dtype
        if x.dtype != dtype or out.dtype != dtype:
            raise ValueError("all calls of a sequence take activations and outputs of one dtype")
        arr[i] = QmmCall(_ptr(x), m, k, nrow, _ptr(w), w.numel(), _ptr(scales), scales.numel(), _ptr(gs), _n(gs),
                         _ptr(out), 1 if after else 0, 0)
        outs.append(out)
        keep.append(gs)
    if n == 0:
        return outs
    check(_lib.nvfp4_qmm_sequence(ctypes.addressof(arr), n, DTYPE_CODE[dtype], _stream(calls[0][0])))
    return outs


def gather_qmm(x, w, scales, rhs, lhs=None, gs=None, sorted_indices=False, out=None):
    """GatherQMM: row r = x[lhs[r]] @ dequantize(w[rhs[r]]).T * gs[rhs[r]]/2688 (zero row if out of range)."""
    _cuda(x, w, scales, rhs, lhs)
    b, k = x.shape
    e, n = w.shape[0], w.shape[1]
    r = rhs.numel()
    gs = _gs_tensor(gs, x.device)
    if out is None:
        out = torch.empty((r, n), dtype=x.dtype, device=x.device)
    check(_lib.nvfp4_gather_qmm(_ptr(x), DTYPE_CODE[x.dtype], b, k, _ptr(lhs), _ptr(rhs), r, int(bool(sorted_indices)),
                                _ptr(w), w.numel(), _ptr(scales), scales.numel(), _ptr(gs), _n(gs), e, n,
                                _ptr(out), _stream(x)))
    return out


def take_device_error():
    """Device error code from a tensor-core kernel's bounded wait (0 = none); synchronises."""
    return int(_lib.nvfp4_take_device_error())


def set_launch_overlap(enable):
    """Let weight-streaming calls start while the previous kernel on the stream
    finishes (the weight planes must not be written by a kernel still running).
    Returns the previous setting."""
    return bool(_lib.nvfp4_set_launch_overlap(int(bool(enable))))


OPTION_CODE = {"tc_tile": 1, "tc_streamk": 2, "nt_decode": 3, "qmv_row_tiles": 4, "gather_group": 5,
               "gather_tc": 6, "gather_tile": 7, "wait_limit_us": 8, "test_withhold": 9}
TILE_CODE = {"auto": 0, "256x256": 1, "256x128": 2, "128x256": 3}


def set_option(name, value):
    """Sets one of the library's process-wide kernel choices (nvfp4_set_option);
    tile options also take "256x256", "256x128" or "128x256"."""
    if isinstance(value, str):
        value = TILE_CODE[value]
    check(_lib.nvfp4_set_option(OPTION_CODE[name], int(value)))


def get_option(name):
    return int(_lib.nvfp4_get_option(OPTION_CODE[name]))


def shutdown():
    """Free the library's workspaces (call with no library work in flight)."""
    _lib.nvfp4_shutdown()


def qmm_crossover(dtype, n, k):
    return int(_lib.nvfp4_qmm_crossover(DTYPE_CODE[dtype], n, k))
