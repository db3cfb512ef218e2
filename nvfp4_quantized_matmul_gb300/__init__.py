"""NVFP4 quantized matmul for GB300 (sm_103a).

The compute path lives in ``libnvfp4.so`` (CUDA kernels behind a C ABI); the
``ops`` attributes below are thin ctypes marshalling over it and are loaded on
first use, so ``synth`` can be imported on machines without the library.
"""
_LAZY = ("transcode", "dequantize", "qmm", "gather_qmm", "library", "qmm_crossover", "take_device_error",
         "set_launch_overlap", "set_option", "get_option", "shutdown", "qmm_noalloc", "qmm_sequence", "qmm_glu", "qmm_batched",
         "qmm_nontransposed", "quantize",
         "transcode_folded")


def __getattr__(name):
    if name in _LAZY:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
