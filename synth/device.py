"""Device-side input generation: seeded expert records written into HBM.

Builds ``synth/_build/libk3synth.so`` from ``fill.cu`` (the same SplitMix64 definition
as :func:`synth.expert_record`) and fills torch uint8 tensors with it.  Input
generation only.
"""
import ctypes
import os
import subprocess

import torch

from . import Config

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fill.cu")
LIB = os.path.join(HERE, "_build", "libk3synth.so")
_L = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", SRC, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


def _lib():
    global _L
    if _L is None:
        _L = ctypes.CDLL(build())
        _L.k3synth_fill_experts.restype = ctypes.c_int
        _L.k3synth_fill_experts.argtypes = [
            ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, ctypes.c_ulonglong,
            ctypes.c_int, ctypes.POINTER(ctypes.c_longlong), ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p]
    return _L


def fill_experts(buf: torch.Tensor, cfg: Config, seed: int, layer: int = 0, stride: int = None,
                 e0: int = 0, ne: int = None, stream=None):
    """Write experts [e0, e0+ne) of ``layer`` into ``buf`` (uint8 CUDA tensor, expert e0 at
    byte 0, records ``stride`` bytes apart)."""
    stride = cfg.record_bytes if stride is None else stride
    ne = cfg.n_experts - e0 if ne is None else ne
    assert buf.is_cuda and buf.dtype == torch.uint8 and buf.numel() >= ne * stride
    off = (ctypes.c_longlong * 7)(*cfg.record_offsets)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = _lib().k3synth_fill_experts(ctypes.c_void_p(buf.data_ptr()), stride, e0, ne, seed,
                                     layer, off, cfg.scale_lo, cfg.scale_hi,
                                     ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError("k3synth_fill_experts failed (%d)" % rc)
