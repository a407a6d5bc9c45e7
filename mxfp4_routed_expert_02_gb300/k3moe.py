"""Python binding of libk3moe (the C ABI declared in ``include/k3moe.h``).

Argument marshalling only: each function takes torch CUDA tensors, checks their dtype,
device and contiguity, and passes raw pointers to the library.  Every step of the MoE
layer runs in the library's CUDA kernels; there is no CPU or PyTorch fallback: if the
library cannot be loaded, every call raises.
"""
import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

K3MOE_OK = 0
STATUS_NAMES = {
    0: "OK", 1: "ERR_ARG", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_WORKSPACE", 5: "ERR_CUDA",
    6: "ERR_TIMEOUT", 7: "ERR_BAD_EXPERT", 8: "ERR_NONFINITE", 9: "ERR_SCRATCH_LIMIT",
    10: "ERR_CACHE_FULL",
}
K3MOE_ERR_CACHE_FULL = 10
K3MOE_ERR_SCRATCH_LIMIT = 9
# MXFP4 terms of the activations in the multi-token path (x, SiTU output); informational.
TC_TERMS_X, TC_TERMS_ACT = 4, 4
# Bytes of the library's static scratch array (K3MOE_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 8 * 1024 * 1024
F32, BF16 = 0, 1

# Every symbol include/k3moe.h declares.
EXPORTS = (
    "k3moe_record_layout", "k3moe_workspace_size", "k3moe_route", "k3moe_expert_ffn_mxfp4",
    "k3moe_layer", "k3moe_layer_static_scratch", "k3moe_decode_stack", "k3moe_rmsnorm_bf16", "k3moe_dequant_mxfp4",
    "k3moe_test_expire_wait", "k3moe_trace_enable", "k3moe_trace_read", "k3moe_status_str",
    "k3moe_latent_layer", "k3moe_latent_workspace_size", "k3moe_cache_create",
    "k3moe_cache_destroy", "k3moe_cache_lookup", "k3moe_cache_stats",
    "k3moe_streamed_workspace_size", "k3moe_layer_streamed",
)


class K3MoeError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (fn, STATUS_NAMES.get(code, "?"), code))


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("group", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("situ_b1", ctypes.c_float), ("situ_b2", ctypes.c_float),
                ("routed_scale", ctypes.c_float), ("renorm", ctypes.c_int32)]


class Experts(ctypes.Structure):
    _fields_ = [("experts", ctypes.c_void_p), ("expert_stride", ctypes.c_int64)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("wr_bf16", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("experts", Experts),
                ("sh_gate", ctypes.c_void_p), ("sh_up", ctypes.c_void_p),
                ("sh_down", ctypes.c_void_p)]


class LatentDimsC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("latent", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("group", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("situ_b1", ctypes.c_float),
                ("situ_b2", ctypes.c_float), ("routed_scale", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("renorm", ctypes.c_int32),
                ("latent_norm", ctypes.c_int32)]


class LatentWeightsC(ctypes.Structure):
    _fields_ = [("wr_bf16", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
                ("latent_norm_w", ctypes.c_void_p), ("experts", Experts),
                ("sh_gate", ctypes.c_void_p), ("sh_up", ctypes.c_void_p),
                ("sh_down", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """Load libk3moe.so (building it first if allowed).  Raises if it is unavailable."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libk3moe.so is not built (%s); run __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    dp = ctypes.POINTER(Dims)
    ep = ctypes.POINTER(Experts)
    L.k3moe_record_layout.restype = i32
    L.k3moe_record_layout.argtypes = [dp, ctypes.POINTER(ctypes.c_int64)]
    L.k3moe_workspace_size.restype = sz
    L.k3moe_workspace_size.argtypes = [dp, i32]
    L.k3moe_route.restype = i32
    L.k3moe_route.argtypes = [dp, vp, vp, vp, i32, vp, vp, vp, sz, vp, vp]
    L.k3moe_expert_ffn_mxfp4.restype = i32
    L.k3moe_expert_ffn_mxfp4.argtypes = [dp, vp, i32, ep, vp, vp, vp, i32, i32, vp, sz, vp, vp]
    L.k3moe_layer.restype = i32
    L.k3moe_layer.argtypes = [dp, vp, i32, vp, vp, ep, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz,
                              vp, vp]
    L.k3moe_layer_static_scratch.restype = i32
    L.k3moe_layer_static_scratch.argtypes = [dp, vp, i32, vp, vp, ep, vp, vp, vp, vp, vp, vp,
                                             i32, i32, vp, vp]
    L.k3moe_decode_stack.restype = i32
    L.k3moe_decode_stack.argtypes = [dp, i32, ctypes.POINTER(LayerWeights), i32, vp,
                                     ctypes.c_float, vp, vp, vp, vp, sz, vp, vp]
    L.k3moe_rmsnorm_bf16.restype = i32
    L.k3moe_rmsnorm_bf16.argtypes = [vp, i32, i32, ctypes.c_float, vp, vp]
    L.k3moe_dequant_mxfp4.restype = i32
    L.k3moe_dequant_mxfp4.argtypes = [vp, vp, i32, i32, vp, vp]
    L.k3moe_test_expire_wait.restype = i32
    L.k3moe_test_expire_wait.argtypes = [i32]
    L.k3moe_trace_enable.restype = i32
    L.k3moe_trace_enable.argtypes = [i32]
    L.k3moe_trace_read.restype = i32
    L.k3moe_trace_read.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p),
                                   ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    L.k3moe_latent_workspace_size.restype = sz
    L.k3moe_latent_workspace_size.argtypes = [ctypes.POINTER(LatentDimsC), i32]
    L.k3moe_latent_layer.restype = i32
    L.k3moe_latent_layer.argtypes = [ctypes.POINTER(LatentDimsC),
                                     ctypes.POINTER(LatentWeightsC), vp, i32, vp, vp, vp, i32,
                                     i32, vp, sz, vp, vp]
    cp = ctypes.c_void_p
    L.k3moe_cache_create.restype = i32
    L.k3moe_cache_create.argtypes = [i32, ctypes.POINTER(ctypes.c_void_p), i32, i64, i64, vp,
                                     i32, i64, ctypes.POINTER(cp)]
    L.k3moe_cache_destroy.restype = i32
    L.k3moe_cache_destroy.argtypes = [cp]
    L.k3moe_cache_lookup.restype = i32
    L.k3moe_cache_lookup.argtypes = [cp, i32, vp, i32, vp, vp]
    L.k3moe_cache_stats.restype = i32
    L.k3moe_cache_stats.argtypes = [cp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                    ctypes.POINTER(i64)]
    L.k3moe_streamed_workspace_size.restype = sz
    L.k3moe_streamed_workspace_size.argtypes = [dp, i32]
    L.k3moe_layer_streamed.restype = i32
    L.k3moe_layer_streamed.argtypes = [dp, cp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                       i32, i32, vp, sz, vp, vp]
    L.k3moe_status_str.restype = ctypes.c_char_p
    L.k3moe_status_str.argtypes = [i32]
    _LIB = L
    return L


@dataclass
class LayerDims:
    hidden: int
    inter: int
    n_experts: int
    topk: int
    shared_inter: int = 0
    situ_b1: float = 4.0
    situ_b2: float = 25.0
    routed_scale: float = 1.0
    renorm: int = 1
    group: int = 32

    def c(self) -> Dims:
        return Dims(self.hidden, self.inter, self.n_experts, self.topk, self.group,
                    self.shared_inter, self.situ_b1, self.situ_b2, self.routed_scale, self.renorm)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, code):
    if code != K3MOE_OK:
        raise K3MoeError(fn, code)


def _bits16(t, name):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype not in (torch.int16, torch.uint16):
        raise TypeError("%s must be bf16 (or its 16-bit pattern)" % name)
    return t


def record_layout(dims: LayerDims):
    off = (ctypes.c_int64 * 7)()
    d = dims.c()
    _check("k3moe_record_layout", lib().k3moe_record_layout(ctypes.byref(d), off))
    return list(off)


def workspace_size(dims: LayerDims, T: int) -> int:
    d = dims.c()
    return int(lib().k3moe_workspace_size(ctypes.byref(d), int(T)))


def new_workspace(dims: LayerDims, T: int, device=None) -> torch.Tensor:
    """A workspace for T tokens, zero-filled as the C ABI requires before first use."""
    n = workspace_size(dims, T)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def k3moe_route(dims: LayerDims, x, wr, bias, idx, w, workspace, status, stream=None):
    d = dims.c()
    x, wr = _bits16(x, "x"), _bits16(wr, "wr")
    T = x.shape[0]
    _check("k3moe_route", lib().k3moe_route(
        ctypes.byref(d), _ptr(x), _ptr(wr), _ptr(bias), T, _ptr(idx), _ptr(w), _ptr(workspace),
        workspace.numel(), _ptr(status), _stream(stream)))


def k3moe_expert_ffn_mxfp4(dims: LayerDims, x, experts, expert_stride: int, idx, w, y,
                           workspace, status, accumulate: bool = False, stream=None):
    d = dims.c()
    x = _bits16(x, "x")
    T = x.shape[0]
    ydt = F32 if y.dtype == torch.float32 else BF16
    if ydt == BF16:
        y = _bits16(y, "y")
    ex = Experts(ctypes.c_void_p(experts.data_ptr()), int(expert_stride))
    _check("k3moe_expert_ffn_mxfp4", lib().k3moe_expert_ffn_mxfp4(
        ctypes.byref(d), _ptr(x), T, ctypes.byref(ex), _ptr(idx), _ptr(w), _ptr(y), ydt,
        int(bool(accumulate)), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream)))


def k3moe_layer(dims: LayerDims, x, wr, bias, experts, expert_stride: int, sh_gate, sh_up,
                sh_down, y, workspace, status, idx_out=None, w_out=None,
                accumulate: bool = False, stream=None):
    d = dims.c()
    x, wr = _bits16(x, "x"), _bits16(wr, "wr")
    if sh_gate is not None:
        sh_gate, sh_up, sh_down = (_bits16(sh_gate, "sh_gate"), _bits16(sh_up, "sh_up"),
                                   _bits16(sh_down, "sh_down"))
    T = x.shape[0]
    ydt = F32 if y.dtype == torch.float32 else BF16
    if ydt == BF16:
        y = _bits16(y, "y")
    ex = Experts(ctypes.c_void_p(experts.data_ptr()), int(expert_stride))
    _check("k3moe_layer", lib().k3moe_layer(
        ctypes.byref(d), _ptr(x), T, _ptr(wr), _ptr(bias), ctypes.byref(ex), _ptr(sh_gate),
        _ptr(sh_up), _ptr(sh_down), _ptr(idx_out), _ptr(w_out), _ptr(y), ydt,
        int(bool(accumulate)), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream)))


def k3moe_layer_static_scratch(dims: LayerDims, x, wr, bias, experts, expert_stride: int,
                               sh_gate, sh_up, sh_down, y, status, idx_out=None, w_out=None,
                               accumulate: bool = False, stream=None):
    """k3moe_layer with the library's static scratch array in place of a workspace: for
    callers that must not allocate device memory while they run the layer."""
    d = dims.c()
    x, wr = _bits16(x, "x"), _bits16(wr, "wr")
    if sh_gate is not None:
        sh_gate, sh_up, sh_down = (_bits16(sh_gate, "sh_gate"), _bits16(sh_up, "sh_up"),
                                   _bits16(sh_down, "sh_down"))
    T = x.shape[0]
    ydt = F32 if y.dtype == torch.float32 else BF16
    if ydt == BF16:
        y = _bits16(y, "y")
    ex = Experts(ctypes.c_void_p(experts.data_ptr()), int(expert_stride))
    _check("k3moe_layer_static_scratch", lib().k3moe_layer_static_scratch(
        ctypes.byref(d), _ptr(x), T, _ptr(wr), _ptr(bias), ctypes.byref(ex), _ptr(sh_gate),
        _ptr(sh_up), _ptr(sh_down), _ptr(idx_out), _ptr(w_out), _ptr(y), ydt,
        int(bool(accumulate)), _ptr(status), _stream(stream)))


def k3moe_decode_stack(dims: LayerDims, layers, h, x_scratch, workspace, status, eps: float = 1e-5,
                       idx_out=None, w_out=None, stream=None):
    """h (float [T][H], updated in place) through the stacked layers; ``layers`` is a
    list of dicts with wr, bias, experts, stride and (optional) sh_gate, sh_up, sh_down."""
    d = dims.c()
    arr = (LayerWeights * len(layers))()
    keep = []
    for i, lw in enumerate(layers):
        wr = _bits16(lw["wr"], "wr")
        sh = [lw.get(k) for k in ("sh_gate", "sh_up", "sh_down")]
        sh = [None if t is None else _bits16(t, k) for t, k in zip(sh, ("sh_gate", "sh_up", "sh_down"))]
        keep += [wr] + sh
        arr[i] = LayerWeights(_ptr(wr), _ptr(lw.get("bias")),
                              Experts(ctypes.c_void_p(lw["experts"].data_ptr()), int(lw["stride"])),
                              *[_ptr(t) for t in sh])
    T = h.shape[0]
    x_scratch = _bits16(x_scratch, "x_scratch")
    _check("k3moe_decode_stack", lib().k3moe_decode_stack(
        ctypes.byref(d), len(layers), arr, T, _ptr(h), float(eps), _ptr(x_scratch),
        _ptr(idx_out), _ptr(w_out), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream)))


def k3moe_rmsnorm_bf16(h, out, eps: float = 1e-5, stream=None):
    T, n = h.shape
    out = _bits16(out, "out")
    _check("k3moe_rmsnorm_bf16", lib().k3moe_rmsnorm_bf16(
        _ptr(h), T, n, float(eps), _ptr(out), _stream(stream)))


def k3moe_dequant_mxfp4(packed, scales, rows: int, cols: int, out, stream=None):
    _check("k3moe_dequant_mxfp4", lib().k3moe_dequant_mxfp4(
        _ptr(packed), _ptr(scales), int(rows), int(cols), _ptr(out), _stream(stream)))


@dataclass
class LatentDims:
    """Shapes of a LatentMoE layer (k3moe_latent_dims)."""
    hidden: int
    latent: int
    inter: int
    n_experts: int
    topk: int
    shared_inter: int = 0
    situ_b1: float = 4.0
    situ_b2: float = 25.0
    routed_scale: float = 1.0
    rms_eps: float = 1e-5
    renorm: int = 1
    latent_norm: int = 1
    group: int = 32

    def c(self) -> LatentDimsC:
        return LatentDimsC(self.hidden, self.latent, self.inter, self.n_experts, self.topk,
                           self.group, self.shared_inter, self.situ_b1, self.situ_b2,
                           self.routed_scale, self.rms_eps, self.renorm, self.latent_norm)


def latent_workspace_size(dims: LatentDims, T: int) -> int:
    d = dims.c()
    return int(lib().k3moe_latent_workspace_size(ctypes.byref(d), int(T)))


def new_latent_workspace(dims: LatentDims, T: int, device=None) -> torch.Tensor:
    n = latent_workspace_size(dims, T)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def k3moe_latent_layer(dims: LatentDims, x, wr, bias, w_down, w_up, norm_w, experts,
                       expert_stride: int, sh_gate, sh_up, sh_down, y, workspace, status,
                       idx_out=None, w_out=None, accumulate: bool = False, stream=None):
    """The LatentMoE layer step (k3moe_latent_layer): tensors on the device, bf16 weights
    and x as bf16 or their 16-bit patterns, norm_w float [L] (or None without the norm)."""
    d = dims.c()
    x, wr = _bits16(x, "x"), _bits16(wr, "wr")
    w_down, w_up = _bits16(w_down, "w_down"), _bits16(w_up, "w_up")
    if sh_gate is not None:
        sh_gate, sh_up, sh_down = (_bits16(sh_gate, "sh_gate"), _bits16(sh_up, "sh_up"),
                                   _bits16(sh_down, "sh_down"))
    T = x.shape[0]
    ydt = F32 if y.dtype == torch.float32 else BF16
    if ydt == BF16:
        y = _bits16(y, "y")
    lw = LatentWeightsC(_ptr(wr), _ptr(bias), _ptr(w_down), _ptr(w_up), _ptr(norm_w),
                        Experts(ctypes.c_void_p(experts.data_ptr()), int(expert_stride)),
                        _ptr(sh_gate), _ptr(sh_up), _ptr(sh_down))
    _check("k3moe_latent_layer", lib().k3moe_latent_layer(
        ctypes.byref(d), ctypes.byref(lw), _ptr(x), T, _ptr(idx_out), _ptr(w_out), _ptr(y), ydt,
        int(bool(accumulate)), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream)))


class ExpertCache:
    """The library's host-side expert cache (k3moe_cache_create): the records of n_layers
    layers in host memory (``host_ptrs``: one address per layer, records ``host_stride``
    apart), ``n_slots`` record-sized slots at device address ``slots_ptr``."""

    def __init__(self, host_ptrs, n_experts: int, record_bytes: int, host_stride: int,
                 slots_ptr: int, n_slots: int, slot_stride: int):
        arr = (ctypes.c_void_p * len(host_ptrs))(*[ctypes.c_void_p(int(p)) for p in host_ptrs])
        self._keep = arr
        h = ctypes.c_void_p()
        _check("k3moe_cache_create", lib().k3moe_cache_create(
            len(host_ptrs), arr, int(n_experts), int(record_bytes), int(host_stride),
            ctypes.c_void_p(int(slots_ptr)), int(n_slots), int(slot_stride), ctypes.byref(h)))
        self.handle = h
        self.n_slots = n_slots

    def lookup(self, layer: int, experts):
        """(slots, load) for one call's experts (host only: the cache's decision, the reads
        taken as done).  Raises K3MoeError (ERR_CACHE_FULL) when they do not fit."""
        import numpy as np
        e = np.ascontiguousarray(experts, dtype=np.int32)
        slots = np.empty_like(e)
        load = np.empty_like(e)
        _check("k3moe_cache_lookup", lib().k3moe_cache_lookup(
            self.handle, int(layer), e.ctypes.data_as(ctypes.c_void_p), e.size,
            slots.ctypes.data_as(ctypes.c_void_p), load.ctypes.data_as(ctypes.c_void_p)))
        return slots, load

    def stats(self):
        h, m, b = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check("k3moe_cache_stats", lib().k3moe_cache_stats(self.handle, ctypes.byref(h),
                                                              ctypes.byref(m), ctypes.byref(b)))
        return {"hits": h.value, "misses": m.value, "bytes_loaded": b.value}

    def close(self):
        if self.handle:
            lib().k3moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def streamed_workspace_size(dims: LayerDims, T: int) -> int:
    d = dims.c()
    return int(lib().k3moe_streamed_workspace_size(ctypes.byref(d), int(T)))


def new_streamed_workspace(dims: LayerDims, T: int, device=None) -> torch.Tensor:
    n = streamed_workspace_size(dims, T)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def k3moe_layer_streamed(dims: LayerDims, cache: ExpertCache, layer: int, x, wr, bias, sh_gate,
                         sh_up, sh_down, y, workspace, status, idx_out=None, w_out=None,
                         accumulate: bool = False, stream=None):
    """k3moe_layer with the routed experts read through the expert cache."""
    d = dims.c()
    x, wr = _bits16(x, "x"), _bits16(wr, "wr")
    if sh_gate is not None:
        sh_gate, sh_up, sh_down = (_bits16(sh_gate, "sh_gate"), _bits16(sh_up, "sh_up"),
                                   _bits16(sh_down, "sh_down"))
    T = x.shape[0]
    ydt = F32 if y.dtype == torch.float32 else BF16
    if ydt == BF16:
        y = _bits16(y, "y")
    _check("k3moe_layer_streamed", lib().k3moe_layer_streamed(
        ctypes.byref(d), cache.handle, int(layer), _ptr(x), T, _ptr(wr), _ptr(bias),
        _ptr(sh_gate), _ptr(sh_up), _ptr(sh_down), _ptr(idx_out), _ptr(w_out), _ptr(y), ydt,
        int(bool(accumulate)), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream)))


def status_str(code: int) -> str:
    return lib().k3moe_status_str(int(code)).decode()


def k3moe_test_expire_wait(on: bool = True):
    """While on, the single-token fused step's second grid dependency cannot complete and its
    wait gives up after ~0.1 s (status K3MOE_ERR_TIMEOUT, output taken as zero)."""
    _check("k3moe_test_expire_wait", lib().k3moe_test_expire_wait(int(bool(on))))


def k3moe_trace_enable(on: bool = True):
    _check("k3moe_trace_enable", lib().k3moe_trace_enable(int(bool(on))))


def k3moe_trace_read() -> dict:
    """{kernel name: (total ms, launches)} for every kernel the library launched."""
    L = lib()
    n = L.k3moe_trace_read(-1, None, None, None)
    out = {}
    for k in range(n):
        name = ctypes.c_char_p()
        ms = ctypes.c_double()
        cnt = ctypes.c_int64()
        L.k3moe_trace_read(k, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(cnt))
        out[name.value.decode()] = (ms.value, cnt.value)
    return out
