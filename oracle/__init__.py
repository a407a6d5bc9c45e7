"""CPU oracle for the Kimi-K3 MoE layer step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  It wraps ``k3moe_oracle.c`` (plain C, fp64 accumulation) through
ctypes and numpy; it shares no code with the CUDA library.

Every function names the passage it follows; "kimi-k3-in-c" is the README of
FareedKhan-dev/kimi-k3-in-c, "Kimi-K3.cpp" the README of Maknee/Kimi-K3.cpp.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``: the
number formats by the page's printed E2M1 table and the closed form of E8M0, the
products and the top-k by brute force on tiny inputs, the router weights, SiTU and the
layer composition by invariants and special cases, the routed sum by sums whose float
result depends on the order of the terms.  None is "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def lib():
    """Load (building first if needed) the oracle shared object."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        c_int, c_float = ctypes.c_int, ctypes.c_float
        sig = {
            "k3o_e2m1": (ctypes.c_double, [c_int]),
            "k3o_e8m0": (ctypes.c_double, [c_int]),
            "k3o_bf16_to_f32": (c_float, [ctypes.c_uint16]),
            "k3o_f32_to_bf16": (ctypes.c_uint16, [c_float]),
            "k3o_dequant_mxfp4": (None, [c_int, c_int, u8p, u8p, f32p]),
            "k3o_mxfp4_gemv": (None, [c_int, c_int, u8p, u8p, f32p, f32p, c_int]),
            "k3o_bf16_gemv": (None, [c_int, c_int, u16p, f32p, f32p, c_int]),
            "k3o_rmsnorm": (None, [c_int, f32p, f32p, c_float, f32p]),
            "k3o_router": (c_int, [c_int, c_int, c_int, c_int, c_int, c_float, u16p, u16p, f32p,
                                   i32p, f32p, f32p, f32p, c_int]),
            "k3o_situ": (None, [c_int, c_float, c_float, f32p, f32p, f32p]),
            "k3o_record_offsets": (None, [c_int, c_int, i64p]),
            "k3o_expert": (None, [c_int, c_int, u8p, f32p, c_float, c_float, f32p, c_int]),
            "k3o_shared_expert": (None, [c_int, c_int, u16p, u16p, u16p, f32p, c_float, c_float,
                                         f32p, c_int]),
            "k3o_moe_token": (None, [c_int, c_int, c_int, c_int, u16p, ctypes.POINTER(u8p), f32p,
                                     u16p, u16p, u16p, c_float, c_float, f32p, c_int]),
            "k3o_combine": (None, [c_int, c_int, f32p, f32p, f32p, f32p]),
            "k3o_latent_moe_token": (None, [c_int, c_int, c_int, c_int, c_int, u16p, u16p, u16p,
                                            f32p, c_int, c_float, ctypes.POINTER(u8p), f32p,
                                            u16p, u16p, u16p, c_float, c_float, f32p, f32p,
                                            f32p, c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _p(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# ----------------------------------------------------------------------------------
# number formats (kimi-k3-in-c, section 4 "Reduction one")
# ----------------------------------------------------------------------------------
def e2m1(code: int) -> float:
    """Value of a 4-bit E2M1 code (the page's printed 16-entry table)."""
    return lib().k3o_e2m1(int(code))


def e8m0(b: int) -> float:
    """Scale of an E8M0 byte: 2^(b-127), with b = 255 mapped to 0."""
    return lib().k3o_e8m0(int(b))


def bf16_to_f32(h) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (kimi-k3-in-c, section 5: a 16-bit shift)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """Round float32 to bf16 bit patterns, nearest-even (through the C routine)."""
    x = np.asarray(x, dtype=np.float32)
    L = lib()
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in, flat_out = x.ravel(), out.ravel()
    for i in range(flat_in.size):
        flat_out[i] = L.k3o_f32_to_bf16(float(flat_in[i]))
    return out


def dequant_mxfp4(packed, scales, rows: int, cols: int) -> np.ndarray:
    """Dequantised float weights [rows][cols] = E2M1(nibble) * E8M0(scale) (exact)."""
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().k3o_dequant_mxfp4(rows, cols, _p(packed, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                            _p(out, ctypes.c_float))
    return out


def mxfp4_gemv(packed, scales, rows: int, cols: int, x, nthreads: int = 0) -> np.ndarray:
    """y = W x read straight from MXFP4 (kimi-k3-in-c, section 4, the nibble product)."""
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    x = _c(x, np.float32)
    y = np.empty(rows, dtype=np.float32)
    lib().k3o_mxfp4_gemv(rows, cols, _p(packed, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                         _p(x, ctypes.c_float), _p(y, ctypes.c_float), nthreads)
    return y


def bf16_gemv(W, x, nthreads: int = 0) -> np.ndarray:
    """y = W x for bf16 W [rows][cols], double accumulation (kimi-k3-in-c, section 5)."""
    W = _c(W, np.uint16)
    x = _c(x, np.float32)
    rows, cols = W.shape
    y = np.empty(rows, dtype=np.float32)
    lib().k3o_bf16_gemv(rows, cols, _p(W, ctypes.c_uint16), _p(x, ctypes.c_float),
                        _p(y, ctypes.c_float), nthreads)
    return y


def rmsnorm(x, w=None, eps: float = 1e-5) -> np.ndarray:
    """RMSNorm with epsilon inside the square root (kimi-k3-in-c, section 5)."""
    x = _c(x, np.float32)
    out = np.empty_like(x)
    wp = None if w is None else _c(w, np.float32)
    lib().k3o_rmsnorm(x.size, _p(x, ctypes.c_float), _p(wp, ctypes.c_float), eps,
                      _p(out, ctypes.c_float))
    return out


def router(x_bf16, wr_bf16, bias, topk: int, renorm: bool = True, routed_scale: float = 1.0,
           nthreads: int = 0):
    """Router for T tokens (kimi-k3-in-c, section 9 "Picking 16 experts of 896").

    Returns ``(idx int32 [T][K], w float32 [T][K], logits float32 [T][E],
    scores float32 [T][E])``; raises ValueError if a score is not finite.
    """
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    wr = _c(wr_bf16, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    assert wr.shape[1] == H
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=np.float32)
    logits = np.empty((T, E), dtype=np.float32)
    scores = np.empty((T, E), dtype=np.float32)
    st = lib().k3o_router(T, H, E, topk, int(bool(renorm)), float(routed_scale),
                          _p(x, ctypes.c_uint16), _p(wr, ctypes.c_uint16),
                          _p(b, ctypes.c_float), _p(idx, ctypes.c_int32), _p(w, ctypes.c_float),
                          _p(logits, ctypes.c_float), _p(scores, ctypes.c_float), nthreads)
    if st != 0:
        raise ValueError("oracle router: non-finite score")
    return idx, w, logits, scores


def situ(g, u, b1: float = 4.0, b2: float = 25.0) -> np.ndarray:
    """SiTU-GLU, the sigmoid on the uncapped gate (kimi-k3-in-c, section 9)."""
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    act = np.empty_like(g)
    lib().k3o_situ(g.size, b1, b2, _p(g, ctypes.c_float), _p(u, ctypes.c_float),
                   _p(act, ctypes.c_float))
    return act


def record_offsets(H: int, I: int):
    """Byte offsets (w1p, w1s, w2p, w2s, w3p, w3s, total) of one expert record."""
    off = np.zeros(7, dtype=np.int64)
    lib().k3o_record_offsets(H, I, _p(off, ctypes.c_int64))
    return [int(v) for v in off]


def expert(rec, x_f32, H: int, I: int, b1: float = 4.0, b2: float = 25.0,
           nthreads: int = 0) -> np.ndarray:
    """One routed expert on one token: W2 SiTU(W1 x, W3 x) (section 9, step 3)."""
    rec = _c(rec, np.uint8)
    x = _c(x_f32, np.float32)
    d = np.empty(H, dtype=np.float32)
    lib().k3o_expert(H, I, _p(rec, ctypes.c_uint8), _p(x, ctypes.c_float), b1, b2,
                     _p(d, ctypes.c_float), nthreads)
    return d


def shared_expert(gate, up, down, x_f32, b1: float = 4.0, b2: float = 25.0,
                  nthreads: int = 0) -> np.ndarray:
    """Shared expert on one token (section 9, step 6), bf16 weights."""
    gate = _c(gate, np.uint16)
    up = _c(up, np.uint16)
    down = _c(down, np.uint16)
    x = _c(x_f32, np.float32)
    SI, H = gate.shape
    ds = np.empty(H, dtype=np.float32)
    lib().k3o_shared_expert(H, SI, _p(gate, ctypes.c_uint16), _p(up, ctypes.c_uint16),
                            _p(down, ctypes.c_uint16), _p(x, ctypes.c_float), b1, b2,
                            _p(ds, ctypes.c_float), nthreads)
    return ds


def combine(w, d, ds=None) -> np.ndarray:
    """Routed sum in router order plus the shared expert (section 9, LatentMoE listing
    steps 3 and 6): acc = 0; acc = acc + w[j] * d[j] for j = 0..K-1 in float, one
    rounding per product and per sum; then acc + ds (one float add) when ds is given.
    d is [K][H]."""
    w = _c(w, np.float32)
    d = _c(np.atleast_2d(d), np.float32)
    K, H = d.shape
    assert w.shape == (K,)
    dsa = None if ds is None else _c(ds, np.float32)
    y = np.empty(H, dtype=np.float32)
    lib().k3o_combine(H, K, _p(w, ctypes.c_float), _p(d, ctypes.c_float),
                      _p(dsa, ctypes.c_float), _p(y, ctypes.c_float))
    return y


def moe_token(x_bf16, recs, w, H: int, I: int, sh_gate=None, sh_up=None, sh_down=None,
              b1: float = 4.0, b2: float = 25.0, nthreads: int = 0) -> np.ndarray:
    """Layer output for one routed token: the float sum of w_j d_j in router order, then
    the shared expert's output added unweighted (``combine``)."""
    x = _c(x_bf16, np.uint16)
    K = len(recs)
    recs = [_c(r, np.uint8) for r in recs]
    arr = (ctypes.POINTER(ctypes.c_uint8) * K)(*[_p(r, ctypes.c_uint8) for r in recs])
    w = _c(w, np.float32)
    SI = 0 if sh_gate is None else int(np.asarray(sh_gate).shape[0])
    g = None if sh_gate is None else _c(sh_gate, np.uint16)
    u = None if sh_up is None else _c(sh_up, np.uint16)
    dn = None if sh_down is None else _c(sh_down, np.uint16)
    y = np.empty(H, dtype=np.float32)
    lib().k3o_moe_token(H, I, K, SI, _p(x, ctypes.c_uint16), arr, _p(w, ctypes.c_float),
                        _p(g, ctypes.c_uint16), _p(u, ctypes.c_uint16), _p(dn, ctypes.c_uint16),
                        b1, b2, _p(y, ctypes.c_float), nthreads)
    return y


def moe_layer(x_bf16, wr_bf16, bias, get_expert, topk: int, H: int, I: int, sh_gate=None,
              sh_up=None, sh_down=None, renorm: bool = True, routed_scale: float = 1.0,
              b1: float = 4.0, b2: float = 25.0, tokens=None, nthreads: int = 0):
    """Full layer step for the tokens listed in ``tokens`` (default: all).

    ``get_expert(e)`` returns the byte record of routed expert ``e``.  Returns
    ``(idx, w, y)`` with y float32 [len(tokens)][H].
    """
    x = np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16))
    if tokens is None:
        tokens = range(x.shape[0])
    tokens = list(tokens)
    idx, w, _, _ = router(x[tokens], wr_bf16, bias, topk, renorm, routed_scale, nthreads)
    y = np.empty((len(tokens), H), dtype=np.float32)
    cache = {}
    for n, t in enumerate(tokens):
        recs = []
        for e in idx[n]:
            e = int(e)
            if e not in cache:
                cache[e] = get_expert(e)
            recs.append(cache[e])
        y[n] = moe_token(x[t], recs, w[n], H, I, sh_gate, sh_up, sh_down, b1, b2, nthreads)
        if len(cache) > 64:
            cache.clear()
    return idx, w, y


def latent_moe_token(x_bf16, recs, w, H: int, L: int, I: int, w_down, w_up, norm_w=None,
                     latent_norm: bool = True, eps: float = 1e-5, sh_gate=None, sh_up=None,
                     sh_down=None, b1: float = 4.0, b2: float = 25.0, nthreads: int = 0,
                     intermediates: bool = False):
    """One routed token through the LatentMoE (kimi-k3-in-c, section 9, LatentMoE listing
    steps 2-6): z = Wdn x; the float router-order sum of w_j expert_j(z) in the latent;
    RMSNorm of that aggregate (weight norm_w, eps) when latent_norm; Wup times it; plus
    the shared experts on the original x, unweighted.  Returns y [H], or (y, z, accL)
    with intermediates=True."""
    x = _c(x_bf16, np.uint16)
    K = len(recs)
    recs = [_c(r, np.uint8) for r in recs]
    arr = (ctypes.POINTER(ctypes.c_uint8) * max(K, 1))(*[_p(r, ctypes.c_uint8) for r in recs])
    w = _c(w, np.float32)
    wdn = _c(w_down, np.uint16)
    wup = _c(w_up, np.uint16)
    assert wdn.shape == (L, H) and wup.shape == (H, L)
    nw = _c(np.ones(L, np.float32) if norm_w is None else norm_w, np.float32)
    SI = 0 if sh_gate is None else int(np.asarray(sh_gate).shape[0])
    g = None if sh_gate is None else _c(sh_gate, np.uint16)
    u = None if sh_up is None else _c(sh_up, np.uint16)
    dn = None if sh_down is None else _c(sh_down, np.uint16)
    y = np.empty(H, dtype=np.float32)
    z = np.empty(L, dtype=np.float32)
    acc = np.empty(L, dtype=np.float32)
    lib().k3o_latent_moe_token(H, L, I, K, SI, _p(x, ctypes.c_uint16), _p(wdn, ctypes.c_uint16),
                               _p(wup, ctypes.c_uint16), _p(nw, ctypes.c_float),
                               int(bool(latent_norm)), float(eps), arr, _p(w, ctypes.c_float),
                               _p(g, ctypes.c_uint16), _p(u, ctypes.c_uint16),
                               _p(dn, ctypes.c_uint16), b1, b2, _p(y, ctypes.c_float),
                               _p(z, ctypes.c_float), _p(acc, ctypes.c_float), nthreads)
    return (y, z, acc) if intermediates else y


def latent_moe_layer(x_bf16, wr_bf16, bias, get_expert, topk: int, H: int, L: int, I: int,
                     w_down, w_up, norm_w=None, latent_norm: bool = True, eps: float = 1e-5,
                     sh_gate=None, sh_up=None, sh_down=None, renorm: bool = True,
                     routed_scale: float = 1.0, b1: float = 4.0, b2: float = 25.0,
                     tokens=None, nthreads: int = 0):
    """The LatentMoE layer for the listed tokens: step 1 routes on the FULL-width x
    (``router``), steps 2-6 are ``latent_moe_token``.  ``get_expert(e)`` returns expert
    e's record of the (L, I) layout.  Returns (idx, w, y [len(tokens)][H])."""
    x = np.atleast_2d(np.asarray(x_bf16, dtype=np.uint16))
    tokens = list(range(x.shape[0]) if tokens is None else tokens)
    idx, w, _, _ = router(x[tokens], wr_bf16, bias, topk, renorm, routed_scale, nthreads)
    y = np.empty((len(tokens), H), dtype=np.float32)
    cache = {}
    for n, t in enumerate(tokens):
        recs = []
        for e in idx[n]:
            e = int(e)
            if e not in cache:
                cache[e] = get_expert(e)
            recs.append(cache[e])
        y[n] = latent_moe_token(x[t], recs, w[n], H, L, I, w_down, w_up, norm_w, latent_norm,
                                eps, sh_gate, sh_up, sh_down, b1, b2, nthreads)
        if len(cache) > 64:
            cache.clear()
    return idx, w, y


def stacked_decode_step(h, layers, topk: int, H: int, I: int, eps: float = 1e-5,
                        renorm: bool = True, routed_scale: float = 1.0, b1: float = 4.0,
                        b2: float = 25.0, nthreads: int = 0):
    """One token through stacked MoE layers with the residual stream between them.

    The decoder loop of kimi-k3-in-c: RMSNorm with weight 1 (section 5 "Kernels with a
    floating point contract"), the layer input rounded to bf16 (the page's layers take
    bf16 activations), the layer step of section 9, and its output added to the residual
    stream in float.  ``layers`` holds dicts with wr, bias, get_expert and (optional)
    sh_gate, sh_up, sh_down.  Returns (h_new, [idx per layer], [w per layer]).
    """
    h = np.array(h, dtype=np.float32)
    idxs, ws = [], []
    for lw in layers:
        x = f32_to_bf16(rmsnorm(h, eps=eps))
        idx, w, y = moe_layer(x[None, :], lw["wr"], lw["bias"], lw["get_expert"], topk, H, I,
                              lw.get("sh_gate"), lw.get("sh_up"), lw.get("sh_down"), renorm,
                              routed_scale, b1, b2, nthreads=nthreads)
        h = (h + y[0]).astype(np.float32)
        idxs.append(idx[0])
        ws.append(w[0])
    return h, idxs, ws


def num_threads() -> int:
    """Threads the oracle's parallel loops use by default (OpenMP)."""
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
