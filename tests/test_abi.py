"""The C ABI library loads and exports every symbol include/k3moe.h declares; host-side
argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

import mxfp4_routed_expert_02_gb300 as k3
from mxfp4_routed_expert_02_gb300 import k3moe as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_\w+)\s*\(", src)))


def test_header_declares_exactly_the_bound_symbols():
    assert header_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = k3.lib()
    for name in header_functions():
        assert hasattr(L, name), name


def test_oracle_is_not_linked_into_the_library():
    L = k3.lib()
    for name in ("k3o_router", "k3o_mxfp4_gemv", "k3o_moe_token"):
        with pytest.raises(AttributeError):
            getattr(L, name)


def test_expiry_hook_needs_no_device():
    # the hook only sets a host flag the next fused launch reads
    L = k3.lib()
    assert L.k3moe_test_expire_wait(1) == 0
    assert L.k3moe_test_expire_wait(0) == 0


def dims(**kw):
    base = dict(hidden=7168, inter=1536, n_experts=896, topk=16, shared_inter=1536)
    base.update(kw)
    return k3.LayerDims(**base)


def test_record_layout_and_workspace_queries():
    assert k3.record_layout(dims()) == [0, 5505024, 5849088, 11354112, 11698176, 17203200,
                                        17547264]
    assert k3.workspace_size(dims(), 0) == 16
    w1, w2, w4096, w5000 = (k3.workspace_size(dims(), t) for t in (1, 2, 4096, 5000))
    # multi-token passes of at most 4096 tokens reuse one workspace
    assert 0 < w1 < w2 < w4096 == w5000
    # shapes the tensor-core path does not take keep the 64-token decode passes
    small = dims(hidden=96, inter=64, n_experts=5, topk=3, shared_inter=64)
    assert k3.workspace_size(small, 64) == k3.workspace_size(small, 65)
    assert k3.workspace_size(dims(hidden=100), 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=100), 2), (dict(inter=40), 2), (dict(topk=0), 2), (dict(topk=33), 2),
    (dict(n_experts=4, topk=5), 2), (dict(group=16), 2), (dict(situ_b1=0.0), 1),
])
def test_bad_dims_are_refused(kw, code):
    d = dims(**kw).c()
    off = (ctypes.c_int64 * 7)()
    assert k3.lib().k3moe_record_layout(ctypes.byref(d), off) == code


def test_null_arguments_are_refused_on_the_host():
    L = k3.lib()
    d = dims().c()
    ex = B.Experts(None, 17547264)
    # every call checks its pointers before touching the device
    assert L.k3moe_layer(ctypes.byref(d), None, 1, None, None, ctypes.byref(ex), None, None, None,
                         None, None, None, 0, 0, None, 0, None, None) == 1
    assert L.k3moe_route(ctypes.byref(d), None, None, None, 1, None, None, None, 0, None,
                         None) == 1
    assert L.k3moe_expert_ffn_mxfp4(ctypes.byref(d), None, 1, ctypes.byref(ex), None, None, None,
                                    0, 0, None, 0, None, None) == 1
    # zero tokens is a no-op
    assert L.k3moe_layer(ctypes.byref(d), None, 0, None, None, ctypes.byref(ex), None, None, None,
                         None, None, None, 0, 0, None, 0, None, None) == 0
    assert L.k3moe_dequant_mxfp4(None, None, 4, 48, None, None) == 2


def test_status_strings():
    for c in range(9):
        assert k3.status_str(c)
    assert k3.status_str(7) == "expert index out of range"
