"""k3moe_layer_static_scratch: the layer step with the library's static scratch array in
place of a caller workspace.  Its results must agree with k3moe_layer's on the same
inputs, call after call (every call shares the one array), and a request larger than the
array must be refused before anything runs.

The file name sorts last so that the GPU test also runs after every other test in one
process; it passes alone in a fresh process as well.
"""
import ctypes
import dataclasses
import os
import re

import pytest
import torch

import synth
import mxfp4_routed_expert_02_gb300 as k3
from mxfp4_routed_expert_02_gb300 import k3moe as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def model_dims(**kw):
    base = dict(hidden=7168, inter=1536, n_experts=896, topk=16, shared_inter=1536)
    base.update(kw)
    return k3.LayerDims(**base)


def test_static_scratch_size_matches_header_and_holds_the_model_shape():
    hdr = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    m = re.search(r"#define\s+K3MOE_STATIC_SCRATCH_BYTES\s+\((\d+)u \* (\d+)u \* (\d+)u\)", hdr)
    assert m, "K3MOE_STATIC_SCRATCH_BYTES not found"
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == k3.STATIC_SCRATCH_BYTES
    # the model shape fits up to nine tokens, the size the header states
    for T in (1, 2, 9):
        assert 0 < k3.workspace_size(model_dims(), T) <= k3.STATIC_SCRATCH_BYTES
    assert k3.workspace_size(model_dims(), 10) > k3.STATIC_SCRATCH_BYTES


def test_static_scratch_refuses_requests_beyond_its_size():
    """Checked on the host before any device work: no pointer is touched."""
    d = model_dims(hidden=8192, inter=8192, n_experts=4096, topk=32, shared_inter=0)
    assert k3.workspace_size(d, 64) > k3.STATIC_SCRATCH_BYTES
    c = d.c()
    ex = B.Experts(None, 0)
    code = k3.lib().k3moe_layer_static_scratch(
        ctypes.byref(c), None, 64, None, None, ctypes.byref(ex), None, None, None, None, None,
        None, B.F32, 0, None, None)
    assert code == B.K3MOE_ERR_SCRATCH_LIMIT
    assert "static" in k3.status_str(code)
    # the model shape at one token is within the limit: the call gets past the size check
    # and then fails on the NULL pointers (ERR_ARG), or without a GPU at the device
    # set-up (ERR_CUDA)
    c = model_dims().c()
    code = k3.lib().k3moe_layer_static_scratch(
        ctypes.byref(c), None, 1, None, None, ctypes.byref(ex), None, None, None, None, None,
        None, B.F32, 0, None, None)
    assert code in (1, 5)


# ------------------------------------------------------------------------------ on GPU
CASES = [
    # name, hidden, inter, experts, topk, shared experts, tokens, output dtype
    ("tiny_f32", 256, 128, 16, 2, 1, 4, torch.float32),
    ("tiny_bf16", 256, 128, 16, 2, 1, 4, torch.bfloat16),
    ("two_passes", 256, 128, 16, 2, 1, 65, torch.float32),
    ("decode_width_t1", 7168, 1536, 40, 16, 1, 1, torch.float32),
    # the largest request within the limit: the model's shape at nine tokens (tensor-core
    # path), 8,157,952 of the array's 8,388,608 bytes
    ("model_t9", 7168, 1536, 896, 16, 1, 9, torch.float32),
]


def _layer_inputs(H, I, E, K, NS, T, seed):
    from parity import Layer
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", hidden=H, inter=I,
                              n_experts=E, topk=K, tokens=T, n_shared=NS)
    return Layer(cfg, seed=seed, device_fill=E * cfg.record_bytes > (64 << 20))


def _run(L, x, ydt, static):
    T, H, K = x.shape[0], L.cfg.hidden, L.cfg.topk
    y = torch.zeros((T, H), dtype=ydt, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    st = k3.new_status()
    if static:
        k3.k3moe_layer_static_scratch(L.dims, x, L.d_wr, L.d_bias, L.experts, L.stride,
                                      L.d_sg, L.d_su, L.d_sd, y, st, idx_out=idx, w_out=w)
    else:
        ws = k3.new_workspace(L.dims, T)
        k3.k3moe_layer(L.dims, x, L.d_wr, L.d_bias, L.experts, L.stride, L.d_sg, L.d_su,
                       L.d_sd, y, ws, st, idx_out=idx, w_out=w)
    return y, idx, w, st


@pytest.mark.gpu
@pytest.mark.parametrize("name,H,I,E,K,NS,T,ydt", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_workspace_call_two_calls_in_a_row(name, H, I, E, K, NS, T, ydt):
    L = _layer_inputs(H, I, E, K, NS, T, seed=11 + T)
    xa = L.d_x
    # a second input with other routes: the tokens in reverse order, and every sign
    # flipped (which negates every router logit)
    xb = torch.flip(L.d_x, dims=[0]).contiguous() ^ -32768
    # the workspace call first, then two static-scratch calls on different inputs in a
    # row: the second overwrites the scratch the first used
    ref_a = _run(L, xa, ydt, static=False)
    ref_b = _run(L, xb, ydt, static=False)
    got_a = _run(L, xa, ydt, static=True)
    got_b = _run(L, xb, ydt, static=True)
    torch.cuda.synchronize()
    # the two inputs route differently, so a read of the first call's scratch would show
    assert not torch.equal(ref_a[1], ref_b[1])
    # the kernels are deterministic: the same inputs give the same bits, whatever memory
    # holds the scratch
    for ref, got in ((ref_a, got_a), (ref_b, got_b)):
        y_r, i_r, w_r, s_r = ref
        y_g, i_g, w_g, s_g = got
        assert int(s_r.item()) == 0 and int(s_g.item()) == 0
        assert torch.equal(i_g, i_r)
        assert torch.equal(w_g, w_r)
        assert torch.equal(y_g, y_r)
