"""Failure detection on the GPU without a fault: a grid-wide dependency that can never
complete makes the fused single-token kernel's bounded wait give up.  The call must end
on its own, report K3MOE_ERR_TIMEOUT in the status word, take the layer's output as zero,
and leave the context and the workspace (whose counters the kernel zeroes on exit) fit
for the next call, which must match the oracle again."""
import time

import numpy as np
import pytest
import torch

import mxfp4_routed_expert_02_gb300 as k3
from parity import fused_layer, rel_l2, REL_L2_F32

pytestmark = pytest.mark.gpu

TIMEOUT = 6  # K3MOE_ERR_TIMEOUT


def call(L, ws, st, y, accumulate=False):
    k3.k3moe_layer(L.dims, L.d_x, L.d_wr, L.d_bias, L.experts, L.stride, L.d_sg, L.d_su,
                   L.d_sd, y, ws, st, accumulate=accumulate)
    torch.cuda.synchronize()
    return int(st.item())


def expired(fn):
    k3.k3moe_test_expire_wait(True)
    try:
        t0 = time.perf_counter()
        out = fn()
        return out, time.perf_counter() - t0
    finally:
        k3.k3moe_test_expire_wait(False)


@pytest.mark.parametrize("n_shared", [1, 0])
def test_expired_wait_reports_timeout_and_the_workspace_stays_usable(n_shared):
    L = fused_layer(41, n_shared=n_shared, topk=8, n_experts=40)
    _, _, oy = L.oracle()
    H = L.cfg.hidden
    ws = k3.new_workspace(L.dims, 1)

    # y = layer: the output is zero
    y = torch.full((1, H), 7.0, device="cuda")
    st = k3.new_status()
    code, dt = expired(lambda: call(L, ws, st, y))
    assert code == TIMEOUT, k3.STATUS_NAMES.get(code)
    assert int(torch.count_nonzero(y)) == 0
    assert dt < 10.0  # one ~0.1 s limit, not a hang

    # y += layer: y is left as it was
    base = torch.randn((1, H), device="cuda")
    y = base.clone()
    st = k3.new_status()
    code, _ = expired(lambda: call(L, ws, st, y, accumulate=True))
    assert code == TIMEOUT
    assert torch.equal(y, base)

    # the same workspace, hook off: a correct result and a clean status
    for _ in range(2):
        y = torch.zeros((1, H), device="cuda")
        st = k3.new_status()
        assert call(L, ws, st, y) == 0
        assert rel_l2(y.cpu().numpy(), oy) <= REL_L2_F32


def test_expired_wait_in_the_stacked_decode_leaves_the_stream_unchanged():
    from test_gpu_stack import Stack
    S = Stack(L=2, E=32, seed=4)
    H = S.cfg.hidden
    g = torch.Generator(device="cpu").manual_seed(9)
    h0 = (torch.randn((1, H), generator=g) * 2).cuda()
    ws, xs = k3.new_workspace(S.dims, 1), torch.empty((1, H), dtype=torch.int16, device="cuda")

    h = h0.clone()
    st = k3.new_status()
    def stack():
        k3.k3moe_decode_stack(S.dims, S.layers, h, xs, ws, st, eps=1e-5)
        torch.cuda.synchronize()
        return int(st.item())
    code, dt = expired(stack)
    assert code == TIMEOUT
    assert torch.equal(h, h0)  # every layer's increment was taken as zero
    assert dt < 20.0

    # hook off, same workspace: the stack matches its layers run one by one
    h_stack, h_manual = h0.clone(), h0.clone()
    st = k3.new_status()
    k3.k3moe_decode_stack(S.dims, S.layers, h_stack, xs, ws, st, eps=1e-5)
    S.manual_step(h_manual, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(h_stack, h_manual)
