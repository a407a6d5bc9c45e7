"""GPU parity of the stacked decode (layers with RMSNorm and the residual stream between
them): layer by layer against the oracle, teacher-forced (the oracle takes the GPU's
stream at each layer boundary, so a rounding difference cannot compound), and
k3moe_decode_stack against the same kernels called one by one."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.device as sd
import mxfp4_routed_expert_02_gb300 as k3
from parity import rel_l2, REL_L2_F32, dims_of

pytestmark = pytest.mark.gpu


class Stack:
    """L full-width layers (hidden 7168, inter 1536) with few experts each."""

    def __init__(self, L=3, E=32, seed=0):
        self.cfg = dataclasses.replace(synth.config("decode1"), name="stack", n_experts=E)
        cfg = self.cfg
        self.dims = dims_of(cfg)
        self.stride = (cfg.record_bytes + 4095) // 4096 * 4096
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.layers, self.host = [], []
        for l in range(L):
            w = synth.layer_weights(cfg, seed, l)
            ex = torch.empty(E * self.stride, dtype=torch.uint8, device="cuda")
            sd.fill_experts(ex, cfg, seed, l, stride=self.stride)
            self.layers.append(dict(wr=t(w["wr"].view(np.int16)), bias=t(w["bias"]), experts=ex,
                                    stride=self.stride, sh_gate=t(w["sh_gate"].view(np.int16)),
                                    sh_up=t(w["sh_up"].view(np.int16)),
                                    sh_down=t(w["sh_down"].view(np.int16))))
            self.host.append(dict(wr=w["wr"], bias=w["bias"], sh_gate=w["sh_gate"],
                                  sh_up=w["sh_up"], sh_down=w["sh_down"],
                                  get_expert=lambda e, l=l: synth.expert_record(cfg, seed, l, e)))

    def manual_step(self, h, ws, st, eps=1e-5):
        """One step with the library's kernels called layer by layer; returns per-layer
        (stream before, bf16 input, idx, w)."""
        T, H, K = h.shape[0], self.cfg.hidden, self.cfg.topk
        trace = []
        for lw in self.layers:
            before = h.clone()
            x = torch.empty((T, H), dtype=torch.int16, device="cuda")
            k3.k3moe_rmsnorm_bf16(h, x, eps)
            idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
            w = torch.empty((T, K), dtype=torch.float32, device="cuda")
            k3.k3moe_layer(self.dims, x, lw["wr"], lw["bias"], lw["experts"], lw["stride"],
                           lw["sh_gate"], lw["sh_up"], lw["sh_down"], h, ws, st, idx_out=idx,
                           w_out=w, accumulate=True)
            trace.append((before, x, idx, w))
        return trace


def test_stack_layer_by_layer_against_the_oracle():
    S = Stack(L=3, E=32, seed=1)
    cfg = S.cfg
    H, I, K = cfg.hidden, cfg.inter, cfg.topk
    xb = synth.activations(cfg, 7, 1).view(np.uint16).astype(np.uint32) << 16
    h = torch.from_numpy(xb.view(np.float32).reshape(1, H).copy()).cuda()
    ws, st = k3.new_workspace(S.dims, 1), k3.new_status()
    for step in range(2):
        trace = S.manual_step(h, ws, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        for l, (before, x, idx, w) in enumerate(trace):
            hb = before.cpu().numpy()[0]
            after = trace[l + 1][0].cpu().numpy()[0] if l + 1 < len(trace) else h.cpu().numpy()[0]
            want_x = oracle.f32_to_bf16(oracle.rmsnorm(hb, eps=1e-5))
            assert np.array_equal(x.cpu().numpy().view(np.uint16)[0], want_x)
            lw = S.host[l]
            oi, ow, oy = oracle.moe_layer(want_x[None, :], lw["wr"], lw["bias"], lw["get_expert"],
                                          K, H, I, lw["sh_gate"], lw["sh_up"], lw["sh_down"])
            assert np.array_equal(idx.cpu().numpy(), oi)
            assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
            # the increment this layer added to the stream, against the oracle's layer output
            assert rel_l2(after.astype(np.float64) - hb, oy[0]) <= REL_L2_F32


@pytest.mark.parametrize("T", [1, 3])
def test_decode_stack_equals_the_layers_one_by_one(T):
    # T = 1: the single-token kernels; T = 3: the multi-token (tensor-core) path
    S = Stack(L=3, E=32, seed=2)
    cfg = S.cfg
    H, K = cfg.hidden, cfg.topk
    g = torch.Generator(device="cpu").manual_seed(3)
    h0 = (torch.randn((T, H), generator=g) * 2).cuda()
    ws, st = k3.new_workspace(S.dims, T), k3.new_status()
    h_manual = h0.clone()
    idx_m = []
    for _ in range(2):
        idx_m += [tr[2].clone() for tr in S.manual_step(h_manual, ws, st)]
    h_stack = h0.clone()
    xs = torch.empty((T, H), dtype=torch.int16, device="cuda")
    idx_s = torch.empty((2, 3, T, K), dtype=torch.int32, device="cuda")
    w_s = torch.empty((2, 3, T, K), dtype=torch.float32, device="cuda")
    for step in range(2):
        k3.k3moe_decode_stack(S.dims, S.layers, h_stack, xs, ws, st, eps=1e-5,
                              idx_out=idx_s[step], w_out=w_s[step])
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(h_stack, h_manual)
    assert torch.equal(idx_s.reshape(6, T, K), torch.stack(idx_m))
