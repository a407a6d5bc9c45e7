"""GPU parity of the LatentMoE layer (k3moe_latent_layer, through the C ABI) against the
oracle (README of FareedKhan-dev/kimi-k3-in-c, section 9, LatentMoE listing steps 1-6):
routes bit-exact, the layer output within the layer step's tolerance (fp32 relative L2
<= 1e-3, bf16 max-relative <= 2e-2), at small shapes with ragged passes and at the
model's shape (hidden 7168, latent 3584, inter 3072, top-16, two shared experts): one token
on the single-token kernels, 2-4 on the tensor-core experts with GEMV projections, more on
tensor-core projections too."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import mxfp4_routed_expert_02_gb300 as k3
from parity import rel_l2, max_rel, REL_L2_F32, MAX_REL_BF16

pytestmark = pytest.mark.gpu


class LatentLayer:
    """One seeded LatentMoE layer: host arrays for the oracle, device tensors for the
    library."""

    def __init__(self, cfg, seed=0, tokens=None, device_fill=None):
        self.cfg, self.seed = cfg, seed
        self.dims = k3.LatentDims(cfg.hidden, cfg.latent, cfg.inter, cfg.n_experts, cfg.topk,
                                  cfg.shared_inter if cfg.n_shared else 0, cfg.situ_b1,
                                  cfg.situ_b2, cfg.routed_scale, cfg.rms_eps, cfg.renorm, 1)
        self.host = synth.layer_weights(cfg, seed)
        self.x = synth.activations(cfg, seed, tokens)
        self.stride = (cfg.record_bytes + 4095) // 4096 * 4096
        self.experts = torch.empty(cfg.n_experts * self.stride, dtype=torch.uint8, device="cuda")
        if device_fill is None:
            device_fill = cfg.n_experts * cfg.record_bytes > (64 << 20)
        self._host_experts = None
        if device_fill:
            import synth.device as sd
            sd.fill_experts(self.experts, cfg, seed, 0, stride=self.stride)
        else:
            self._host_experts = synth.all_experts(cfg, seed)
            self.experts.view(cfg.n_experts, self.stride)[:, :cfg.record_bytes].copy_(
                torch.from_numpy(self._host_experts))
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        h = self.host
        self.d = {k: t(h[k].view(np.int16)) for k in ("wr", "w_down", "w_up")}
        self.d["bias"] = t(h["bias"])
        self.d["norm_w"] = t(h["norm_w"])
        for k in ("sh_gate", "sh_up", "sh_down"):
            self.d[k] = t(h[k].view(np.int16)) if cfg.n_shared else None
        self.d_x = t(self.x.view(np.int16))

    def expert_record(self, e):
        if self._host_experts is not None:
            return self._host_experts[e]
        return synth.expert_record(self.cfg, self.seed, 0, e)

    def run(self, x=None, ydt=torch.float32, accumulate=False, y=None, dims=None):
        x = self.d_x if x is None else x
        dims = dims or self.dims
        T, H, K = x.shape[0], self.cfg.hidden, self.cfg.topk
        if y is None:
            y = torch.zeros((T, H), dtype=ydt, device="cuda")
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        ws = k3.new_latent_workspace(dims, T)
        st = k3.new_status()
        d = self.d
        k3.k3moe_latent_layer(dims, x, d["wr"], d["bias"], d["w_down"], d["w_up"], d["norm_w"],
                              self.experts, self.stride, d["sh_gate"], d["sh_up"], d["sh_down"],
                              y, ws, st, idx_out=idx, w_out=w, accumulate=accumulate)
        torch.cuda.synchronize()
        return y, idx, w, int(st.item())

    def oracle(self, tokens=None, latent_norm=True):
        h, c = self.host, self.cfg
        sh = (h.get("sh_gate"), h.get("sh_up"), h.get("sh_down"))
        return oracle.latent_moe_layer(self.x, h["wr"], h["bias"], self.expert_record, c.topk,
                                       c.hidden, c.latent, c.inter, h["w_down"], h["w_up"],
                                       h["norm_w"], latent_norm, c.rms_eps, *sh,
                                       renorm=bool(c.renorm), routed_scale=c.routed_scale,
                                       b1=c.situ_b1, b2=c.situ_b2, tokens=tokens)


def custom(H, L, I, E, K, NS, T):
    return dataclasses.replace(synth.config("latent_tiny"), name="custom", hidden=H, latent=L,
                               inter=I, n_experts=E, topk=K, n_shared=NS, tokens=T)


def check(L, tokens=None, ydt=torch.float32):
    y, idx, w, st = L.run(ydt=ydt)
    assert st == 0
    oi, ow, oy = L.oracle(tokens=tokens)
    sel = slice(None) if tokens is None else tokens
    assert np.array_equal(idx.cpu().numpy()[sel], oi)
    assert np.allclose(w.cpu().numpy()[sel], ow, rtol=2e-7, atol=0)
    gy = y.float().cpu().numpy()[sel]
    if ydt == torch.float32:
        err = rel_l2(gy, oy)
        assert err <= REL_L2_F32, err
    else:
        err = max_rel(gy, oy)
        assert err <= MAX_REL_BF16, err
    return y, err


SHAPES = [
    # hidden, latent, inter, experts, top-k, shared experts, tokens
    (256, 128, 128, 16, 2, 2, 4),
    (256, 128, 128, 16, 2, 2, 1),
    (256, 128, 128, 16, 2, 0, 3),       # no shared expert: the up-projection writes y
    (256, 128, 128, 16, 2, 2, 65),      # two passes of the 64-token workspace
    (1024, 512, 512, 24, 6, 2, 3),
    (768, 384, 256, 12, 5, 1, 7),       # odd top-k, one shared expert; projections and
                                        # experts on the tensor cores (more than 4 tokens)
    (1024, 512, 512, 24, 6, 2, 67),     # a 64-token pass on the tensor cores, then 3 tokens
    (2048, 1024, 512, 24, 6, 2, 1),     # one token on the single-token kernels (ring gate/up,
    (2048, 1024, 1024, 24, 5, 0, 1),    # whole-expert down stages), odd top-k, no shared
]


@pytest.mark.parametrize("H,L,I,E,K,NS,T", SHAPES)
def test_latent_layer_shapes(H, L, I, E, K, NS, T):
    check(LatentLayer(custom(H, L, I, E, K, NS, T), seed=H + L + T))


def test_latent_layer_bf16_accumulate_determinism_and_no_norm():
    L = LatentLayer(synth.config("latent_tiny"), seed=3)
    y1, _ = check(L)
    y2, _, _, _ = L.run()
    assert torch.equal(y1, y2)                        # bitwise reproducible
    base = torch.randn_like(y1)
    y3, _, _, st = L.run(y=base.clone(), accumulate=True)
    assert st == 0 and torch.equal(y3, base + y1)     # y += layer, one float add
    check(L, ydt=torch.bfloat16)
    # without the latent RMSNorm
    nd = dataclasses.replace(L.dims, latent_norm=0)
    y4, idx, _, st = L.run(dims=nd)
    assert st == 0
    _, _, oy = L.oracle(latent_norm=False)
    assert rel_l2(y4.cpu().numpy(), oy) <= REL_L2_F32


def test_latent_layer_nan_bias_sets_nonfinite_status():
    L = LatentLayer(synth.config("latent_tiny"), seed=4)
    bias = L.d["bias"].clone()
    bias[3] = float("nan")
    L.d["bias"] = bias
    _, _, _, st = L.run()
    assert st == 8


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 2, 8])
def test_latent_layer_at_the_model_shape(T):
    cfg = dataclasses.replace(synth.config("latent_decode1"), n_experts=64, tokens=T)
    L = LatentLayer(cfg, seed=50 + T, device_fill=True)
    k3.k3moe_trace_enable(True)
    _, err = check(L)
    trace = k3.k3moe_trace_read()
    k3.k3moe_trace_enable(False)
    print("latent layer at the model shape, T=%d: relative L2 error %.3e" % (T, err))
    if T == 1:  # one token: the experts' gate/up on the tensor cores
        assert trace.get("k_gateup_tc1", (0, 0))[1] >= 1
