"""Shared helpers of the GPU parity tests: build a seeded layer on the device, run the
library through its C ABI, run the oracle on the same inputs, compare.

Tolerances (fp32 output: relative L2 error <= 1e-3 over the [T][H] output; bf16 output:
max |y - y_ref| / max |y_ref| <= 2e-2) are those the layer step is specified to; expert
indices must match exactly.
"""
import dataclasses

import numpy as np
import torch

import oracle
import synth
import mxfp4_routed_expert_02_gb300 as k3

REL_L2_F32 = 1e-3
MAX_REL_BF16 = 2e-2


def rel_l2(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def max_rel(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-300))


def dims_of(cfg: synth.Config) -> "k3.LayerDims":
    return k3.LayerDims(cfg.hidden, cfg.inter, cfg.n_experts, cfg.topk,
                        cfg.shared_inter if cfg.n_shared > 0 else 0, cfg.situ_b1, cfg.situ_b2,
                        cfg.routed_scale, cfg.renorm)


class Layer:
    """One seeded layer: host arrays for the oracle, device tensors for the library."""

    def __init__(self, cfg: synth.Config, seed: int = 0, layer: int = 0, device_fill=None,
                 tokens=None):
        self.cfg, self.seed, self.layer = cfg, seed, layer
        self.overrides = {}
        self.dims = dims_of(cfg)
        w = synth.layer_weights(cfg, seed, layer)
        self.host = w
        self.x = synth.activations(cfg, seed, tokens)
        dev = torch.device("cuda")
        self.rec_bytes = cfg.record_bytes
        self.stride = (self.rec_bytes + 4095) // 4096 * 4096
        n = cfg.n_experts * self.stride
        self.experts = torch.empty(n, dtype=torch.uint8, device=dev)
        big = cfg.n_experts * self.rec_bytes > (1 << 30)
        if device_fill is None:
            device_fill = big
        if device_fill:
            import synth.device as sd
            sd.fill_experts(self.experts, cfg, seed, layer, stride=self.stride)
            self._host_experts = None
        else:
            allx = synth.all_experts(cfg, seed, layer)
            self._host_experts = allx
            view = self.experts.view(cfg.n_experts, self.stride)
            view[:, :self.rec_bytes].copy_(torch.from_numpy(allx))
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.d_x = t(self.x.view(np.int16))
        self.d_wr = t(w["wr"].view(np.int16))
        self.d_bias = t(w["bias"])
        if cfg.n_shared > 0:
            self.d_sg = t(w["sh_gate"].view(np.int16))
            self.d_su = t(w["sh_up"].view(np.int16))
            self.d_sd = t(w["sh_down"].view(np.int16))
        else:
            self.d_sg = self.d_su = self.d_sd = None

    def expert_record(self, e: int) -> np.ndarray:
        if e in self.overrides:
            return self.overrides[e]
        if self._host_experts is not None:
            return self._host_experts[e]
        return synth.expert_record(self.cfg, self.seed, self.layer, e)

    def set_expert(self, e: int, rec: np.ndarray):
        """Replace expert e's record on the device and for the oracle."""
        rec = np.ascontiguousarray(rec, np.uint8)
        self.experts.view(self.cfg.n_experts, self.stride)[e, :self.rec_bytes].copy_(
            torch.from_numpy(rec))
        self.overrides[int(e)] = rec

    def set_router(self, wr=None, bias=None):
        """Replace the router weights and/or the correction bias (device and oracle)."""
        if wr is not None:
            self.host["wr"] = wr
            self.d_wr = torch.from_numpy(np.ascontiguousarray(wr).view(np.int16)).cuda()
        if bias is not None:
            self.host["bias"] = bias
            self.d_bias = torch.from_numpy(np.ascontiguousarray(bias)).cuda()

    def run(self, x=None, ydt=torch.float32, accumulate=False, y=None):
        x = self.d_x if x is None else x
        T = x.shape[0]
        H, K = self.cfg.hidden, self.cfg.topk
        ws = k3.new_workspace(self.dims, T)
        st = k3.new_status()
        if y is None:
            y = torch.zeros((T, H), dtype=ydt, device="cuda")
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        k3.k3moe_layer(self.dims, x, self.d_wr, self.d_bias, self.experts, self.stride,
                       self.d_sg, self.d_su, self.d_sd, y, ws, st, idx_out=idx, w_out=w,
                       accumulate=accumulate)
        torch.cuda.synchronize()
        return y, idx, w, int(st.item())

    def oracle(self, tokens=None, nthreads=0):
        h, cfg = self.host, self.cfg
        sh = (h.get("sh_gate"), h.get("sh_up"), h.get("sh_down"))
        return oracle.moe_layer(self.x, h["wr"], h["bias"], self.expert_record, cfg.topk,
                                cfg.hidden, cfg.inter, *sh, renorm=bool(cfg.renorm),
                                routed_scale=cfg.routed_scale, b1=cfg.situ_b1, b2=cfg.situ_b2,
                                tokens=tokens, nthreads=nthreads)


def fused_layer(seed, **kw):
    """A one-token layer at a shape the fused single-token kernel takes."""
    base = dict(hidden=1024, inter=512, n_experts=24, topk=6, tokens=1, n_shared=1)
    base.update(kw)
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", **base)
    return Layer(cfg, seed=seed)
