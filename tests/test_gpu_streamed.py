"""GPU parity of the host-tier streamed layer (k3moe_layer_streamed): the routed experts'
records live in pinned host memory and are read into a small pool of device slots by the
expert cache (README of FareedKhan-dev/kimi-k3-in-c, section 12 "An LRU cache for the
experts"; README of Maknee/Kimi-K3.cpp, "The consumer-memory idea").  The layer output
must match the oracle's on the same inputs, and a call whose experts were all resident
must give the same bits as the call that read them."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import mxfp4_routed_expert_02_gb300 as k3
from mxfp4_routed_expert_02_gb300 import k3moe as B
from parity import Layer, rel_l2, REL_L2_F32

pytestmark = pytest.mark.gpu


class Streamed:
    """A seeded layer whose expert records sit in pinned host memory, and a cache of
    n_slots device slots in front of them."""

    def __init__(self, cfg, seed, n_slots, tokens=None):
        self.L = Layer(cfg, seed=seed, tokens=tokens, device_fill=cfg.n_experts * cfg.record_bytes > (64 << 20))
        L = self.L
        self.host = torch.empty(cfg.n_experts * L.stride, dtype=torch.uint8).pin_memory()
        self.host.copy_(L.experts.cpu())
        self.slots = torch.empty(n_slots * L.stride, dtype=torch.uint8, device="cuda")
        self.cache = k3.ExpertCache([self.host.data_ptr()], cfg.n_experts, cfg.record_bytes,
                                    L.stride, self.slots.data_ptr(), n_slots, L.stride)

    def run(self, x, ydt=torch.float32):
        L, T = self.L, x.shape[0]
        y = torch.zeros((T, L.cfg.hidden), dtype=ydt, device="cuda")
        idx = torch.empty((T, L.cfg.topk), dtype=torch.int32, device="cuda")
        w = torch.empty((T, L.cfg.topk), dtype=torch.float32, device="cuda")
        st = k3.new_status()
        k3.k3moe_layer_streamed(L.dims, self.cache, 0, x, L.d_wr, L.d_bias, L.d_sg, L.d_su,
                                L.d_sd, y, k3.new_streamed_workspace(L.dims, T), st,
                                idx_out=idx, w_out=w)
        torch.cuda.synchronize()
        return y, idx, w, int(st.item())


def custom(H, I, E, K, NS, T):
    return dataclasses.replace(synth.config("tiny"), name="custom", hidden=H, inter=I,
                               n_experts=E, topk=K, tokens=T, n_shared=NS)


@pytest.mark.parametrize("H,I,E,K,NS,T,slots", [
    (256, 128, 16, 2, 1, 6, 3),      # tiny layer, 3 slots: one token per call
    (1024, 512, 24, 6, 1, 4, 14),    # two tokens per call
    (512, 256, 12, 4, 0, 6, 12),     # no shared expert, three tokens per call
])
def test_streamed_layer_matches_the_oracle_through_hits_and_misses(H, I, E, K, NS, T, slots):
    S = Streamed(custom(H, I, E, K, NS, T), seed=H + E, n_slots=slots)
    L = S.L
    per = slots // K                 # tokens per call: their distinct experts always fit
    oi, ow, oy = L.oracle()
    outs = []
    for t0 in range(0, T, per):
        y, idx, w, st = S.run(L.d_x[t0:t0 + per])
        assert st == 0
        assert np.array_equal(idx.cpu().numpy(), oi[t0:t0 + per])
        assert np.allclose(w.cpu().numpy(), ow[t0:t0 + per], rtol=2e-7, atol=0)
        outs.append(y.cpu().numpy())
    assert rel_l2(np.concatenate(outs), oy) <= REL_L2_F32
    s0 = S.cache.stats()
    assert s0["misses"] > 0 and s0["bytes_loaded"] == s0["misses"] * L.rec_bytes
    # the last call again: every expert is resident now, and the bits are the same
    y1, _, _, _ = S.run(L.d_x[t0:t0 + per])
    y2, _, _, st = S.run(L.d_x[t0:t0 + per])
    assert st == 0 and torch.equal(y1, y2)
    s1 = S.cache.stats()
    assert s1["misses"] == s0["misses"] and s1["hits"] > s0["hits"]
    assert np.array_equal(y1.cpu().numpy(), outs[-1])


def test_streamed_layer_refuses_a_call_that_does_not_fit():
    S = Streamed(custom(256, 128, 16, 2, 1, 4), seed=3, n_slots=3)
    with pytest.raises(k3.K3MoeError) as ei:
        S.run(S.L.d_x[0:4])            # up to 8 distinct experts, 3 slots
    assert ei.value.code == B.K3MOE_ERR_CACHE_FULL


@pytest.mark.slow
def test_streamed_layer_at_the_model_width():
    cfg = dataclasses.replace(synth.config("decode1"), n_experts=64, tokens=3)
    S = Streamed(cfg, seed=61, n_slots=24)
    L = S.L
    oi, ow, oy = L.oracle()
    for t in range(3):
        y, idx, w, st = S.run(L.d_x[t:t + 1])
        assert st == 0
        assert np.array_equal(idx.cpu().numpy(), oi[t:t + 1])
        err = rel_l2(y.cpu().numpy(), oy[t:t + 1])
        print("streamed layer at hidden 7168, token %d: relative L2 error %.3e" % (t, err))
        assert err <= REL_L2_F32
    st = S.cache.stats()
    assert st["hits"] + st["misses"] == 3 * 16     # counted per distinct expert of a call
