"""GPU parity of the router-order combine, the bf16 output at the model's width and the
non-finite router check, on every path the layer takes, through the C ABI.

* Router order (README of FareedKhan-dev/kimi-k3-in-c, section 9, LatentMoE listing
  step 3; README of Maknee/Kimi-K3.cpp, "The consumer-memory idea", item 7): the probe
  records of ``order_probe`` make each output row's float sum exactly zero or exactly one
  small term, depending only on where that term sits in router order.  The router is set
  up so that the probe experts win in a known order that is not their index order.  A
  kernel that summed the slots in another order, or in a wider type, gives nonzero rows
  where the oracle's float router-order sum gives zero, or the other way round.
* bf16 output (round to nearest even) at hidden 7168 on the single-token kernel and the
  tensor-core path, against the 2e-2 max-relative bound.
* A NaN correction bias through the single-token fused kernel and through the tensor-core
  router: status K3MOE_ERR_NONFINITE (host-injected; nothing faults).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import order_probe
import synth
from parity import Layer, rel_l2, max_rel, REL_L2_F32, MAX_REL_BF16

pytestmark = pytest.mark.gpu


def custom(H, I, E, K, NS, T):
    return dataclasses.replace(synth.config("tiny"), name="custom", hidden=H, inter=I,
                               n_experts=E, topk=K, tokens=T, n_shared=NS)


def probe_layer(H, I, E, K, T, seed):
    """A layer whose router picks K probe experts, in an order unlike their indices, for
    every token, with equal weights."""
    cfg = custom(H, I, E, K, 0, T)
    L = Layer(cfg, seed=seed, device_fill=E * cfg.record_bytes > (64 << 20))
    recs, pattern = order_probe.records(H, I, K, seed)
    ids = np.random.default_rng(seed + 1).permutation(E)[:K]  # expert at position j
    wr = L.host["wr"].copy()
    wr[ids] = wr[ids[0]]                     # equal logits -> equal scores -> equal weights
    bias = L.host["bias"].copy()
    bias[ids] = 2.0 - 0.01 * np.arange(K, dtype=np.float32)   # router order = position
    L.set_router(wr=wr, bias=bias)
    for j, e in enumerate(ids):
        L.set_expert(int(e), recs[j])
    return L, ids, pattern


ORDER_SHAPES = [
    # hidden, inter, experts, top-k, tokens: which combine runs
    (256, 128, 16, 4, 1),      # one token, CUDA-core kernels (register down kernel)
    (256, 128, 16, 4, 3),      # several tokens, CUDA-core kernels
    (1024, 512, 24, 5, 1),     # one token, single-token gate/up + bulk-copy down kernel
    (1024, 512, 24, 6, 1),     # one token, the fused single-token kernel
    (512, 256, 12, 4, 5),      # several tokens, tensor-core GEMMs + the combine kernel
    (7168, 1536, 64, 16, 1),   # the model's width, fused kernel, 1680 triples
    (7168, 1536, 64, 16, 2),   # the model's width, tensor-core path
]


@pytest.mark.parametrize("H,I,E,K,T", ORDER_SHAPES)
def test_layer_sums_the_routed_outputs_in_router_order(H, I, E, K, T):
    L, ids, pattern = probe_layer(H, I, E, K, T, seed=H + K + T)
    y, idx, w, st = L.run()
    assert st == 0
    gi = idx.cpu().numpy()
    assert (gi == ids[None, :]).all()
    oi, ow, oy = L.oracle()
    assert np.array_equal(gi, oi)
    assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
    zero = order_probe.zero_rows(pattern)
    gy = y.cpu().numpy()
    assert np.all(oy[:, zero] == 0.0)          # the oracle's float router-order sum
    assert np.all(gy[:, zero] == 0.0)          # the kernels': the same rows vanish
    assert np.all(gy[:, ~zero] != 0.0)         # and the others keep their small term
    assert rel_l2(gy, oy) <= REL_L2_F32


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 3])
def test_bf16_output_at_the_model_width(T):
    # T = 1: the fused single-token kernel; T = 3: the tensor-core path
    cfg = dataclasses.replace(synth.config("decode1"), n_experts=64, tokens=T)
    L = Layer(cfg, seed=40 + T, device_fill=True)
    yb, idx, w, st = L.run(ydt=torch.bfloat16)
    assert st == 0
    oi, ow, oy = L.oracle()
    assert np.array_equal(idx.cpu().numpy(), oi)
    err = max_rel(yb.float().cpu().numpy(), oy)
    print("bf16 max-relative error at hidden 7168, T=%d: %.3e" % (T, err))
    assert err <= MAX_REL_BF16
    # the bf16 output is the fp32 output rounded once (nearest even)
    yf, _, _, st = L.run()
    assert st == 0
    want = oracle.f32_to_bf16(yf.cpu().numpy())
    assert np.array_equal(yb.view(torch.int16).cpu().numpy().view(np.uint16), want)


@pytest.mark.parametrize("H,I,E,K,T", [
    (1024, 512, 24, 6, 1),     # fused single-token kernel
    (512, 256, 12, 4, 4),      # tensor-core router (screening, then exact candidates)
    (256, 128, 16, 2, 1),      # single-token CUDA-core router
])
def test_nan_bias_sets_nonfinite_status(H, I, E, K, T):
    L = Layer(custom(H, I, E, K, 1, T), seed=7 + T)
    bias = L.host["bias"].copy()
    bias[5] = np.float32("nan")
    L.set_router(bias=bias)
    _, _, _, st = L.run()
    assert st == 8
    # the next call with a finite bias on fresh buffers is clean again
    bias[5] = 0.0
    L.set_router(bias=bias)
    y, idx, _, st = L.run()
    assert st == 0
    oi, _, oy = L.oracle()
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert rel_l2(y.cpu().numpy(), oy) <= REL_L2_F32
