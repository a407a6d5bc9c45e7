"""Pins of the oracle's stacked decode step (the decoder loop of kimi-k3-in-c: RMSNorm of
section 5 with weight 1, the layer step of section 9, the residual stream between
layers): each check fails for a plausible slip in the composition -- a dropped residual,
the residual added to the normalised value, a layer fed an unnormalised input, layers
applied out of order."""
import numpy as np

import oracle
import synth


def _layers(cfg, n, seed=0):
    out = []
    for l in range(n):
        w = synth.layer_weights(cfg, seed, l)
        allx = synth.all_experts(cfg, seed, l)
        out.append(dict(wr=w["wr"], bias=w["bias"], get_expert=lambda e, a=allx: a[e],
                        sh_gate=w["sh_gate"], sh_up=w["sh_up"], sh_down=w["sh_down"],
                        _allx=allx))
    return out


def _step(h, layers, cfg, eps=1e-5):
    return oracle.stacked_decode_step(h, layers, cfg.topk, cfg.hidden, cfg.inter, eps=eps)


def test_silent_layer_leaves_the_stream_unchanged():
    # every routed group scaled by 255 (contributes nothing) and a zero shared gate
    # (SiTU(0, u) = 0): the layer adds exactly zero, so h passes through bit for bit
    cfg = synth.config("tiny")
    lay = _layers(cfg, 1)[0]
    off = cfg.record_offsets
    allx = lay["_allx"].copy()
    for op in (1, 3, 5):
        allx[:, off[op]:off[op + 1]] = 255
    lay["get_expert"] = lambda e: allx[e]
    lay["sh_gate"] = np.zeros_like(lay["sh_gate"])
    h = np.random.default_rng(0).standard_normal(cfg.hidden).astype(np.float32) * 3
    h2, idx, w = _step(h, [lay], cfg)
    assert np.array_equal(h2, h)
    assert len(idx) == 1 and idx[0].shape == (cfg.topk,)


def test_residual_adds_the_unnormalised_stream():
    # with eps = 0, scaling h by 4 (a power of two) leaves the layer input unchanged, so
    # the increment is the same: h'(4h) - 4h == h'(h) - h up to the rounding of the two
    # float adds (adding to the normalised value instead would be off by 3h)
    cfg = synth.config("tiny")
    lay = _layers(cfg, 1)
    h = np.random.default_rng(1).standard_normal(cfg.hidden).astype(np.float32)
    a, ia, _ = _step(h, lay, cfg, eps=0.0)
    b, ib, _ = _step(4 * h, lay, cfg, eps=0.0)
    assert np.array_equal(ia[0], ib[0])
    da = a.astype(np.float64) - h
    db = b.astype(np.float64) - 4.0 * h
    bound = 2.0 ** -22 * (np.abs(4.0 * h) + np.abs(da))
    assert np.all(np.abs(db - da) <= bound)
    assert np.abs(da).max() > 1e-3


def test_each_layer_sees_a_normalised_bf16_input():
    # the increment of layer l equals the layer step on bf16(RMSNorm(h_l)) computed
    # directly, for a stream of very different scales
    cfg = synth.config("tiny")
    lays = _layers(cfg, 2, seed=3)
    h = (np.random.default_rng(2).standard_normal(cfg.hidden) * 1000).astype(np.float32)
    h2, idx, w = _step(h, lays, cfg)
    h_l = h
    for l, lay in enumerate(lays):
        n = oracle.rmsnorm(h_l, eps=1e-5)
        rms = float(np.sqrt(np.mean(n.astype(np.float64) ** 2)))
        assert abs(rms - 1.0) < 1e-3           # the layer input is unit-RMS
        x = oracle.f32_to_bf16(n)
        i1, w1, y = oracle.moe_layer(x[None, :], lay["wr"], lay["bias"], lay["get_expert"],
                                     cfg.topk, cfg.hidden, cfg.inter, lay["sh_gate"],
                                     lay["sh_up"], lay["sh_down"])
        assert np.array_equal(i1[0], idx[l]) and np.array_equal(w1[0], w[l])
        h_l = (h_l + y[0]).astype(np.float32)
    assert np.array_equal(h_l, h2)


def test_layer_order_matters():
    cfg = synth.config("tiny")
    lays = _layers(cfg, 2, seed=5)
    h = np.random.default_rng(4).standard_normal(cfg.hidden).astype(np.float32)
    a, _, _ = _step(h, lays, cfg)
    b, _, _ = _step(h, lays[::-1], cfg)
    assert not np.array_equal(a, b)
