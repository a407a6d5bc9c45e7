"""Pins of the oracle's expert record, expert FFN and layer composition
(kimi-k3-in-c, 'The problem: a model that does not fit' census, section 9 LatentMoE
listing; Kimi-K3.cpp 'The consumer-memory idea', item 7)."""
import json
import math
import os

import numpy as np

import oracle
import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


def test_record_size_matches_the_census():
    g = GOLD["expert_record"]
    off = oracle.record_offsets(7168, 1536)
    assert off[6] == g["bytes_per_expert"] == 17547264
    assert off[6] == g["pages_of_4096"] * 4096
    assert g["params_per_expert"] * g["bytes_per_param"] == off[6]
    # three matrices of 7168 x 1536 weights; half a byte each plus one byte per 32
    sizes = np.diff(off)
    assert sizes.tolist() == [5505024, 344064] * 3
    assert all(o % 4096 == 0 for o in off)
    # the page's LatentMoE shape (latent 3584, inter 3072) has the same record size
    assert oracle.record_offsets(3584, 3072)[6] == off[6]


def test_checkpoint_tensor_shape_is_consistent():
    c = GOLD["checkpoint_mxfp4_tensor"]
    assert c["packed_cols"] * 2 == c["logical_width"]
    assert c["scale_cols"] * c["group_size"] == c["logical_width"]


def test_generator_layout_agrees_with_oracle():
    for H, I in [(7168, 1536), (256, 128), (96, 64)]:
        assert synth.record_offsets(H, I) == oracle.record_offsets(H, I)


def _expert(H, I, gate, up, down, gs=127, us=127, ds=127):
    """Record from per-operand code matrices (one code per weight) and uniform scales."""
    def pack(codes):
        codes = np.asarray(codes, np.uint8)
        return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    off = oracle.record_offsets(H, I)
    rec = np.zeros(off[6], np.uint8)
    rec[off[0]:off[1]] = pack(gate).ravel()
    rec[off[1]:off[2]] = gs
    rec[off[2]:off[3]] = pack(down).ravel()
    rec[off[3]:off[4]] = ds
    rec[off[4]:off[5]] = pack(up).ravel()
    rec[off[5]:off[6]] = us
    return rec


def test_operand_roles_gate_up_down():
    # gate weights all +6 (g huge -> a = b1), up weights: row i is +0.5 at column i only
    H = I = 32
    gate = np.full((I, H), 7)
    up = np.zeros((I, H), int)
    np.fill_diagonal(up, 1)
    down = np.zeros((H, I), int)
    np.fill_diagonal(down, 2)              # down = identity
    rec = _expert(H, I, gate, up, down)
    x = np.full(H, 0.1, np.float32)
    x[3] = 2.0
    d = oracle.expert(rec, x, H, I)
    g = 6.0 * x.sum()
    for i in (0, 3):
        u = 0.5 * x[i]
        want = 4 * math.tanh(g / 4) / (1 + math.exp(-g)) * 25 * math.tanh(u / 25)
        assert abs(d[i] - want) <= 1e-6 * abs(want)
    # swapping the gate and up roles would give a very different value
    u_sw = 6.0 * x.sum()
    g_sw = 0.5 * x[3]
    wrong = 4 * math.tanh(g_sw / 4) / (1 + math.exp(-g_sw)) * 25 * math.tanh(u_sw / 25)
    assert abs(d[3] - wrong) > 0.1 * abs(wrong)


def _tiny_layer(seed=0, E=6, K=3, H=64, I=32):
    rng = np.random.default_rng(seed)
    x = oracle.f32_to_bf16(rng.standard_normal((2, H)).astype(np.float32))
    wr = oracle.f32_to_bf16((rng.standard_normal((E, H)) / 8).astype(np.float32))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    off = oracle.record_offsets(H, I)
    recs = []
    for e in range(E):
        r = rng.integers(0, 256, off[6], dtype=np.uint8)
        for a, b in ((1, 2), (3, 4), (5, 6)):
            r[off[a]:off[b]] = rng.integers(122, 127, off[b] - off[a])
        recs.append(r)
    return x, wr, bias, recs


def test_identical_experts_with_renorm_give_one_expert():
    x, wr, bias, recs = _tiny_layer(1)
    same = [recs[0]] * len(recs)
    idx, w, y = oracle.moe_layer(x, wr, bias, lambda e: same[e], 3, 64, 32)
    for t in range(2):
        d = oracle.expert(same[0], oracle.bf16_to_f32(x[t]), 64, 32)
        assert np.allclose(y[t], d, rtol=1e-5, atol=1e-6)


def test_down_scale_plus_one_doubles_the_routed_sum_exactly():
    x, wr, bias, recs = _tiny_layer(2)
    off = oracle.record_offsets(64, 32)
    up1 = []
    for r in recs:
        r2 = r.copy()
        r2[off[3]:off[4]] += 1
        up1.append(r2)
    _, _, y = oracle.moe_layer(x, wr, bias, lambda e: recs[e], 3, 64, 32)
    _, _, y2 = oracle.moe_layer(x, wr, bias, lambda e: up1[e], 3, 64, 32)
    assert np.array_equal(y2, 2 * y)


def test_router_order_weighted_sum_and_unweighted_shared():
    x, wr, bias, recs = _tiny_layer(3)
    H, I, SI = 64, 32, 32
    rng = np.random.default_rng(9)
    sg = oracle.f32_to_bf16((rng.standard_normal((SI, H)) / 8).astype(np.float32))
    su = oracle.f32_to_bf16((rng.standard_normal((SI, H)) / 8).astype(np.float32))
    sd = oracle.f32_to_bf16((rng.standard_normal((H, SI)) / 6).astype(np.float32))
    idx, w, y = oracle.moe_layer(x, wr, bias, lambda e: recs[e], 3, H, I, sg, su, sd)
    _, _, y0 = oracle.moe_layer(x, wr, bias, lambda e: recs[e], 3, H, I)
    for t in range(2):
        ds = oracle.shared_expert(sg, su, sd, oracle.bf16_to_f32(x[t]))
        # shared output is added with weight 1, independent of the route
        # (both outputs are rounded to float once: compare within a few of their ulps)
        tol = 4 * np.spacing(np.float32(np.abs(y[t]).max()))
        assert np.all(np.abs((y[t] - y0[t]) - ds) <= tol)
        # K = 1 without renormalisation: the routed sum is sc * d of the best expert
    idx1, w1, y1 = oracle.moe_layer(x, wr, bias, lambda e: recs[e], 1, H, I, renorm=False)
    for t in range(2):
        d = oracle.expert(recs[idx1[t][0]], oracle.bf16_to_f32(x[t]), H, I)
        assert np.allclose(y1[t], np.float64(w1[t][0]) * d, rtol=1e-6, atol=1e-7)


def test_combine_is_a_float_sum_in_router_order():
    # kimi-k3-in-c, section 9, LatentMoE listing steps 3 and 6: acc += w[j] * d_j[i] in
    # float, j in router order, then the shared output added.  2^24 + 1 rounds back to
    # 2^24, so the three terms sum to 0 left to right and to 1 right to left (and in
    # double).
    big = 2.0 ** 24
    assert oracle.combine([1, 1, 1], [[big], [1.0], [-big]])[0] == 0.0
    assert oracle.combine([1, 1, 1], [[-big], [1.0], [big]])[0] == 1.0
    # each product is rounded to float before it is added (no fused multiply-add):
    # (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 rounds to 1 + 2^-11
    a = 1.0 + 2.0 ** -12
    assert oracle.combine([-1.0, a], [[1.0], [a]])[0] == 2.0 ** -11
    # the shared expert's output comes after the routed sum: added first, 1 + 2^24 would
    # round away the 1
    assert oracle.combine([1, 1], [[big], [-big]], ds=[1.0])[0] == 1.0
    assert oracle.combine([1, 1], [[big], [-big]])[0] == 0.0


def test_routed_sum_in_router_order_through_the_layer():
    # records built so that each output row's float sum is exactly 0 or exactly the one
    # small term, depending only on where that term sits in the router order
    import order_probe
    H, I, K = 96, 64, 4
    recs, pat = order_probe.records(H, I, K, seed=11)
    rng = np.random.default_rng(12)
    x = oracle.f32_to_bf16(rng.standard_normal(H).astype(np.float32))
    xf = oracle.bf16_to_f32(x)
    w = np.full(K, 0.25, np.float32)
    y = oracle.moe_token(x, list(recs), w, H, I)
    zero = order_probe.zero_rows(pat)
    assert zero.any() and (~zero).any()
    assert np.all(y[zero] == 0.0)
    r = order_probe.small_term_position(pat)
    d = np.stack([oracle.expert(recs[k], xf, H, I) for k in range(K)])
    want = w[r] * d[r, np.arange(H)]            # one float32 product per row
    assert want.dtype == np.float32 and np.all(want[~zero] != 0)
    assert np.array_equal(y[~zero], want[~zero])
    # the same experts in another order: the rows that vanish follow the new order
    perm = [2, 0, 3, 1]                          # position n holds expert perm[n]
    y2 = oracle.moe_token(x, [recs[k] for k in perm], w, H, I)
    pos = np.argsort(perm)                       # expert k sits at position pos[k]
    zero2 = order_probe.zero_rows(pos[pat])
    assert not np.array_equal(zero, zero2)
    assert np.all(y2[zero2] == 0.0)
    assert np.array_equal(y2[~zero2], want[~zero2])
