"""GPU parity: the CUDA path (through the C ABI) against the oracle on the same seeded
inputs.  Expert indices and dequantised weights bit-exact; layer outputs within the
stated tolerance (fp32 relative L2 <= 1e-3, bf16 max-relative <= 2e-2)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import mxfp4_routed_expert_02_gb300 as k3
from parity import Layer, fused_layer, rel_l2, max_rel, REL_L2_F32, MAX_REL_BF16, dims_of

pytestmark = pytest.mark.gpu


def f32bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ------------------------------------------------------------------------------ dequant
def test_dequant_exhaustive_bitwise():
    rows, cols = 256, 32
    codes = np.arange(32) % 16
    packed = np.tile((codes[0::2] | (codes[1::2] << 4)).astype(np.uint8), (rows, 1))
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    want = oracle.dequant_mxfp4(packed, scales, rows, cols)
    out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    k3.k3moe_dequant_mxfp4(torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda(),
                           rows, cols, out)
    torch.cuda.synchronize()
    assert np.array_equal(f32bits(out.cpu().numpy()), f32bits(want))


def test_dequant_tiny_expert_all_operands_bitwise():
    cfg = synth.config("tiny")
    rec = synth.expert_record(cfg, 0, 0, 5)
    off = cfg.record_offsets
    H, I = cfg.hidden, cfg.inter
    for (p, s, rows, cols) in ((0, 1, I, H), (2, 3, H, I), (4, 5, I, H)):
        packed = rec[off[p]:off[s]].reshape(rows, cols // 2)
        scales = rec[off[s]:off[s + 1]].reshape(rows, cols // 32)
        want = oracle.dequant_mxfp4(packed, scales, rows, cols)
        out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
        k3.k3moe_dequant_mxfp4(torch.from_numpy(packed.copy()).cuda(),
                               torch.from_numpy(scales.copy()).cuda(), rows, cols, out)
        torch.cuda.synchronize()
        assert np.array_equal(f32bits(out.cpu().numpy()), f32bits(want))


# ------------------------------------------------------------------------------ router
@pytest.mark.parametrize("name,T", [("tiny", 4), ("decode1", 3)])
def test_route_matches_oracle(name, T):
    cfg = synth.config(name)
    L = Layer(cfg, seed=1, tokens=T, device_fill=True)
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.topk), dtype=torch.float32, device="cuda")
    ws = k3.new_workspace(L.dims, T)
    st = k3.new_status()
    k3.k3moe_route(L.dims, L.d_x, L.d_wr, L.d_bias, idx, w, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    oi, ow, _, _ = oracle.router(L.x, L.host["wr"], L.host["bias"], cfg.topk)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)


def test_route_ties_and_bias_only_selects():
    cfg = synth.config("tiny")
    H, E, K = cfg.hidden, cfg.n_experts, cfg.topk
    dims = dims_of(cfg)
    x = torch.from_numpy(oracle.f32_to_bf16(np.ones((2, H), np.float32)).view(np.int16)).cuda()
    wr = torch.zeros((E, H), dtype=torch.int16, device="cuda")   # every score 0.5: all tied
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    bias[9] = 0.01
    idx = torch.empty((2, K), dtype=torch.int32, device="cuda")
    w = torch.empty((2, K), dtype=torch.float32, device="cuda")
    st = k3.new_status()
    k3.k3moe_route(dims, x, wr, bias, idx, w, k3.new_workspace(dims, 2), st)
    torch.cuda.synchronize()
    assert idx.cpu().numpy().tolist() == [[9, 0], [9, 0]]   # bias picks 9, tie -> lowest
    assert np.all(w.cpu().numpy() == np.float32(0.5))         # unbiased, renormalised 0.5/1.0


def test_layer_tensor_core_router_ties_and_bias():
    # multi-token path: duplicated router rows give equal selection scores (the lower
    # index must win), a large bias on one expert forces it in without changing weights
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", hidden=512, inter=256,
                              n_experts=24, topk=5, tokens=33, n_shared=1)
    L = Layer(cfg, seed=21)
    wr = L.host["wr"].copy()
    wr[7] = wr[3]
    wr[12] = wr[3]
    wr[20] = wr[9]
    bias = L.host["bias"].copy()
    bias[3] = bias[7] = bias[12] = 0.05
    bias[17] = 2.0
    L.host["wr"], L.host["bias"] = wr, bias
    L.d_wr = torch.from_numpy(wr.view(np.int16)).cuda()
    L.d_bias = torch.from_numpy(bias).cuda()
    y, idx, w, st = L.run()
    assert st == 0
    oi, ow, oy = L.oracle()
    gi = idx.cpu().numpy()
    assert np.array_equal(gi, oi)
    assert (gi == 17).any(axis=1).all()
    assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
    assert rel_l2(y.cpu().numpy(), oy) <= REL_L2_F32


def test_route_nonfinite_sets_status():
    cfg = synth.config("tiny")
    dims = dims_of(cfg)
    L = Layer(cfg, seed=0, tokens=1)
    bias = L.d_bias.clone()
    bias[3] = float("nan")
    idx = torch.empty((1, cfg.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((1, cfg.topk), dtype=torch.float32, device="cuda")
    st = k3.new_status()
    k3.k3moe_route(dims, L.d_x, L.d_wr, bias, idx, w, k3.new_workspace(dims, 1), st)
    torch.cuda.synchronize()
    assert st.item() == 8


# ------------------------------------------------------------------------------ layer
def check_layer(L, T_sample=None, ydt=torch.float32, nthreads=0):
    y, idx, w, st = L.run(ydt=ydt)
    assert st == 0
    T = y.shape[0]
    tokens = list(range(T)) if T_sample is None else T_sample
    oi, ow, oy = L.oracle(tokens=tokens, nthreads=nthreads)
    gi = idx.cpu().numpy()[tokens]
    assert np.array_equal(gi, oi)
    assert np.allclose(w.cpu().numpy()[tokens], ow, rtol=2e-7, atol=0)
    gy = y.float().cpu().numpy()[tokens]
    if ydt == torch.float32:
        err = rel_l2(gy, oy)
        assert err <= REL_L2_F32, err
    else:
        err = max_rel(gy, oy)
        assert err <= MAX_REL_BF16, err
    return err


@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_layer_tiny(ydt):
    err = check_layer(Layer(synth.config("tiny"), seed=0), ydt=ydt)
    if ydt == torch.float32:
        assert err < 1e-4   # the fp32 path sits far inside the bound


SHAPES = [
    # hidden, inter, experts, topk, shared experts (each inter wide), tokens: ragged
    # tiles, both gate/up thread mappings (H/32 a power of two <= 16, or not), 1..8
    # groups per down lane, the 64-token decode pass boundary, two shared experts.
    (96, 64, 5, 3, 1, 1),
    (96, 64, 5, 3, 2, 3),
    (512, 96, 9, 4, 0, 7),
    (256, 128, 16, 2, 1, 64),
    (256, 128, 16, 2, 1, 65),
    (1024, 256, 24, 6, 2, 130),
    (2048, 512, 33, 8, 1, 2),
    # tensor-core path (two tokens and up, H and I multiples of 64, at least 256): ragged
    # 128-row tiles (I 320, H 320), a partial last 128-byte K chunk (H/2 = 160, I/2 = 160),
    # more than 128 pairs on one expert (T 300 over 4 experts), no shared expert; B tiles
    # of 32, 48, 64 and 128 rows (several activation terms side by side in one MMA, or one)
    (256, 256, 8, 2, 1, 5),
    (320, 320, 6, 3, 1, 40),
    (512, 384, 4, 2, 1, 300),
    (768, 256, 12, 4, 0, 64),
    (256, 320, 8, 2, 1, 150),
    (384, 256, 8, 2, 0, 200),
    # one token through the fused single-token kernel (H a multiple of 1024, I of 512, top-k
    # even): 1..7 consumer warps per row parity, 1..2 groups per down lane, an odd number of
    # down stages per tile (top-6), top-16, two shared experts or none, more experts than
    # top-k threads (200)
    (1024, 512, 24, 6, 1, 1),
    (2048, 512, 40, 16, 2, 1),
    (3072, 1024, 40, 4, 0, 1),
    (1024, 512, 200, 8, 1, 1),
]


@pytest.mark.parametrize("H,I,E,K,NS,T", SHAPES)
def test_layer_shapes(H, I, E, K, NS, T):
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", hidden=H, inter=I,
                              n_experts=E, topk=K, tokens=T, n_shared=NS)
    check_layer(Layer(cfg, seed=H + T))


def test_fused_single_token_ties_bias_bf16_accumulate():
    # equal selection scores (duplicated router rows: the lower index wins), a large bias
    # that forces one expert in without changing the weights, bf16 output, y += layer,
    # and bitwise reproducibility across calls
    L = fused_layer(31)
    wr = L.host["wr"].copy()
    wr[7] = wr[3]
    wr[12] = wr[3]
    wr[20] = wr[9]
    bias = L.host["bias"].copy()
    bias[3] = bias[7] = bias[12] = 1.5
    bias[17] = 3.0
    L.host["wr"], L.host["bias"] = wr, bias
    L.d_wr = torch.from_numpy(wr.view(np.int16)).cuda()
    L.d_bias = torch.from_numpy(bias).cuda()
    oi, ow, oy = L.oracle()
    assert oi[0, :4].tolist() == [17, 3, 7, 12]
    y1, idx, w, st = L.run()
    assert st == 0
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
    assert rel_l2(y1.cpu().numpy(), oy) <= REL_L2_F32
    y2, _, _, _ = L.run()
    assert torch.equal(y1, y2)
    base = torch.randn_like(y1)
    y3, _, _, st = L.run(y=base.clone(), accumulate=True)
    assert st == 0 and torch.equal(y3, base + y1)
    yb, _, _, st = L.run(ydt=torch.bfloat16)
    assert st == 0 and max_rel(yb.float().cpu().numpy(), oy) <= MAX_REL_BF16


def test_fused_topk_one_lane_holds_most_of_the_selection():
    # The single-token kernel's top-k lane l scans experts l, l + 32, ... and keeps its
    # four best; boosting every expert 5 + 32 i puts the first 12 picks in one lane, which
    # must rescan for more three times.  The rest of the selection comes from the others.
    L = fused_layer(34, n_experts=384, topk=16)
    bias = L.host["bias"].copy()
    for i in range(12):
        bias[5 + 32 * i] = 10.0 + i
    L.host["bias"] = bias
    L.d_bias = torch.from_numpy(bias).cuda()
    oi, ow, oy = L.oracle()
    assert oi[0, :12].tolist() == [5 + 32 * i for i in range(11, -1, -1)]
    check_layer(L)


@pytest.mark.parametrize("E,K", [(37, 6), (1100, 8)])
def test_fused_single_token_expert_counts(E, K):
    # 37: the score copy for the top-k includes the workspace's padding (37 * 4 bytes is
    # not a multiple of 16); 1100: the scores exceed the shared-memory copy and the top-k
    # warp reads them from the workspace
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", hidden=1024, inter=512,
                              n_experts=E, topk=K, tokens=1, n_shared=1)
    check_layer(Layer(cfg, seed=35 + K, device_fill=E > 64))


def test_fused_single_token_scale_255_and_0_groups():
    L = fused_layer(32, topk=8, n_experts=16, n_shared=0)
    cfg = L.cfg
    off = cfg.record_offsets
    rec = L._host_experts
    rng = np.random.default_rng(5)
    for op in (1, 3, 5):
        seg = rec[:, off[op]:off[op + 1]]
        seg[rng.random(seg.shape) < 0.05] = 255
        seg[rng.random(seg.shape) < 0.05] = 0
    view = L.experts.view(cfg.n_experts, L.stride)
    view[:, :L.rec_bytes].copy_(torch.from_numpy(rec))
    check_layer(L)


def test_layer_accumulate_and_determinism():
    L = Layer(synth.config("tiny"), seed=3)
    y1, _, _, _ = L.run()
    y2, _, _, _ = L.run()
    assert torch.equal(y1, y2)                       # bitwise reproducible
    base = torch.randn_like(y1)
    y3, _, _, _ = L.run(y=base.clone(), accumulate=True)
    assert torch.equal(y3, base + y1)                # y += layer, one float add


def test_scale_255_and_0_groups():
    cfg = synth.config("tiny")
    L = Layer(cfg, seed=4)
    off = cfg.record_offsets
    rec = L._host_experts
    rng = np.random.default_rng(0)
    for op in (1, 3, 5):
        seg = rec[:, off[op]:off[op + 1]]
        m = rng.random(seg.shape) < 0.05
        seg[m] = 255
        m = rng.random(seg.shape) < 0.05
        seg[m] = 0
    view = L.experts.view(cfg.n_experts, L.stride)
    view[:, :L.rec_bytes].copy_(torch.from_numpy(rec))
    check_layer(L)


def test_expert_ffn_bad_index_reports_and_drops_the_slot():
    cfg = synth.config("tiny")
    L = Layer(cfg, seed=5)
    T, K, H = cfg.tokens, cfg.topk, cfg.hidden
    oi, ow, _, _ = oracle.router(L.x, L.host["wr"], L.host["bias"], K)
    bad = oi.copy()
    bad[1, 1] = cfg.n_experts + 7
    idx = torch.from_numpy(bad).cuda()
    w = torch.from_numpy(ow).cuda()
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    st = k3.new_status()
    k3.k3moe_expert_ffn_mxfp4(L.dims, L.d_x, L.experts, L.stride, idx, w, y,
                              k3.new_workspace(L.dims, T), st)
    torch.cuda.synchronize()
    assert st.item() == 7
    gy = y.cpu().numpy()
    for t in range(T):
        keep = [j for j in range(K) if 0 <= bad[t, j] < cfg.n_experts]
        want = oracle.moe_token(L.x[t], [L.expert_record(int(bad[t, j])) for j in keep],
                                ow[t, keep], H, cfg.inter)
        assert rel_l2(gy[t], want) <= REL_L2_F32


def test_expert_ffn_tensor_core_bad_index_reports_and_drops_the_slot():
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", hidden=512, inter=256,
                              n_experts=8, topk=3, tokens=20, n_shared=0)
    L = Layer(cfg, seed=9)
    T, K, H = cfg.tokens, cfg.topk, cfg.hidden
    oi, ow, _, _ = oracle.router(L.x, L.host["wr"], L.host["bias"], K)
    bad = oi.copy()
    bad[3, 2] = -1
    bad[11, 0] = cfg.n_experts
    idx = torch.from_numpy(bad).cuda()
    w = torch.from_numpy(ow).cuda()
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    st = k3.new_status()
    k3.k3moe_expert_ffn_mxfp4(L.dims, L.d_x, L.experts, L.stride, idx, w, y,
                              k3.new_workspace(L.dims, T), st)
    torch.cuda.synchronize()
    assert st.item() == 7
    gy = y.cpu().numpy()
    for t in range(T):
        keep = [j for j in range(K) if 0 <= bad[t, j] < cfg.n_experts]
        want = oracle.moe_token(L.x[t], [L.expert_record(int(bad[t, j])) for j in keep],
                                ow[t, keep], H, cfg.inter)
        assert rel_l2(gy[t], want) <= REL_L2_F32


def test_tensor_core_path_scale_255_and_0_groups():
    # scale byte 255 (the group contributes nothing) and 0 (2^-127) in every operand
    cfg = dataclasses.replace(synth.config("tiny"), name="custom", hidden=512, inter=256,
                              n_experts=6, topk=2, tokens=9, n_shared=1)
    L = Layer(cfg, seed=12)
    off = cfg.record_offsets
    rec = L._host_experts
    rng = np.random.default_rng(3)
    for op in (1, 3, 5):
        seg = rec[:, off[op]:off[op + 1]]
        m = rng.random(seg.shape) < 0.05
        seg[m] = 255
        m = rng.random(seg.shape) < 0.05
        seg[m] = 0
    view = L.experts.view(cfg.n_experts, L.stride)
    view[:, :L.rec_bytes].copy_(torch.from_numpy(rec))
    check_layer(L)


def test_rmsnorm_bf16():
    rng = np.random.default_rng(0)
    h = (rng.standard_normal((3, 7168)) * 3).astype(np.float32)
    out = torch.empty((3, 7168), dtype=torch.int16, device="cuda")
    k3.k3moe_rmsnorm_bf16(torch.from_numpy(h).cuda(), out, 1e-5)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    for t in range(3):
        want = oracle.f32_to_bf16(oracle.rmsnorm(h[t], eps=1e-5))
        assert np.array_equal(got[t], want)


def test_device_fill_matches_host_generator():
    import synth.device as sd
    cfg = synth.config("tiny")
    stride = (cfg.record_bytes + 4095) // 4096 * 4096
    buf = torch.empty(cfg.n_experts * stride, dtype=torch.uint8, device="cuda")
    sd.fill_experts(buf, cfg, 7, 2, stride=stride)
    torch.cuda.synchronize()
    got = buf.view(-1)[:cfg.n_experts * stride].view(cfg.n_experts, stride)[:, :cfg.record_bytes]
    assert np.array_equal(got.cpu().numpy(), synth.all_experts(cfg, 7, 2))


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.slow
def test_decode1_full_layer():
    cfg = synth.config("decode1")
    L = Layer(cfg, seed=0, tokens=4)
    # each token is one decode step: run them one at a time, like the decode workload
    for t in range(4):
        y, idx, w, st = L.run(x=L.d_x[t:t + 1])
        assert st == 0
        oi, ow, oy = oracle.moe_layer(L.x[t:t + 1], L.host["wr"], L.host["bias"],
                                      L.expert_record, 16, 7168, 1536, L.host["sh_gate"],
                                      L.host["sh_up"], L.host["sh_down"])
        assert np.array_equal(idx.cpu().numpy(), oi)
        assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
        err = rel_l2(y.cpu().numpy(), oy)
        print("decode1 token %d: relative L2 error %.3e" % (t, err))
        assert err <= REL_L2_F32


def test_single_token_tensor_core_gate_up_at_model_width():
    """Top-15 (the fused kernel takes an even top-k only), one token at a time: the router
    kernel, the single-token gate/up on the tensor cores (k_gateup_tc1, the route taken
    in-kernel) and the down kernel, against the oracle."""
    cfg = synth.config("decode1", topk=15)
    L = Layer(cfg, seed=1, tokens=2)
    for t in range(2):
        k3.k3moe_trace_enable(True)
        y, idx, w, st = L.run(x=L.d_x[t:t + 1])
        trace = k3.k3moe_trace_read()
        k3.k3moe_trace_enable(False)
        assert st == 0
        assert trace.get("k_gateup_tc1", (0, 0))[1] >= 1
        assert trace.get("k_gateup_t1", (0, 0))[1] == 0
        oi, ow, oy = oracle.moe_layer(L.x[t:t + 1], L.host["wr"], L.host["bias"],
                                      L.expert_record, 15, 7168, 1536, L.host["sh_gate"],
                                      L.host["sh_up"], L.host["sh_down"])
        assert np.array_equal(idx.cpu().numpy(), oi)
        assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
        err = rel_l2(y.cpu().numpy(), oy)
        print("top-15 token %d through the tensor-core gate/up: relative L2 error %.3e" % (t, err))
        assert err <= REL_L2_F32


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode64_zipf", "decode64_uniform"])
def test_decode64_sampled(name):
    cfg = synth.config(name)
    L = Layer(cfg, seed=0)
    y, idx, w, st = L.run()
    assert st == 0
    # every token's route against the oracle router, outputs on a sample of tokens
    oi, ow, _, _ = oracle.router(L.x, L.host["wr"], L.host["bias"], 16)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
    tokens = [0, 17, 40, 63]
    _, _, oy = L.oracle(tokens=tokens)
    assert rel_l2(y.cpu().numpy()[tokens], oy) <= REL_L2_F32


@pytest.mark.slow
def test_prefill4096_sampled():
    cfg = synth.config("prefill4096")
    L = Layer(cfg, seed=0)
    y, idx, w, st = L.run()
    assert st == 0
    # every token's route against the oracle router, outputs on a sample of tokens
    oi, ow, _, _ = oracle.router(L.x, L.host["wr"], L.host["bias"], 16)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.allclose(w.cpu().numpy(), ow, rtol=2e-7, atol=0)
    tokens = [0, 1, 1000, 2047, 4095]
    _, _, oy = L.oracle(tokens=tokens)
    assert rel_l2(y.cpu().numpy()[tokens], oy) <= REL_L2_F32
