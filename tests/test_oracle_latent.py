"""Pins of the oracle's LatentMoE (README of FareedKhan-dev/kimi-k3-in-c, section 9,
LatentMoE listing steps 1-6; section 2, K3Cfg fields latent, n_shared, latent_norm;
section 5 for RMSNorm and the bf16 weight products).

Each step is checked against something other than the oracle's own code: a textbook
double matvec in numpy for the projections, the RMS of the normed aggregate (1 by the
norm's definition, which per-expert norming does not give), exact special cases (a zero
down-projection leaves exactly the shared experts' output), and the page's own claim that
norming each expert and then summing is a different function.
"""
import numpy as np

import oracle

H, L, I, K, SI = 96, 64, 64, 3, 64


def widen(b):
    return oracle.bf16_to_f32(b).astype(np.float64)


def setup(seed):
    rng = np.random.default_rng(seed)
    bf = lambda a: oracle.f32_to_bf16(np.asarray(a, np.float32))
    x = bf(rng.standard_normal(H))
    wdn = bf(rng.standard_normal((L, H)) / np.sqrt(H))
    wup = bf(rng.standard_normal((H, L)) / np.sqrt(L))
    off = oracle.record_offsets(L, I)
    recs = []
    for _ in range(K):
        r = rng.integers(0, 256, off[6], dtype=np.uint8)
        for a, b in ((1, 2), (3, 4), (5, 6)):
            r[off[a]:off[b]] = rng.integers(122, 127, off[b] - off[a])
        recs.append(r)
    w = rng.dirichlet(np.ones(K)).astype(np.float32)
    sh = (bf(rng.standard_normal((SI, H)) / np.sqrt(H)), bf(rng.standard_normal((SI, H)) / np.sqrt(H)),
          bf(rng.standard_normal((H, SI)) / np.sqrt(SI)))
    nw = (1.0 + 0.25 * rng.standard_normal(L)).astype(np.float32)
    return x, wdn, wup, recs, w, sh, nw


def test_down_projection_is_the_bf16_matvec_of_the_full_width_input():
    x, wdn, wup, recs, w, sh, nw = setup(1)
    _, z, _ = oracle.latent_moe_token(x, recs, w, H, L, I, wdn, wup, nw, intermediates=True)
    want = (widen(wdn) @ widen(x)).astype(np.float32)   # double sum, one rounding
    assert np.array_equal(z, want)


def test_experts_run_in_the_latent_and_sum_in_router_order():
    x, wdn, wup, recs, w, sh, nw = setup(2)
    _, z, acc = oracle.latent_moe_token(x, recs, w, H, L, I, wdn, wup, nw, latent_norm=False,
                                        intermediates=True)
    d = [oracle.expert(r, z, L, I) for r in recs]
    want = np.zeros(L, np.float32)
    for j in range(K):                                   # float, j in router order
        want = want + w[j] * d[j]
    assert np.array_equal(acc, want)


def test_norm_is_on_the_aggregate_not_on_each_expert():
    x, wdn, wup, recs, w, sh, _ = setup(3)
    ones = np.ones(L, np.float32)
    _, z, acc = oracle.latent_moe_token(x, recs, w, H, L, I, wdn, wup, ones, intermediates=True)
    # RMSNorm with weight 1 leaves the aggregate at RMS 1 (eps 1e-5 against a mean square
    # of order 1 moves it by ~5e-6)
    rms = np.sqrt(np.mean(acc.astype(np.float64) ** 2))
    assert abs(rms - 1.0) < 2e-5
    # the page: norming each expert first and summing is a different function
    d = [oracle.expert(r, z, L, I).astype(np.float64) for r in recs]
    per_expert = sum(w[j] * d[j] / np.sqrt(np.mean(d[j] ** 2) + 1e-5) for j in range(K))
    assert np.sqrt(np.mean(per_expert ** 2)) < 0.99      # a convex sum of unit vectors
    assert np.abs(acc - per_expert).max() > 1e-2
    # the norm's weight multiplies element by element: weight 2 doubles the latent exactly
    _, _, acc2 = oracle.latent_moe_token(x, recs, w, H, L, I, wdn, wup, 2 * ones,
                                         intermediates=True)
    assert np.array_equal(acc2, 2 * acc)


def test_up_projection_and_unweighted_shared_experts_on_the_original_input():
    x, wdn, wup, recs, w, sh, nw = setup(4)
    y, z, acc = oracle.latent_moe_token(x, recs, w, H, L, I, wdn, wup, nw, sh_gate=sh[0],
                                        sh_up=sh[1], sh_down=sh[2], intermediates=True)
    up = (widen(wup) @ acc.astype(np.float64)).astype(np.float32)
    ds = oracle.shared_expert(sh[0], sh[1], sh[2], oracle.bf16_to_f32(x))
    assert np.array_equal(y, up + ds)                    # one float add per element
    # the shared experts see the full-width x, not the latent: with the down-projection
    # zeroed the latent is zero (SiTU(0, 0) = 0, RMSNorm(0) = 0) and y is exactly shared(x)
    y0 = oracle.latent_moe_token(x, recs, w, H, L, I, np.zeros_like(wdn), wup, nw,
                                 sh_gate=sh[0], sh_up=sh[1], sh_down=sh[2])
    assert np.array_equal(y0, ds) and np.abs(ds).max() > 0


def test_layer_routes_on_the_full_width_input():
    x, wdn, wup, recs, w, sh, nw = setup(5)
    rng = np.random.default_rng(6)
    E = 8
    X = oracle.f32_to_bf16(rng.standard_normal((3, H)).astype(np.float32))
    wr = oracle.f32_to_bf16((rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    off = oracle.record_offsets(L, I)
    pool = [recs[e % K] if e < K else rng.integers(0, 256, off[6], dtype=np.uint8) for e in range(E)]
    for r in pool[K:]:
        for a, b in ((1, 2), (3, 4), (5, 6)):
            r[off[a]:off[b]] = rng.integers(122, 127, off[b] - off[a])
    idx, wt, y = oracle.latent_moe_layer(X, wr, bias, lambda e: pool[e], K, H, L, I, wdn, wup, nw)
    ri, rw, _, _ = oracle.router(X, wr, bias, K)
    assert np.array_equal(idx, ri) and np.array_equal(wt, rw)
    for t in range(3):
        want = oracle.latent_moe_token(X[t], [pool[e] for e in ri[t]], rw[t], H, L, I, wdn, wup, nw)
        assert np.array_equal(y[t], want)
