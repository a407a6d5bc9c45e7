"""Pins of the oracle router (kimi-k3-in-c, section 9 "Picking 16 experts of 896"; "Three
invariants", item 3): top-k against a full sort and brute force, tie-breaking, the bias
steering selection only, renormalisation."""
import itertools

import numpy as np
import pytest

import oracle


def sigmoid_f(z):
    return np.float32(1.0 / (1.0 + np.exp(-np.float64(z))))


def make(E, H, seed, bias_scale=0.1):
    rng = np.random.default_rng(seed)
    x = oracle.f32_to_bf16(rng.standard_normal((1, H)).astype(np.float32))
    wr = oracle.f32_to_bf16((rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32))
    bias = rng.uniform(-bias_scale, bias_scale, E).astype(np.float32)
    return x, wr, bias


def test_logits_are_double_dot_rounded_to_float():
    x, wr, bias = make(12, 64, 0)
    _, _, logits, scores = oracle.router(x, wr, bias, 3)
    xd = oracle.bf16_to_f32(x).astype(np.float64)[0]
    wd = oracle.bf16_to_f32(wr).astype(np.float64)
    want = (wd @ xd).astype(np.float32)
    assert np.array_equal(logits[0], want)
    assert np.array_equal(scores[0], np.array([sigmoid_f(v) for v in want], np.float32))


@pytest.mark.parametrize("seed", range(6))
def test_topk_equals_full_sort_by_choice_desc_index_asc(seed):
    E, K = 40, 7
    x, wr, bias = make(E, 96, seed)
    idx, w, _, sc = oracle.router(x, wr, bias, K)
    ch = (sc[0] + bias).astype(np.float32)
    order = np.lexsort((np.arange(E), -ch.astype(np.float64)))
    assert idx[0].tolist() == order[:K].tolist()


@pytest.mark.parametrize("E,K", [(5, 1), (6, 2), (8, 3)])
def test_topk_brute_force_over_all_subsets(E, K):
    for seed in range(4):
        x, wr, bias = make(E, 32, 100 + seed)
        idx, _, _, sc = oracle.router(x, wr, bias, K)
        ch = (sc[0] + bias).astype(np.float32)
        # the chosen set is the unique K-subset whose every member beats every outsider
        # under (ch desc, index asc)
        def beats(a, b):
            return ch[a] > ch[b] or (ch[a] == ch[b] and a < b)
        winners = [s for s in itertools.combinations(range(E), K)
                   if all(beats(a, b) for a in s for b in range(E) if b not in s)]
        assert len(winners) == 1
        assert sorted(idx[0].tolist()) == list(winners[0])
        # and the order is descending by the same key
        assert all(beats(idx[0][i], idx[0][i + 1]) for i in range(K - 1))


def test_ties_go_to_the_lower_index():
    E, H = 8, 32
    x = oracle.f32_to_bf16(np.ones((1, H), np.float32))
    wr = np.zeros((E, H), np.uint16)          # every logit 0 -> every score 0.5
    bias = np.zeros(E, np.float32)
    idx, w, _, _ = oracle.router(x, wr, bias, 3)
    assert idx[0].tolist() == [0, 1, 2]
    bias[5] = bias[6] = 0.25                  # two equal winners: lower index first
    idx, _, _, _ = oracle.router(x, wr, bias, 3)
    assert idx[0].tolist() == [5, 6, 0]


def test_bias_changes_selection_but_not_the_weights_of_chosen_experts():
    E, H, K = 16, 64, 4
    x, wr, _ = make(E, H, 11)
    zero = np.zeros(E, np.float32)
    idx0, w0, _, sc = oracle.router(x, wr, zero, K, renorm=False)
    # push the 5th-ranked expert (by score) into the top set
    order = np.argsort(-sc[0], kind="stable")
    bias = zero.copy()
    bias[order[K]] = 1.0
    idx1, w1, _, _ = oracle.router(x, wr, bias, K, renorm=False)
    assert idx1[0][0] == order[K] and set(idx1[0]) != set(idx0[0])
    # weights are the UNBIASED scores of the chosen experts
    assert np.array_equal(w1[0], sc[0][idx1[0]])


def test_renorm_sums_to_routed_scale_and_zero_sum_guard():
    E, H, K = 20, 64, 5
    x, wr, bias = make(E, H, 12)
    _, w, _, _ = oracle.router(x, wr, bias, K, renorm=True, routed_scale=2.5)
    assert abs(float(w[0].astype(np.float64).sum()) - 2.5) < 1e-5
    # all scores 0 (logits -> -inf): the s > 0 guard leaves the weights at 0, no NaN
    xb = oracle.f32_to_bf16(np.full((1, H), 1.0, np.float32))
    wrb = oracle.f32_to_bf16(np.full((E, H), -1e30, np.float32))
    _, w2, _, sc2 = oracle.router(xb, wrb, np.zeros(E, np.float32), K)
    assert np.all(sc2 == 0.0) and np.all(w2 == 0.0)


def test_nonfinite_score_is_refused():
    E, H = 6, 32
    x = oracle.f32_to_bf16(np.ones((1, H), np.float32))
    wr = np.zeros((E, H), np.uint16)
    bias = np.zeros(E, np.float32)
    bias[2] = np.inf
    with pytest.raises(ValueError):
        oracle.router(x, wr, bias, 2)
