"""Expert records whose routed sum depends on the order of its terms.

The layer's routed sum is a float sum taken in router order (README of
FareedKhan-dev/kimi-k3-in-c, section 9, LatentMoE listing step 3; README of
Maknee/Kimi-K3.cpp, "The consumer-memory idea", item 7).  Float addition is not
associative, so the order shows in the result when the terms are chosen for it:

  * every probe expert has the same gate and up operands, so all of them see the same
    SiTU activations;
  * output row i names three router positions (p, q, r).  Expert p's down row i is a
    random MXFP4 row at a large scale, expert q's is the same row with every code's sign
    flipped (E2M1 code ^ 8), so w_p d_p[i] = -w_q d_q[i] exactly when w_p = w_q; expert
    r's is a random row about 2^60 smaller; every other expert's row i has zero codes and
    scale byte 255 and contributes exactly zero;
  * summed left to right, S + b rounds to S while b is below half an ulp of S, so the
    row's sum is exactly 0 unless position r comes after both p and q, in which case it
    is exactly fl(w_r d_r[i]) (the big pair cancels first).

Over all triples (p, q, r) these rows pin the order of the terms: any order other than
router order (up to swapping the first two terms, which a float sum from zero cannot
tell apart) turns some row from zero to nonzero or back.  A sum accumulated in double, or
in any order that lets the pair cancel before the small term is added, gives the small
term in every row.

The construction only writes bytes (codes, scale bytes); it computes nothing of the
method.
"""
import itertools

import numpy as np

import synth

BIG = 127 + 20     # scale byte of the cancelling pair: 2^20
SMALL = 127 - 40   # scale byte of the small term: 2^-40


def triples(K):
    """Every (p, q, r) with p < q and r outside {p, q}."""
    return [(p, q, r) for p, q in itertools.combinations(range(K), 2) for r in range(K)
            if r not in (p, q)]


def records(H, I, K, seed):
    """K expert records of the (H, I) layout and the triple of every output row.

    Returns (recs uint8 [K][record bytes], pattern int [H][3])."""
    off = synth.record_offsets(H, I)
    rng = np.random.default_rng(seed)
    recs = np.zeros((K, off[6]), np.uint8)
    gate = rng.integers(0, 256, off[1] - off[0], dtype=np.uint8)
    gate_s = rng.integers(122, 127, off[2] - off[1], dtype=np.uint8)
    up = rng.integers(0, 256, off[5] - off[4], dtype=np.uint8)
    up_s = rng.integers(122, 127, off[6] - off[5], dtype=np.uint8)
    tr = triples(K)
    pattern = np.array([tr[i % len(tr)] for i in range(H)], dtype=np.int64)
    rowb, rows_s = I // 2, I // 32
    # background rows: code 0 with scale byte 255, exactly zero on every path (a path
    # that reads byte 255 as 2^-127 still multiplies it by zero codes)
    down = np.zeros((K, H, rowb), np.uint8)
    down_s = np.full((K, H, rows_s), 255, np.uint8)
    base = rng.integers(0, 256, (H, rowb), dtype=np.uint8)
    small = rng.integers(0, 256, (H, rowb), dtype=np.uint8)
    for i, (p, q, r) in enumerate(pattern):
        down[p, i] = base[i]
        down[q, i] = base[i] ^ 0x88          # both nibbles' sign bits: exactly -row
        down_s[p, i] = BIG
        down_s[q, i] = BIG
        down[r, i] = small[i]
        down_s[r, i] = SMALL
    for k in range(K):
        recs[k, off[0]:off[1]] = gate
        recs[k, off[1]:off[2]] = gate_s
        recs[k, off[2]:off[3]] = down[k].ravel()
        recs[k, off[3]:off[4]] = down_s[k].ravel()
        recs[k, off[4]:off[5]] = up
        recs[k, off[5]:off[6]] = up_s
    return recs, pattern


def zero_rows(pattern):
    """Rows whose router-order sum is exactly zero: the small term's position r comes
    before at least one of the cancelling pair's."""
    p, q, r = pattern[:, 0], pattern[:, 1], pattern[:, 2]
    return r < np.maximum(p, q)


def small_term_position(pattern):
    """Position r of each row (its sum, where nonzero, is exactly w_r d_r[i])."""
    return pattern[:, 2]
