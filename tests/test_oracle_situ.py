"""Pins of the oracle's SiTU-GLU (kimi-k3-in-c, section 9, activation listing): the cap
|act| <= b1 b2 = 100 reached at large inputs, the sigmoid on the UNCAPPED gate, odd
symmetry in the up input."""
import json
import math
import os

import numpy as np

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


def test_bound_and_its_attainment():
    cap = GOLD["situ_bound"]["max_abs_out"]
    b1, b2 = GOLD["moe_config"]["situ_b1"], GOLD["moe_config"]["situ_b2"]
    assert b1 * b2 == cap
    v = np.concatenate([np.geomspace(0.1, 1000.0, 24), -np.geomspace(0.1, 1000.0, 24)])
    g, u = np.meshgrid(v, v)
    act = oracle.situ(g.ravel().astype(np.float32), u.ravel().astype(np.float32), b1, b2)
    assert np.all(np.abs(act) <= cap)
    # the page's fixture drives |out| to the analytic cap: g = u = 1000
    top = oracle.situ(np.float32([1000.0]), np.float32([1000.0]), b1, b2)[0]
    assert top == np.float32(100.0)


def test_sigmoid_takes_the_uncapped_gate():
    b1, b2 = 4.0, 25.0
    g, u = 8.0, 3.0
    got = float(oracle.situ(np.float32([g]), np.float32([u]), b1, b2)[0])
    uncapped = b1 * math.tanh(g / b1) / (1 + math.exp(-g)) * b2 * math.tanh(u / b2)
    capped_g = b1 * math.tanh(g / b1)
    capped = capped_g / (1 + math.exp(-capped_g)) * b2 * math.tanh(u / b2)
    assert abs(got - uncapped) <= 1e-6 * abs(uncapped)
    assert abs(got - capped) > 1e-2 * abs(capped)   # the wrong reading differs by ~2%


def test_odd_in_up_and_small_input_limit():
    g = np.float32([0.5, -1.5, 3.0])
    u = np.float32([0.25, 2.0, -7.0])
    assert np.array_equal(oracle.situ(g, -u), -oracle.situ(g, u))
    # near zero the caps are the identity: act ~ g * sigmoid(g) * u
    gs, us = np.float32([1e-3]), np.float32([2e-3])
    want = 1e-3 / (1 + math.exp(-1e-3)) * 2e-3
    assert abs(float(oracle.situ(gs, us)[0]) - want) <= 1e-6 * want
