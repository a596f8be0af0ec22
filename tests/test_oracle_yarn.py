"""Pins of the oracle's YaRN context extension (RoPE frequencies and the
attention temperature), against the figures printed in section 3.2 of the
DeepSeek-V2 analysis page and against closed forms and brute force."""
import json
import math
import os

import numpy as np

import oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "yarn.json")))
G = {v["name"]: v for v in GOLDEN["values"]}


def page_theta():
    return O.yarn_theta(G["rope_dims"]["value"], 10000.0, G["factor_s"]["value"], G["alpha"]["value"],
                        G["beta"]["value"], G["original_window"]["value"])


def test_printed_temperatures_and_window():
    s = G["factor_s"]["value"]
    for coef, name in (("v2_coef", "v2_temperature_at_s40"), ("yarn_coef", "yarn_temperature_at_s40")):
        t = O.yarn_temperature(s, G[coef]["value"])
        assert abs(t - G[name]["value"]) <= G[name]["tolerance"], (name, t)
    assert G["original_window"]["value"] * s == G["target_window"]["value"]


def test_softmax_scale_carries_the_square_of_the_temperature():
    # YaRN scales q and k each by sqrt(1/t): the logit q.k by its square
    m = O.yarn_temperature(40.0, 0.0707)
    assert math.isclose(O.yarn_softmax_scale(0.5, 40.0, 0.0707), 0.5 * m * m, rel_tol=1e-15)
    assert O.yarn_softmax_scale(0.5, 1.0, 0.0707) == 0.5
    # same effect as rotating q and k with sqrt(1/t)-scaled cos/sin on a pure-RoPE dot product
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    qs, ks = O.rope(q, 100, 10000.0) * m, O.rope(k, 7, 10000.0) * m
    assert math.isclose(float(qs @ ks) * 0.5, float(O.rope(q, 100, 10000.0) @ O.rope(k, 7, 10000.0)) *
                        O.yarn_softmax_scale(0.5, 40.0, 0.0707), rel_tol=1e-12)


def test_factor_one_is_plain_rope():
    for d_r in (16, 64):
        th = O.yarn_theta(d_r, 10000.0, 1.0, 1.0, 32.0, 4096)
        i = np.arange(d_r // 2)
        assert np.array_equal(th, 10000.0 ** (-2.0 * i / d_r))


def turns_brute_force(theta, window):
    """Full turns a pair makes over positions 0..window: counted by stepping the angle."""
    ang = 0.0
    turns = 0
    for _ in range(window):
        ang += theta
        while ang >= 2 * math.pi:
            ang -= 2 * math.pi
            turns += 1
    return turns


def test_regimes_by_counted_turns():
    """Pairs turning more than beta times over the 4K window keep their
    frequency, pairs turning less than alpha times are divided by s, the rest
    lie strictly between (turns counted by brute force, not by the formula)."""
    base, d_r, s, a, b, L = 10000.0, 64, 40.0, 1.0, 32.0, 4096
    plain = O.rope_theta(d_r, base)
    th = page_theta()
    seen = set()
    for i in range(d_r // 2):
        n = turns_brute_force(plain[i], L)
        if n >= b + 1:                       # certainly more than beta turns
            assert th[i] == plain[i], i
            seen.add("keep")
        elif n == 0 and plain[i] * L < 2 * math.pi * a * 0.99:   # less than alpha turns
            assert math.isclose(th[i], plain[i] / s, rel_tol=1e-15), i
            seen.add("interp")
        elif a + 1 <= n <= b - 1:            # inside the ramp
            assert plain[i] / s < th[i] < plain[i], i
            seen.add("ramp")
    assert seen == {"keep", "interp", "ramp"}


def test_ramp_is_monotone_and_continuous():
    # a dense sweep of frequencies through both ends of the ramp
    base, s, a, b, L = 10000.0, 40.0, 1.0, 32.0, 4096
    d_r = 2048
    plain = O.rope_theta(d_r, base)
    th = O.yarn_theta(d_r, base, s, a, b, L)
    ratio = th / plain                     # 1 at high frequency, 1/s at low, non-increasing in i
    assert ratio[0] == 1.0 and math.isclose(ratio[-1], 1.0 / s, rel_tol=1e-12)
    assert np.all(np.diff(ratio) <= 1e-15)
    assert np.max(np.abs(np.diff(ratio))) < 0.02   # no jump at either end of the ramp


def test_rope_invariants_hold_with_yarn_frequencies():
    th = page_theta()
    rng = np.random.default_rng(5)
    x = rng.standard_normal(64)
    assert np.array_equal(O.rope(x, 0, 10000.0, th), x)                 # position 0: identity
    y = O.rope(x, 131071, 10000.0, th)
    assert np.allclose(np.hypot(y[0::2], y[1::2]), np.hypot(x[0::2], x[1::2]), rtol=1e-13)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d1 = O.rope(q, 5000, 10000.0, th) @ O.rope(k, 4000, 10000.0, th)
    d2 = O.rope(q, 101000, 10000.0, th) @ O.rope(k, 100000, 10000.0, th)
    assert math.isclose(d1, d2, rel_tol=1e-9)                             # depends on the offset only
