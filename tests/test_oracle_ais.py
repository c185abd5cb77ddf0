"""Pins of the oracle's AIS mixing coefficient (CPU only).

AIS summary, section 2.1 "混合係数": alpha = clip(alpha_ess - beta alpha_var, 0, 1) alpha_mis with
alpha_ess = (1 + CV^2(w))^-1/2, alpha_mis = min(1, dbar / delta), alpha_var = max(0, (dsigma - gamma) /
gamma); section 2.2: w~_i = 1 + alpha (min(rho_i, C) - 1), and alpha -> 0 gives vanilla GRPO (all
weights 1). Each case below has a closed form that the oracle does not use (two-valued weights,
constant weights, saturation), or an invariance of the definition.
"""
import math

import numpy as np
import pytest

import oracle


def _batch(lr, lt, adv):
    return (np.asarray(lr, np.float32), np.asarray(lt, np.float32), np.asarray(adv, np.float32))


def test_no_mismatch_is_vanilla_grpo():
    rng = np.random.default_rng(0)
    lr = -rng.exponential(1.0, 1000).astype(np.float32)
    adv = rng.standard_normal(1000).astype(np.float32)
    st, w = oracle.ais(lr, lr, adv, C=2.0, delta=0.05, gamma=0.5, beta=1.0)
    assert st["alpha"] == 0.0 and st["alpha_mis"] == 0.0 and st["dbar"] == 0.0
    assert st["alpha_ess"] == 1.0 and st["cv2"] == 0.0 and st["dsigma"] == 0.0
    assert np.all(w == 1.0)


def test_two_valued_weights_closed_form():
    # half the tokens at ratio a, half at ratio b (below C): CV^2 = ((a - b) / (a + b))^2
    lt = np.array([0.25, -0.5] * 50, np.float32)
    lr = np.zeros(100, np.float32)
    adv = np.array([1.0, 1.0] * 50, np.float32)  # constant advantages: std(A) = 0, dsigma = 0
    a, b = math.exp(float(np.float32(0.25))), math.exp(float(np.float32(-0.5)))
    st, w = oracle.ais(lr, lt, adv, C=10.0, delta=1.0, gamma=0.5, beta=1.0)
    cv2 = ((a - b) / (a + b)) ** 2
    assert st["cv2"] == pytest.approx(cv2, rel=1e-12)
    assert st["alpha_ess"] == pytest.approx((1 + cv2) ** -0.5, rel=1e-12)
    dbar = (0.25 + 0.5) / 2
    assert st["dbar"] == pytest.approx(dbar, rel=1e-12)
    assert st["alpha_mis"] == pytest.approx(dbar / 1.0, rel=1e-12)  # below the saturation threshold
    assert st["dsigma"] == 0.0 and st["alpha_var"] == 0.0
    alpha = (1 + cv2) ** -0.5 * dbar
    assert st["alpha"] == pytest.approx(alpha, rel=1e-12)
    assert w[0] == pytest.approx(1 + alpha * (a - 1), rel=1e-12)
    assert w[1] == pytest.approx(1 + alpha * (b - 1), rel=1e-12)


def test_truncation_and_saturation():
    # every ratio far above C: all weights truncate to C, CV = 0, and dbar >> delta saturates alpha_mis
    lr = np.full(64, -9.0, np.float32)
    lt = np.full(64, -1.0, np.float32)
    adv = np.array([1.0, -1.0] * 32, np.float32)
    st, w = oracle.ais(lr, lt, adv, C=2.0, delta=0.1, gamma=4.0, beta=1.0)
    assert st["mean_w"] == 2.0 and st["cv2"] == 0.0 and st["alpha_ess"] == 1.0
    assert st["alpha_mis"] == 1.0 and st["dbar"] == 8.0
    # std(w A) / std(A) = C exactly: dsigma = C - 1 = 1 < gamma: no variance penalty
    assert st["dsigma"] == pytest.approx(1.0, rel=1e-15) and st["alpha_var"] == 0.0
    assert st["alpha"] == 1.0 and np.all(w == 2.0)


@pytest.mark.parametrize("k,gamma,beta", [(3.0, 0.5, 0.25), (3.0, 0.5, 1.0), (1.2, 0.5, 1.0), (5.0, 1.0, 0.1)])
def test_variance_penalty_closed_form(k, gamma, beta):
    # constant ratio k (below C) and advantages +-1: CV = 0, std(kA)/std(A) = k, dsigma = k - 1
    lk = float(np.float32(math.log(k)))
    lr = np.zeros(40, np.float32)
    lt = np.full(40, lk, np.float32)
    adv = np.array([1.0, -1.0] * 20, np.float32)
    st, w = oracle.ais(lr, lt, adv, C=100.0, delta=0.01, gamma=gamma, beta=beta)
    kk = math.exp(lk)
    a_var = max(0.0, (kk - 1 - gamma) / gamma)
    assert st["dsigma"] == pytest.approx(kk - 1, rel=1e-12)
    assert st["alpha_var"] == pytest.approx(a_var, rel=1e-12, abs=1e-15)
    alpha = min(1.0, max(0.0, 1.0 - beta * a_var)) * 1.0
    assert st["alpha"] == pytest.approx(alpha, rel=1e-12, abs=1e-15)
    assert np.allclose(w, 1 + alpha * (kk - 1), rtol=1e-12)


def test_invariances():
    rng = np.random.default_rng(3)
    n = 777
    lr = -rng.exponential(2.0, n).astype(np.float32)
    lt = (lr + rng.normal(0, 0.1, n)).astype(np.float32)
    adv = rng.standard_normal(n).astype(np.float32)
    base, w = oracle.ais(lr, lt, adv, 2.0, 0.05, 0.3, 0.5)
    p = rng.permutation(n)
    st_p, w_p = oracle.ais(lr[p], lt[p], adv[p], 2.0, 0.05, 0.3, 0.5)
    for k in base:
        assert st_p[k] == pytest.approx(base[k], rel=1e-12, abs=1e-15)
    assert np.allclose(w_p, w[p], rtol=1e-12)
    # scaling the advantages by a power of two changes no statistic (dsigma is a ratio of spreads)
    st_s, _ = oracle.ais(lr, lt, (adv * 4).astype(np.float32), 2.0, 0.05, 0.3, 0.5)
    for k in base:
        assert st_s[k] == pytest.approx(base[k], rel=1e-12, abs=1e-15)
    # weights lie between 1 and min(rho, C): w~ - 1 = alpha (w - 1), 0 <= alpha <= 1
    assert 0.0 <= base["alpha"] <= 1.0
    rho = np.minimum(np.exp(lt.astype(np.float64) - lr.astype(np.float64)), 2.0)
    assert np.allclose(w - 1, base["alpha"] * (rho - 1), rtol=1e-12, atol=1e-15)


def test_penalty_clips_at_zero():
    # a large variance penalty drives alpha_ess - beta alpha_var below zero: alpha = 0, weights 1
    lr = np.zeros(8, np.float32)
    lt = np.full(8, np.float32(math.log(4.0)), np.float32)
    adv = np.array([1, -1] * 4, np.float32)
    st, w = oracle.ais(lr, lt, adv, C=100.0, delta=0.01, gamma=0.5, beta=2.0)
    assert st["alpha_var"] > 1 and st["alpha"] == 0.0 and np.all(w == 1.0)
