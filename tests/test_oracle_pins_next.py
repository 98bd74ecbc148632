"""Pins of the oracle's dense-path, logits-backward, GRPO-loss and greedy
functions to facts other than the oracle itself: library routines (numpy
matmul, scipy, torch fp64 autograd of log_softmax), closed forms, finite
differences and constructed ties."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from invariant_rl_logprob_gb300 import synth


def test_lm_head_vs_numpy(oracle_mod):
    g = synth.generator(50)
    W = synth.normal_bf16(g, (37, 48), 0.5)
    h = synth.normal_bf16(g, (5, 48), 1.0)
    z = oracle_mod.lm_head(synth.bf16_bits(h), synth.bf16_bits(W))
    np.testing.assert_allclose(z, h.double().numpy() @ W.double().numpy().T, atol=1e-12, rtol=0)


def test_logits_bwd_vs_autograd_and_sum(oracle_mod):
    z, tg, _ = synth.logits_batch(T=6, V=300, seed=12)
    gr = np.array([1.0, -0.5, 2.0, 0.0, 3.0, -1.0])
    dz = oracle_mod.logits_bwd(synth.bf16_bits(z), tg.numpy(), gr)
    zz = z.double().clone().requires_grad_(True)
    ls = torch.log_softmax(zz, dim=1)
    (ls[torch.arange(6), tg] * torch.from_numpy(gr)).sum().backward()
    np.testing.assert_allclose(dz, zz.grad.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-12)      # g (1 - sum p) = 0


def test_logits_bwd_finite_differences(oracle_mod):
    rng = np.random.default_rng(9)
    V = 11
    z = rng.normal(0, 2, (1, V))
    tg = np.array([4])
    dz = oracle_mod.logits_bwd(z, tg, np.array([1.0]))[0]
    eps = 1e-6
    for v in range(V):
        zp, zm = z.copy(), z.copy()
        zp[0, v] += eps
        zm[0, v] -= eps
        fd = (oracle_mod.logp_from_logits(zp, tg)[0][0] - oracle_mod.logp_from_logits(zm, tg)[0][0]) / (2 * eps)
        assert abs(fd - dz[v]) < 1e-7


def test_logits_bwd_masking(oracle_mod):
    z = np.zeros((3, 5))
    out = oracle_mod.logits_bwd(z, np.array([1, -100, 2]), np.ones(3))
    assert np.all(out[1] == 0)
    np.testing.assert_allclose(out[0], [-0.2, 0.8, -0.2, -0.2, -0.2], atol=1e-15)


# ---- GRPO per-token loss ----

def test_grpo_on_policy_closed_form(oracle_mod):
    lp = np.array([-1.0, -2.5, -0.1])
    a = np.array([0.7, -1.3, 2.0])
    o = oracle_mod.grpo_token(lp, lp, a, eps_low=0.2, eps_high=0.28)
    np.testing.assert_allclose(o["ratio"], 1.0, atol=0)
    np.testing.assert_allclose(o["loss"], -a, atol=1e-15)
    np.testing.assert_allclose(o["grad"], -a, atol=1e-15)


def test_grpo_clipping_cases(oracle_mod):
    lp_old = np.zeros(4)
    lp = np.array([math.log(1.5), math.log(0.5), math.log(1.5), math.log(0.5)])
    a = np.array([1.0, -1.0, -1.0, 1.0])
    o = oracle_mod.grpo_token(lp, lp_old, a, eps_low=0.2, eps_high=0.2)
    # A>0, ratio above 1.2: clipped term 1.2 * A is the min, no gradient
    assert abs(o["loss"][0] + 1.2) < 1e-15 and o["grad"][0] == 0.0
    # A<0, ratio below 0.8: clipped term 0.8 * A = -0.8 is the min, no gradient
    assert abs(o["loss"][1] - 0.8) < 1e-15 and o["grad"][1] == 0.0
    # A<0, ratio above 1.2: unclipped term -1.5 is the min, gradient -A*ratio
    assert abs(o["loss"][2] - 1.5) < 1e-12 and abs(o["grad"][2] - 1.5) < 1e-12
    # A>0, ratio below 0.8: unclipped term 0.5 is the min, gradient -A*ratio
    assert abs(o["loss"][3] + 0.5) < 1e-12 and abs(o["grad"][3] + 0.5) < 1e-12


def test_grpo_kl_properties(oracle_mod):
    rng = np.random.default_rng(3)
    lp = rng.normal(-2, 1, 50)
    o0 = oracle_mod.grpo_token(lp, lp, np.zeros(50), logp_ref=lp, beta=0.1)
    assert np.all(o0["kl"] == 0) and np.all(o0["grad"] == 0) and np.all(o0["loss"] == 0)
    ref = lp + rng.normal(0, 0.5, 50)
    o = oracle_mod.grpo_token(lp, lp, np.zeros(50), logp_ref=ref, beta=1.0)
    assert np.all(o["kl"] >= 0)
    d = ref - lp
    np.testing.assert_allclose(o["kl"], np.expm1(d) - d, rtol=1e-12, atol=1e-15)


def test_grpo_finite_differences(oracle_mod):
    rng = np.random.default_rng(4)
    n = 40
    lp_old = rng.normal(-2, 1, n)
    lp = lp_old + rng.normal(0, 0.3, n)
    ref = lp + rng.normal(0, 0.3, n)
    a = rng.normal(0, 1, n)
    kw = dict(eps_low=0.2, eps_high=0.28, beta=0.05, scale=0.5)
    o = oracle_mod.grpo_token(lp, lp_old, a, logp_ref=ref, **kw)
    eps = 1e-6
    lo_b, hi_b = math.log(0.8), math.log(1.28)
    for i in range(n):
        dlr = lp[i] - lp_old[i]
        if abs(dlr - lo_b) < 1e-4 or abs(dlr - hi_b) < 1e-4:
            continue                                          # kink of the clip
        p1, m1 = lp.copy(), lp.copy()
        p1[i] += eps
        m1[i] -= eps
        fd = (oracle_mod.grpo_token(p1, lp_old, a, logp_ref=ref, **kw)["loss"][i]
              - oracle_mod.grpo_token(m1, lp_old, a, logp_ref=ref, **kw)["loss"][i]) / (2 * eps)
        assert abs(fd - o["grad"][i]) < 1e-7, i


def test_grpo_masking(oracle_mod):
    lp = np.array([-1.0, -2.0, -3.0])
    o = oracle_mod.grpo_token(lp, lp - 0.1, np.ones(3), targets=np.array([3, -100, 5]))
    assert o["loss"][1] == 0 and o["grad"][1] == 0 and o["loss"][0] != 0


# ---- greedy decoding step ----

def test_greedy_vs_library(oracle_mod):
    g = synth.generator(60)
    W = synth.normal_bf16(g, (300, 32), 0.5)
    h = synth.normal_bf16(g, (7, 32), 1.0)
    tok, lp, zm = oracle_mod.linear_greedy(synth.bf16_bits(h), synth.bf16_bits(W))
    z = h.double().numpy() @ W.double().numpy().T
    np.testing.assert_array_equal(tok, np.argmax(z, axis=1))
    np.testing.assert_allclose(lp, z.max(axis=1) - scipy.special.logsumexp(z, axis=1), atol=1e-12)
    np.testing.assert_allclose(zm, z.max(axis=1), atol=1e-12)
    lp2, _ = oracle_mod.linear_logp(synth.bf16_bits(h), synth.bf16_bits(W), tok)
    np.testing.assert_allclose(lp, lp2, atol=0, rtol=0)            # re-score = decode


def test_greedy_ties_take_lowest_index(oracle_mod):
    W = np.zeros((10, 8))
    W[3, 0] = W[7, 0] = 2.0
    h = np.zeros((1, 8))
    h[0, 0] = 1.0
    tok, lp, _ = oracle_mod.linear_greedy(h, W)
    assert tok[0] == 3
    assert abs(lp[0] - (2.0 - math.log(2 * math.exp(2.0) + 8))) < 1e-12


# ---- dW ----

@pytest.mark.parametrize("H,V,T", [(16, 7, 5), (32, 40, 9)])
def test_dw_vs_torch_autograd(oracle_mod, H, V, T):
    g = synth.generator(400 + H + V)
    W = synth.normal_bf16(g, (V, H), 0.5)
    h = synth.normal_bf16(g, (T, H), 1.0)
    tg = synth.uniform_targets(g, T, V)
    gr = torch.randn(T, generator=g, dtype=torch.float64)
    dW = oracle_mod.linear_logp_dw(synth.bf16_bits(h), synth.bf16_bits(W), tg.numpy(), gr.numpy())
    WW = W.double().clone().requires_grad_(True)
    ls = torch.log_softmax(h.double() @ WW.T, dim=1)
    (ls[torch.arange(T), tg] * gr).sum().backward()
    np.testing.assert_allclose(dW, WW.grad.numpy(), atol=1e-12, rtol=0)


def test_dw_finite_differences_and_columns(oracle_mod):
    rng = np.random.default_rng(21)
    H, V, T = 6, 5, 4
    W = rng.normal(0, 0.7, (V, H))
    h = rng.normal(0, 1, (T, H))
    tg = rng.integers(0, V, T)
    gr = rng.normal(0, 1, T)
    dW = oracle_mod.linear_logp_dw(h, W, tg, gr)
    eps = 1e-6

    def f(WW):
        lp, _ = oracle_mod.linear_logp(h, WW, tg)
        return float(np.dot(gr, lp))
    for v in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            assert abs((f(Wp) - f(Wm)) / (2 * eps) - dW[v, k]) < 1e-7
    # sum over v of dW[v, :] = sum_t g_t (1 - 1) h_t = 0
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-12)


def test_dw_masking(oracle_mod):
    rng = np.random.default_rng(22)
    W = rng.normal(0, 1, (5, 4))
    h = rng.normal(0, 1, (3, 4))
    full = oracle_mod.linear_logp_dw(h, W, np.array([1, 2, 3]), np.ones(3))
    part = oracle_mod.linear_logp_dw(h, W, np.array([1, -100, 3]), np.ones(3))
    only = oracle_mod.linear_logp_dw(h[[0, 2]], W, np.array([1, 3]), np.ones(2))
    np.testing.assert_allclose(part, only, atol=1e-15)
    assert not np.allclose(full, part)
