"""Pins of the fp64 oracle to facts other than itself.

The pages print no worked numeric example for the selected-token logprob, so
the oracle is pinned to closed forms, invariants, library routines and finite
differences, chosen so that a plausible slip (a dropped max shift, a wrong
target index, a transposed W, a missing one-hot term or a wrong sign in the
backward, a broken mask) fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from invariant_rl_logprob_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def bf16(x) -> np.ndarray:
    """bf16 bits of x (values must be exactly representable)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float32)), "value not exact in bf16"
    return synth.bf16_bits(t)


# --------------------------------------------------------------------------
# 1. Uniform logits give -log V exactly
# --------------------------------------------------------------------------

@pytest.mark.parametrize("c", [1.5, 1024.0])          # exp(1024) overflows fp64 without the shift
@pytest.mark.parametrize("V", [1, 2, 7, 4096, 32000])
def test_uniform_logits_row(oracle_mod, V, c):
    z = bf16(np.full((3, V), c))
    tg = np.array([0, V // 2, V - 1], dtype=np.int64)
    logp, lse = oracle_mod.logp_from_logits(z, tg)
    np.testing.assert_allclose(logp, -math.log(V), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, c + math.log(V), rtol=0, atol=1e-12)


def test_zero_hidden_gives_uniform(oracle_mod):
    rng = np.random.default_rng(0)
    H, V = 64, 300
    W = bf16(np.round(rng.normal(0, 0.02, (V, H)) * 256) / 256)
    h = bf16(np.zeros((2, H)))
    logp, lse = oracle_mod.linear_logp(h, W, np.array([5, 299]))
    np.testing.assert_allclose(logp, -math.log(V), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, math.log(V), atol=1e-12, rtol=0)


def test_identical_weight_rows_give_uniform(oracle_mod):
    rng = np.random.default_rng(1)
    H, V = 64, 257
    w = np.round(rng.normal(0, 0.5, H) * 64) / 64
    W = bf16(np.tile(w, (V, 1)))
    h = bf16(np.round(rng.normal(0, 1, (4, H)) * 16) / 16)
    logp, _ = oracle_mod.linear_logp(h, W, np.array([0, 1, 100, 256]))
    np.testing.assert_allclose(logp, -math.log(V), atol=1e-12, rtol=0)


# --------------------------------------------------------------------------
# 2. One dominant logit
# --------------------------------------------------------------------------

@pytest.mark.parametrize("delta", [1.0, 5.0, 20.0])
def test_dominant_logit_closed_form(oracle_mod, delta):
    V, c = 32000, -3.0
    z = np.full((2, V), c)
    z[0, 123] += delta        # dominant logit is the target
    z[1, 7] += delta          # dominant logit elsewhere, target at a plain column
    tg = np.array([123, 4000])
    logp, _ = oracle_mod.logp_from_logits(bf16(z), tg)
    on_target = -math.log1p((V - 1) * math.exp(-delta))
    off_target = -delta - math.log1p((V - 1) * math.exp(-delta))
    # sequential fp64 summation of V terms of size <= 1: error <= (V-1) * 2^-53 * sum
    bound = (V - 1) * 2.0 ** -53 * 2.0 + 1e-14
    np.testing.assert_allclose(logp[0], on_target, atol=bound, rtol=0)
    np.testing.assert_allclose(logp[1], off_target, atol=bound, rtol=0)
    if delta == 20.0:
        assert -7e-5 < logp[0] < -6e-5      # about -6.6e-5: "dominant logit gives ~0"


# --------------------------------------------------------------------------
# 3. Normalisation: the selected logprobs over all targets sum to one
# --------------------------------------------------------------------------

def test_normalisation_over_all_targets_linear(oracle_mod):
    g = synth.generator(11)
    H, V = 64, 512
    W = synth.bf16_bits(synth.normal_bf16(g, (V, H), 0.3))
    h1 = synth.bf16_bits(synth.normal_bf16(g, (1, H), 1.0))
    h = np.repeat(h1, V, axis=0)
    logp, lse = oracle_mod.linear_logp(h, W, np.arange(V))
    assert abs(math.fsum(np.exp(logp)) - 1.0) < 1e-12
    assert np.all(lse == lse[0])


def test_normalisation_over_all_targets_logits(oracle_mod):
    zrow, _, _ = synth.logits_batch(T=1, V=4096, seed=5)
    z = np.repeat(synth.bf16_bits(zrow), 4096, axis=0)
    logp, _ = oracle_mod.logp_from_logits(z, np.arange(4096))
    assert abs(math.fsum(np.exp(logp)) - 1.0) < 1e-12


# --------------------------------------------------------------------------
# 4. Library routines on tiny inputs (a different algorithm: scipy's
#    log_softmax of a numpy matmul; and torch's fp64 autograd)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("H,V,T", [(16, 5, 3), (64, 64, 8), (32, 50, 6)])
def test_linear_logp_vs_library(oracle_mod, H, V, T):
    g = synth.generator(100 + H + V)
    W = synth.normal_bf16(g, (V, H), 0.5)
    h = synth.normal_bf16(g, (T, H), 1.0)
    tg = synth.uniform_targets(g, T, V).numpy()
    logp, lse = oracle_mod.linear_logp(synth.bf16_bits(h), synth.bf16_bits(W), tg)
    z = h.double().numpy() @ W.double().numpy().T
    ls = scipy.special.log_softmax(z, axis=1)
    np.testing.assert_allclose(logp, ls[np.arange(T), tg], atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=1), atol=1e-12, rtol=0)


def test_logits_vs_library(oracle_mod):
    z, tg, spikes = synth.logits_batch(T=16, V=1000, seed=9)
    logp, lse = oracle_mod.logp_from_logits(synth.bf16_bits(z), tg.numpy())
    zz = z.double().numpy()
    ls = scipy.special.log_softmax(zz, axis=1)
    np.testing.assert_allclose(logp, ls[np.arange(16), tg.numpy()], atol=1e-12, rtol=0)


@pytest.mark.parametrize("H,V,T", [(16, 5, 3), (32, 40, 5)])
def test_backward_vs_torch_autograd(oracle_mod, H, V, T):
    g = synth.generator(300 + H)
    W = synth.normal_bf16(g, (V, H), 0.5)
    h = synth.normal_bf16(g, (T, H), 1.0)
    tg = synth.uniform_targets(g, T, V)
    gr = torch.randn(T, generator=g, dtype=torch.float64)
    dh = oracle_mod.linear_logp_bwd(synth.bf16_bits(h), synth.bf16_bits(W), tg.numpy(), gr.numpy())
    hh = h.double().clone().requires_grad_(True)
    ls = torch.log_softmax(hh @ W.double().T, dim=1)
    (ls[torch.arange(T), tg] * gr).sum().backward()
    np.testing.assert_allclose(dh, hh.grad.numpy(), atol=1e-12, rtol=0)


# --------------------------------------------------------------------------
# 5. V = 1
# --------------------------------------------------------------------------

def test_single_vocab(oracle_mod):
    rng = np.random.default_rng(3)
    H = 32
    W = bf16(np.round(rng.normal(0, 1, (1, H)) * 8) / 8)
    h = bf16(np.round(rng.normal(0, 1, (3, H)) * 8) / 8)
    logp, _ = oracle_mod.linear_logp(h, W, np.zeros(3, dtype=np.int64))
    assert np.all(logp == 0.0)
    dh = oracle_mod.linear_logp_bwd(h, W, np.zeros(3, dtype=np.int64), np.array([1.0, -2.0, 0.5]))
    assert np.all(dh == 0.0)


# --------------------------------------------------------------------------
# 6. Shift invariance of the logits path
# --------------------------------------------------------------------------

def test_shift_invariance(oracle_mod):
    rng = np.random.default_rng(4)
    V = 3000
    z = rng.integers(-40, 40, (4, V)).astype(np.float64) / 4.0      # exact in bf16
    tg = rng.integers(0, V, 4)
    a, _ = oracle_mod.logp_from_logits(bf16(z), tg)
    b, lse_b = oracle_mod.logp_from_logits(bf16(z + 16.0), tg)
    np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)


# --------------------------------------------------------------------------
# 7. Backward: finite differences, identical rows, sum of (onehot - p)
# --------------------------------------------------------------------------

def test_backward_finite_differences(oracle_mod):
    rng = np.random.default_rng(5)
    H, V = 12, 9
    W = rng.normal(0, 0.7, (V, H))
    h = rng.normal(0, 1.0, (1, H))
    tg = np.array([4])
    gr = np.array([1.7])
    dh = oracle_mod.linear_logp_bwd(h, W, tg, gr)[0]
    eps = 1e-6
    fd = np.empty(H)
    for k in range(H):
        hp, hm = h.copy(), h.copy()
        hp[0, k] += eps
        hm[0, k] -= eps
        lp, _ = oracle_mod.linear_logp(hp, W, tg)
        lm, _ = oracle_mod.linear_logp(hm, W, tg)
        fd[k] = gr[0] * (lp[0] - lm[0]) / (2 * eps)
    np.testing.assert_allclose(dh, fd, rtol=1e-6, atol=1e-9)


def test_backward_identical_rows_vanish(oracle_mod):
    rng = np.random.default_rng(6)
    H, V = 16, 33
    W = np.tile(rng.normal(0, 1, H), (V, 1))
    h = rng.normal(0, 1, (3, H))
    dh = oracle_mod.linear_logp_bwd(h, W, np.array([0, 5, 32]), np.array([1.0, 2.0, -3.0]))
    np.testing.assert_allclose(dh, 0.0, atol=1e-13)


def test_backward_probabilities_sum_to_one(oracle_mod):
    # A constant-one column in W turns dh[:, that column] into g * (1 - sum_v p_v) = 0,
    # while the other columns stay nonzero.
    rng = np.random.default_rng(7)
    H, V = 8, 40
    W = rng.normal(0, 1, (V, H))
    W[:, 3] = 1.0
    h = rng.normal(0, 1, (5, H))
    dh = oracle_mod.linear_logp_bwd(h, W, rng.integers(0, V, 5), rng.normal(0, 1, 5))
    np.testing.assert_allclose(dh[:, 3], 0.0, atol=1e-13)
    assert np.all(np.abs(np.delete(dh, 3, axis=1)) > 0)


# --------------------------------------------------------------------------
# 8. Masking
# --------------------------------------------------------------------------

def test_masking_rows(oracle_mod):
    pool = synth.make_pool(32, 100, [3, 4], seed=8, with_grad=True)
    lay = synth.packed(pool, [0, 1], lead_pad=2)
    t = lay.targets.numpy().copy()
    t[3] = -100                                  # an ignored token inside a sequence
    h = synth.bf16_bits(lay.h)
    W = synth.bf16_bits(pool.W)
    logp, lse = oracle_mod.linear_logp(h, W, t, lay.cu_seqlens.numpy())
    act = oracle_mod.active_rows(t, lay.cu_seqlens.numpy())
    assert list(np.nonzero(~act)[0]) == [0, 1, 3]
    assert np.all(logp[~act] == 0) and np.all(lse[~act] == 0)
    assert np.all(np.isfinite(logp[act])) and np.all(logp[act] < 0)
    dh = oracle_mod.linear_logp_bwd(h, W, t, lay.g.numpy(), lay.cu_seqlens.numpy())
    assert np.all(dh[~act] == 0) and np.all(np.isfinite(dh))
    # cu_seqlens bounds: rows past cu_seqlens[-1] are inactive even with a valid target
    cu = np.array([2, 5], dtype=np.int32)
    act2 = oracle_mod.active_rows(lay.targets.numpy(), cu)
    assert list(np.nonzero(act2)[0]) == [2, 3, 4]


def test_out_of_range_target_is_an_error(oracle_mod):
    z = bf16(np.zeros((1, 8)))
    with pytest.raises(ValueError):
        oracle_mod.logp_from_logits(z, np.array([8]))


# --------------------------------------------------------------------------
# 9. The stored worked example of the tiny workload is reproduced
# --------------------------------------------------------------------------

def test_tiny_golden_snapshot(oracle_mod):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_linear_logp_oracle.json")
    with open(path) as f:
        gold = json.load(f)
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    logp, lse = oracle_mod.linear_logp(synth.bf16_bits(lay.h), synth.bf16_bits(pool.W),
                                       lay.targets.numpy(), lay.cu_seqlens.numpy())
    np.testing.assert_allclose(logp, gold["logp"], atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, gold["lse"], atol=1e-12, rtol=0)
    # the snapshot itself obeys the closed-form bound logp <= 0 and lse >= log V - max|z|
    assert max(gold["logp"]) < 0
