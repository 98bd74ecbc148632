"""A seeded sweep of random shapes and masks against the oracle.

Each case draws T, H and V (with V at and around the 8- and 256-column
boundaries as well as in between), masks rows both by target (-100) and by
cu_seqlens (leading and trailing rows outside the sequences), and checks:
  - the forward against the oracle (|d logp| <= 1e-3 + 1e-3 |logp|, same for lse);
  - the recompute backward and the saved-terms backward against the oracle
    (|d dh| <= 1e-3 + 1e-3 max |dh|), and inactive rows exactly 0;
  - the saved-terms forward and the forward with the GRPO loss give the plain
    forward's logp and lse bits;
  - on every fourth case, dW of the saved full backward against the oracle.
"""
import numpy as np
import pytest
import torch

from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import cuda, bits_np, oracle_bwd, oracle_dw, oracle_linear, same_bits

pytestmark = pytest.mark.gpu

V_CHOICES = [1, 2, 7, 8, 9, 255, 256, 257, 511, 1000, 2049, 4095]


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


def _case(i):
    rng = np.random.default_rng(7000 + i)
    T = int(rng.integers(1, 4)) if rng.random() < 0.3 else int(rng.integers(4, 400))
    H = int(64 * rng.integers(1, 7))
    V = int(V_CHOICES[i % len(V_CHOICES)] if i < len(V_CHOICES) else rng.integers(1, 4000))
    lead = int(rng.integers(0, min(3, T - 1) + 1)) if T > 1 else 0
    trail = int(rng.integers(0, min(3, T - 1 - lead) + 1)) if T - lead > 1 else 0
    # sequence boundaries between lead and T - trail
    inner = T - lead - trail
    cuts = sorted(set(int(x) for x in rng.integers(1, max(inner, 2), size=3))) if inner > 2 else []
    cu = [lead] + [lead + c for c in cuts if 0 < c < inner] + [lead + inner]
    return T, H, V, np.array(cu, dtype=np.int32), rng


@pytest.mark.parametrize("i", range(48))
def test_random_shape_and_mask_vs_oracle(rk, i):
    T, H, V, cu, rng = _case(i)
    gen = synth.generator(9100 + i)
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    drop = rng.random(T) < 0.1
    tg[torch.as_tensor(drop)] = -100
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    cud = cuda(torch.as_tensor(cu))
    desc = f"T={T} H={H} V={V} cu={cu.tolist()}"

    logp, lse = rk.linear_logp(hd, Wd, tgd, cud)
    hb, Wb = bits_np(h), bits_np(W)
    ref_lp, ref_lse = oracle_linear(hb, Wb, tg.numpy(), cu)
    for got, ref, name in ((logp, ref_lp, "logp"), (lse, ref_lse, "lse")):
        err = np.abs(got.cpu().double().numpy() - ref)
        assert np.all(err <= 1e-3 + 1e-3 * np.abs(ref)), (desc, name, float(err.max()))

    ref_dh = oracle_bwd(hb, Wb, tg.numpy(), g.double().numpy(), cu)
    inactive = np.ones(T, dtype=bool)
    inactive[cu[0]:cu[-1]] = False
    inactive |= tg.numpy() < 0
    dh = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd, cud)
    chk = contract.check_gradient_accuracy(dh.cpu().numpy(), ref_dh)
    assert chk.passed, (desc, "recompute", chk)

    lp_s, lse_s, saved = rk.linear_logp_fwd_saved(hd, Wd, tgd, cud)
    assert same_bits(lp_s, logp) and same_bits(lse_s, lse), desc
    dh_s = rk.linear_logp_bwd_saved(hd, Wd, tgd, lse_s, gd, saved, cud)
    chk = contract.check_gradient_accuracy(dh_s.cpu().numpy(), ref_dh)
    assert chk.passed, (desc, "saved", chk)
    for d in (dh, dh_s):
        assert bool((d.cpu()[torch.as_tensor(inactive)] == 0).all()), desc

    # the forward with the per-token GRPO loss in its merge: same logp / lse
    old = logp + 0.05 * torch.randn(T, device=logp.device)
    adv = torch.randn(T, device=logp.device)
    out = rk.linear_logp_grpo(hd, Wd, tgd, old, adv, cu_seqlens=cud)
    assert same_bits(out["logp"], logp) and same_bits(out["lse"], lse), desc

    if i % 4 == 0:
        _, lse_f, saved_f = rk.linear_logp_fwd_saved(hd, Wd, tgd, cud)
        _, dW = rk.linear_logp_bwd_full_saved(hd, Wd, tgd, lse_f, gd, saved_f, cud)
        ref_dw = oracle_dw(hb, Wb, tg.numpy(), g.double().numpy(), cu)
        chk = contract.check_gradient_accuracy(dW.cpu().numpy(), ref_dw)
        assert chk.passed, (desc, "dW", chk)
    assert rk.get_device_error() == 0


LOGITS_V = [1, 2, 7, 8, 9, 63, 64, 65, 255, 256, 257, 1000, 8191, 8192, 8193, 32000, 100003]


@pytest.mark.parametrize("i", range(len(LOGITS_V)))
def test_random_logits_path_vs_oracle(rk, i):
    # the logits path and its backward on random shapes and masks, V across
    # the 8-value group and the 64-value batch boundaries of the row kernel
    import oracle
    V = LOGITS_V[i]
    rng = np.random.default_rng(7500 + i)
    T = int(rng.integers(1, 300))
    gen = synth.generator(9500 + i)
    z = (torch.randn((T, V), generator=gen) * 2.0).to(torch.bfloat16)
    tg = synth.uniform_targets(gen, T, V)
    tg[torch.as_tensor(rng.random(T) < 0.1)] = -100
    lead = int(rng.integers(0, min(3, T) + 1))
    cu = np.array([lead, max(lead, T - int(rng.integers(0, 3)))], dtype=np.int32)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    zd, tgd, cud, gd = cuda(z), cuda(tg), cuda(torch.as_tensor(cu)), cuda(g)
    desc = f"T={T} V={V} cu={cu.tolist()}"
    logp, lse = rk.logp_from_logits(zd, tgd, cud)
    zb = bits_np(z)
    ref_lp, ref_lse = oracle.logp_from_logits(zb, tg.numpy(), cu)
    for got, ref, name in ((logp, ref_lp, "logp"), (lse, ref_lse, "lse")):
        err = np.abs(got.cpu().double().numpy() - ref)
        assert np.all(err <= 1e-3 + 1e-3 * np.abs(ref)), (desc, name, float(err.max()))
    dz = rk.logp_from_logits_bwd(zd, tgd, lse, gd, cud)
    ref_dz = oracle.logits_bwd(zb, tg.numpy(), g.double().numpy(), cu)
    chk = contract.check_gradient_accuracy(dz.cpu().numpy(), ref_dz)
    assert chk.passed, (desc, chk)
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("i", range(12))
def test_random_lm_head_and_greedy_vs_oracle(rk, i):
    # the dense path's bf16 logits and the greedy step on random shapes:
    #  - lm_head within one bf16 rounding of the fp32 accumulation, whose own
    #    error is bounded by z_error_bound;
    #  - the greedy token within the bounds of the maximum, the oracle's
    #    argmax wherever it is unambiguous, and logp of the chosen token
    import oracle
    from tests.helpers import oracle_lm_head, z_error_bound
    rng = np.random.default_rng(7700 + i)
    T = int(rng.integers(1, 300))
    H = int(64 * rng.integers(1, 9))
    V = int(V_CHOICES[i] if i < len(V_CHOICES) else rng.integers(1, 5000))
    gen = synth.generator(9700 + i)
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    hd, Wd = cuda(h), cuda(W)
    hb, Wb = bits_np(h), bits_np(W)
    desc = f"T={T} H={H} V={V}"
    ref = oracle_lm_head(hb, Wb, list(range(T)))
    acc = z_error_bound(hb, Wb, list(range(T)))
    z = rk.lm_head(hd, Wd).float().cpu().numpy()
    assert np.all(np.abs(z - ref) <= 2.0 ** -8 * (np.abs(ref) + acc) + acc), desc
    tok, lp, _ = rk.linear_greedy(hd, Wd)
    j = tok.cpu().numpy()
    r = np.arange(T)
    a = ref.argmax(axis=1)
    assert np.all(ref[r, j] >= ref[r, a] - acc[r, j] - acc[r, a]), desc
    hi = ref + acc
    hi[r, a] = -np.inf
    clear = (ref[r, a] - acc[r, a]) > hi.max(axis=1)
    assert np.all(j[clear] == a[clear]), desc
    ref_lp, _ = oracle.linear_logp(hb, Wb, j)
    err = np.abs(lp.cpu().double().numpy() - ref_lp)
    assert np.all(err <= 1e-3 + 1e-3 * np.abs(ref_lp)), (desc, float(err.max()))
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("i", range(40))
def test_random_layout_invariance(rk, i):
    # a random pool of sequences in random layouts (packed, permuted behind
    # random lead padding, right- and left-padded to the longest, a random
    # subset packed): every active row's logp, lse and dh, from both the
    # recompute and the saved-terms backward, bitwise equal to the packed
    # layout's
    rng = np.random.default_rng(7900 + i)
    H = int(64 * rng.integers(1, 7))
    V = int(rng.choice([7, 256, 257, 1000, 3001, 16384]))
    n = int(rng.integers(1, 7))
    lengths = [int(x) for x in rng.integers(1, 600, size=n)]
    pool = synth.make_pool(H, V, lengths, seed=9900 + i, with_grad=True)
    W = cuda(pool.W)
    seqs = list(range(n))

    def run(lay):
        h, tg, g = cuda(lay.h), cuda(lay.targets), cuda(lay.g)
        cu = cuda(lay.cu_seqlens)
        logp, lse = rk.linear_logp(h, W, tg, cu)
        dh = rk.linear_logp_bwd(h, W, tg, lse, g, cu)
        lp_s, lse_s, saved = rk.linear_logp_fwd_saved(h, W, tg, cu)
        dh_s = rk.linear_logp_bwd_saved(h, W, tg, lse_s, g, saved, cu)
        return {"logp": logp.cpu(), "lse": lse.cpu(), "dh": dh.cpu(), "logp_s": lp_s.cpu(),
                "dh_s": dh_s.cpu()}

    base = synth.packed(pool, seqs)
    bout = run(base)
    perm = [int(x) for x in rng.permutation(n)]
    sub = sorted(int(x) for x in rng.choice(n, size=int(rng.integers(1, n + 1)), replace=False))
    longest = max(lengths)
    layouts = [(synth.packed(pool, perm, lead_pad=int(rng.integers(0, 300))), seqs),
               (synth.padded(pool, seqs, longest, side="right"), seqs),
               (synth.padded(pool, seqs, longest + int(rng.integers(0, 40)), side="left"), seqs),
               (synth.packed(pool, sub), sub)]
    for lay, ids in layouts:
        out = run(lay)
        for s_id in ids:
            a, b = lay.rows_of[s_id], base.rows_of[s_id]
            for k in out:
                assert torch.equal(out[k][a].view(torch.int32), bout[k][b].view(torch.int32)), \
                    (k, lay.description, s_id)

    # dW over the whole sample set, named in canonical (sequence, position)
    # order: the same bits from every layout that holds all sequences, from
    # rk_linear_logp_dw and from the saved full backward
    def dw_of(lay):
        order = cuda(torch.tensor([r for s_id in seqs for r in lay.rows_of[s_id]],
                                  dtype=torch.int64))
        h, tg, g = cuda(lay.h), cuda(lay.targets), cuda(lay.g)
        cu = cuda(lay.cu_seqlens)
        _, lse = rk.linear_logp(h, W, tg, cu)
        dw = rk.linear_logp_dw(h, W, tg, lse, g, cu, row_order=order).cpu()
        _, lse_s, saved = rk.linear_logp_fwd_saved(h, W, tg, cu)
        dw_s = rk.linear_logp_bwd_full_saved(h, W, tg, lse_s, g, saved, cu, row_order=order)[1]
        return dw, dw_s.cpu()

    if i % 2 == 0:
        dw0, dws0 = dw_of(base)
        for lay, ids in layouts[:3]:
            dw, dws = dw_of(lay)
            assert torch.equal(dw.view(torch.int32), dw0.view(torch.int32)), lay.description
            assert torch.equal(dws.view(torch.int32), dws0.view(torch.int32)), lay.description
    assert rk.get_device_error() == 0
