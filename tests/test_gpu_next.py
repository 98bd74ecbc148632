"""GPU parity and invariance of the widened rows: the dense path (lm_head +
logits path) against the indexed path, the logits-path backward, the
per-token GRPO loss feeding the linear_logp backward, and greedy decoding
re-scored by prefill."""
import numpy as np
import pytest
import torch

import oracle
from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import (DEV, bits_np, cuda, oracle_lm_head, oracle_linear, same_bits,
                           z_error_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


# --------------------------------------------------------------------------
# dense path: lm_head
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,V", [(64, 256, 4096), (300, 192, 1001), (257, 512, 769)])
def test_lm_head_vs_oracle(rk, T, H, V):
    gen = synth.generator(3000 + T + V)
    W = synth.normal_bf16(gen, (V, H), 0.02)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    z = rk.lm_head(cuda(h), cuda(W)).float().cpu().numpy()
    ref = oracle.lm_head(bits_np(h), bits_np(W))
    # one rounding to bf16 (at most 2^-8 relative) of an fp32 accumulation
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5
    assert np.all(np.abs(z - ref) <= bound), float(np.max(np.abs(z - ref) - bound))
    assert rk.get_device_error() == 0


@pytest.mark.slow
def test_lm_head_multi_wave_sampled_rows(rk):
    # 16 x 125 pair tiles, several waves of the resident pairs: sampled rows
    # against fp64 z, within one bf16 rounding of an fp32 accumulation whose
    # own error is bounded by z_error_bound
    T, H, V = 4096, 1024, 32000
    gen = synth.generator(3200)
    W = synth.normal_bf16(gen, (V, H), 0.02)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    z = rk.lm_head(cuda(h), cuda(W)).float().cpu().numpy()
    rows = synth.sample_rows(T, 128, seed=32)
    hb, Wb = bits_np(h), bits_np(W)
    ref = oracle_lm_head(hb, Wb, rows)
    acc = z_error_bound(hb, Wb, rows)
    # bf16 keeps 8 significant bits: round to nearest moves a value by at
    # most 2^-8 of its magnitude
    bound = 2.0 ** -8 * (np.abs(ref) + acc) + acc
    err = np.abs(z[rows] - ref)
    print(f"lm_head T=4096 H=1024 V=32000, 128 rows: max |dz| {err.max():.3g}, "
          f"max |dz| / bound {np.max(err / bound):.3g}")
    assert np.all(err <= bound), float(np.max(err - bound))
    assert rk.get_device_error() == 0


def test_lm_head_tile_order(rk):
    # tiles taken from the workspace counter or from fixed per-pair lists:
    # the same bits
    gen = synth.generator(3100)
    W = synth.normal_bf16(gen, (9000, 256), 0.02)
    h = synth.normal_bf16(gen, (1500, 256), 1.0)
    hd, Wd = cuda(h), cuda(W)
    a = rk.lm_head(hd, Wd)
    lib = rk.load_library()
    b = torch.empty_like(a)
    st = lib.rk_lm_head(hd.data_ptr(), Wd.data_ptr(), 1500, 256, 9000, b.data_ptr(), b.stride(0),
                        None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert torch.equal(a.view(torch.int16).cpu(), b.view(torch.int16).cpu())


def test_dense_vs_indexed_paths(rk):
    # P-relation: logp from bf16 logits (dense) vs logp fused on fp32 z
    # (indexed).  The dense path rounds every z to bf16 (8 significant bits,
    # so |dz| <= 2^-8 |z|), hence |d logp| <= 2^-8 (|z_target| + max_v |z_v|)
    # up to fp32 rounding.
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    h, W, tg = cuda(lay.h), cuda(pool.W), cuda(lay.targets)
    lp_idx, lse_idx = rk.linear_logp(h, W, tg)
    logits = rk.lm_head(h, W)
    lp_dense, _ = rk.logp_from_logits(logits.contiguous(), tg)
    z = oracle.lm_head(bits_np(lay.h), bits_np(pool.W))
    ztg = z[np.arange(lay.T), lay.targets.numpy()]
    bound = 2.0 ** -8 * (np.abs(ztg) + np.abs(z).max(axis=1)) + 1e-5
    diff = np.abs(lp_dense.cpu().numpy() - lp_idx.cpu().numpy())
    assert np.all(diff <= bound), float(np.max(diff - bound))
    # and the dense path is exact for its own (rounded) logits
    ref_dense, _ = oracle.logp_from_logits(bits_np(logits.contiguous().cpu()), lay.targets.numpy())
    assert contract.check_forward_accuracy(lp_dense.cpu().numpy(), ref_dense).passed


def test_lm_head_row_invariance(rk):
    pool = synth.tiny_pool()
    base = synth.packed(pool, [0, 1, 2, 3])
    W = cuda(pool.W)
    zb = rk.lm_head(cuda(base.h), W).cpu()
    for off in (1, 77, 128, 200):
        lay = synth.packed(pool, [3, 1, 0, 2], lead_pad=off)
        zl = rk.lm_head(cuda(lay.h), W).cpu()
        for i in range(4):
            assert torch.equal(zb[base.rows_of[i]].view(torch.int16), zl[lay.rows_of[i]].view(torch.int16))


# --------------------------------------------------------------------------
# logits-path backward
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,V", [(2048, 32000), (50, 1001), (17, 5)])
def test_logits_bwd_vs_oracle(rk, T, V):
    z, tg, _ = synth.logits_batch(T=T, V=V, seed=T + 11 * V)
    gen = synth.generator(V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    tg[::13] = -100
    zd, tgd = cuda(z), cuda(tg)
    _, lse = rk.logp_from_logits(zd, tgd)
    dz = rk.logp_from_logits_bwd(zd, tgd, lse, cuda(g)).cpu().numpy()
    rows = synth.sample_rows(T, 64, seed=5)
    ref = oracle.logits_bwd(bits_np(z), tg.numpy(), g.double().numpy(), rows=rows)
    chk = contract.check_gradient_accuracy(dz[rows], ref)
    assert chk.passed, chk
    act = oracle.active_rows(tg.numpy())
    assert np.all(dz[~act] == 0)
    np.testing.assert_allclose(dz[act].sum(axis=1), 0.0, atol=1e-4)   # g (1 - sum p)
    assert rk.get_device_error() == 0


def test_logits_bwd_invariance(rk):
    z, tg, _ = synth.logits_batch(T=256, V=32000, seed=8)
    g = torch.randn(256, generator=synth.generator(9), dtype=torch.float32)
    zd, tgd, gd = cuda(z), cuda(tg), cuda(g)
    _, lse = rk.logp_from_logits(zd, tgd)
    base = rk.logp_from_logits_bwd(zd, tgd, lse, gd).cpu()
    perm = torch.randperm(256, generator=synth.generator(10))
    pd = perm.to(DEV)
    got = rk.logp_from_logits_bwd(zd[pd].contiguous(), tgd[pd].contiguous(), lse[pd].contiguous(),
                                  gd[pd].contiguous()).cpu()
    assert same_bits(got, base[perm])
    one = rk.logp_from_logits_bwd(zd[5:6].contiguous(), tgd[5:6].contiguous(), lse[5:6].contiguous(),
                                  gd[5:6].contiguous()).cpu()
    assert same_bits(one[0], base[5])


def test_logits_bwd_output_alignment(rk):
    # an output only 16-byte aligned takes the element-wise store path; the
    # bits are the same as from the 32-byte store path
    z, tg, _ = synth.logits_batch(T=64, V=4096, seed=12)
    g = torch.randn(64, generator=synth.generator(13), dtype=torch.float32)
    zd, tgd, gd = cuda(z), cuda(tg), cuda(g)
    _, lse = rk.logp_from_logits(zd, tgd)
    base = rk.logp_from_logits_bwd(zd, tgd, lse, gd)
    buf = torch.empty(64 * 4096 + 4, dtype=torch.float32, device=DEV)
    out = buf[4:].view(64, 4096)
    assert out.data_ptr() % 32 == 16
    rk.logp_from_logits_bwd(zd, tgd, lse, gd, out=out)
    assert same_bits(out, base)


# --------------------------------------------------------------------------
# per-token GRPO loss, and the chain logp -> loss -> dh
# --------------------------------------------------------------------------

def _grpo_inputs(T, seed):
    gen = synth.generator(seed)
    lp_old = -torch.rand(T, generator=gen, dtype=torch.float64) * 5
    lp = lp_old + 0.3 * torch.randn(T, generator=gen, dtype=torch.float64)
    ref = lp + 0.3 * torch.randn(T, generator=gen, dtype=torch.float64)
    adv = torch.randn(T, generator=gen, dtype=torch.float64)
    tg = torch.randint(0, 100, (T,), generator=gen)
    tg[::9] = -100
    return lp.float(), lp_old.float(), ref.float(), adv.float(), tg


def test_grpo_token_vs_oracle(rk):
    lp, lo, ref, adv, tg = _grpo_inputs(5000, 1)
    kw = dict(eps_low=0.2, eps_high=0.28, beta=0.04, scale=1.0)
    out = rk.grpo_token_loss(cuda(lp), cuda(lo), cuda(adv), cuda(tg), logp_ref=cuda(ref), **kw)
    o = oracle.grpo_token(lp.double().numpy(), lo.double().numpy(), adv.double().numpy(),
                          logp_ref=ref.double().numpy(), targets=tg.numpy(), **kw)
    for k in ("loss", "grad", "ratio", "kl"):
        chk = contract.check_forward_accuracy(out[k].cpu().numpy(), o[k])
        assert chk.passed, (k, chk)


def test_grpo_token_invariance(rk):
    lp, lo, ref, adv, tg = _grpo_inputs(3000, 2)
    args = [cuda(x) for x in (lp, lo, adv, tg)]
    base = rk.grpo_token_loss(*args, logp_ref=cuda(ref), beta=0.1)
    perm = torch.randperm(3000, generator=synth.generator(3)).to(DEV)
    got = rk.grpo_token_loss(*[x[perm].contiguous() for x in args],
                             logp_ref=cuda(ref)[perm].contiguous(), beta=0.1)
    for k in base:
        assert same_bits(got[k], base[k][perm]), k


def test_fused_forward_loss_matches_separate_calls(rk):
    # rk_linear_logp_grpo: the forward's merge applies the loss; every output
    # has the bits of rk_linear_logp followed by rk_grpo_token_loss, with
    # masked rows, an out-of-range target (NaN), and with / without the KL term
    pool = synth.make_pool(256, 5000, [300, 200, 157], seed=95)
    lay = synth.packed(pool, [0, 1, 2], lead_pad=11)
    tg = lay.targets.clone()
    tg[40] = -100
    tg[77] = 5000
    h, W, tgd, cu = cuda(lay.h), cuda(pool.W), cuda(tg), cuda(lay.cu_seqlens)
    gen = synth.generator(96)
    T = lay.T
    lp_old = cuda(-torch.rand(T, generator=gen) * 9 - 1)
    adv = cuda(torch.randn(T, generator=gen))
    lp_ref = cuda(-torch.rand(T, generator=gen) * 9 - 1)
    for ref in (lp_ref, None):
        kw = dict(logp_ref=ref, eps_low=0.2, eps_high=0.28, beta=0.04, scale=1.0 / T)
        rk.get_device_error()
        fused = rk.linear_logp_grpo(h, W, tgd, lp_old, adv, cu, **kw)
        assert rk.get_device_error() & rk.DEVERR_TARGET_RANGE
        logp, lse = rk.linear_logp(h, W, tgd, cu)
        sep = rk.grpo_token_loss(logp, lp_old, adv, tgd, cu, **kw)
        rk.get_device_error()
        assert same_bits(fused["logp"], logp) and same_bits(fused["lse"], lse)
        for k in ("loss", "grad", "ratio", "kl"):
            assert same_bits(fused[k], sep[k]), k
        f = {k: v.cpu() for k, v in fused.items()}
        # the out-of-range row's NaN logp goes through the same loss
        # arithmetic as in the separate call (compared bitwise above)
        assert torch.isnan(f["logp"][77]) and torch.isnan(f["ratio"][77])
        assert f["loss"][40] == 0 and f["grad"][:11].abs().sum() == 0


def test_chain_logp_loss_backward(rk):
    # linear_logp -> GRPO per-token loss -> dh, against the same chain in the oracle
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    h, W, tg, cu = cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.cu_seqlens)
    gen = synth.generator(70)
    lp_old = -torch.rand(lay.T, generator=gen) * 9 - 1
    adv = torch.randn(lay.T, generator=gen)
    logp, lse = rk.linear_logp(h, W, tg, cu)
    out = rk.grpo_token_loss(logp, cuda(lp_old), cuda(adv), tg, cu, eps_low=0.2, eps_high=0.28,
                             scale=1.0 / lay.T)
    dh = rk.linear_logp_bwd(h, W, tg, lse, out["grad"], cu)
    hb, Wb = bits_np(lay.h), bits_np(pool.W)
    ref_lp, _ = oracle.linear_logp(hb, Wb, lay.targets.numpy(), lay.cu_seqlens.numpy())
    o = oracle.grpo_token(ref_lp, lp_old.double().numpy(), adv.double().numpy(),
                          targets=lay.targets.numpy(), cu_seqlens=lay.cu_seqlens.numpy(),
                          eps_low=0.2, eps_high=0.28, scale=1.0 / lay.T)
    ref_dh = oracle.linear_logp_bwd(hb, Wb, lay.targets.numpy(), o["grad"], lay.cu_seqlens.numpy())
    assert contract.check_forward_accuracy(out["loss"].cpu().numpy(), o["loss"]).passed
    chk = contract.check_gradient_accuracy(dh.cpu().numpy(), ref_dh)
    assert chk.passed, chk


# --------------------------------------------------------------------------
# greedy decoding and generate-then-re-score
# --------------------------------------------------------------------------

def _greedy_case(name):
    if name == "tiny":
        pool = synth.tiny_pool()
        return pool.h, pool.W, None
    # several waves of pair tiles (16 x 125), with sampled rows
    T, H, V = 4096, 1024, 32000
    gen = synth.generator(3300)
    W = synth.normal_bf16(gen, (V, H), 0.02)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    return h, W, synth.sample_rows(T, 256, seed=33)


@pytest.mark.parametrize("name", ["tiny", "multi_wave"])
def test_greedy_vs_oracle(rk, name):
    # Several tokens can be correct where the top logits lie within the fp32
    # error of z.  With B[v] the bound of |z_gpu[v] - z[v]| (z_error_bound):
    #  - every row's token j must satisfy z[j] >= max z - B[j] - B[argmax]
    #    (the GPU saw z_gpu[j] >= z_gpu[argmax]);
    #  - where the oracle's argmax a beats every other column even after the
    #    bounds (z[a] - B[a] > z[v] + B[v] for all v != a), j must be a;
    #  - logp must match the oracle's logp of the chosen token.
    h, W, rows = _greedy_case(name)
    tok, lp, lse = rk.linear_greedy(cuda(h), cuda(W))
    tok, lp = tok.cpu().numpy(), lp.cpu().numpy()
    hb, Wb = bits_np(h), bits_np(W)
    rows = list(range(h.shape[0])) if rows is None else rows
    z = oracle_lm_head(hb, Wb, rows)
    B = z_error_bound(hb, Wb, rows)
    r = np.arange(len(rows))
    j = tok[rows]
    a = z.argmax(axis=1)
    assert np.all(z[r, j] >= z[r, a] - B[r, j] - B[r, a])
    hi = z + B
    hi[r, a] = -np.inf
    clear = (z[r, a] - B[r, a]) > hi.max(axis=1)
    assert np.all(j[clear] == a[clear])
    ref_lp, _ = oracle_linear(hb, Wb, tok, rows=rows)
    chk = contract.check_forward_accuracy(lp[rows], ref_lp)
    print(f"greedy {name}: {clear.sum()} of {len(rows)} rows unambiguous, "
          f"{np.sum(j == a)} match the oracle argmax; logp {chk}")
    assert chk.passed, chk
    # the oracle's own greedy step picks the same argmax (the lowest index of the maximum)
    rtok, _, rzm = oracle.linear_greedy(hb, Wb, rows=rows)
    assert np.array_equal(rtok, a) and np.allclose(rzm, z[r, a], rtol=0, atol=0)


def test_generate_then_rescore(rk):
    # decode: one row at a time (T = 1 launches), each step's greedy token
    # and logprob recorded; re-score: the whole sequence at once through
    # rk_linear_logp with the generated tokens.  Selected logprobs and lse
    # must agree bit for bit.
    pool = synth.grpo_pool(n_seqs=1)
    H = pool.H
    seq = cuda(pool.h[:96])
    W = cuda(pool.W)
    toks, lps, lses = [], [], []
    for t in range(seq.shape[0]):
        tk, lp, ls = rk.linear_greedy(seq[t:t + 1].contiguous(), W)
        toks.append(tk)
        lps.append(lp)
        lses.append(ls)
    toks = torch.cat(toks)
    dec_lp, dec_lse = torch.cat(lps).cpu(), torch.cat(lses).cpu()
    cu = torch.tensor([0, seq.shape[0]], dtype=torch.int32, device=DEV)
    re_lp, re_lse = rk.linear_logp(seq, W, toks, cu)
    assert same_bits(re_lp, dec_lp) and same_bits(re_lse, dec_lse)
    # and a prefill-shaped greedy pass makes the same choices
    tk2, lp2, _ = rk.linear_greedy(seq, W)
    assert torch.equal(tk2.cpu(), toks.cpu()) and same_bits(lp2, dec_lp)
    # the scores are the oracle's within tolerance
    ref, _ = oracle_linear(bits_np(pool.h[:96]), bits_np(pool.W), toks.cpu().numpy())
    assert contract.check_forward_accuracy(re_lp.cpu().numpy(), ref).passed
