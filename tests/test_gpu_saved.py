"""The forward that keeps its softmax terms and the backward that uses them
(rk_linear_logp_fwd_saved / rk_linear_logp_bwd_saved): the forward's logp and
lse are bitwise rk_linear_logp's; dh matches the fp64 oracle (relation A) on
every shape, mask and peaked regime the recompute path is checked on; and dh
is bitwise invariant under the batch transforms (relation I; PR #264
"docs(ws1): batch-invariance contract RFC", T1-T6)."""
import numpy as np
import pytest
import torch

import oracle
from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import DEV, bits_np, cuda, oracle_bwd, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


def _saved_fwd_bwd(rk, h, W, tg, g, cu=None):
    logp, lse, saved = rk.linear_logp_fwd_saved(h, W, tg, cu)
    dh = rk.linear_logp_bwd_saved(h, W, tg, lse, g, saved, cu)
    return logp, lse, dh


@pytest.mark.parametrize("T,H,V", [(300, 64, 1000), (129, 192, 4097), (1, 128, 5), (257, 256, 769),
                                   (700, 128, 2001), (64, 256, 4096), (513, 512, 20000)])
def test_saved_path_vs_oracle(rk, T, H, V):
    gen = synth.generator(8000 + T + H + V)
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    tg[::13] = -100
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    logp, lse, dh = _saved_fwd_bwd(rk, hd, Wd, tgd, gd)
    lp0, lse0 = rk.linear_logp(hd, Wd, tgd)
    assert same_bits(logp, lp0) and same_bits(lse, lse0)
    ref = oracle_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dh.cpu().numpy(), ref)
    assert chk.passed, chk
    assert torch.all(dh.cpu()[::13] == 0)
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("w_std,argmax_targets", [(0.25, True), (0.4, True), (0.4, False)])
def test_saved_path_peaked_softmax(rk, w_std, argmax_targets):
    # logit std ~6-9: the target (or another column) holds most of the mass;
    # those columns come from an exact z, so dh stays inside the tolerance
    T, H, V = 512, 512, 4096
    gen = synth.generator(123)
    W = synth.normal_bf16(gen, (V, H), w_std)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    z = oracle.lm_head(bits_np(h), bits_np(W))
    tg = torch.as_tensor(z.argmax(axis=1), dtype=torch.int64) if argmax_targets else \
        synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    _, _, dh = _saved_fwd_bwd(rk, cuda(h), cuda(W), cuda(tg), cuda(g))
    ref = oracle.linear_logp_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dh.cpu().numpy(), ref)
    print(f"saved path, peaked w_std={w_std} argmax={argmax_targets}: {chk}")
    assert chk.passed, chk
    assert rk.get_device_error() == 0


def test_saved_path_masking_and_bad_target(rk):
    pool = synth.make_pool(128, 1500, [30, 50], seed=41, with_grad=True)
    lay = synth.packed(pool, [0, 1], lead_pad=7)
    tg = lay.targets.clone()
    tg[20] = 1500                                   # out of range: NaN row + error bit
    h, W, tgd, cu, g = cuda(lay.h), cuda(pool.W), cuda(tg), cuda(lay.cu_seqlens), cuda(lay.g)
    rk.get_device_error()
    _, _, dh = _saved_fwd_bwd(rk, h, W, tgd, g, cu)
    assert rk.get_device_error() & rk.DEVERR_TARGET_RANGE
    d = dh.cpu()
    assert torch.all(d[:7] == 0) and torch.all(torch.isnan(d[20]))
    ok = torch.ones(lay.T, dtype=torch.bool)
    ok[20] = False
    assert torch.all(torch.isfinite(d[ok]))
    act = oracle.active_rows(tg.numpy(), lay.cu_seqlens.numpy()) & (tg.numpy() < 1500)
    ref = oracle_bwd(bits_np(lay.h), bits_np(pool.W), np.where(act, tg.numpy(), -100),
                     np.nan_to_num(lay.g.double().numpy()), lay.cu_seqlens.numpy())
    assert contract.check_gradient_accuracy(d[ok].numpy(), ref[ok.numpy()]).passed


def test_saved_path_invariance_tiny(rk):
    # every transform class of the tiny workload: dh bitwise equal to the
    # packed baseline on the logical rows
    pool = synth.tiny_pool()
    W = cuda(pool.W)

    def run(lay):
        h, tg, cu, g = cuda(lay.h), cuda(lay.targets), cuda(lay.cu_seqlens), cuda(lay.g)
        logp, lse, dh = _saved_fwd_bwd(rk, h, W, tg, g, cu)
        return {"logp": logp.cpu(), "lse": lse.cpu(), "dh": dh.cpu()}

    base_lay = synth.packed(pool, [0, 1, 2, 3])
    base = run(base_lay)
    layouts = [(synth.packed(pool, [i]), [i]) for i in range(4)]
    layouts += [(synth.packed(pool, [3, 2, 1, 0]), [0, 1, 2, 3]),
                (synth.packed(pool, [0, 1, 2, 3], lead_pad=77), [0, 1, 2, 3]),
                (synth.padded(pool, [0, 1, 2, 3], 40, side="left"), [0, 1, 2, 3]),
                (synth.padded(pool, [0, 1, 2, 3], 160, side="right"), [0, 1, 2, 3]),
                (synth.packed(synth.replace_neighbours(pool, [1], seed=synth.NEIGHBOUR_SEED_OFFSET),
                              [0, 1, 2, 3]), [1])]
    for lay, seqs in layouts:
        out = run(lay)
        for i in seqs:
            b = torch.tensor(base_lay.rows_of[i])
            v = torch.tensor(lay.rows_of[i])
            for k in base:
                assert torch.equal(out[k][v].view(torch.int32), base[k][b].view(torch.int32)), \
                    (lay.description, i, k)
    # the same physical batch twice: the same bits (the saved state is rebuilt)
    again = run(base_lay)
    assert all(same_bits(again[k], base[k]) for k in base)
    assert rk.get_device_error() == 0


@pytest.mark.slow
def test_saved_path_grpo_sampled_rows(rk):
    # the GRPO group at full size (T = 65536, H = 4096, V = 128256): sampled
    # rows of dh against the oracle, and the decode-shaped launches (rows
    # alone, T = 1 and 64) equal to the prefill rows bit for bit
    pool = synth.grpo_pool()
    lay = synth.packed(pool, list(range(len(pool.lengths))))
    h, W, tg, g = cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.g)
    logp, lse, dh = _saved_fwd_bwd(rk, h, W, tg, g)
    assert rk.last_row_blocks("dh") == 2
    rows = synth.sample_rows(lay.T, 64, seed=14)
    ref = oracle_bwd(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(), lay.g.double().numpy(),
                     rows=rows)
    chk = contract.check_gradient_accuracy(dh.cpu()[rows].numpy(), ref)
    print(f"saved path, grpo 64 sampled rows: dh {chk}")
    assert chk.passed, chk
    dh_c = dh.cpu()
    for n in (1, 64):
        sub = torch.arange(5000, 5000 + n, device=DEV)
        _, _, dh1 = _saved_fwd_bwd(rk, h[sub].contiguous(), W, tg[sub].contiguous(),
                                   g[sub].contiguous())
        assert same_bits(dh1.cpu(), dh_c[5000:5000 + n]), n
    assert rk.get_device_error() == 0


def _saved_terms(rk, saved, T, H, V):
    """The saved state's bf16 terms as raw bytes [T, ld * 2] (after the forward workspace)."""
    ws = rk.linear_logp_workspace_size(T, H, V)
    ld = (V + 7) // 8 * 8
    return saved[ws:ws + T * ld * 2].view(T, ld * 2)


@pytest.mark.parametrize("all_pad,H,V", [(False, 256, 3000), (True, 256, 3000),
                                          (False, 2048, 16384)])
def test_padding_blocks_are_skipped(rk, all_pad, H, V):
    # Sequences right-padded to 1024 rows: a block of 256 rows holding no
    # active row gets no tensor work.  Visible: the forward leaves the block's
    # saved terms as the buffer held them, and the backward writes dh = 0 there
    # over a NaN-filled output.  logp and lse are 0 there, and the active rows
    # are the packed layout's bits.  At V = 16384, H = 2048 the dh GEMM takes
    # its 8 H tiles per row block in rounds (two rounds of the resident
    # pairs), skipping the dead blocks' tiles within them.
    pool = synth.make_pool(H, V, [300, 40, 700, 129], seed=93, with_grad=True)
    seqs = [0, 1, 2, 3]
    lay = synth.padded(pool, seqs, 1024)
    if all_pad:
        lay.targets[:] = -100
    T = lay.T
    W = cuda(pool.W)

    def run(l, sentinel):
        h, tg, g = cuda(l.h), cuda(l.targets), cuda(l.g)
        saved = torch.full((rk.linear_logp_saved_size(l.T, H, V),), sentinel, dtype=torch.uint8,
                           device=DEV)
        lp, lse, saved = rk.linear_logp_fwd_saved(h, W, tg, saved=saved)
        terms = _saved_terms(rk, saved, l.T, H, V).clone()  # the backward rewrites them
        dh = torch.full((l.T, H), float("nan"), device=DEV)
        rk.linear_logp_bwd_saved(h, W, tg, lse, g, saved, dh=dh)
        return lp.cpu(), lse.cpu(), dh.cpu(), terms.cpu()

    lp, lse, dh, terms = run(lay, 0xAB)
    if V >= 16384 and not all_pad:
        assert rk.last_tile_order("dh") in (1, 2)  # 2: rounds, unless refused
    dead = (lay.targets.view(-1, 256) < 0).all(dim=1)
    assert int(dead.sum()) == (16 if all_pad else 9)
    for b in range(T // 256):
        rows = slice(256 * b, 256 * b + 256)
        if dead[b]:
            assert bool((terms[rows] == 0xAB).all()), f"block {b} was computed"
        else:
            assert not bool((terms[rows] == 0xAB).all())
    inactive = lay.targets < 0
    assert bool((lp[inactive] == 0).all()) and bool((lse[inactive] == 0).all())
    assert bool((dh[inactive] == 0).all())
    if not all_pad:
        pk = synth.packed(pool, seqs)
        lp_p, lse_p, dh_p, _ = run(pk, 0)
        for i in seqs:
            a, b = lay.rows_of[i], pk.rows_of[i]
            assert same_bits(lp[a], lp_p[b]) and same_bits(lse[a], lse_p[b])
            assert same_bits(dh[a], dh_p[b])
    assert rk.get_device_error() == 0


def test_padding_blocks_are_skipped_recompute(rk):
    # The same for the recompute backward (rk_linear_logp_bwd), one chunk:
    # the dZ rows of blocks without an active row keep what the workspace
    # held, their dh is 0 over a NaN-filled output, and the active rows are
    # the packed layout's bits.
    H, V = 256, 3000
    pool = synth.make_pool(H, V, [300, 40, 700, 129], seed=94, with_grad=True)
    seqs = [0, 1, 2, 3]
    lay = synth.padded(pool, seqs, 1024)
    W = cuda(pool.W)
    ld = (V + 7) // 8 * 8
    r256 = lambda x: (x + 255) // 256 * 256

    def run(l):
        h, tg, g = cuda(l.h), cuda(l.targets), cuda(l.g)
        _, lse = rk.linear_logp(h, W, tg)
        ws = torch.full((rk.linear_logp_bwd_workspace_size(l.T, H, V),), 0xAB, dtype=torch.uint8,
                        device=DEV)
        dh = torch.full((l.T, H), float("nan"), device=DEV)
        rk.linear_logp_bwd(h, W, tg, lse, g, dh=dh, workspace=ws)
        off = 256 + r256(l.T * 4) + r256(l.T * 65 * 8)
        return dh.cpu(), ws[off:off + l.T * ld * 2].view(l.T, ld * 2).cpu()

    dh, dz = run(lay)
    dead = (lay.targets.view(-1, 256) < 0).all(dim=1)
    assert int(dead.sum()) == 9
    for b in range(lay.T // 256):
        rows = slice(256 * b, 256 * b + 256)
        assert bool((dz[rows] == 0xAB).all()) == bool(dead[b]), f"block {b}"
    assert bool((dh[lay.targets < 0] == 0).all())
    pk = synth.packed(pool, seqs)
    dh_p, _ = run(pk)
    for i in seqs:
        assert same_bits(dh[lay.rows_of[i]], dh_p[pk.rows_of[i]])
    assert rk.get_device_error() == 0


# --------------------------------------------------------------------------
# dh and dW together from the saved terms (rk_linear_logp_bwd_full_saved)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,V,kind", [(300, 128, 1001, "uniform"), (700, 256, 2001, "masked"),
                                        (600, 256, 128256, "zipf"), (512, 512, 4096, "peaked")])
def test_saved_full_backward_vs_oracle(rk, T, H, V, kind):
    gen = synth.generator(8500 + T + V)
    W = synth.normal_bf16(gen, (V, H), 0.25 if kind == "peaked" else 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    if kind == "zipf":
        p = np.arange(1, V + 1, dtype=np.float64) ** -1.1
        tg = torch.as_tensor(np.random.default_rng(85).choice(V, size=T, p=p / p.sum()))
    if kind == "masked":
        tg[::7] = -100
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse, saved = rk.linear_logp_fwd_saved(hd, Wd, tgd)
    dh, dW = rk.linear_logp_bwd_full_saved(hd, Wd, tgd, lse, gd, saved)
    # dh is the saved-terms backward's, bit for bit (that call consumes `saved`)
    dh_s = rk.linear_logp_bwd_saved(hd, Wd, tgd, lse, gd, saved)
    assert same_bits(dh, dh_s)
    from tests.helpers import oracle_dw
    ref = oracle_dw(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dW.cpu().numpy(), ref)
    print(f"saved full backward dW T={T} V={V} {kind}: {chk}")
    assert chk.passed, chk
    assert rk.get_device_error() == 0


def test_saved_full_backward_layout_invariance(rk):
    # the same sample set in packed, padded and permuted layouts, each named
    # in canonical (sequence, position) order: dW bitwise equal
    pool = synth.make_pool(128, 3000, [40, 70, 25, 33], seed=91, with_grad=True)
    W = cuda(pool.W)
    seqs = [0, 1, 2, 3]

    def dw_of(lay):
        order = torch.tensor([r for i in seqs for r in lay.rows_of[i]], dtype=torch.int64)
        h, tg, g = cuda(lay.h), cuda(lay.targets), cuda(lay.g)
        _, lse, saved = rk.linear_logp_fwd_saved(h, W, tg)
        return rk.linear_logp_bwd_full_saved(h, W, tg, lse, g, saved, row_order=cuda(order))[1].cpu()

    base = dw_of(synth.packed(pool, seqs))
    for lay in (synth.padded(pool, seqs, 80, side="right"), synth.padded(pool, seqs, 80, side="left"),
                synth.packed(pool, [3, 2, 1, 0], lead_pad=37), synth.packed(pool, [2, 0, 3, 1])):
        assert same_bits(dw_of(lay), base), lay.description
    assert rk.get_device_error() == 0


@pytest.mark.slow
def test_saved_full_backward_grpo(rk):
    # full size: dW within the tolerance of the recompute path's dW, the
    # projection identity with dh, and dh bitwise the saved-terms backward's
    from tests.test_gpu_dw import _projection_identity
    pool = synth.grpo_pool()
    h, W, tg, g = cuda(pool.h), cuda(pool.W), cuda(pool.targets), cuda(pool.g)
    _, lse, saved = rk.linear_logp_fwd_saved(h, W, tg)
    dh, dW = rk.linear_logp_bwd_full_saved(h, W, tg, lse, g, saved)
    assert rk.last_row_blocks("dw") == 2
    rel = _projection_identity(h, W, dh, dW)
    print(f"saved full backward, GRPO projection identity residual {rel:.3g}")
    assert rel < 1e-4, rel
    dW_r = rk.linear_logp_dw(h, W, tg, lse, g)
    chk = contract.check_gradient_accuracy(dW.cpu().numpy(), dW_r.double().cpu().numpy())
    print(f"saved full backward dW vs recompute dW: {chk}")
    assert chk.passed, chk
    del dW_r
    dh_s = rk.linear_logp_bwd_saved(h, W, tg, lse, g, saved)
    assert torch.equal(dh_s.view(torch.int32), dh.view(torch.int32))
    assert rk.get_device_error() == 0


@pytest.mark.slow
def test_saved_path_llama_t1_t2_t3(rk):
    # the Llama-shaped batch (T = 8192 varlen, H = 4096, V = 128256): logp,
    # lse and dh of the picked sequences bitwise under T1 (a sequence alone),
    # T2 (sequences reversed behind 77 pad rows) and T3 (neighbours redrawn)
    pool = synth.llama_pool(with_grad=True)
    W = cuda(pool.W)
    n = len(pool.lengths)

    def run(p, seqs, lead_pad=0):
        lay = synth.packed(p, seqs, lead_pad=lead_pad)
        h, tg, cu, g = cuda(lay.h), cuda(lay.targets), cuda(lay.cu_seqlens), cuda(lay.g)
        logp, lse, dh = _saved_fwd_bwd(rk, h, W, tg, g, cu)
        return lay, {"logp": logp.cpu(), "lse": lse.cpu(), "dh": dh.cpu()}

    base_lay, base = run(pool, list(range(n)))
    picks = [0, n // 2, n - 1]
    variants = [(run(pool, [i]), [i]) for i in picks]
    variants.append((run(pool, list(reversed(range(n))), lead_pad=77), picks))
    other = synth.replace_neighbours(pool, picks, seed=2 + synth.NEIGHBOUR_SEED_OFFSET)
    variants.append((run(other, list(range(n))), picks))
    for (lay, out), seqs in variants:
        for i in seqs:
            b = torch.tensor(base_lay.rows_of[i])
            v = torch.tensor(lay.rows_of[i])
            for k in base:
                assert torch.equal(out[k][v].view(torch.int32), base[k][b].view(torch.int32)), \
                    (lay.description, i, k)
    assert rk.get_device_error() == 0
