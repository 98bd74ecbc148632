"""dW of linear_logp on the GPU: parity with the fp64 oracle, the one-hot
term's edge cases, and bitwise invariance over the same complete sample set
in canonical order (issue #244 "[WS1 Test] ...", Workstream 3)."""
import numpy as np
import pytest
import torch

import oracle
from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import DEV, bits_np, cuda, oracle_bwd, oracle_dw, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


def _case(T, H, V, seed, w_std=0.05):
    gen = synth.generator(seed)
    W = synth.normal_bf16(gen, (V, H), w_std)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    return h, W, tg, g


def _gpu_dw(rk, h, W, tg, g, cu=None, order=None):
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd, cuda(cu))
    return rk.linear_logp_dw(hd, Wd, tgd, lse, gd, cuda(cu), row_order=cuda(order))


@pytest.mark.parametrize("T,H,V", [(64, 256, 4096), (300, 128, 1001), (129, 192, 700), (7, 64, 5),
                                   (200, 8192, 1500)])
def test_dw_vs_oracle(rk, T, H, V):
    h, W, tg, g = _case(T, H, V, 5000 + T + V)
    tg[::11] = -100
    dW = _gpu_dw(rk, h, W, tg, g).cpu().numpy()
    ref = oracle.linear_logp_dw(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dW, ref)
    assert chk.passed, chk
    assert rk.get_device_error() == 0


def test_dw_all_tokens_one_target_and_empty(rk):
    h, W, tg, g = _case(200, 128, 1000, 77)
    tg[:] = 513                                            # one bucket of 200 tokens
    dW = _gpu_dw(rk, h, W, tg, g).cpu().numpy()
    ref = oracle.linear_logp_dw(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    assert contract.check_gradient_accuracy(dW, ref).passed
    tg[:] = -100                                           # no active token
    dW0 = _gpu_dw(rk, h, W, tg, g).cpu()
    assert torch.all(dW0 == 0)


def test_dw_canonical_order_invariance(rk):
    # the same sample set, physical layouts: packed, padded (left/right), with
    # neighbours outside the set redrawn, sequences reversed -- each given the
    # canonical order (sequence id, position) of its active tokens
    pool = synth.make_pool(128, 3000, [40, 70, 25, 33], seed=90, with_grad=True)
    W = cuda(pool.W)

    def dw_of(lay, seqs):
        order = torch.tensor([r for i in seqs for r in lay.rows_of[i]], dtype=torch.int64)
        h, tg, g = cuda(lay.h), cuda(lay.targets), cuda(lay.g)
        _, lse = rk.linear_logp(h, W, tg)
        return rk.linear_logp_dw(h, W, tg, lse, g, row_order=cuda(order)).cpu()

    seqs = [0, 1, 2, 3]
    base = dw_of(synth.packed(pool, seqs), seqs)
    variants = [synth.padded(pool, seqs, 80, side="right"), synth.padded(pool, seqs, 80, side="left"),
                synth.packed(pool, [3, 2, 1, 0], lead_pad=37), synth.packed(pool, [2, 0, 3, 1])]
    for lay in variants:
        assert same_bits(dw_of(lay, seqs), base), lay.description
    # and against the oracle in the same canonical order
    lay = synth.packed(pool, seqs)
    ref = oracle.linear_logp_dw(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(),
                                np.nan_to_num(lay.g.double().numpy()))
    assert contract.check_gradient_accuracy(base.numpy(), ref).passed


def test_dw_run_to_run(rk):
    h, W, tg, g = _case(500, 256, 4096, 31)
    a = _gpu_dw(rk, h, W, tg, g)
    b = _gpu_dw(rk, h, W, tg, g)
    assert same_bits(a, b)


def test_full_backward_matches_separate_calls(rk):
    # one shared softmax pass gives the same dh as rk_linear_logp_bwd and the
    # same dW as rk_linear_logp_dw, bit for bit; masked rows 0, bad targets NaN
    pool = synth.make_pool(192, 2500, [50, 90, 41], seed=93, with_grad=True)
    lay = synth.packed(pool, [0, 1, 2], lead_pad=9)
    tg = lay.targets.clone()
    tg[30] = 2500                                          # out of range: NaN row + error bit
    h, W, tgd, cu, g = cuda(lay.h), cuda(pool.W), cuda(tg), cuda(lay.cu_seqlens), cuda(lay.g)
    _, lse = rk.linear_logp(h, W, tgd, cu)
    rk.get_device_error()
    dh_sep = rk.linear_logp_bwd(h, W, tgd, lse, g, cu)
    dw_sep = rk.linear_logp_dw(h, W, tgd, lse, g, cu)
    assert rk.get_device_error() & rk.DEVERR_TARGET_RANGE
    dh_full, dw_full = rk.linear_logp_bwd_full(h, W, tgd, lse, g, cu)
    assert rk.get_device_error() & rk.DEVERR_TARGET_RANGE
    assert same_bits(dh_full, dh_sep) and same_bits(dw_full, dw_sep)
    d = dh_full.cpu()
    assert torch.all(d[:9] == 0) and torch.all(torch.isnan(d[30]))
    act = oracle.active_rows(tg.numpy(), lay.cu_seqlens.numpy()) & (tg.numpy() < 2500)
    ref = oracle.linear_logp_dw(bits_np(lay.h), bits_np(pool.W), np.where(act, tg.numpy(), -100),
                                np.nan_to_num(lay.g.double().numpy()), lay.cu_seqlens.numpy())
    assert contract.check_gradient_accuracy(dw_full.cpu().numpy(), ref).passed


def test_one_and_two_row_blocks_per_tile_agree(rk):
    # Long K loops with many tiles run the dh and dW GEMMs with two row blocks
    # per tile; short ones with one.  Each accumulator sees the same MMAs
    # either way, so the bits must agree.
    T, H, V = 20480, 4096, 20480
    h, W, tg, g = _case(T, H, V, 57, w_std=0.02)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    # dh: the whole group (two blocks per tile) vs 128-row chunks (one)
    dh_two = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
    wmin = torch.empty(rk.linear_logp_bwd_min_workspace_size(H, V), dtype=torch.uint8, device=DEV)
    dh_one = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd, workspace=wmin)
    assert same_bits(dh_two, dh_one)
    # dW: 10000 active tokens named alone (K = 10000 tokens, one block per
    # tile) vs the same tokens among 20480 candidates (two blocks per tile)
    tg2 = tgd.clone()
    tg2[10000:] = -100
    dw_one = rk.linear_logp_dw(hd, Wd, tg2, lse, gd, row_order=torch.arange(10000, device=DEV))
    dw_two = rk.linear_logp_dw(hd, Wd, tg2, lse, gd)
    assert same_bits(dw_one, dw_two)
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("w_std,argmax_targets", [(0.25, True), (0.4, True), (0.4, False)])
def test_peaked_softmax_gradients(rk, w_std, argmax_targets):
    # Logits with std ~6-9: most rows put p > 0.5 on one column.  With the
    # target there (a confident, correct policy) dh = g (1 - p_t) (W_t - ...)
    # is a small difference of large terms; with a random target two large
    # terms compete.  The target and every column with p >= 1/64 are kept in
    # fp32, so dh and dW stay inside the tolerance in both regimes.
    T, H, V = 512, 512, 4096
    gen = synth.generator(123)
    W = synth.normal_bf16(gen, (V, H), w_std)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    z = oracle.lm_head(bits_np(h), bits_np(W))
    if argmax_targets:
        tg = torch.as_tensor(z.argmax(axis=1), dtype=torch.int64)
    else:
        tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    dh = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd).cpu().numpy()
    ref = oracle.linear_logp_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dh, ref)
    assert chk.passed, ("dh", chk)
    dW = rk.linear_logp_dw(hd, Wd, tgd, lse, gd).cpu().numpy()
    refw = oracle.linear_logp_dw(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dW, refw)
    assert chk.passed, ("dW", chk)
    # and the fused full backward gives the same bits
    dh2, dW2 = rk.linear_logp_bwd_full(hd, Wd, tgd, lse, gd)
    assert same_bits(dh2.cpu(), torch.from_numpy(dh)) and same_bits(dW2.cpu(), torch.from_numpy(dW))
    assert rk.get_device_error() == 0


def test_foreign_lse_is_flagged(rk):
    # an lse that does not belong to the inputs (here 10 too small) makes far
    # more than 64 columns per row look like p >= 1/64: the call still
    # finishes and raises RK_DEVERR_LSE
    h, W, tg, g = _case(64, 256, 4096, 7)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    rk.get_device_error()
    rk.linear_logp_bwd(hd, Wd, tgd, lse - 10.0, gd)
    assert rk.get_device_error() & rk.DEVERR_LSE
    assert rk.get_device_error() == 0


def test_skewed_targets(rk):
    # Half the tokens share one target and a few others repeat hundreds of
    # times (as common tokens do in real batches): long per-row entry lists
    # for the fp32 term, which runs in batches of 32 entries.
    T, H, V = 3000, 256, 2048
    h, W, _, g = _case(T, H, V, 61)
    gen = synth.generator(62)
    tg = torch.randint(0, V, (T,), generator=gen)
    tg[: T // 2] = 7
    tg[T // 2: T // 2 + 400] = 1999
    tg[T // 2 + 400: T // 2 + 433] = 0
    tg = tg[torch.randperm(T, generator=gen)]
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    dW = rk.linear_logp_dw(hd, Wd, tgd, lse, gd)
    ref = oracle.linear_logp_dw(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(dW.cpu().numpy(), ref)
    assert chk.passed, chk
    dh2, dW2 = rk.linear_logp_bwd_full(hd, Wd, tgd, lse, gd)
    assert same_bits(dW2, dW)
    assert rk.get_device_error() == 0


# --------------------------------------------------------------------------
# the paths dW and the fused backward take at full size
# --------------------------------------------------------------------------

def _zipf_targets(gen, T, V, a=1.1):
    # seeded Zipf(a) over the vocabulary: common tokens repeat, as in real text
    p = np.arange(1, V + 1, dtype=np.float64) ** -a
    rng = np.random.default_rng(int(torch.randint(0, 2**31 - 1, (1,), generator=gen).item()))
    return torch.as_tensor(rng.choice(V, size=T, p=p / p.sum()), dtype=torch.int64)


@pytest.mark.parametrize("kind", ["uniform", "zipf", "peaked"])
def test_dw_large_vocabulary_vs_oracle(rk, kind):
    # V = 128256: column indices take 17 bits, so the stable column sort of
    # the fp32 entries runs 4 radix passes of 5 bits (V <= 32768 runs at most
    # 3), and most entries sit in columns >= 32768.  "peaked" (logit std ~5)
    # adds a few columns per row with p >= 1/64 at random places.
    T, H, V = 600, 256, 128256
    h, W, tg, g = _case(T, H, V, 7100 + len(kind), w_std=0.3 if kind == "peaked" else 0.02)
    if kind == "zipf":
        tg = _zipf_targets(synth.generator(7200), T, V)
    tg[::17] = -100
    assert (tg >= 32768).sum() > (T // 4 if kind != "zipf" else 0)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    dW = rk.linear_logp_dw(hd, Wd, tgd, lse, gd)
    assert rk.last_row_blocks("dw") == 1            # K = 600 tokens: a short K loop
    hb, Wb, g64 = bits_np(h), bits_np(W), g.double().numpy()
    ref = oracle_dw(hb, Wb, tg.numpy(), g64)
    chk = contract.check_gradient_accuracy(dW.cpu().numpy(), ref)
    print(f"dW V=128256 {kind}: {chk}")
    assert chk.passed, chk
    dh2, dW2 = rk.linear_logp_bwd_full(hd, Wd, tgd, lse, gd)
    assert same_bits(dW2, dW)
    ref_dh = oracle_bwd(hb, Wb, tg.numpy(), g64)
    chk = contract.check_gradient_accuracy(dh2.cpu().numpy(), ref_dh)
    print(f"dh (full backward) V=128256 {kind}: {chk}")
    assert chk.passed, chk
    assert rk.get_device_error() == 0


_LONG_K = {}


def _long_k_reference():
    # 16384 canonical tokens: the dW GEMM's K loop is 256 stages of 64 (the
    # length from which the launcher takes two row blocks per tile)
    if not _LONG_K:
        T, H, V = 16384, 128, 4096
        h, W, tg, g = _case(T, H, V, 7300, w_std=0.1)
        tg[::29] = -100
        _LONG_K["in"] = (h, W, tg, g)
        _LONG_K["dW"] = oracle_dw(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    return _LONG_K["in"], _LONG_K["dW"]


@pytest.mark.parametrize("blocks", [1, 2])
def test_dw_long_token_axis_vs_oracle(rk, blocks):
    # both GEMM forms on a 256-stage K loop, forced (the launcher alone picks
    # two blocks only when there are also ~8 tiles per resident pair, far
    # beyond what the oracle finishes in seconds), against the oracle and
    # against each other bit for bit
    (h, W, tg, g), ref = _long_k_reference()
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    rk.set_row_blocks(blocks)
    try:
        dW = rk.linear_logp_dw(hd, Wd, tgd, lse, gd)
        assert rk.last_row_blocks("dw") == blocks
        dh, dW_full = rk.linear_logp_bwd_full(hd, Wd, tgd, lse, gd)
        assert rk.last_row_blocks("dw") == blocks and rk.last_row_blocks("dh") == blocks
    finally:
        rk.set_row_blocks(0)
    chk = contract.check_gradient_accuracy(dW.cpu().numpy(), ref)
    print(f"dW K=16384 blocks={blocks}: {chk}")
    assert chk.passed, chk
    assert same_bits(dW_full, dW)
    _LONG_K.setdefault("bits", {})[blocks] = dW.cpu()
    if len(_LONG_K["bits"]) == 2:
        assert same_bits(_LONG_K["bits"][1], _LONG_K["bits"][2])
    assert rk.get_device_error() == 0


def test_dh_two_row_blocks_vs_oracle(rk):
    # the dh GEMM's K loop is the vocabulary: V = 20000 gives 313 stages;
    # two row blocks per tile (forced) against the oracle on every row, and
    # bit for bit against one block
    T, H, V = 1500, 256, 20000
    h, W, tg, g = _case(T, H, V, 7400)
    tg[::23] = -100
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    out = {}
    try:
        for blocks in (2, 1):
            rk.set_row_blocks(blocks)
            out[blocks] = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
            assert rk.last_row_blocks("dh") == blocks
    finally:
        rk.set_row_blocks(0)
    assert same_bits(out[1], out[2])
    ref = oracle_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    chk = contract.check_gradient_accuracy(out[2].cpu().numpy(), ref)
    print(f"dh V=20000 blocks=2: {chk}")
    assert chk.passed, chk
    assert rk.get_device_error() == 0


def _projection_identity(h, W, dh, dW, n_pairs=4, seed=7500):
    """For any a, b in R^H: sum_t (h_t.a)(dh_t.b) = sum_v (W_v.b)(dW_v.a).

    Both sides equal sum_{t,v} D[t,v] (h_t.a)(W_v.b) with D = dlogp/dz, since
    dh = D W and dW = D^T h.  Returns the worst |lhs - rhs| / sum|terms|."""
    gen = torch.Generator(device=h.device)
    gen.manual_seed(seed)
    worst = 0.0
    H = h.shape[1]
    for _ in range(n_pairs):
        a = torch.randn(H, generator=gen, device=h.device, dtype=torch.float64)
        b = torch.randn(H, generator=gen, device=h.device, dtype=torch.float64)
        ha = torch.cat([h[i:i + 8192].double() @ a for i in range(0, h.shape[0], 8192)])
        db = torch.cat([dh[i:i + 8192].double() @ b for i in range(0, dh.shape[0], 8192)])
        wb = torch.cat([W[i:i + 8192].double() @ b for i in range(0, W.shape[0], 8192)])
        da = torch.cat([dW[i:i + 8192].double() @ a for i in range(0, dW.shape[0], 8192)])
        lhs, rhs = (ha * db).sum().item(), (wb * da).sum().item()
        scale = (ha * db).abs().sum().item() + (wb * da).abs().sum().item()
        worst = max(worst, abs(lhs - rhs) / scale)
    return worst


@pytest.mark.slow
def test_grpo_full_size_dw(rk):
    # The GRPO group itself (T = 65536, H = 4096, V = 128256): here the
    # launcher picks two row blocks per tile for both GEMMs on its own, and
    # the column sort runs 4 passes.  The oracle cannot compute dW at this
    # size (every token's softmax over 128256 columns), so:
    #  - dW of the fused backward equals rk_linear_logp_dw's and the forced
    #    one-block form's, bit for bit;
    #  - dh (checked against the oracle on sampled rows elsewhere) and dW
    #    satisfy the projection identity of dh = D W, dW = D^T h;
    #  - dW rows of vocabulary entries no token targets are -sum_t g_t p h_t
    #    and so tiny; every value is finite.
    pool = synth.grpo_pool()
    h, W, tg, g = cuda(pool.h), cuda(pool.W), cuda(pool.targets), cuda(pool.g)
    _, lse = rk.linear_logp(h, W, tg)
    dh, dW = rk.linear_logp_bwd_full(h, W, tg, lse, g)
    assert rk.last_row_blocks("dw") == 2 and rk.last_row_blocks("dh") == 2
    assert rk.last_tile_order("dw") in (1, 2) and rk.last_tile_order("dh") in (1, 2)
    assert torch.isfinite(dW).all() and torch.isfinite(dh).all()
    dW_sep = rk.linear_logp_dw(h, W, tg, lse, g)
    assert rk.last_row_blocks("dw") == 2
    assert torch.equal(dW_sep.view(torch.int32), dW.view(torch.int32))
    del dW_sep
    rk.set_row_blocks(1)
    try:
        dW_one = rk.linear_logp_dw(h, W, tg, lse, g)
        assert rk.last_row_blocks("dw") == 1
    finally:
        rk.set_row_blocks(0)
    assert torch.equal(dW_one.view(torch.int32), dW.view(torch.int32))
    del dW_one
    rel = _projection_identity(h, W, dh, dW)
    print(f"GRPO dW projection identity: worst relative residual {rel:.3g}")
    assert rel < 1e-4, rel
    hit = torch.zeros(pool.V, dtype=torch.bool, device=DEV)
    hit[tg] = True
    untargeted = dW[~hit].abs().max().item()
    targeted = dW[hit].abs().max().item()
    assert untargeted < 0.1 * targeted, (untargeted, targeted)
    assert rk.get_device_error() == 0
