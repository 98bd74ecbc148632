"""GPU kernels against the fp64 oracle (relation A), through the C ABI.

Tolerance (the forward_accuracy / gradient_accuracy rows of the contract):
|logp - ref| <= 1e-3 + 1e-3 |ref| per row; |dh - ref| <= 1e-3 + 1e-3 max|ref|.
Sizes span several tiles and ragged tails; the full-size workloads are checked
on seeded row samples.
"""
import numpy as np
import pytest
import torch

import oracle
from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import (DEV, bits_np, cuda, oracle_bwd, oracle_linear, oracle_logits,
                           same_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.get_device_error()  # clear
    return m


def _check_fwd(logp, lse, ref_logp, ref_lse, what):
    c1 = contract.check_forward_accuracy(logp.cpu().numpy(), ref_logp)
    c2 = contract.check_forward_accuracy(lse.cpu().numpy(), ref_lse)
    assert c1.passed, f"{what} logp: {c1}"
    assert c2.passed, f"{what} lse: {c2}"
    return c1, c2


# --------------------------------------------------------------------------
# linear_logp forward
# --------------------------------------------------------------------------

def test_tiny_linear_logp_all_rows(rk):
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    logp, lse = rk.linear_logp(cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.cu_seqlens))
    ref_logp, ref_lse = oracle.linear_logp(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(),
                                           lay.cu_seqlens.numpy())
    c1, _ = _check_fwd(logp, lse, ref_logp, ref_lse, "tiny")
    assert c1.max_abs_error < 1e-4, c1          # far inside the bound (fp32 accumulation)
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("T,H,V", [
    (300, 64, 1000),        # 3 row tiles (ragged), 4 vocab tiles (ragged), K = one stage
    (129, 192, 4097),       # one row past a tile, V one past a tile multiple
    (1, 128, 5),            # decode-shaped, V far below a tile
    (257, 256, 769),        # ragged everywhere
    (256, 512, 8192),       # exact tiles, 8 K stages
    (64, 64, 1),            # V = 1: logp = 0
])
def test_linear_logp_shapes(rk, T, H, V):
    gen = synth.generator(1000 + T + H + V)
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    logp, lse = rk.linear_logp(cuda(h), cuda(W), cuda(tg))
    ref_logp, ref_lse = oracle_linear(bits_np(h), bits_np(W), tg.numpy())
    _check_fwd(logp, lse, ref_logp, ref_lse, f"T={T} H={H} V={V}")
    if V == 1:
        assert torch.all(logp.cpu() == 0)
    assert rk.get_device_error() == 0


def test_linear_logp_masking_and_nan_pads(rk):
    pool = synth.make_pool(128, 3000, [40, 70, 25], seed=21)
    lay = synth.packed(pool, [0, 1, 2], lead_pad=13)
    tg = lay.targets.clone()
    tg[20] = -100                                   # ignored token inside a sequence
    cu = lay.cu_seqlens.clone()
    cu[-1] -= 5                                     # last 5 rows fall outside cu_seqlens
    logp, lse = rk.linear_logp(cuda(lay.h), cuda(pool.W), cuda(tg), cuda(cu))
    ref_logp, ref_lse = oracle.linear_logp(bits_np(lay.h), bits_np(pool.W), tg.numpy(), cu.numpy())
    act = oracle.active_rows(tg.numpy(), cu.numpy())
    assert (~act).sum() == 13 + 1 + 5
    _check_fwd(logp, lse, ref_logp, ref_lse, "masked")
    assert torch.all(logp.cpu()[~torch.from_numpy(act)] == 0)
    assert torch.all(torch.isfinite(logp.cpu()))


def test_linear_logp_zero_rows_and_bad_args(rk):
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device=DEV)
    h = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    logp, _ = rk.linear_logp(h, W, torch.zeros(0, dtype=torch.int64, device=DEV))
    assert logp.numel() == 0
    h = torch.zeros((4, 96), dtype=torch.bfloat16, device=DEV)     # H % 64 != 0
    W2 = torch.zeros((100, 96), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rk.RkError, match="UNSUPPORTED"):
        rk.linear_logp(h, W2, torch.zeros(4, dtype=torch.int64, device=DEV))
    h = torch.zeros((4, 64), dtype=torch.bfloat16, device=DEV)
    small = torch.empty(8, dtype=torch.uint8, device=DEV)
    with pytest.raises(rk.RkError, match="WORKSPACE"):
        rk.linear_logp(h, W, torch.zeros(4, dtype=torch.int64, device=DEV), workspace=small)


def test_linear_logp_out_of_range_target(rk):
    gen = synth.generator(5)
    W = synth.normal_bf16(gen, (300, 64), 0.05)
    h = synth.normal_bf16(gen, (8, 64), 1.0)
    tg = synth.uniform_targets(gen, 8, 300)
    tg[3] = 300
    rk.get_device_error()
    logp, lse = rk.linear_logp(cuda(h), cuda(W), cuda(tg))
    assert rk.get_device_error() & rk.DEVERR_TARGET_RANGE
    lp = logp.cpu()
    assert torch.isnan(lp[3]) and torch.all(torch.isfinite(lp[[0, 1, 2, 4, 5, 6, 7]]))
    assert rk.get_device_error() == 0                       # cleared by the read


def test_linear_logp_normalisation_and_shared_lse(rk):
    # V copies of one row with targets 0..V-1: every lse is bitwise the same
    # (positions differ, content does not) and the probabilities sum to one.
    gen = synth.generator(77)
    V, H = 4096, 256
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h1 = synth.normal_bf16(gen, (1, H), 1.0)
    h = h1.repeat(V, 1)
    tg = torch.arange(V, dtype=torch.int64)
    logp, lse = rk.linear_logp(cuda(h), cuda(W), cuda(tg))
    lse = lse.cpu()
    assert torch.all(lse.view(torch.int32) == lse[0].view(torch.int32))
    total = torch.exp(logp.cpu().double()).sum().item()
    assert abs(total - 1.0) < 1e-4


@pytest.mark.slow
def test_llama_shape_sampled_rows(rk):
    pool = synth.llama_pool()
    lay = synth.packed(pool, list(range(len(pool.lengths))))
    logp, lse = rk.linear_logp(cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.cu_seqlens))
    rows = synth.sample_rows(lay.T, 256, seed=2)
    ref_logp, ref_lse = oracle_linear(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(),
                                      lay.cu_seqlens.numpy(), rows=rows)
    c1, c2 = _check_fwd(logp.cpu()[rows], lse.cpu()[rows], ref_logp, ref_lse, "llama sampled")
    print(f"llama 256 sampled rows: logp {c1}; lse {c2}")
    # properties at full size: logp <= 0 on every active row, all finite
    lp = logp.cpu()
    assert torch.all(torch.isfinite(lp)) and torch.all(lp <= 0)
    assert rk.get_device_error() == 0


# --------------------------------------------------------------------------
# logits path
# --------------------------------------------------------------------------

def test_logits_path_full_config_all_rows(rk):
    z, tg, spikes = synth.logits_batch()
    logp, lse = rk.logp_from_logits(cuda(z), cuda(tg))
    ref_logp, ref_lse = oracle_logits(bits_np(z), tg.numpy())
    c1, _ = _check_fwd(logp, lse, ref_logp, ref_lse, "logits T=2048 V=32000")
    assert c1.max_abs_error < 1e-4, c1
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("T,V", [(37, 1), (64, 7), (100, 1001), (33, 4096), (5, 40000), (16, 262144)])
def test_logits_path_shapes(rk, T, V):
    z, tg, _ = synth.logits_batch(T=T, V=V, seed=T + V)
    logp, lse = rk.logp_from_logits(cuda(z), cuda(tg))
    ref_logp, ref_lse = oracle_logits(bits_np(z), tg.numpy())
    _check_fwd(logp, lse, ref_logp, ref_lse, f"logits T={T} V={V}")


def test_logits_path_address_independent(rk):
    # the same rows at a 2-byte-offset address (2-byte loads instead of
    # 16-byte loads) must give the same bits
    z, tg, _ = synth.logits_batch(T=64, V=32000, seed=3)
    zd = cuda(z)
    buf = torch.empty(64 * 32000 + 8, dtype=torch.bfloat16, device=DEV)
    zoff = buf[1:1 + 64 * 32000].view(64, 32000)
    zoff.copy_(zd)
    a, la = rk.logp_from_logits(zd, cuda(tg))
    b, lb = rk.logp_from_logits(zoff, cuda(tg))
    assert same_bits(a, b) and same_bits(la, lb)


def test_logits_path_masking(rk):
    z, tg, _ = synth.logits_batch(T=50, V=3000, seed=4)
    tg[7] = -1
    cu = torch.tensor([5, 20, 45], dtype=torch.int32)
    z[0:5] = float("nan")
    logp, lse = rk.logp_from_logits(cuda(z), cuda(tg), cuda(cu))
    ref_logp, ref_lse = oracle.logp_from_logits(bits_np(z), tg.numpy(), cu.numpy())
    _check_fwd(logp, lse, ref_logp, ref_lse, "logits masked")


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def _check_bwd(dh, ref, what):
    c = contract.check_gradient_accuracy(dh.cpu().numpy(), ref)
    assert c.passed, f"{what}: {c}"
    return c


def test_tiny_backward_all_rows(rk):
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    h, W, tg, cu, g = cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.cu_seqlens), cuda(lay.g)
    _, lse = rk.linear_logp(h, W, tg, cu)
    dh = rk.linear_logp_bwd(h, W, tg, lse, g, cu)
    ref = oracle_bwd(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(), lay.g.double().numpy(),
                     lay.cu_seqlens.numpy())
    _check_bwd(dh, ref, "tiny bwd")
    assert rk.get_device_error() == 0


# (700, ...) gives three 256-row blocks: the dh GEMM's last two-block tile is
# half outside the rows
@pytest.mark.parametrize("T,H,V", [(200, 192, 1000), (130, 320, 4097), (3, 64, 9), (700, 128, 2001)])
def test_backward_shapes(rk, T, H, V):
    gen = synth.generator(2000 + T + H + V)
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    dh = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
    ref = oracle_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    _check_bwd(dh, ref, f"bwd T={T} H={H} V={V}")


def test_backward_chunking_is_invisible(rk):
    gen = synth.generator(31)
    T, H, V = 700, 128, 2000
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    _, lse = rk.linear_logp(hd, Wd, tgd)
    full = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
    wmin = torch.empty(rk.linear_logp_bwd_min_workspace_size(H, V), dtype=torch.uint8, device=DEV)
    chunked = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd, workspace=wmin)
    assert same_bits(full, chunked)


def test_wide_hidden_size(rk):
    # H = 16384: 256 K stages per forward tile and 64 H tiles in the dh GEMM
    # (four raster groups of 16)
    gen = synth.generator(99)
    T, H, V = 300, 16384, 3000
    W = synth.normal_bf16(gen, (V, H), 0.01)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    logp, lse = rk.linear_logp(hd, Wd, tgd)
    dh = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
    rows = synth.sample_rows(T, 24, seed=4)
    ref_logp, ref_lse = oracle_linear(bits_np(h), bits_np(W), tg.numpy(), rows=rows)
    _check_fwd(logp[rows], lse[rows], ref_logp, ref_lse, "H=16384")
    ref_dh = oracle_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy(), rows=rows)
    _check_bwd(dh[rows], ref_dh, "H=16384")
    assert rk.get_device_error() == 0


def test_largest_hidden_size(rk):
    # H = 65536, the largest the kernels accept: 1024 K stages per forward tile
    gen = synth.generator(100)
    T, H, V = 40, 65536, 700
    W = synth.normal_bf16(gen, (V, H), 0.005)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    logp, lse = rk.linear_logp(hd, Wd, tgd)
    dh = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
    ref_logp, ref_lse = oracle_linear(bits_np(h), bits_np(W), tg.numpy())
    _check_fwd(logp, lse, ref_logp, ref_lse, "H=65536")
    ref_dh = oracle_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy())
    _check_bwd(dh, ref_dh, "H=65536")
    assert rk.get_device_error() == 0


def test_many_short_tiles(rk):
    # H = 64 gives one K stage per forward / dZ tile, so the producer runs
    # many tiles ahead of the epilogue and the tile queue wraps many times
    gen = synth.generator(88)
    T, H, V = 2048, 64, 20000
    W = synth.normal_bf16(gen, (V, H), 0.1)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    logp, lse = rk.linear_logp(hd, Wd, tgd)
    dh = rk.linear_logp_bwd(hd, Wd, tgd, lse, gd)
    rows = synth.sample_rows(T, 48, seed=3)
    ref_logp, ref_lse = oracle_linear(bits_np(h), bits_np(W), tg.numpy(), rows=rows)
    _check_fwd(logp[rows], lse[rows], ref_logp, ref_lse, "H=64 many tiles")
    ref_dh = oracle_bwd(bits_np(h), bits_np(W), tg.numpy(), g.double().numpy(), rows=rows)
    _check_bwd(dh[rows], ref_dh, "H=64 many tiles")
    # and the same rows alone give the same bits
    sub = torch.as_tensor(rows, device=DEV)
    lp1, lse1 = rk.linear_logp(hd[sub].contiguous(), Wd, tgd[sub].contiguous())
    assert same_bits(lp1, logp[sub]) and same_bits(lse1, lse[sub])
    assert rk.get_device_error() == 0


def test_workspace_contents_are_ignored(rk):
    # the workspaces hold the tile counters the launches zero themselves:
    # garbage in them changes nothing
    gen = synth.generator(77)
    T, H, V = 600, 128, 3000
    W = synth.normal_bf16(gen, (V, H), 0.05)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    g = torch.randn(T, generator=gen, dtype=torch.float32)
    hd, Wd, tgd, gd = cuda(h), cuda(W), cuda(tg), cuda(g)
    lp0, lse0 = rk.linear_logp(hd, Wd, tgd)
    dh0 = rk.linear_logp_bwd(hd, Wd, tgd, lse0, gd)
    wf = torch.full((rk.linear_logp_workspace_size(T, H, V),), 0xA5, dtype=torch.uint8, device=DEV)
    wb = torch.full((rk.linear_logp_bwd_workspace_size(T, H, V),), 0x5A, dtype=torch.uint8,
                    device=DEV)
    for _ in range(2):   # the second call finds the first call's counters
        lp1, lse1 = rk.linear_logp(hd, Wd, tgd, workspace=wf)
        dh1 = rk.linear_logp_bwd(hd, Wd, tgd, lse1, gd, workspace=wb)
        assert same_bits(lp1, lp0) and same_bits(lse1, lse0) and same_bits(dh1, dh0)
    assert rk.get_device_error() == 0


def test_backward_masking(rk):
    pool = synth.make_pool(128, 1500, [30, 50], seed=41, with_grad=True)
    lay = synth.packed(pool, [0, 1], lead_pad=7)
    h, W, tg, cu, g = cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.cu_seqlens), cuda(lay.g)
    _, lse = rk.linear_logp(h, W, tg, cu)
    dh = rk.linear_logp_bwd(h, W, tg, lse, g, cu).cpu()
    assert torch.all(dh[:7] == 0) and torch.all(torch.isfinite(dh))
    ref = oracle_bwd(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(),
                     np.nan_to_num(lay.g.double().numpy()), lay.cu_seqlens.numpy())
    _check_bwd(dh, ref, "bwd masked")


@pytest.mark.slow
def test_grpo_shape_sampled_rows(rk):
    pool = synth.grpo_pool()
    lay = synth.packed(pool, list(range(len(pool.lengths))))
    h, W, tg, g = cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.g)
    logp, lse = rk.linear_logp(h, W, tg)
    dh = rk.linear_logp_bwd(h, W, tg, lse, g)
    # the launch the bench times: one pass over all rows, two row blocks per
    # dh tile (K = 2004 stages of the vocabulary), tiles taken in rounds
    assert rk.last_row_blocks("dh") == 2
    # rounds (2) unless the device refused the cooperative launch (1)
    assert rk.last_tile_order("dh") in (1, 2)
    print(f"GRPO dh tile order: {rk.last_tile_order('dh')}")
    rows = synth.sample_rows(lay.T, 64, seed=4)
    hb, Wb = bits_np(lay.h), bits_np(pool.W)
    ref_logp, ref_lse = oracle_linear(hb, Wb, lay.targets.numpy(), rows=rows)
    c1, c2 = _check_fwd(logp.cpu()[rows], lse.cpu()[rows], ref_logp, ref_lse, "grpo fwd sampled")
    ref_dh = oracle_bwd(hb, Wb, lay.targets.numpy(), lay.g.double().numpy(), rows=rows)
    c3 = _check_bwd(dh.cpu()[rows], ref_dh, "grpo bwd sampled")
    print(f"grpo 64 sampled rows: logp {c1}; lse {c2}; dh {c3}")
    assert rk.get_device_error() == 0


@pytest.mark.slow
def test_qwen_shape_padded_sampled_rows(rk):
    # [8, 2048] right-padded batch of the Qwen-shaped pool (pads NaN, target
    # -100): sampled active rows against the oracle, inactive rows exactly 0
    pool = synth.qwen_pool()
    lay = synth.padded(pool, list(range(8)), 2048)
    logp, lse = rk.linear_logp(cuda(lay.h), cuda(pool.W), cuda(lay.targets))
    act = oracle.active_rows(lay.targets.numpy())
    rows = [r for r in synth.sample_rows(lay.T, 96, seed=3) if act[r]][:48]
    ref_logp, ref_lse = oracle_linear(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(),
                                      rows=rows)
    _check_fwd(logp.cpu()[rows], lse.cpu()[rows], ref_logp, ref_lse, "qwen padded sampled")
    lp = logp.cpu()
    assert torch.all(lp[~torch.from_numpy(act)] == 0)
    assert torch.all(torch.isfinite(lp))


@pytest.mark.slow
@pytest.mark.parametrize("T,V", [(1024, 152064), (65536, 32000)])
def test_logits_path_large_sampled(rk, T, V):
    # the Qwen vocabulary (not a multiple of 256) and a 4.2 GB batch: sampled
    # rows against the oracle, properties on every row
    z, tg, _ = synth.logits_batch(T=T, V=V, seed=T + V)
    logp, lse = rk.logp_from_logits(cuda(z), cuda(tg))
    rows = synth.sample_rows(T, 64, seed=V)
    ref_logp, ref_lse = oracle_logits(bits_np(z), tg.numpy(), rows=rows)
    _check_fwd(logp.cpu()[rows], lse.cpu()[rows], ref_logp, ref_lse, f"logits T={T} V={V}")
    lp = logp.cpu()
    assert torch.all(torch.isfinite(lp)) and torch.all(lp <= 0)
    assert rk.get_device_error() == 0
