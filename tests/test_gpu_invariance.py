"""Bitwise batch-invariance matrix (relation I, atol = rtol = 0) on the GPU.

For one logical token set, every transform of the batch around it must leave
its logp, lse and dh bit-for-bit unchanged (PR #264 "docs(ws1):
batch-invariance contract RFC", transform taxonomy T1-T6; issue #244
"[WS1 Test] ...", Workstream 3, logical-workload identity).  Baseline and
variants are built from the same logical tensors by exact indexing; outputs
are extracted by exact indexing in canonical (sequence, position) order and
compared as bit patterns.  A failure carries the drift record of the contract.
T5 (execution schedule: chunked prefill) concerns attention and has no
counterpart here; decode-shaped single-row launches stand in for the
prefill / decode split.
"""
import json

import pytest
import torch

from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import DEV, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


def arch_key() -> str:
    cc = torch.cuda.get_device_capability(DEV)
    return f"sm{cc[0]}{cc[1]}"


class Runner:
    """Runs the three operators on a layout and extracts logical rows."""

    def __init__(self, rk, pool, with_bwd=True, bwd_workspace=None, saved=False):
        self.rk = rk
        self.pool = pool
        self.W = cuda(pool.W)
        self.with_bwd = with_bwd and pool.g is not None
        self.bwd_workspace = bwd_workspace
        self.saved = saved  # the forward that keeps its terms + the backward from them

    def run(self, lay):
        h, tg = cuda(lay.h), cuda(lay.targets)
        cu = cuda(lay.cu_seqlens)
        if self.saved:
            logp, lse, sv = self.rk.linear_logp_fwd_saved(h, self.W, tg, cu)
            out = {"logp": logp, "lse": lse}
            if self.with_bwd:
                out["dh"] = self.rk.linear_logp_bwd_saved(h, self.W, tg, lse, cuda(lay.g), sv, cu)
            torch.cuda.synchronize()
            return {k: v.cpu() for k, v in out.items()}
        logp, lse = self.rk.linear_logp(h, self.W, tg, cu)
        out = {"logp": logp, "lse": lse}
        if self.with_bwd:
            ws = None
            if self.bwd_workspace is not None:
                ws = torch.empty(self.bwd_workspace, dtype=torch.uint8, device=DEV)
            out["dh"] = self.rk.linear_logp_bwd(h, self.W, tg, lse, cuda(lay.g), cu, workspace=ws)
        torch.cuda.synchronize()
        return {k: v.cpu() for k, v in out.items()}

    @staticmethod
    def extract(lay, out, seq_ids):
        rows = [r for i in seq_ids for r in lay.rows_of[i]]
        idx = torch.tensor(rows, dtype=torch.int64)
        seq = [i for i in seq_ids for _ in lay.rows_of[i]]
        pos = [p for i in seq_ids for p in range(len(lay.rows_of[i]))]
        return {k: v[idx] for k, v in out.items()}, rows, seq, pos


def assert_invariant(runner, base_lay, base_out, var_lay, var_out, seq_ids, tclass, tname,
                     workload, seed):
    b, brows, seq, pos = Runner.extract(base_lay, base_out, seq_ids)
    v, vrows, _, _ = Runner.extract(var_lay, var_out, seq_ids)
    for key in b:
        rec = contract.compare_invariance(
            operator="linear_logp", direction="backward" if key == "dh" else "forward",
            transform_class=tclass, transform_name=tname, baseline_desc=base_lay.description,
            variant_desc=var_lay.description, seed=seed, workload=workload,
            base_vals=b[key].numpy(), var_vals=v[key].numpy(), seq_ids=seq, positions=pos,
            base_rows=brows, var_rows=vrows,
            launch={"batch_size": var_lay.T, "seq_len": None, "chunk_size": None,
                    "padding_side": None},
            arch_key=arch_key(), device=str(DEV))
        assert rec["status"] == "pass", f"{key} drift: " + json.dumps(rec)
    # the rows compared were all active and finite
    assert torch.all(torch.isfinite(b["logp"])) and torch.all(b["logp"] < 0)


# --------------------------------------------------------------------------
# tiny workload: every transform class on all tokens
# --------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny(rk):
    pool = synth.tiny_pool()
    runner = Runner(rk, pool)
    base = synth.packed(pool, [0, 1, 2, 3])
    return pool, runner, base, runner.run(base)


def test_tiny_t1_batch_population(rk, tiny):
    pool, runner, base, bout = tiny
    for group in ([0], [1], [2], [3], [0, 1], [2, 3]):          # B = 1, B = 2
        lay = synth.packed(pool, group)
        assert_invariant(runner, base, bout, lay, runner.run(lay), group, "T1",
                         f"B={len(group)}", "tiny", 0)


def test_tiny_t2_order_and_offsets(rk, tiny):
    pool, runner, base, bout = tiny
    rev = synth.packed(pool, [3, 2, 1, 0])
    assert_invariant(runner, base, bout, rev, runner.run(rev), [0, 1, 2, 3], "T2",
                     "reversed_sequences", "tiny", 0)
    # full row reversal: every token at a new position (row r -> T-1-r)
    rows = torch.arange(base.T - 1, -1, -1)
    rl = synth.Layout(h=base.h[rows].clone(), targets=base.targets[rows].clone(),
                      g=base.g[rows].clone(), cu_seqlens=None, src=base.src[rows].clone(),
                      rows_of={i: [base.T - 1 - r for r in base.rows_of[i]] for i in base.rows_of},
                      description="row-reversed")
    assert_invariant(runner, base, bout, rl, runner.run(rl), [0, 1, 2, 3], "T2", "row_reversal",
                     "tiny", 0)


def test_tiny_t2_offset_sweep(rk, tiny):
    # 0..255 NaN pad rows in front: each token visits every position of a
    # 128-row tile and both tiles of a 2-tile span
    pool, runner, base, bout = tiny
    r2 = Runner(rk, pool, with_bwd=False)
    for off in range(256):
        lay = synth.packed(pool, [0, 1, 2, 3], lead_pad=off)
        assert_invariant(r2, base, {k: bout[k] for k in ("logp", "lse")}, lay, r2.run(lay),
                         [0, 1, 2, 3], "T2", f"lead_pad={off}", "tiny", 0)


def test_tiny_t2_offset_sweep_backward(rk, tiny):
    pool, runner, base, bout = tiny
    for off in (1, 7, 31, 64, 100, 127, 128, 129, 200):
        lay = synth.packed(pool, [0, 1, 2, 3], lead_pad=off)
        assert_invariant(runner, base, bout, lay, runner.run(lay), [0, 1, 2, 3], "T2",
                         f"lead_pad={off}", "tiny", 0)


def test_tiny_t3_neighbour_content(rk, tiny):
    pool, runner, base, bout = tiny
    for keep in ([0], [2], [1, 3]):
        other = synth.replace_neighbours(pool, keep, seed=synth.NEIGHBOUR_SEED_OFFSET)
        lay = synth.packed(other, [0, 1, 2, 3])
        assert_invariant(runner, base, bout, lay, runner.run(lay), keep, "T3",
                         f"neighbours_redrawn keep={keep}", "tiny", 0)
    # neighbours replaced by NaN rows
    lay = synth.packed(pool, [0, 1, 2, 3])
    for i in (1, 3):
        lay.h[lay.rows_of[i]] = synth._nan_rows(len(lay.rows_of[i]), pool.H)
    assert_invariant(runner, base, bout, lay, runner.run(lay), [0, 2], "T3", "neighbours_nan",
                     "tiny", 0)


def test_tiny_t4_padding(rk, tiny):
    pool, runner, base, bout = tiny
    for side in ("right", "left"):
        for max_len in (16, 40, 160):
            lay = synth.padded(pool, [0, 1, 2, 3], max_len, side=side)
            assert_invariant(runner, base, bout, lay, runner.run(lay), [0, 1, 2, 3], "T4",
                             f"padded {side} max_len={max_len}", "tiny", 0)


def test_tiny_t6_selection(rk, tiny):
    pool, runner, base, bout = tiny
    lay = synth.packed(pool, [2, 0])
    assert_invariant(runner, base, bout, lay, runner.run(lay), [0, 2], "T6", "subset_packed",
                     "tiny", 0)


def test_tiny_decode_rows(rk, tiny):
    # single-token launches (T = 1) reproduce the prefill rows
    pool, runner, base, bout = tiny
    for i in range(4):
        for p in (0, 7, 15):
            r = pool.offsets[i] + p
            lay = synth._assemble(pool, [r], [0, 1], {i: [0]}, f"decode seq={i} pos={p}")
            out = runner.run(lay)
            b = base.rows_of[i][p]
            for k in out:
                assert torch.equal(out[k][0].view(torch.int32), bout[k][b].view(torch.int32)), (k, i, p)


def test_tiny_run_to_run(rk, tiny):
    pool, runner, base, bout = tiny
    for _ in range(3):
        again = runner.run(base)
        for k in bout:
            assert torch.equal(again[k].view(torch.int32), bout[k].view(torch.int32)), k


def test_backward_chunking_invariance(rk, tiny):
    pool, runner, base, bout = tiny
    r2 = Runner(rk, pool, bwd_workspace=rk.linear_logp_bwd_min_workspace_size(pool.H, pool.V))
    lay = synth.packed(pool, [0, 1, 2, 3], lead_pad=150)   # 214 rows, 2 chunks of 128
    assert_invariant(r2, base, bout, lay, r2.run(lay), [0, 1, 2, 3], "T1", "bwd_row_chunks",
                     "tiny", 0)


# --------------------------------------------------------------------------
# logits path
# --------------------------------------------------------------------------

def test_logits_path_transforms(rk):
    z, tg, _ = synth.logits_batch()
    zd, tgd = cuda(z), cuda(tg)
    base, blse = rk.logp_from_logits(zd, tgd)
    base, blse = base.cpu(), blse.cpu()
    checks = []
    sel = torch.tensor([5, 77, 1000, 2047, 0])
    a, la = rk.logp_from_logits(zd[sel].contiguous(), tgd[sel].contiguous())  # T1 / T6 subset
    checks.append(("subset", a.cpu(), la.cpu(), sel))
    rev = torch.arange(2047, -1, -1)
    a, la = rk.logp_from_logits(zd[rev].contiguous(), tgd[rev].contiguous())  # T2 reversal
    checks.append(("reversed", a.cpu(), la.cpu(), rev))
    for i in (3, 1999):                                                       # T1 alone
        a, la = rk.logp_from_logits(zd[i:i + 1].contiguous(), tgd[i:i + 1].contiguous())
        checks.append((f"alone {i}", a.cpu(), la.cpu(), torch.tensor([i])))
    for off in range(32):                                                     # T2/T4 pads
        pad = torch.full((off, z.shape[1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        zz = torch.cat([pad, zd[:64]])
        tt = torch.cat([torch.full((off,), -100, dtype=torch.int64, device=DEV), tgd[:64]])
        a, la = rk.logp_from_logits(zz, tt)
        checks.append((f"lead_pad {off}", a.cpu()[off:], la.cpu()[off:], torch.arange(64)))
    zn = zd[:128].clone()                                                    # T3 neighbours
    zn[1::2] = torch.randn_like(zn[1::2], dtype=torch.float32).to(torch.bfloat16)
    a, la = rk.logp_from_logits(zn, tgd[:128].contiguous())
    checks.append(("neighbours", a.cpu()[0::2], la.cpu()[0::2], torch.arange(0, 128, 2)))
    for name, a, la, idx in checks:
        assert torch.equal(a.view(torch.int32), base[idx].view(torch.int32)), name
        assert torch.equal(la.view(torch.int32), blse[idx].view(torch.int32)), name


# --------------------------------------------------------------------------
# full-size workloads (sampled sequences)
# --------------------------------------------------------------------------

@pytest.mark.slow
def test_llama_t1_t2_t3(rk):
    # logp, lse and dh of the picked sequences, bitwise, under T1-T3
    pool = synth.llama_pool(with_grad=True)
    runner = Runner(rk, pool)
    n = len(pool.lengths)
    base = synth.packed(pool, list(range(n)))
    bout = runner.run(base)
    picks = [0, n // 2, n - 1]
    for i in picks:                                              # T1: sequence alone
        lay = synth.packed(pool, [i])
        assert_invariant(runner, base, bout, lay, runner.run(lay), [i], "T1", "B=1", "llama", 2)
    perm = list(reversed(range(n)))                              # T2: permutation + shift
    lay = synth.packed(pool, perm, lead_pad=77)
    assert_invariant(runner, base, bout, lay, runner.run(lay), picks, "T2",
                     "reversed+lead_pad=77", "llama", 2)
    other = synth.replace_neighbours(pool, picks, seed=2 + synth.NEIGHBOUR_SEED_OFFSET)
    lay = synth.packed(other, list(range(n)))                    # T3: neighbours redrawn
    assert_invariant(runner, base, bout, lay, runner.run(lay), picks, "T3", "neighbours_redrawn",
                     "llama", 2)


@pytest.mark.slow
@pytest.mark.parametrize("saved", [False, True])
def test_qwen_padding_vs_packing(rk, saved):
    # logp, lse and dh of the active tokens, bitwise: B = 8 and B = 32
    # right-padded, B = 1 padded, against the varlen pack (T4 / T6, T1); with
    # the recompute backward and with the saved-terms forward and backward
    # (whose dh GEMM skips the padding blocks and takes its tiles in rounds)
    pool = synth.qwen_pool(with_grad=True)
    runner = Runner(rk, pool, saved=saved)
    base = synth.packed(pool, list(range(8)))                    # varlen pack of seqs 0-7
    bout = runner.run(base)
    b8 = synth.padded(pool, list(range(8)), 2048)                # [8, 2048] right-padded
    assert_invariant(runner, base, bout, b8, runner.run(b8), list(range(8)), "T4", "B=8 padded",
                     "qwen", 3)
    b32 = synth.padded(pool, list(range(32)), 2048)              # [32, 2048]
    assert_invariant(runner, base, bout, b32, runner.run(b32), list(range(8)), "T1",
                     "B=32 padded", "qwen", 3)
    for i in (0, 5):                                             # B = 1
        lay = synth.padded(pool, [i], 2048)
        assert_invariant(runner, base, bout, lay, runner.run(lay), [i], "T1", "B=1 padded",
                         "qwen", 3)


@pytest.mark.slow
def test_grpo_decode_rows_match_prefill(rk):
    pool = synth.grpo_pool(n_seqs=8)
    runner = Runner(rk, pool)
    base = synth.packed(pool, list(range(8)))
    bout = runner.run(base)
    gen = synth.generator(44)
    for i in range(8):
        picks = [0, pool.lengths[i] - 1, int(torch.randint(1, pool.lengths[i] - 1, (1,), generator=gen))]
        for n_rows in (1, 3, 64):
            # decode-shaped launch of n_rows rows: the picked rows followed by
            # further rows of the same sequence
            extra = [p for p in range(pool.lengths[i]) if p not in picks][: max(0, n_rows - 3)]
            pos = (picks + extra)[:n_rows]
            src = [pool.offsets[i] + p for p in pos]
            lay = synth._assemble(pool, src, [0, len(src)], {i: list(range(len(src)))},
                                  f"decode seq={i} rows={n_rows}")
            out = runner.run(lay)
            for j, p in enumerate(pos):
                b = base.rows_of[i][p]
                for k in out:
                    assert torch.equal(out[k][j].view(torch.int32), bout[k][b].view(torch.int32)), \
                        (k, i, p, n_rows)


@pytest.mark.slow
def test_qwen_dw_padding_packing_permutation(rk):
    # dW over the same complete sample set (the active tokens of sequences
    # 0-7 of the Qwen-shaped pool, in canonical (sequence, position) order),
    # from a right-padded [8, 2048] batch, a left-padded one, the varlen pack
    # and a permuted pack behind 37 pad rows: bitwise equal (issue #244,
    # Workstream 3, logical-workload identity).  The fused backward gives the
    # same dW bits.
    pool = synth.qwen_pool(with_grad=True)
    W = cuda(pool.W)
    seqs = list(range(8))

    def dw_of(lay, full=False):
        order = torch.tensor([r for i in seqs for r in lay.rows_of[i]], dtype=torch.int64)
        h, tg, g = cuda(lay.h), cuda(lay.targets), cuda(lay.g)
        _, lse = rk.linear_logp(h, W, tg)
        if full:
            return rk.linear_logp_bwd_full(h, W, tg, lse, g, row_order=cuda(order))[1]
        return rk.linear_logp_dw(h, W, tg, lse, g, row_order=cuda(order))

    base = dw_of(synth.packed(pool, seqs)).cpu()
    assert torch.isfinite(base).all()
    for lay, full in ((synth.padded(pool, seqs, 2048, side="right"), False),
                      (synth.padded(pool, seqs, 2048, side="left"), False),
                      (synth.packed(pool, [7, 3, 5, 1, 0, 6, 2, 4], lead_pad=37), False),
                      (synth.padded(pool, seqs, 2048, side="right"), True)):
        got = dw_of(lay, full).cpu()
        assert torch.equal(got.view(torch.int32), base.view(torch.int32)), (lay.description, full)
    assert rk.get_device_error() == 0


@pytest.mark.slow
def test_qwen_dw_saved_padding_packing_permutation(rk):
    # The same sample set through the forward that keeps its softmax terms
    # and rk_linear_logp_bwd_full_saved: dW (canonical order) and the active
    # rows' dh bitwise equal across right- and left-padded batches and a
    # permuted pack behind 37 pad rows.
    pool = synth.qwen_pool(with_grad=True)
    W = cuda(pool.W)
    seqs = list(range(8))

    def grads_of(lay):
        order = torch.tensor([r for i in seqs for r in lay.rows_of[i]], dtype=torch.int64)
        h, tg, g = cuda(lay.h), cuda(lay.targets), cuda(lay.g)
        _, lse, saved = rk.linear_logp_fwd_saved(h, W, tg)
        dh, dW = rk.linear_logp_bwd_full_saved(h, W, tg, lse, g, saved, row_order=cuda(order))
        return dh[cuda(order)].cpu(), dW.cpu()

    dh0, dw0 = grads_of(synth.packed(pool, seqs))
    assert torch.isfinite(dw0).all() and torch.isfinite(dh0).all()
    for lay in (synth.padded(pool, seqs, 2048, side="right"),
                synth.padded(pool, seqs, 2048, side="left"),
                synth.packed(pool, [7, 3, 5, 1, 0, 6, 2, 4], lead_pad=37)):
        dh, dw = grads_of(lay)
        assert torch.equal(dw.view(torch.int32), dw0.view(torch.int32)), lay.description
        assert torch.equal(dh.view(torch.int32), dh0.view(torch.int32)), lay.description
    assert rk.get_device_error() == 0
