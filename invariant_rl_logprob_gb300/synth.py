"""Seeded synthetic workloads for the selected-token logprob path.

This module only draws random numbers, rounds them to bf16 and lays rows out
(packed, padded, permuted, regenerated neighbours).  It holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it: every tensor is produced on the CPU from a ``torch.Generator`` seeded per
workload, rounded to bf16 with round-to-nearest-even, and the very same bits
are handed to both sides.

Fixture rules followed (PR #264 "docs(ws1): batch-invariance contract RFC",
InvarianceFixture, requirements 1-4): the baseline and every transformed
layout are built from the same logical tensors by exact indexing -- nothing is
regenerated per case; the layout records which rows are active; and a case is
fully described by its workload name and seed.

Workloads (the value distributions and shapes of the five configurations this
library is measured and checked on):

* tiny      -- 4 packed sequences x 16 tokens, H=256, V=4096, seed 0
* logits    -- T=2048 materialised bf16 logits, V=32000, N(0, std 2), 1% of
               rows with one logit raised by +20, seed 1
* llama     -- H=4096, V=128256, T=8192 packed varlen, lengths U{128..2048}, seed 2
* qwen      -- H=3584, V=152064, pool of 32 sequences (lengths U{128..2048}),
               padded [B, 2048] or packed, seed 3
* grpo      -- 64 completions x 1024 tokens (T=65536), H=4096, V=128256,
               upstream gradient g ~ N(0,1) per token, seed 4

h ~ N(0, 1) and W ~ N(0, 0.02) (sigma is the standard deviation); targets are
uniform in [0, V).  Pad rows hold NaN in h and g and target -100.
"""
from __future__ import annotations

import dataclasses

import torch

BF16_NAN_BITS = 0x7FC0
IGNORE_TARGET = -100

WORKLOADS = {
    "tiny": dict(H=256, V=4096, seed=0, n_seqs=4, seq_len=16),
    "logits": dict(T=2048, V=32000, seed=1, std=2.0, spike_frac=0.01, spike=20.0),
    "llama": dict(T=8192, H=4096, V=128256, seed=2, len_lo=128, len_hi=2048),
    "qwen": dict(H=3584, V=152064, seed=3, pool=32, max_len=2048, len_lo=128, len_hi=2048),
    "grpo": dict(H=4096, V=128256, seed=4, n_seqs=64, seq_len=1024),
}

NEIGHBOUR_SEED_OFFSET = 1000


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(gen: torch.Generator, shape, std: float, chunk_rows: int = 8192) -> torch.Tensor:
    """N(0, std) drawn in fp32, scaled, rounded to bf16 (RNE); drawn in row chunks."""
    rows = shape[0]
    out = torch.empty(shape, dtype=torch.bfloat16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[r0:r1] = x.to(torch.bfloat16)
    return out


def uniform_targets(gen: torch.Generator, n: int, V: int) -> torch.Tensor:
    return torch.randint(0, V, (n,), generator=gen, dtype=torch.int64)


def varlen_lengths(gen: torch.Generator, total: int, lo: int, hi: int) -> list[int]:
    """Lengths drawn from U{lo..hi} until their sum reaches ``total``; the last
    is truncated so that the sum is exactly ``total`` (it may fall below lo)."""
    out: list[int] = []
    acc = 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor (the exact bits the GPU receives)."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view("uint16")


@dataclasses.dataclass
class Pool:
    """Logical token rows of a set of sequences plus the shared weight W.

    Sequence i owns pool rows [offsets[i], offsets[i] + lengths[i]).
    """
    h: torch.Tensor            # [N, H] bf16
    targets: torch.Tensor      # [N] int64
    g: torch.Tensor | None     # [N] fp32 upstream gradient of logp (or None)
    W: torch.Tensor            # [V, H] bf16
    lengths: list[int]
    offsets: list[int]

    @property
    def H(self) -> int:
        return self.h.shape[1]

    @property
    def V(self) -> int:
        return self.W.shape[0]

    def seq_rows(self, i: int) -> range:
        return range(self.offsets[i], self.offsets[i] + self.lengths[i])


@dataclasses.dataclass
class Layout:
    """A physical batch built from a Pool by exact indexing.

    ``src[r]`` is the pool row that physical row r holds, or -1 for a pad row.
    ``rows_of[i]`` lists, for logical sequence i, the physical rows of its
    tokens in token order (the canonical (sequence, position) coordinates).
    """
    h: torch.Tensor
    targets: torch.Tensor
    g: torch.Tensor | None
    cu_seqlens: torch.Tensor | None   # int32 [num_seqs + 1] or None
    src: torch.Tensor                 # int64 [T]
    rows_of: dict[int, list[int]]
    description: str

    @property
    def T(self) -> int:
        return self.h.shape[0]


def _offsets(lengths):
    offs, acc = [], 0
    for n in lengths:
        offs.append(acc)
        acc += n
    return offs


def make_pool(H: int, V: int, lengths: list[int], seed: int, with_grad: bool = False,
              W: torch.Tensor | None = None) -> Pool:
    """Draw a pool: W first (unless given), then h, targets, g, all from one seed."""
    gen = generator(seed)
    if W is None:
        W = normal_bf16(gen, (V, H), 0.02)
    n = int(sum(lengths))
    h = normal_bf16(gen, (n, H), 1.0)
    targets = uniform_targets(gen, n, V)
    g = torch.randn(n, generator=gen, dtype=torch.float32) if with_grad else None
    return Pool(h=h, targets=targets, g=g, W=W, lengths=list(lengths), offsets=_offsets(lengths))


def replace_neighbours(pool: Pool, keep: list[int], seed: int) -> Pool:
    """T3 neighbour content: sequences not in ``keep`` are redrawn from another
    seed (same lengths); kept sequences keep their exact rows."""
    other = make_pool(pool.H, pool.V, pool.lengths, seed, with_grad=pool.g is not None, W=pool.W)
    h = other.h.clone()
    targets = other.targets.clone()
    g = other.g.clone() if other.g is not None else None
    for i in keep:
        rr = list(pool.seq_rows(i))
        h[rr] = pool.h[rr]
        targets[rr] = pool.targets[rr]
        if g is not None:
            g[rr] = pool.g[rr]
    return Pool(h=h, targets=targets, g=g, W=pool.W, lengths=pool.lengths, offsets=pool.offsets)


def _nan_rows(n: int, H: int) -> torch.Tensor:
    return torch.full((n, H), BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16)


def _assemble(pool: Pool, src: list[int], cu: list[int] | None, rows_of, desc) -> Layout:
    src_t = torch.tensor(src, dtype=torch.int64)
    T = len(src)
    real = src_t >= 0
    h = _nan_rows(T, pool.H)
    targets = torch.full((T,), IGNORE_TARGET, dtype=torch.int64)
    g = torch.full((T,), float("nan"), dtype=torch.float32) if pool.g is not None else None
    if real.any():
        idx = src_t[real]
        h[real] = pool.h[idx]
        targets[real] = pool.targets[idx]
        if g is not None:
            g[real] = pool.g[idx]
    cu_t = torch.tensor(cu, dtype=torch.int32) if cu is not None else None
    return Layout(h=h, targets=targets, g=g, cu_seqlens=cu_t, src=src_t, rows_of=rows_of,
                  description=desc)


def packed(pool: Pool, seq_ids: list[int], lead_pad: int = 0) -> Layout:
    """Varlen packing of ``seq_ids`` in the given order, after ``lead_pad`` NaN
    pad rows; cu_seqlens marks the packed sequences (it starts at lead_pad)."""
    src = [-1] * lead_pad
    cu = [lead_pad]
    rows_of = {}
    for i in seq_ids:
        start = len(src)
        rr = list(pool.seq_rows(i))
        src.extend(rr)
        rows_of[i] = list(range(start, start + len(rr)))
        cu.append(len(src))
    return _assemble(pool, src, cu, rows_of,
                     f"packed seqs={list(seq_ids)} lead_pad={lead_pad}")


def padded(pool: Pool, seq_ids: list[int], max_len: int, side: str = "right") -> Layout:
    """Padded [B, max_len] layout (rows flattened), pad rows NaN / target -100,
    no cu_seqlens (masking by target only)."""
    src: list[int] = []
    rows_of = {}
    for i in seq_ids:
        rr = list(pool.seq_rows(i))
        assert len(rr) <= max_len
        npad = max_len - len(rr)
        if side == "left":
            src.extend([-1] * npad)
        start = len(src)
        src.extend(rr)
        rows_of[i] = list(range(start, start + len(rr)))
        if side == "right":
            src.extend([-1] * npad)
    return _assemble(pool, src, None, rows_of,
                     f"padded seqs={list(seq_ids)} max_len={max_len} side={side}")


# ----------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------

def tiny_pool() -> Pool:
    c = WORKLOADS["tiny"]
    return make_pool(c["H"], c["V"], [c["seq_len"]] * c["n_seqs"], c["seed"], with_grad=True)


def logits_batch(T: int | None = None, V: int | None = None, seed: int | None = None):
    """Materialised logits: (logits bf16 [T,V], targets int64 [T], spike_rows).

    N(0, std 2) in fp32; round(0.01*T) rows, chosen by a seeded permutation,
    get +20 added at one seeded column before the bf16 cast."""
    c = WORKLOADS["logits"]
    T = c["T"] if T is None else T
    V = c["V"] if V is None else V
    seed = c["seed"] if seed is None else seed
    gen = generator(seed)
    z = torch.randn((T, V), generator=gen, dtype=torch.float32).mul_(c["std"])
    n_spike = int(round(c["spike_frac"] * T))
    spike_rows = torch.randperm(T, generator=gen)[:n_spike]
    spike_cols = torch.randint(0, V, (n_spike,), generator=gen, dtype=torch.int64)
    z[spike_rows, spike_cols] += c["spike"]
    targets = uniform_targets(gen, T, V)
    return z.to(torch.bfloat16), targets, spike_rows


def llama_pool(T: int | None = None, with_grad: bool = False) -> Pool:
    """The Llama-shaped workload; ``with_grad`` also draws g ~ N(0, 1) per
    token (after h and the targets, which it leaves unchanged)."""
    c = WORKLOADS["llama"]
    T = c["T"] if T is None else T
    gen = generator(c["seed"] + 500)
    lengths = varlen_lengths(gen, T, c["len_lo"], c["len_hi"])
    return make_pool(c["H"], c["V"], lengths, c["seed"], with_grad=with_grad)


def qwen_pool(with_grad: bool = False) -> Pool:
    """The Qwen-shaped pool of 32 sequences; ``with_grad`` as for llama_pool."""
    c = WORKLOADS["qwen"]
    gen = generator(c["seed"] + 500)
    lengths = [int(torch.randint(c["len_lo"], c["len_hi"] + 1, (1,), generator=gen).item())
               for _ in range(c["pool"])]
    return make_pool(c["H"], c["V"], lengths, c["seed"], with_grad=with_grad)


def grpo_pool(n_seqs: int | None = None) -> Pool:
    c = WORKLOADS["grpo"]
    n = c["n_seqs"] if n_seqs is None else n_seqs
    return make_pool(c["H"], c["V"], [c["seq_len"]] * n, c["seed"], with_grad=True)


def sample_rows(n_total: int, k: int, seed: int) -> list[int]:
    """Seeded sample of k distinct row indices, sorted."""
    gen = generator(seed + 777)
    k = min(k, n_total)
    return sorted(torch.randperm(n_total, generator=gen)[:k].tolist())


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def round_up(a: int, b: int) -> int:
    return ceil_div(a, b) * b

