"""Shared helpers for the GPU tests: device transfer, oracle on row samples
(run in threads -- the oracle's C calls release the GIL), bit comparison."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
from invariant_rl_logprob_gb300 import synth

DEV = torch.device("cuda:0")


def cuda(t: torch.Tensor | None):
    return None if t is None else t.to(DEV)


def bits_np(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t.cpu() if t.device.type != "cpu" else t)


def oracle_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _split(rows, n):
    rows = list(rows)
    k = max(1, (len(rows) + n - 1) // n)
    return [rows[i:i + k] for i in range(0, len(rows), k)]


def oracle_linear(h_bits, W_bits, targets, cu=None, rows=None):
    """(logp, lse) for `rows` (all rows if None), parallel over rows."""
    targets = np.asarray(targets, dtype=np.int64)
    rows = list(range(targets.shape[0])) if rows is None else list(rows)
    parts = _split(rows, oracle_threads())
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda rr: oracle.linear_logp(h_bits, W_bits, targets, cu, rows=rr), parts))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def oracle_bwd(h_bits, W_bits, targets, g, cu=None, rows=None):
    targets = np.asarray(targets, dtype=np.int64)
    rows = list(range(targets.shape[0])) if rows is None else list(rows)
    parts = _split(rows, oracle_threads())
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda rr: oracle.linear_logp_bwd(h_bits, W_bits, targets, g, cu, rows=rr),
                          parts))
    return np.concatenate(res, axis=0)


def oracle_dw(h_bits, W_bits, targets, g, cu=None, rows=None, max_threads: int = 8):
    """dW [V, H] in float64 over `rows` (all rows if None, in that order).

    dW is a sum over tokens, so the tokens are split into consecutive runs,
    each run's dW is computed by the oracle in its own thread, and the
    partials are added in run order.  This only regroups an fp64 sum (the
    result moves by rounding at the 1e-16 level), and caps the threads
    because every partial is a full [V, H] fp64 matrix."""
    targets = np.asarray(targets, dtype=np.int64)
    rows = list(range(targets.shape[0])) if rows is None else list(rows)
    parts = _split(rows, max(1, min(max_threads, oracle_threads())))
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda rr: oracle.linear_logp_dw(h_bits, W_bits, targets, g, cu, rows=rr),
                          parts))
    out = res[0]
    for r in res[1:]:
        out += r
    return out


def oracle_lm_head(h, W, rows=None):
    """z = h W^T in float64 for `rows` (all by default), parallel over rows.
    h and W are bf16 bits or float64 (e.g. |h| and |W| for error bounds)."""
    rows = list(range(h.shape[0])) if rows is None else list(rows)
    parts = _split(rows, oracle_threads())
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda rr: oracle.lm_head(h, W, rows=rr), parts))
    return np.concatenate(res, axis=0)


def z_error_bound(h_bits, W_bits, rows=None):
    """Per-element bound on |z_gpu - z| for z = h W^T accumulated in fp32 from
    exact bf16 x bf16 products, whatever the order of the K additions:
    H * 2^-23 * sum_k |h_k W_vk| (each of the at most H additions rounds by at
    most 2^-23 of a partial sum, and every partial sum is bounded by
    sum_k |h_k W_vk|; 2^-23 rather than 2^-24 leaves room for truncating
    adders)."""
    ha = np.abs(oracle.bf16_bits_to_f64(h_bits))
    Wa = np.abs(oracle.bf16_bits_to_f64(W_bits))
    return h_bits.shape[1] * 2.0 ** -23 * oracle_lm_head(ha, Wa, rows)


def oracle_logits(z_bits, targets, cu=None, rows=None):
    targets = np.asarray(targets, dtype=np.int64)
    rows = list(range(targets.shape[0])) if rows is None else list(rows)
    parts = _split(rows, oracle_threads())
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda rr: oracle.logp_from_logits(z_bits, targets, cu, rows=rr), parts))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    a = a.detach().float().contiguous().cpu()
    b = b.detach().float().contiguous().cpu()
    return a.shape == b.shape and torch.equal(a.view(torch.int32), b.view(torch.int32))


def first_diff(a: torch.Tensor, b: torch.Tensor):
    a = a.detach().float().contiguous().cpu().view(torch.int32)
    b = b.detach().float().contiguous().cpu().view(torch.int32)
    bad = (a != b)
    if bad.dim() > 1:
        bad = bad.any(dim=1)
    idx = torch.nonzero(bad).flatten()
    return None if idx.numel() == 0 else int(idx[0])
