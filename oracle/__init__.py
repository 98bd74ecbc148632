"""fp64 CPU oracle for the selected-token logprob path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``invariant_rl_logprob_gb300``) never imports,
links or executes anything here, and this package imports nothing from it:
the two share no code.

The arithmetic lives in ``rk_oracle.c`` (plain C, fp64, sequential sums,
compiled with ``-O2 -fno-fast-math -ffp-contract=off``).  This module compiles
it with gcc, marshals numpy arrays into it, and applies the masking rule.

Inputs are either bf16 bit patterns (``numpy.uint16``; upcast exactly to
double inside the C code) or ``numpy.float64`` arrays (used by the pins, e.g.
finite differences, that need inputs bf16 cannot hold).

Masking (who counts as an active token).  The pages make the active-token set
an explicit input of every comparison -- PR #264 "docs(ws1): batch-invariance
contract RFC", InvarianceFixture ("action_mask ... defines the active token
set") and its requirement 3, and issue #244 "[WS1 Test] ...", Workstream 3,
Logical-workload identity ("Exclude padding tokens from output / loss / grad
comparisons").  They do not fix an encoding.  Reading used here: row t is
active iff ``targets[t] >= 0`` and, when ``cu_seqlens`` is given,
``cu_seqlens[0] <= t < cu_seqlens[num_seqs]``.  Inactive rows produce
``logp = lse = 0`` and ``dh = 0``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_F64, _BF16 = 0, 1
_lib = None


def build(force: bool = False) -> str:
    """Compile rk_oracle.c into oracle/_build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_linear_logp.argtypes = [vp, i32, vp, i32, vp, vp, i64, i64, i64, vp, vp]
        lib.oracle_linear_logp.restype = i32
        lib.oracle_logp_from_logits.argtypes = [vp, i32, vp, vp, i64, i64, vp, vp]
        lib.oracle_logp_from_logits.restype = i32
        lib.oracle_linear_logp_bwd.argtypes = [vp, i32, vp, i32, vp, vp, vp, i64, i64, i64, vp]
        lib.oracle_linear_logp_bwd.restype = i32
        lib.oracle_lm_head.argtypes = [vp, i32, vp, i32, vp, i64, i64, i64, vp]
        lib.oracle_lm_head.restype = i32
        lib.oracle_logits_bwd.argtypes = [vp, i32, vp, vp, vp, i64, i64, vp]
        lib.oracle_logits_bwd.restype = i32
        d = ctypes.c_double
        lib.oracle_grpo_token.argtypes = [vp, vp, vp, vp, i64, d, d, d, d, vp, vp, vp, vp]
        lib.oracle_grpo_token.restype = None
        lib.oracle_linear_greedy.argtypes = [vp, i32, vp, i32, vp, i64, i64, i64, vp, vp, vp]
        lib.oracle_linear_greedy.restype = i32
        lib.oracle_linear_logp_dw.argtypes = [vp, i32, vp, i32, vp, vp, vp, i64, i64, i64, vp]
        lib.oracle_linear_logp_dw.restype = i32
        _lib = lib
    return _lib


def _as_matrix(a) -> tuple[np.ndarray, int]:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, _BF16
    if a.dtype == np.float64:
        return a, _F64
    raise TypeError(f"oracle inputs are bf16 bits (uint16) or float64, got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def active_rows(targets, cu_seqlens=None, T: int | None = None) -> np.ndarray:
    """Boolean [T] mask of active rows (see the module docstring)."""
    targets = np.asarray(targets, dtype=np.int64)
    T = targets.shape[0] if T is None else T
    act = targets >= 0
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        idx = np.arange(T)
        act &= (idx >= cu[0]) & (idx < cu[-1])
    return act


def _rows_to_run(targets, cu_seqlens, rows):
    T = targets.shape[0]
    act = active_rows(targets, cu_seqlens, T)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    return rows, act[rows]


def linear_logp(h, W, targets, cu_seqlens=None, rows=None):
    """(logp, lse) in float64 for the selected rows (all rows by default).

    h: [T,H], W: [V,H] (uint16 bf16 bits or float64); targets: int64 [T].
    """
    h, hk = _as_matrix(h)
    W, wk = _as_matrix(W)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    T, H = h.shape
    V = W.shape[0]
    assert W.shape[1] == H and targets.shape == (T,)
    rows, act = _rows_to_run(targets, cu_seqlens, rows)
    logp = np.zeros(rows.shape[0], dtype=np.float64)
    lse = np.zeros(rows.shape[0], dtype=np.float64)
    run = np.ascontiguousarray(rows[act])
    if run.size:
        o_logp = np.empty(run.size, dtype=np.float64)
        o_lse = np.empty(run.size, dtype=np.float64)
        rc = _load().oracle_linear_logp(_ptr(h), hk, _ptr(W), wk, _ptr(targets), _ptr(run),
                                        run.size, H, V, _ptr(o_logp), _ptr(o_lse))
        if rc != 0:
            raise ValueError("oracle_linear_logp: target out of range or out of memory")
        logp[act] = o_logp
        lse[act] = o_lse
    return logp, lse


def logp_from_logits(logits, targets, cu_seqlens=None, rows=None):
    """(logp, lse) in float64 from materialised logits [T,V]."""
    z, zk = _as_matrix(logits)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    T, V = z.shape
    assert targets.shape == (T,)
    rows, act = _rows_to_run(targets, cu_seqlens, rows)
    logp = np.zeros(rows.shape[0], dtype=np.float64)
    lse = np.zeros(rows.shape[0], dtype=np.float64)
    run = np.ascontiguousarray(rows[act])
    if run.size:
        o_logp = np.empty(run.size, dtype=np.float64)
        o_lse = np.empty(run.size, dtype=np.float64)
        rc = _load().oracle_logp_from_logits(_ptr(z), zk, _ptr(targets), _ptr(run), run.size,
                                             V, _ptr(o_logp), _ptr(o_lse))
        if rc != 0:
            raise ValueError("oracle_logp_from_logits: target out of range or out of memory")
        logp[act] = o_logp
        lse[act] = o_lse
    return logp, lse


def linear_logp_bwd(h, W, targets, grad_logp, cu_seqlens=None, rows=None):
    """dh [n_rows, H] in float64: g * (W[target] - softmax(h W^T) W)."""
    h, hk = _as_matrix(h)
    W, wk = _as_matrix(W)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    g = np.ascontiguousarray(grad_logp, dtype=np.float64)
    T, H = h.shape
    V = W.shape[0]
    assert W.shape[1] == H and targets.shape == (T,) and g.shape == (T,)
    rows, act = _rows_to_run(targets, cu_seqlens, rows)
    dh = np.zeros((rows.shape[0], H), dtype=np.float64)
    run = np.ascontiguousarray(rows[act])
    if run.size:
        out = np.empty((run.size, H), dtype=np.float64)
        rc = _load().oracle_linear_logp_bwd(_ptr(h), hk, _ptr(W), wk, _ptr(targets), _ptr(g),
                                            _ptr(run), run.size, H, V, _ptr(out))
        if rc != 0:
            raise ValueError("oracle_linear_logp_bwd: target out of range or out of memory")
        dh[act] = out
    return dh


def lm_head(h, W, rows=None) -> np.ndarray:
    """z = h W^T in float64 for the selected rows: [n_rows, V] (no rounding)."""
    h, hk = _as_matrix(h)
    W, wk = _as_matrix(W)
    T, H = h.shape
    V = W.shape[0]
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    z = np.empty((rows.size, V), dtype=np.float64)
    if rows.size and _load().oracle_lm_head(_ptr(h), hk, _ptr(W), wk, _ptr(rows), rows.size,
                                            H, V, _ptr(z)) != 0:
        raise MemoryError("oracle_lm_head")
    return z


def logits_bwd(logits, targets, grad_logp, cu_seqlens=None, rows=None) -> np.ndarray:
    """d(g * logp)/d logits = g * (onehot - softmax) in float64, [n_rows, V];
    zero rows for inactive tokens."""
    z, zk = _as_matrix(logits)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    g = np.ascontiguousarray(grad_logp, dtype=np.float64)
    T, V = z.shape
    rows, act = _rows_to_run(targets, cu_seqlens, rows)
    out = np.zeros((rows.shape[0], V), dtype=np.float64)
    run = np.ascontiguousarray(rows[act])
    if run.size:
        o = np.empty((run.size, V), dtype=np.float64)
        if _load().oracle_logits_bwd(_ptr(z), zk, _ptr(targets), _ptr(g), _ptr(run), run.size,
                                     V, _ptr(o)) != 0:
            raise ValueError("oracle_logits_bwd: target out of range or out of memory")
        out[act] = o
    return out


def grpo_token(logp, logp_old, adv, logp_ref=None, targets=None, cu_seqlens=None, *,
               eps_low=0.2, eps_high=0.2, beta=0.0, scale=1.0):
    """Per-token GRPO loss: dict of float64 arrays loss, grad, ratio, kl
    (zeros on inactive tokens; all tokens active when targets is None)."""
    logp = np.ascontiguousarray(logp, dtype=np.float64)
    n = logp.shape[0]
    lo = np.ascontiguousarray(logp_old, dtype=np.float64)
    a = np.ascontiguousarray(adv, dtype=np.float64)
    ref = None if logp_ref is None else np.ascontiguousarray(logp_ref, dtype=np.float64)
    act = np.ones(n, dtype=bool) if targets is None else active_rows(targets, cu_seqlens, n)
    out = {k: np.zeros(n, dtype=np.float64) for k in ("loss", "grad", "ratio", "kl")}
    idx = np.nonzero(act)[0]
    if idx.size:
        x_lp = np.ascontiguousarray(logp[idx])
        x_lo = np.ascontiguousarray(lo[idx])
        x_a = np.ascontiguousarray(a[idx])
        x_ref = np.ascontiguousarray(ref[idx]) if ref is not None else None
        o = {k: np.empty(idx.size, dtype=np.float64) for k in out}
        _load().oracle_grpo_token(_ptr(x_lp), _ptr(x_lo),
                                  _ptr(x_ref) if x_ref is not None else None, _ptr(x_a), idx.size,
                                  eps_low, eps_high, beta, scale, _ptr(o["loss"]),
                                  _ptr(o["grad"]), _ptr(o["ratio"]), _ptr(o["kl"]))
        for k in out:
            out[k][idx] = o[k]
    return out


def linear_greedy(h, W, rows=None):
    """(token int64, logp float64, zmax float64) of the greedy step per row."""
    h, hk = _as_matrix(h)
    W, wk = _as_matrix(W)
    T, H = h.shape
    V = W.shape[0]
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    tok = np.empty(rows.size, dtype=np.int64)
    lp = np.empty(rows.size, dtype=np.float64)
    zm = np.empty(rows.size, dtype=np.float64)
    if rows.size and _load().oracle_linear_greedy(_ptr(h), hk, _ptr(W), wk, _ptr(rows), rows.size,
                                                  H, V, _ptr(tok), _ptr(lp), _ptr(zm)) != 0:
        raise MemoryError("oracle_linear_greedy")
    return tok, lp, zm


def linear_logp_dw(h, W, targets, grad_logp, cu_seqlens=None, rows=None) -> np.ndarray:
    """dW [V, H] in float64 = sum over the active rows (in the given order) of
    g (onehot - softmax(h W^T))^T h."""
    h, hk = _as_matrix(h)
    W, wk = _as_matrix(W)
    targets = np.ascontiguousarray(targets, dtype=np.int64)
    g = np.ascontiguousarray(grad_logp, dtype=np.float64)
    T, H = h.shape
    V = W.shape[0]
    rows, act = _rows_to_run(targets, cu_seqlens, rows)
    run = np.ascontiguousarray(rows[act])
    dW = np.zeros((V, H), dtype=np.float64)
    if run.size and _load().oracle_linear_logp_dw(_ptr(h), hk, _ptr(W), wk, _ptr(targets), _ptr(g),
                                                  _ptr(run), run.size, H, V, _ptr(dW)) != 0:
        raise ValueError("oracle_linear_logp_dw: target out of range or out of memory")
    return dW


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact upcast of bf16 bit patterns to float64 (for building pins)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
