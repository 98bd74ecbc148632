"""The numerical contract the library is checked against, in one place.

Relations (RL-Kernel issue #101 "[RFC] Batch-Invariant RL Kernel Suite for
Train-Inference Consistency", maintainer comment, relation table; PR #264
"docs(ws1): batch-invariance contract RFC"):

* I (invariance) -- the kernel against itself under a batch-shape transform:
  bitwise, atol = rtol = 0, on active tokens.
* A (accuracy)   -- the kernel against the fp64 oracle within a tolerance.

Four judgments, each with its own threshold (issue #244 "[WS1 Test] ...",
"Sole definition of aligned" table; gradient thresholds do not inherit the
forward ones):

* forward_accuracy:   |logp - ref| <= 1e-3 + 1e-3 |ref|          (elementwise)
* gradient_accuracy:  |dh - ref|   <= 1e-3 + 1e-3 max|ref|        (max over the row set)
* forward_invariance, gradient_invariance: bitwise equality.

Transform classes (PR #264, transform taxonomy): T1 population (batch size),
T2 position, T3 neighbour content, T4 padding, T5 execution schedule (attention
only -- not applicable to these operators), T6 selection / packing.

The drift record follows the schema of PR #264 "Drift Report", with
``first_mismatch`` given as the logical sequence id, the token position and the
baseline and variant physical rows (the reviewers' reading of that field for
per-token outputs); ``vocab_index`` is kept and is null for per-token outputs.
"""
from __future__ import annotations

import dataclasses
import hashlib
import json

import numpy as np

TOLERANCES = {
    "forward_accuracy": {"atol": 1e-3, "rtol": 1e-3, "rtol_of": "elementwise |ref|"},
    "gradient_accuracy": {"atol": 1e-3, "rtol": 1e-3, "rtol_of": "max |ref| over the checked rows"},
    "forward_invariance": {"atol": 0.0, "rtol": 0.0},
    "gradient_invariance": {"atol": 0.0, "rtol": 0.0},
}

TRANSFORMS = {
    "T1": "batch_population",
    "T2": "position",
    "T3": "neighbour_content",
    "T4": "padding",
    "T5": "execution_schedule",
    "T6": "selection_packing",
}

CHAIN_INDEX = {"lm_head": 6, "linear_logp": 7, "batch_invariant_logp": 8}


@dataclasses.dataclass
class OutputCheck:
    """Accuracy check record (the fields of the pages' OutputCheck)."""
    max_abs_error: float
    mean_abs_error: float
    max_rel_error: float
    passed: bool
    n_checked: int
    worst_index: int


def check_forward_accuracy(got, ref) -> OutputCheck:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = TOLERANCES["forward_accuracy"]
    err = np.abs(got - ref)
    bound = tol["atol"] + tol["rtol"] * np.abs(ref)
    ok = bool(np.all(err <= bound)) and bool(np.all(np.isfinite(got)))
    rel = err / np.maximum(np.abs(ref), 1e-30)
    return OutputCheck(float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0,
                       float(rel.max(initial=0.0)), ok, int(err.size),
                       int(np.argmax(err)) if err.size else -1)


def check_gradient_accuracy(got, ref) -> OutputCheck:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = TOLERANCES["gradient_accuracy"]
    err = np.abs(got - ref)
    scale = float(np.abs(ref).max(initial=0.0))
    bound = tol["atol"] + tol["rtol"] * scale
    ok = bool(np.all(err <= bound)) and bool(np.all(np.isfinite(got)))
    rel = err / max(scale, 1e-30)
    return OutputCheck(float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0,
                       float(rel.max(initial=0.0)), ok, int(err.size),
                       int(np.argmax(err)) if err.size else -1)


def bits(a) -> np.ndarray:
    """Raw float32 bit patterns (NaN-exact comparison)."""
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def fixture_id(op: str, workload: str, seed: int, transform: str) -> str:
    h = hashlib.sha1(f"{op}|{workload}|{seed}|{transform}".encode()).hexdigest()[:6]
    return f"{op}-bf16-cuda-{h}"


def compare_invariance(*, operator: str, direction: str, transform_class: str,
                       transform_name: str, baseline_desc, variant_desc, seed: int,
                       workload: str, base_vals, var_vals, seq_ids, positions,
                       base_rows, var_rows, launch: dict, arch_key: str, device: str):
    """Bitwise comparison of one logical token set under a transform.

    ``base_vals`` / ``var_vals`` are the outputs of the same logical tokens
    (rows extracted by exact indexing, in canonical (sequence, position)
    order); the other arguments describe them.  Returns a drift record (dict)
    whose ``status`` is "pass" or "fail"."""
    b = np.asarray(base_vals, dtype=np.float32)
    v = np.asarray(var_vals, dtype=np.float32)
    assert b.shape == v.shape
    bb = bits(b).reshape(b.shape[0], -1)
    vb = bits(v).reshape(v.shape[0], -1)
    row_bad = np.any(bb != vb, axis=1)
    diff = np.abs(b.astype(np.float64) - v.astype(np.float64)).reshape(b.shape[0], -1)
    diff = np.where(np.isnan(diff), np.inf, diff)
    n_bad = int(row_bad.sum())
    first = None
    if n_bad:
        i = int(np.argmax(row_bad))   # lowest (sequence, position) in canonical order
        first = {"sequence_id": int(seq_ids[i]), "token_position": int(positions[i]),
                 "baseline_row": int(base_rows[i]), "variant_row": int(var_rows[i]),
                 "vocab_index": None}
    return {
        "relation": "invariance",
        "status": "fail" if n_bad else "pass",
        "fixture_id": fixture_id(operator, workload, seed, f"{transform_class}:{transform_name}"),
        "operator": operator,
        "op_class": "logprob",
        "chain_index": CHAIN_INDEX.get(operator),
        "transform": {"class": transform_class, "name": transform_name,
                      "baseline": baseline_desc, "variant": variant_desc},
        "backend": "cuda",
        "arch_key": arch_key,
        "device": device,
        "dtype": "torch.bfloat16",
        "direction": direction,
        "threshold": {"atol": 0.0, "rtol": 0.0},
        "max_abs_error": float(diff.max(initial=0.0)),
        "mean_abs_error": float(diff.mean()) if diff.size else 0.0,
        "n_mismatched": n_bad,
        "n_active": int(b.shape[0]),
        "first_mismatch": first,
        "launch": launch,
        "seed": seed,
    }


def dumps(record: dict) -> str:
    return json.dumps(record, sort_keys=False)
