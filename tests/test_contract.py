"""The contract module: tolerances of the four judgments and the drift
record, checked against the schema the pages print (PR #264 "docs(ws1):
batch-invariance contract RFC", Drift Report) -- host-only."""
import json
import os

import numpy as np

from invariant_rl_logprob_gb300 import contract

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "drift_report_example.json")


def _record(base, var):
    return contract.compare_invariance(
        operator="batch_invariant_logp", direction="forward", transform_class="T1",
        transform_name="batch_population", baseline_desc=1, variant_desc=16, seed=123,
        workload="logits", base_vals=base, var_vals=var, seq_ids=[0, 0, 1, 1],
        positions=[0, 1, 0, 1], base_rows=[0, 1, 2, 3], var_rows=[5, 6, 9, 10],
        launch={"batch_size": 16, "seq_len": 256, "chunk_size": None, "padding_side": "right"},
        arch_key="sm103", device="cuda:0")


def test_drift_record_has_the_pages_schema():
    with open(GOLDEN) as f:
        example = json.load(f)["example"]
    rec = _record(np.array([1.0, 2.0, 3.0, 4.0]), np.array([1.0, 2.0, 3.5, 4.0]))
    assert set(example) == set(rec)
    assert set(example["transform"]) == set(rec["transform"])
    assert set(example["launch"]) == set(rec["launch"])
    assert rec["threshold"] == example["threshold"] == {"atol": 0.0, "rtol": 0.0}
    assert rec["chain_index"] == example["chain_index"] == 8
    # first_mismatch: the lowest (sequence, position) that differs, with the
    # logical sequence id and both physical rows (vocab_index kept, null for
    # per-token outputs)
    assert rec["status"] == "fail" and rec["n_mismatched"] == 1 and rec["n_active"] == 4
    assert rec["first_mismatch"] == {"sequence_id": 1, "token_position": 0, "baseline_row": 2,
                                     "variant_row": 9, "vocab_index": None}
    assert rec["max_abs_error"] == 0.5


def test_drift_record_pass_and_nan_bits():
    same = _record(np.array([1.0, np.nan]), np.array([1.0, np.nan]))
    assert same["status"] == "pass" and same["first_mismatch"] is None
    # -0.0 and +0.0 differ bitwise: the I-relation is bit equality, not ==
    z = _record(np.array([0.0]), np.array([-0.0]))
    assert z["status"] == "fail"


def test_accuracy_judgments():
    ok = contract.check_forward_accuracy([-1.0005, -10.01], [-1.0, -10.0])
    assert ok.passed
    bad = contract.check_forward_accuracy([-1.0025], [-1.0])
    assert not bad.passed
    # gradient bound scales with max |ref| over the checked set, not per element
    g = contract.check_gradient_accuracy([10.0, 0.005], [10.0, 0.0])
    assert g.passed
    assert not contract.check_gradient_accuracy([10.0, 0.02], [10.0, 0.0]).passed
    assert contract.TOLERANCES["forward_invariance"] == {"atol": 0.0, "rtol": 0.0}
    assert contract.TOLERANCES["gradient_invariance"] == {"atol": 0.0, "rtol": 0.0}
