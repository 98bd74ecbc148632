"""Failure detection without a GPU fault.

A pipeline wait that cannot complete must end in an error status the host
can read, not in a hang (issue #244 "[WS1 Test] ...", #150: silent fallback or
silent failure is not a pass).  A self-test kernel waits on an mbarrier that
nothing ever completes, through the same bounded wait the tile kernels use,
with a 50 ms limit; the error word must report the timeout and the context
must stay usable afterwards.
"""
import time

import pytest
import torch

import oracle
from invariant_rl_logprob_gb300 import contract, synth
from tests.helpers import bits_np, cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


def test_bounded_wait_reports_timeout_and_context_survives(rk):
    t0 = time.perf_counter()
    rk.selftest_wait_timeout(50_000_000)
    err = rk.get_device_error()
    dt = time.perf_counter() - t0
    assert err & rk.DEVERR_TIMEOUT
    assert dt < 5.0
    assert rk.get_device_error() == 0                 # read clears it
    # the context still computes correct results
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    logp, _ = rk.linear_logp(cuda(lay.h), cuda(pool.W), cuda(lay.targets), cuda(lay.cu_seqlens))
    ref, _ = oracle.linear_logp(bits_np(lay.h), bits_np(pool.W), lay.targets.numpy(),
                                lay.cu_seqlens.numpy())
    assert contract.check_forward_accuracy(logp.cpu().numpy(), ref).passed
    assert rk.get_device_error() == 0


def test_selftest_rejects_bad_limits(rk):
    with pytest.raises(rk.RkError, match="INVALID_ARG"):
        rk.selftest_wait_timeout(0)
    with pytest.raises(rk.RkError, match="INVALID_ARG"):
        rk.selftest_wait_timeout(11_000_000_000)
