"""rk_linear_logp_noalloc: the forward for callers that cannot allocate.

Callers that own all device memory through a fixed-budget arena or pool, or
that sit behind a plugin-style interface handing over only input/output
pointers and a stream, cannot give the library a workspace or let it call
cudaMalloc (which could fail against the budget, fragment the pool, or stall
the device mid-loop).  This entry point keeps its scratch in a fixed array
inside the library instead.  The test calls it through the C ABI and checks
that it reproduces the workspace-taking entry point within the forward
accuracy tolerance the other tests use (and, since it runs the same kernels,
bit for bit), on two calls in a row, and that requests larger than the array
are refused before anything runs.

The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

from invariant_rl_logprob_gb300 import contract, synth

pytestmark = pytest.mark.gpu

RK_OK, RK_ERR_WORKSPACE = 0, 3
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    from invariant_rl_logprob_gb300 import build
    path = build.build()
    import invariant_rl_logprob_gb300 as rk
    rk.load_library()
    l = ctypes.CDLL(path)
    f = l.rk_linear_logp_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int32] + [ctypes.c_int64] * 3 + \
        [ctypes.c_void_p] * 3
    return l


def call_noalloc(lib, h, W, tg, cu, logp, lse):
    ns = 0 if cu is None else cu.numel() - 1
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.rk_linear_logp_noalloc(p(h), p(W), p(tg), p(cu), ns, h.shape[0], h.shape[1],
                                      W.shape[0], p(logp), p(lse), stream)


def workload(T, H, V, seed, varlen=False):
    gen = synth.generator(seed)
    W = synth.normal_bf16(gen, (V, H), 0.02)
    h = synth.normal_bf16(gen, (T, H), 1.0)
    tg = synth.uniform_targets(gen, T, V)
    tg[::37] = -100
    cu = None
    if varlen:
        lens = synth.varlen_lengths(gen, T - 3, 50, 400)
        cu = torch.tensor([3] + [3 + sum(lens[:i + 1]) for i in range(len(lens))], dtype=torch.int32)
    d = torch.device("cuda:0")
    return h.to(d), W.to(d), tg.to(d), (cu.to(d) if cu is not None else None)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    import invariant_rl_logprob_gb300 as rk
    cases = [workload(3000, 512, 32000, seed=91, varlen=True),     # first call
             workload(1000, 4096, 128256, seed=92)]                # second call, other shape
    for h, W, tg, cu in cases:
        ref_logp, ref_lse = rk.linear_logp(h, W, tg, cu)
        logp = torch.full_like(ref_logp, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert call_noalloc(lib, h, W, tg, cu, logp, lse) == RK_OK
        torch.cuda.synchronize()
        for got, ref in ((logp, ref_logp), (lse, ref_lse)):
            chk = contract.check_forward_accuracy(got.cpu().numpy(), ref.cpu().numpy())
            assert chk.passed, chk
            assert torch.equal(got.cpu().view(torch.int32), ref.cpu().view(torch.int32))
    assert rk.get_device_error() == 0


def test_noalloc_allocates_no_device_memory(lib):
    # After one warm-up call (which looks up the array's address and loads
    # the kernels), further calls of other shapes leave both the CUDA driver's
    # free-memory count and PyTorch's allocator exactly where they were.
    h, W, tg, cu = workload(2048, 256, 50000, seed=93, varlen=True)
    h2, W2, tg2, _ = workload(700, 512, 9000, seed=94)
    logp = torch.empty(2048, dtype=torch.float32, device=h.device)
    lse = torch.empty(2048, dtype=torch.float32, device=h.device)
    assert call_noalloc(lib, h, W, tg, cu, logp, lse) == RK_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(3):
        assert call_noalloc(lib, h2, W2, tg2, None, logp[:700], lse[:700]) == RK_OK
        assert call_noalloc(lib, h, W, tg, cu, logp, lse) == RK_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == reserved0


def test_noalloc_refuses_requests_beyond_its_scratch(lib):
    # V = 128256: 8363 rows fit in 32 MiB, 8364 do not
    import invariant_rl_logprob_gb300 as rk
    V, H = 128256, 64
    assert rk.linear_logp_workspace_size(8363, H, V) <= SCRATCH_BYTES
    assert rk.linear_logp_workspace_size(8364, H, V) > SCRATCH_BYTES
    d = torch.device("cuda:0")
    W = torch.zeros((V, H), dtype=torch.bfloat16, device=d)
    h = torch.zeros((8364, H), dtype=torch.bfloat16, device=d)
    tg = torch.zeros(8364, dtype=torch.int64, device=d)
    logp = torch.empty(8364, dtype=torch.float32, device=d)
    assert call_noalloc(lib, h, W, tg, None, logp, None) == RK_ERR_WORKSPACE
    assert call_noalloc(lib, h[:8363], W, tg[:8363], None, logp[:8363], None) == RK_OK
    torch.cuda.synchronize()
    assert torch.allclose(logp[:8363].cpu(), torch.full((8363,), -float(torch.log(torch.tensor(V * 1.0)))),
                          atol=1e-5)
