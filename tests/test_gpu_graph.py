"""The operators inside CUDA graphs.

Every call is stream-ordered, allocates no device memory inside the library
and never synchronises the host, so a step captured once replays with the bits
of the eager calls: a training loop can capture its logprob step, a serving
loop its greedy decode step."""
import pytest
import torch

from invariant_rl_logprob_gb300 import synth
from tests.helpers import DEV, cuda, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rk():
    from invariant_rl_logprob_gb300 import build
    build.build()
    import invariant_rl_logprob_gb300 as m
    m.load_library()
    m.get_device_error()
    return m


def _capture(fn, stream):
    # warm-up on the capture stream (kernel attributes, occupancy queries),
    # then capture
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    return graph


def test_grpo_step_graph_replays_eager_bits(rk):
    H, V = 256, 3000
    p1 = synth.make_pool(H, V, [300, 212, 97], seed=71, with_grad=True)
    p2 = synth.make_pool(H, V, [300, 212, 97], seed=72, with_grad=True, W=p1.W)
    T = p1.h.shape[0]
    W = cuda(p1.W)
    h, tg, g = cuda(p1.h), cuda(p1.targets), cuda(p1.g)
    z, zt, _ = synth.logits_batch(T=64, V=V, seed=5)
    z, zt = cuda(z), cuda(zt)
    logp = torch.empty(T, device=DEV)
    lse = torch.empty(T, device=DEV)
    saved = torch.empty(rk.linear_logp_saved_size(T, H, V), dtype=torch.uint8, device=DEV)
    ws = torch.empty(rk.linear_logp_bwd_saved_workspace_size(T, H, V), dtype=torch.uint8,
                     device=DEV)
    dh = torch.empty((T, H), device=DEV)
    zl = torch.empty(64, device=DEV)
    zs = torch.empty(64, device=DEV)
    cs = torch.cuda.Stream()

    def step():
        rk.linear_logp_fwd_saved(h, W, tg, out=logp, lse=lse, saved=saved, stream=cs)
        rk.linear_logp_bwd_saved(h, W, tg, lse, g, saved, dh=dh, workspace=ws, stream=cs)
        rk.logp_from_logits(z, zt, out=zl, lse=zs, stream=cs)

    graph = _capture(step, cs)
    for pool in (p1, p2):  # new inputs copied into the captured buffers
        h.copy_(cuda(pool.h))
        tg.copy_(cuda(pool.targets))
        g.copy_(cuda(pool.g))
        torch.cuda.synchronize()
        with torch.cuda.stream(cs):
            graph.replay()
        cs.synchronize()
        he, te = cuda(pool.h), cuda(pool.targets)
        lp_e, ls_e, sv = rk.linear_logp_fwd_saved(he, W, te)
        dh_e = rk.linear_logp_bwd_saved(he, W, te, ls_e, cuda(pool.g), sv)
        assert same_bits(logp, lp_e) and same_bits(lse, ls_e)
        assert same_bits(dh, dh_e)
    zl_e, zs_e = rk.logp_from_logits(z, zt)
    assert same_bits(zl, zl_e) and same_bits(zs, zs_e)
    assert rk.get_device_error() == 0


def test_greedy_decode_graph_replays_eager_bits(rk):
    # one new token for each of 64 sequences
    H, V = 512, 5000
    pool = synth.make_pool(H, V, [64], seed=73)
    W, h = cuda(pool.W), cuda(pool.h)
    ws = torch.empty(rk.linear_greedy_workspace_size(64, H, V), dtype=torch.uint8, device=DEV)
    cs = torch.cuda.Stream()
    out = {}

    def step():
        out["tok"], out["logp"], out["lse"] = rk.linear_greedy(h, W, workspace=ws, stream=cs)

    graph = _capture(step, cs)
    h2 = cuda(synth.make_pool(H, V, [64], seed=74, W=pool.W).h)
    for src in (h.clone(), h2):
        h.copy_(src)
        torch.cuda.synchronize()
        with torch.cuda.stream(cs):
            graph.replay()
        cs.synchronize()
        tok, lp, ls = rk.linear_greedy(src, W)
        assert torch.equal(out["tok"], tok)
        assert same_bits(out["logp"], lp) and same_bits(out["lse"], ls)
    assert rk.get_device_error() == 0


@pytest.mark.parametrize("blocks", [1, 2])
def test_rounds_and_counter_tile_orders_agree(rk, blocks):
    # V = 16384: the dh GEMM's K loop has 256 stages, so an eager call takes
    # its tiles in rounds (a cooperative launch; 128 one-block tiles are two
    # rounds of the resident pairs); inside a graph capture the same GEMM
    # takes them from the counter.  Same bits, in either tile form.
    H, V = 2048, 16384
    pool = synth.make_pool(H, V, [1500, 1000, 1596], seed=75, with_grad=True)
    T = pool.h.shape[0]
    W, h, tg, g = cuda(pool.W), cuda(pool.h), cuda(pool.targets), cuda(pool.g)
    _, lse = rk.linear_logp(h, W, tg)
    rk.set_row_blocks(blocks)
    try:
        dh_rounds = rk.linear_logp_bwd(h, W, tg, lse, g)
        assert rk.last_row_blocks("dh") == blocks
        if rk.last_tile_order("dh") != 2:
            pytest.skip("the device refused the cooperative launch: tiles came from the counter")
        ws = torch.empty(rk.linear_logp_bwd_workspace_size(T, H, V), dtype=torch.uint8,
                         device=DEV)
        dh = torch.empty((T, H), device=DEV)
        cs = torch.cuda.Stream()
        graph = _capture(lambda: rk.linear_logp_bwd(h, W, tg, lse, g, dh=dh, workspace=ws,
                                                    stream=cs), cs)
        assert rk.last_tile_order("dh") == 1
    finally:
        rk.set_row_blocks(0)
    dh.fill_(float("nan"))
    with torch.cuda.stream(cs):
        graph.replay()
    cs.synchronize()
    assert same_bits(dh, dh_rounds)
    assert rk.get_device_error() == 0
