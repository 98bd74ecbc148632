"""The C-ABI library builds, loads and exports every symbol include/rk.h
declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(rk_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from invariant_rl_logprob_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_operators():
    names = declared_symbols()
    for n in ("rk_linear_logp", "rk_logp_from_logits", "rk_linear_logp_bwd",
              "rk_linear_logp_workspace_size", "rk_linear_logp_bwd_workspace_size",
              "rk_get_device_error", "rk_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls(lib):
    lib.rk_status_string.restype = ctypes.c_char_p
    lib.rk_status_string.argtypes = [ctypes.c_int]
    assert lib.rk_status_string(0) == b"RK_OK"
    assert lib.rk_status_string(3) == b"RK_ERR_WORKSPACE"
    lib.rk_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.rk_version()
    lib.rk_linear_logp_workspace_size.restype = ctypes.c_size_t
    lib.rk_linear_logp_workspace_size.argtypes = [ctypes.c_int64] * 3
    f = lib.rk_linear_logp_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64] * 3
    # T rows x ceil(V/256) tiles x 8 bytes + T x 4 bytes + one live flag per
    # 256 rows, each rounded to 256, + 256 bytes for the tile counter
    assert f(8192, 4096, 128256) == 8192 * 501 * 8 + 8192 * 4 + 256 + 256
    assert f(100, 64, 1001) == 256 * ((100 * 4 * 8 + 255) // 256) + 512 + 256 + 256
    assert f(0, 4096, 128256) == 0
    g = lib.rk_linear_logp_bwd_workspace_size
    g.restype = ctypes.c_size_t
    g.argtypes = [ctypes.c_int64] * 3
    # tile counter, then per 128-row chunk: entry counts, entry lists
    # (65 slots of 8 bytes), dZ, a live flag per 256 rows; each part rounded
    # to 256 bytes
    assert g(100, 64, 1001) == 256 + 512 + 128 * 65 * 8 + 128 * 1008 * 2 + 256


def test_argument_errors_return_before_any_launch(lib):
    # invalid sizes are rejected on the host, without touching a device
    f = lib.rk_linear_logp
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int32] + [ctypes.c_int64] * 3 + \
        [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]
    assert f(None, None, None, None, 0, -1, 64, 10, None, None, None, 0, None) == 1
    assert f(None, None, None, None, 0, 0, 64, 10, None, None, None, 0, None) == 0   # T = 0
    assert f(None, None, None, None, 0, 4, 64, 10, None, None, None, 0, None) == 1   # NULL h
    g = lib.rk_logp_from_logits
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int32] + [ctypes.c_int64] * 2 + \
        [ctypes.c_void_p] * 3
    assert g(None, None, None, 0, 5, 0, None, None, None) == 1                         # V = 0


def test_argument_errors_of_the_widened_rows(lib):
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lh = lib.rk_lm_head
    lh.restype = ctypes.c_int
    lh.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, sz, vp]
    assert lh(None, None, -1, 64, 10, None, 16, None, 0, None) == 1   # T < 0
    assert lh(None, None, 0, 64, 10, None, 16, None, 0, None) == 0    # T = 0: nothing to do
    fake = ctypes.c_void_p(4096)                                       # never dereferenced
    assert lh(fake, fake, 4, 64, 10, fake, 8, None, 0, None) == 1     # ld < V
    assert lh(fake, fake, 4, 96, 10, fake, 16, None, 0, None) == 2    # H % 64 != 0
    assert lh(fake, fake, 4, 64, 10, fake, 16, fake, 8, None) == 3    # workspace too small
    lws = lib.rk_lm_head_workspace_size
    lws.restype = sz
    assert lws() == 256
    gl = lib.rk_grpo_token_loss
    gl.restype = ctypes.c_int
    gl.argtypes = [vp] * 6 + [i32, i64, f32, f32, f32, f32] + [vp] * 5
    assert gl(fake, fake, None, fake, fake, None, 0, 8, 1.5, 0.2, 0.0, 1.0, fake, fake, None, None, None) == 1
    assert gl(fake, fake, None, fake, fake, None, 0, 8, 0.2, 0.2, -1.0, 1.0, fake, fake, None, None, None) == 1
    assert gl(fake, None, None, fake, fake, None, 0, 8, 0.2, 0.2, 0.0, 1.0, fake, fake, None, None, None) == 1
    dw = lib.rk_linear_logp_dw
    dw.restype = ctypes.c_int
    dw.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, i64, vp, vp, sz, vp]
    assert dw(fake, fake, fake, None, 0, 8, 64, 100, fake, fake, fake, -1, fake, fake, 1 << 30, None) == 1
    assert dw(fake, fake, fake, None, 0, 8, 64, 100, fake, fake, None, 0, fake, None, 0, None) == 3
    q = lib.rk_linear_logp_dw_workspace_size
    q.restype = sz
    q.argtypes = [i64, i64, i64]
    assert q(0, 64, 100) == 0 and q(100, 64, 1000) > 100 * 1008 * 2
    qf = lib.rk_linear_logp_bwd_full_workspace_size
    qf.restype = sz
    qf.argtypes = [i64, i64, i64]
    # the full backward holds dZ^T [V, round_up(n, 8)] bf16 beside the dW buffers
    assert qf(0, 64, 100) == 0
    assert qf(100, 64, 1000) >= q(100, 64, 1000) + 1000 * 104 * 2
    gr = lib.rk_linear_greedy
    gr.restype = ctypes.c_int
    gr.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, sz, vp]
    assert gr(fake, fake, None, 0, 8, 64, 100, fake, fake, None, None, 0, None) == 3
    st = lib.rk_selftest_wait_timeout
    st.restype = ctypes.c_int
    st.argtypes = [i64, vp]
    assert st(0, None) == 1 and st(20_000_000_000, None) == 1
    # the forward that keeps its softmax terms and the backwards from them:
    # argument errors found on the host
    ss = lib.rk_linear_logp_saved_size
    ss.restype, ss.argtypes = sz, [i64, i64, i64]
    # the forward workspace, then the terms: round_up(V, 8) bf16 per row
    assert ss(100, 64, 1001) == lib.rk_linear_logp_workspace_size(100, 64, 1001) + \
        ((100 * 1008 * 2 + 255) // 256) * 256
    assert ss(0, 64, 1001) == 0
    fs = lib.rk_linear_logp_fwd_saved
    fs.restype = ctypes.c_int
    fs.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, sz, vp]
    assert fs(fake, fake, fake, None, 0, 8, 64, 100, fake, None, None, 0, None) == 3   # no state
    assert fs(fake, fake, fake, None, 0, 8, 64, 100, fake, None, ctypes.c_void_p(4096 + 16),
              1 << 30, None) == 1                                               # misaligned
    bs = lib.rk_linear_logp_bwd_saved
    bs.restype = ctypes.c_int
    bs.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, sz, vp, vp, sz, vp]
    assert bs(fake, fake, fake, None, 0, 8, 96, 100, fake, fake, fake, 1 << 30, fake, fake,
              1 << 30, None) == 2                                               # H % 64 != 0
    assert bs(fake, fake, fake, None, 0, 8, 64, 100, fake, fake, fake, 16, fake, fake,
              1 << 30, None) == 3                                               # state too small
    bws = lib.rk_linear_logp_bwd_saved_workspace_size
    bws.restype, bws.argtypes = sz, [i64, i64, i64]
    assert bws(100, 64, 1001) == 256 + 512 + ((100 * 65 * 8 + 255) // 256) * 256
    gp = lib.rk_linear_logp_grpo
    gp.restype = ctypes.c_int
    gp.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, f32, f32, f32, f32] + [vp] * 6 + \
        [vp, sz, vp]
    assert gp(fake, fake, fake, None, 0, 8, 64, 100, fake, None, fake, 1.5, 0.2, 0.0, 1.0,
              fake, None, fake, fake, None, None, fake, 1 << 30, None) == 1     # eps_low >= 1
    # the dh / dW GEMM form: host-side setting and query only
    sr, lr = lib.rk_set_row_blocks, lib.rk_last_row_blocks
    sr.restype, sr.argtypes = ctypes.c_int, [i32]
    lr.restype, lr.argtypes = i32, [i32]
    assert sr(3) == 1 and sr(-1) == 1
    assert sr(2) == 0 and sr(1) == 0 and sr(0) == 0
    assert lr(0) == 0 and lr(1) == 0 and lr(2) == -1    # no GEMM launched in this thread
    lt = lib.rk_last_tile_order
    lt.restype, lt.argtypes = i32, [i32]
    assert lt(0) == 0 and lt(1) == 0 and lt(-1) == -1
