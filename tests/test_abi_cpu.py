"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/tpmlp.h declares, and rejects bad arguments on the host before
anything is launched (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")

INVALID, NOT_DIV, UNSUP, WORKSPACE = -1, -2, -3, -4


@pytest.fixture(scope="module")
def lib():
    from sp_partitioned_transformer_gb300 import build

    build.build()
    import sp_partitioned_transformer_gb300 as tpmlp

    return tpmlp.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(tpmlp_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tpmlp_forward", "tpmlp_backward", "tpmlp_split_dim0", "tpmlp_gather_dim0",
              "tpmlp_reduce_scatter_dim0", "tpmlp_workspace_size", "tpmlp_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.tpmlp_abi_version() == 4


def _ws(lib, *a):
    return lib.tpmlp_workspace_size(*a)


def test_layernorm_backward_workspace_formula(lib):
    """2·⌈s·b/8⌉·h float32 partial rows: room for one dγ and one dβ partial per
    CTA of the streamed pass (at most one CTA per 8 tokens)."""
    f = lib.tpmlp_sp_layernorm_backward_workspace
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64] * 3
    assert f(4096, 1, 6144) == 2 * 512 * 6144 * 4
    assert f(9, 1, 5) == 2 * 2 * 5 * 4
    assert f(0, 1, 64) == 0
    assert f(-1, 1, 64) == 0


def test_workspace_size_formula(lib):
    # [s,b,h] = [512,4,1024], f=4096, tp=4, SP, bf16: 512-row sequence chunks are read in
    # place by the GEMMs (all-gather fused into the loads), so no gather buffers ...
    M, h = 512 * 4, 1024
    assert _ws(lib, 512, 4, 1024, 4096, 4, 1, 2, 0, 1) == 0
    # ... and PARTIALS mode needs only the tp float32 partials
    assert _ws(lib, 512, 4, 1024, 4096, 4, 1, 2, 0, 0) == 4 * M * h * 4
    # 96-row chunks (not whole 128-row blocks): gathered X and dZ, each M·h·2 bytes
    M2, h2 = 96 * 2, 136
    g = ((M2 * h2 * 2 + 255) // 256) * 256
    assert _ws(lib, 96, 2, 136, 272, 2, 1, 2, 0, 1) == 2 * g
    # float32 path always gathers
    assert _ws(lib, 512, 4, 1024, 4096, 4, 1, 0, 0, 1) == 2 * M * h * 4
    # SP off, fused: no workspace
    assert _ws(lib, 1024, 8, 3072, 12288, 8, 0, 1, 0, 1) == 0
    # invalid -> 0 with a message
    assert _ws(lib, 16, 2, 64, 250, 4, 0, 0, 0, 1) == 0
    assert b"divisible" in lib.tpmlp_last_error()


def _vp(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


FAKE = 0x10000  # never dereferenced: every case below fails validation first


def _fwd(lib, s=16, b=2, h=64, f=256, tp=2, sp=0, dt=2, act=0, mode=1, x=None, w1=FAKE, w2=FAKE, u=FAKE,
         y=FAKE, z=None, ws=None, ws_bytes=0):
    n = tp if sp else 1
    x = x if x is not None else _vp(*([FAKE] * n))
    z = z if z is not None else _vp(*([FAKE] * n))
    return lib.tpmlp_forward(s, b, h, f, tp, sp, dt, act, mode, x, w1, w2, u, y, z, ws, ws_bytes, None)


def test_forward_rejects_bad_arguments_on_the_host(lib):
    assert _fwd(lib, f=250, tp=4) == NOT_DIV  # f % tp
    assert _fwd(lib, s=15, tp=2, sp=1) == NOT_DIV  # s % tp under SP
    assert b"First dimension" in lib.tpmlp_last_error()
    assert _fwd(lib, tp=0) == INVALID
    assert _fwd(lib, tp=65) == INVALID
    assert _fwd(lib, dt=7) == INVALID
    assert _fwd(lib, act=9) == INVALID
    assert _fwd(lib, mode=5) == INVALID
    assert _fwd(lib, h=0) == INVALID
    assert _fwd(lib, s=-1) == INVALID
    assert _fwd(lib, w1=None) == INVALID
    assert _fwd(lib, z=_vp(None)) == INVALID
    assert _fwd(lib, h=60) == UNSUP  # tensor-core path: h % 8
    assert _fwd(lib, f=2 * 12, tp=2) == UNSUP  # f/tp = 12, not a multiple of 8
    assert _fwd(lib, w2=FAKE + 2) == UNSUP  # 16-byte alignment of the tensor-core path
    assert _fwd(lib, dt=0, w2=FAKE + 2) == INVALID  # float32 path wants 4-byte alignment
    # SP needs workspace for the gathered input
    assert _fwd(lib, sp=1, ws=None, ws_bytes=0) == WORKSPACE
    assert _fwd(lib, sp=1, ws=FAKE, ws_bytes=100) == WORKSPACE
    assert b"workspace" in lib.tpmlp_last_error()
    assert _fwd(lib, mode=0, ws=FAKE + 16, ws_bytes=1 << 30) == UNSUP  # ws must be 256-byte aligned


def test_forward_workspace_leaves_out_the_backward_dz_slot(lib):
    """The forward gathers only X: its workspace is the gathered X (when SP
    chunks are not whole 128-row blocks) plus, in PARTIALS mode, the tp float32
    partials; the backward also gathers dZ.  (That tpmlp_forward runs on
    exactly the forward's size is checked on the GPU, by the allocation-free
    forward whose built-in scratch sits between the two sizes.)"""
    fws = lib.tpmlp_forward_workspace_size
    fws.restype = ctypes.c_size_t
    fws.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int] * 5
    M, h = 96 * 2, 136
    g = ((M * h * 2 + 255) // 256) * 256
    p = 2 * M * h * 4
    assert fws(96, 2, 136, 272, 2, 1, 2, 0, 1) == g
    assert _ws(lib, 96, 2, 136, 272, 2, 1, 2, 0, 1) == 2 * g
    assert fws(96, 2, 136, 272, 2, 1, 2, 0, 0) == g + p
    assert _ws(lib, 96, 2, 136, 272, 2, 1, 2, 0, 0) == 2 * g + p
    assert fws(512, 4, 1024, 4096, 4, 1, 2, 0, 1) == 0  # chunks read in place
    assert fws(16, 2, 64, 250, 4, 0, 0, 0, 1) == 0  # invalid -> 0
    # one byte less than the forward's size is refused before anything runs
    assert _fwd(lib, s=96, b=2, h=136, f=272, sp=1, ws=FAKE * 256, ws_bytes=g - 1) == WORKSPACE
    assert str(g).encode() in lib.tpmlp_last_error()


def test_backward_and_dim0_ops_reject_bad_arguments(lib):
    vp1 = _vp(FAKE)
    rc = lib.tpmlp_backward(16, 2, 64, 256, 2, 0, 2, 0, 1, vp1, FAKE, FAKE, FAKE, FAKE, vp1, _vp(None), FAKE,
                            FAKE, FAKE, None, 0, None)
    assert rc == INVALID
    rc = lib.tpmlp_backward(16, 2, 64, 256, 3, 0, 2, 0, 1, vp1, FAKE, FAKE, FAKE, FAKE, vp1, vp1, FAKE, FAKE,
                            FAKE, None, 0, None)
    assert rc == NOT_DIV
    assert lib.tpmlp_split_dim0(FAKE, _vp(FAKE, FAKE, FAKE), 10, 1, 8, 3, 2, None) == NOT_DIV
    assert lib.tpmlp_gather_dim0(_vp(FAKE, None), FAKE, 10, 1, 8, 2, 2, None) == INVALID
    assert lib.tpmlp_reduce_scatter_dim0(FAKE, _vp(FAKE), 10, 1, 8, 3, 1, 2, None) == NOT_DIV
    assert lib.tpmlp_reduce_scatter_dim0(FAKE, _vp(FAKE), 10, 1, 8, 3, 2, 2, None) == INVALID
    assert lib.tpmlp_wait_timeout_selftest(0, None) == INVALID


def test_binding_refuses_to_run_without_the_library(tmp_path):
    import sp_partitioned_transformer_gb300 as tpmlp

    saved = tpmlp._lib
    tpmlp._lib = None
    try:
        with pytest.raises(ImportError):
            tpmlp.load(str(tmp_path / "missing.so"))
    finally:
        tpmlp._lib = saved


def _attn_fwd(lib, s=256, b=1, h=256, heads=2, tp=2, sp=1, dt=2, causal=0, wqkv=FAKE, lse=FAKE, ws=None,
              ws_bytes=0, kv=None):
    n = tp if sp else 1
    x = _vp(*([FAKE] * n))
    z = _vp(*([FAKE] * n))
    f = lib.tpmlp_attn_forward
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 7 + [ctypes.c_void_p,
                                                                                       ctypes.c_size_t,
                                                                                       ctypes.c_void_p]
    return f(s, b, h, heads, heads if kv is None else kv, tp, sp, dt, causal, x, wqkv, FAKE, FAKE, FAKE, lse, z, ws,
             ws_bytes, None)


def test_attention_rejects_bad_arguments_on_the_host(lib):
    assert _attn_fwd(lib, heads=3, h=384, tp=2) == NOT_DIV  # heads % tp
    assert b"heads" in lib.tpmlp_last_error()
    assert _attn_fwd(lib, s=255) == NOT_DIV  # s % tp under SP
    assert _attn_fwd(lib, h=320) == UNSUP  # head width 160: only 128 and 96
    assert _attn_fwd(lib, h=128, heads=2) == UNSUP  # head width 64
    assert _attn_fwd(lib, heads=4, h=512, kv=3) == NOT_DIV  # heads % kv_heads
    assert b"kv heads" in lib.tpmlp_last_error()
    assert _attn_fwd(lib, heads=4, h=512, kv=1, tp=2) == NOT_DIV  # kv_heads % tp: a shard needs whole groups
    assert b"query groups" in lib.tpmlp_last_error()
    assert _attn_fwd(lib, heads=4, h=512, kv=0) == INVALID
    assert _attn_fwd(lib, heads=4, h=512, kv=8) == INVALID
    assert _attn_fwd(lib, dt=0) == UNSUP  # float32 storage
    assert _attn_fwd(lib, causal=2) == INVALID
    assert _attn_fwd(lib, tp=0) == INVALID
    assert _attn_fwd(lib, wqkv=None) == INVALID
    assert _attn_fwd(lib, lse=FAKE + 4) == UNSUP  # 16-byte alignment
    # 96-row chunks (s/tp·b = 96) are gathered through the workspace
    assert _attn_fwd(lib, s=192, ws=None) == WORKSPACE
    assert b"workspace" in lib.tpmlp_last_error()


def test_attention_workspace_formula(lib):
    f = lib.tpmlp_attn_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int] * 6

    def a256(x):
        return (x + 255) // 256 * 256

    def ds_tiles(s, causal):
        """16 KB dSᵀ tiles per (sequence, query head): key tile kt visits the
        64-query tiles from 2·kt (causal) or 0 to the last, counted here one by one."""
        nk, nq = -(-s // 128), -(-s // 64)
        return sum(nq - (2 * kt if causal else 0) for kt in range(nk))

    # 128-row chunks read in place: Δ and −lse2, each [b][heads][s_pad] float32, then dSᵀ
    for causal in (0, 1):
        assert f(256, 1, 256, 2, 2, 2, 1, 2, causal) == a256(2 * 1 * 2 * 256 * 4) + 2 * ds_tiles(256, causal) * 16384
    # 96-row chunks: gathered X and dZ, then Δ and −lse2 (s_pad = 256), then dSᵀ
    assert f(192, 1, 256, 2, 2, 2, 1, 2, 1) == (2 * a256(192 * 256 * 2) + a256(2 * 2 * 256 * 4)
                                                + 2 * ds_tiles(192, True) * 16384)
    # ragged s = 100 (one key tile, two query tiles), b = 3, 2 heads, no SP
    assert f(100, 3, 256, 2, 2, 1, 0, 2, 1) == a256(2 * 3 * 2 * 128 * 4) + 3 * 2 * 2 * 16384
    assert ds_tiles(4096, True) == 1056 and ds_tiles(4096, False) == 2048
    # grouped-query attention: the per-query-head statistics and dSᵀ tiles do not
    # depend on the number of key/value heads; the dK/dV partials of the r query
    # heads of every group follow, float32 [r][s·b][kv_heads][2][d]
    r, kv, d = 2, 2, 128
    assert f(256, 1, 512, 4, kv, 2, 1, 2, 1) == f(256, 1, 512, 4, 4, 2, 1, 2, 1) + r * 256 * kv * 2 * d * 4
    # head width 96 (h = 96·heads) is accepted and sized like 128
    assert f(256, 1, 384, 4, 4, 2, 1, 2, 1) == f(256, 1, 512, 4, 4, 2, 1, 2, 1)
    assert f(192, 1, 320, 2, 2, 2, 1, 2, 0) == 0  # invalid (head width 160) -> 0
    assert f(192, 1, 256, 2, 2, 2, 1, 2, 2) == 0  # invalid causal flag -> 0
    assert f(192, 1, 512, 4, 3, 2, 1, 2, 0) == 0  # kv_heads does not divide heads -> 0
