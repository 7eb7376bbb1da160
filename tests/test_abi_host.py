"""The C-ABI library on the host: it loads, exports every call include/mhc.h declares, and its
argument validation rejects bad calls before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mhc.h")


@pytest.fixture(scope="module")
def M():
    from stream_residual_fusion_gb300 import build
    build.build()
    import stream_residual_fusion_gb300.mhc as m
    return m


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mhc_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(M):
    names = _declared()
    assert "mhc_fused_step" in names and "mhc_rmsnorm" in names
    lib = ctypes.CDLL(M.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), f"{name} declared but not exported"
        assert name in M.SIGNATURES, f"{name} has no binding signature"


def test_status_codes_match_header(M):
    text = open(HEADER).read()
    codes = dict((k, int(v)) for k, v in re.findall(r"#define (MHC_[A-Z_]+)\s+(-?\d+)\b", text))
    for k, v in codes.items():
        if hasattr(M, k):
            assert getattr(M, k) == v
    for code in range(-7, 1):
        assert M.lib.mhc_strerror(code)
    assert M.lib.mhc_strerror(-99) == b"unknown status code"


def test_sizes(M):
    B = M.lib.mhc_packed_block_columns()
    assert B in (16, 32, 64)
    # d/B blocks x 4 streams x 80 rows (72 = 3 planes x 24 mix rows, 8 zero) x B bf16
    assert M.lib.mhc_packed_weights_bytes(4, 5120) == (5120 // B) * 4 * 80 * B * 2
    assert M.lib.mhc_packed_weights_bytes(4, B + 8) == 0
    assert M.lib.mhc_workspace_bytes(4, 5120) >= M.lib.mhc_packed_weights_bytes(4, 5120)
    assert M.lib.mhc_packed_weights_bytes(3, 5120) == 0


# Fake device addresses: validation runs before any CUDA call, so these are never dereferenced.
A = 1 << 32


def _addr(i):
    return ctypes.c_void_p(A + i * (1 << 28))


def _fused(M, N=256, n=4, d=5120, iters=20, flags=0, ptrs=None, ws=None, ws_bytes=None):
    p = [_addr(i) for i in range(15)] if ptrs is None else ptrs
    ws = _addr(20) if ws is None else ws
    wsb = M.lib.mhc_workspace_bytes(4, 5120) if ws_bytes is None else ws_bytes
    return M.lib.mhc_fused_step(*p, N, n, d, iters, 1e-6, 1e-6, flags, ws, wsb, None)


def test_fused_validation(M):
    assert _fused(M, n=3) == M.MHC_ERR_SHAPE
    assert _fused(M, N=-1) == M.MHC_ERR_SHAPE
    assert _fused(M, iters=0) == M.MHC_ERR_SHAPE
    assert _fused(M, d=5000) == M.MHC_ERR_SHAPE          # not a multiple of the tile width (16*8)
    assert _fused(M, d=24576) == M.MHC_ERR_SHAPE         # over 640 columns per CTA even at split 32
    assert _fused(M, N=0, d=8192) == M.MHC_OK            # 16 CTAs of 512 columns
    assert _fused(M, flags=7 << 8) == M.MHC_ERR_SHAPE    # split 64 is not offered
    assert _fused(M, flags=M.split_flag(4)) == M.MHC_ERR_SHAPE   # 1280 columns per CTA: too wide
    assert _fused(M, N=0, flags=M.split_flag(16)) == M.MHC_OK    # 320 columns per CTA
    assert _fused(M, N=0, flags=M.split_flag(32)) == M.MHC_OK    # 160 columns: 5 slots
    assert _fused(M, flags=M.split_flag(32) | M.tile_flag(16)) == M.MHC_ERR_SHAPE  # 16 % 32 != 0
    assert _fused(M, flags=M.split_flag(16) | M.tile_flag(8)) == M.MHC_ERR_SHAPE  # 8 % 16 != 0
    assert _fused(M, N=0, d=4096, flags=M.split_flag(32)) == M.MHC_OK        # 128 columns per CTA
    assert [M.split_flag(v) >> 8 for v in (0, 1, 2, 4, 8, 16, 32)] == [0, 1, 2, 3, 4, 5, 6]
    assert _fused(M, flags=17 << 16) == M.MHC_ERR_SHAPE   # tile of 136 tokens: over 128
    assert _fused(M, N=0, flags=M.tile_flag(96)) == M.MHC_OK
    assert M.tile_flag(96) == 12 << 16
    assert _fused(M, flags=M.split_flag(1)) == M.MHC_ERR_SHAPE   # 5120 columns do not fit one CTA
    p = [_addr(i) for i in range(15)]
    p[0] = ctypes.c_void_p(A + 8)
    assert _fused(M, ptrs=p) == M.MHC_ERR_ALIGN
    p = [_addr(i) for i in range(15)]
    p[1] = None
    assert _fused(M, ptrs=p) == M.MHC_ERR_NULL
    assert _fused(M, ws=ctypes.c_void_p(0)) == M.MHC_ERR_WORKSPACE
    assert _fused(M, ws_bytes=100) == M.MHC_ERR_WORKSPACE
    p = [_addr(i) for i in range(15)]
    p[10] = ctypes.c_void_p(p[1].value + 4096)          # y_out inside F
    assert _fused(M, ptrs=p) == M.MHC_ERR_ALIAS
    p = [_addr(i) for i in range(15)]
    p[9] = p[0]                                          # X_out == X: in place is allowed
    assert _fused(M, N=0, ptrs=p) == M.MHC_OK
    p = [_addr(i) for i in range(15)]
    p[9] = ctypes.c_void_p(p[0].value + 16)              # partial overlap is not
    assert _fused(M, ptrs=p) == M.MHC_ERR_ALIAS
    assert _fused(M, ws=p[3]) == M.MHC_ERR_ALIAS         # workspace over an input
    assert _fused(M, N=0) == M.MHC_OK                    # nothing to do, nothing launched


def _mx(M, N=256, d=5120, ptrs=None):
    p = [_addr(i) for i in range(16)] if ptrs is None else ptrs
    return M.lib.mhc_fused_step_mxfp8(*p, N, 4, d, 20, 1e-6, 1e-6, 0, _addr(21), 1 << 26, None)


def test_mxfp8_validation(M):
    """The MXFP8-y entry: its scale pointer is required and aligned, and the codes take one byte
    per element when overlaps are checked (host-side checks, before any device call)."""
    assert _mx(M, N=0) == M.MHC_OK
    p = [_addr(i) for i in range(16)]
    p[11] = None                                         # y_scale
    assert _mx(M, ptrs=p) == M.MHC_ERR_NULL
    p = [_addr(i) for i in range(16)]
    p[11] = ctypes.c_void_p(p[11].value + 4)
    assert _mx(M, ptrs=p) == M.MHC_ERR_ALIGN
    N, d = 256, 5120
    p = [_addr(i) for i in range(16)]
    p[11] = ctypes.c_void_p(p[10].value + N * d - 16)     # scales inside the codes
    assert _mx(M, ptrs=p) == M.MHC_ERR_ALIAS
    p = [_addr(i) for i in range(16)]
    p[11] = ctypes.c_void_p(p[10].value + N * d)          # right after them: no overlap
    assert _mx(M, ptrs=p) != M.MHC_ERR_ALIAS
    p = [_addr(i) for i in range(16)]
    p[12] = ctypes.c_void_p(p[11].value + N * d // 32 - 16)   # pre_out inside the scales
    assert _mx(M, ptrs=p) == M.MHC_ERR_ALIAS
    p = [_addr(i) for i in range(16)]
    p[10] = ctypes.c_void_p(p[1].value - N * d)           # codes end where F begins
    assert _mx(M, ptrs=p) != M.MHC_ERR_ALIAS


def test_split_choices(M):
    B = M.lib.mhc_packed_block_columns()
    # d/split a multiple of 32 (whole pipeline slots) in [128, 640] for some split <= 32
    ok = {4 * B: M.MHC_OK, 160: M.MHC_OK, 256: M.MHC_OK, 512: M.MHC_OK, 640: M.MHC_OK,
          704: M.MHC_OK, 1024: M.MHC_OK, 2048: M.MHC_OK, 5120: M.MHC_OK, 5632: M.MHC_OK,
          6144: M.MHC_OK, 7168: M.MHC_OK, 20480: M.MHC_OK,
          2 * B: M.MHC_ERR_SHAPE, 100: M.MHC_ERR_SHAPE, 24576: M.MHC_ERR_SHAPE,
          20992: M.MHC_ERR_SHAPE, 5000: M.MHC_ERR_SHAPE}
    for d, want in ok.items():
        assert _fused(M, N=0, d=d, ws_bytes=1 << 40) == want, d


def test_other_calls_validation(M):
    p = [_addr(i) for i in range(8)]
    lib = M.lib
    assert lib.mhc_sinkhorn(*p[:6], 10, 4, 0, 1e-6, None) == M.MHC_ERR_SHAPE
    assert lib.mhc_sinkhorn(*p[:6], 0, 4, 20, 1e-6, None) == M.MHC_OK
    assert lib.mhc_sinkhorn(None, *p[1:6], 10, 4, 20, 1e-6, None) == M.MHC_ERR_NULL
    assert lib.mhc_sinkhorn(None, *p[1:6], 0, 4, 20, 1e-6, None) == M.MHC_OK  # empty: no address needed
    assert lib.mhc_rmsnorm(*p[:3], 10, 100, 1e-6, None) == M.MHC_ERR_SHAPE
    assert lib.mhc_rmsnorm(p[0], p[1], p[0], 0, 128, 1e-6, None) == M.MHC_OK   # in place
    q = [ctypes.c_void_p(A + 4), p[1], p[2]]
    assert lib.mhc_rmsnorm(*q, 10, 128, 1e-6, None) == M.MHC_ERR_ALIGN
    assert lib.mhc_hc_post(*p[:5], 10, 2, 128, 0, None) == M.MHC_ERR_SHAPE
    assert lib.mhc_hc_pre(p[0], p[1], ctypes.c_void_p(p[0].value + 32), 10, 4, 128, None) == M.MHC_ERR_ALIAS
    assert lib.mhc_pack_weights(p[0], ctypes.c_void_p(p[0].value + 64), 4, 128, None) == M.MHC_ERR_ALIAS
    assert lib.mhc_pack_weights(p[0], p[1], 4, 8, None) == M.MHC_ERR_SHAPE
    assert lib.mhc_mixes(*p[:8], 10, 4, 5120, 20, 1e-6, 1e-6, 0, None, 0, None) == M.MHC_ERR_WORKSPACE
    assert lib.mhc_mixes(*p[:8], 0, 4, 5120, 20, 1e-6, 1e-6, 0, p[7], 1 << 30, None) == M.MHC_OK


def _host(M, N=256, n=4, d=5120, iters=20, flags=0, ptrs=None, staging=None, nbytes=1 << 40,
          chunk=128):
    p = [_addr(i) for i in range(15)] if ptrs is None else ptrs
    st = _addr(20) if staging is None else staging
    return M.lib.mhc_fused_step_host(*p, N, n, d, iters, 1e-6, 1e-6, flags, st, nbytes, chunk,
                                     None)


def test_host_pipeline_validation(M):
    lib = M.lib
    assert _host(M, chunk=0) == M.MHC_ERR_SHAPE
    assert _host(M, n=3) == M.MHC_ERR_SHAPE
    assert _host(M, N=-1) == M.MHC_ERR_SHAPE
    assert _host(M, d=5000) == M.MHC_ERR_SHAPE           # the device step's shape rules
    assert _host(M, iters=0) == M.MHC_ERR_SHAPE
    assert _host(M, N=0) == M.MHC_OK
    p = [_addr(i) for i in range(15)]
    p[5] = None                                          # W_mix
    assert _host(M, ptrs=p) == M.MHC_ERR_NULL
    p = [_addr(i) for i in range(15)]
    p[10] = ctypes.c_void_p(p[1].value + 4096)           # host y_out inside host F
    assert _host(M, ptrs=p) == M.MHC_ERR_ALIAS
    p = [_addr(i) for i in range(15)]
    p[14] = ctypes.c_void_p(p[13].value + 64)            # mixes_out over comb_out
    assert _host(M, ptrs=p) == M.MHC_ERR_ALIAS
    assert _host(M, staging=ctypes.c_void_p(0)) == M.MHC_ERR_WORKSPACE
    need = lib.mhc_host_staging_bytes(4, 5120, 128, 1)
    assert need > 0 and lib.mhc_host_staging_bytes(4, 5120, 0, 1) == 0
    assert lib.mhc_host_staging_bytes(4, 5120, 128, 0) < need
    assert _host(M, nbytes=need - 1) == M.MHC_ERR_WORKSPACE
    assert _host(M, staging=ctypes.c_void_p(A + 16)) == M.MHC_ERR_ALIGN
    # three staging slots of 128 tokens, each at least the tokens' inputs and outputs
    assert need >= M.lib.mhc_workspace_bytes(4, 5120) + 3 * 128 * (2 * 51200 + 2 * 96 + 96)


def _chunks_by_definition(N, c):
    """The chunk rule as the header states it, written out."""
    r = [c // 8, c // 4, c // 2]
    if c >= 8 and N >= 2 * sum(r) + c:
        mid = N - 2 * sum(r)
        return r + [c] * (mid // c) + ([mid % c] if mid % c else []) + r[::-1]
    return [c] * (N // c) + ([N % c] if N % c else [])


def test_host_chunk_plan(M):
    assert M.lib.mhc_host_chunks(-1, 8, None, 0) == M.MHC_ERR_SHAPE
    assert M.lib.mhc_host_chunks(10, 0, None, 0) == M.MHC_ERR_SHAPE
    assert M.host_chunks(0, 128) == []
    assert M.host_chunks(1500, 256) == [32, 64, 128, 256, 256, 256, 256, 28, 128, 64, 32]
    assert M.host_chunks(703, 256) == [256, 256, 191]
    assert M.host_chunks(704, 256) == [32, 64, 128, 256, 128, 64, 32]
    for N in list(range(0, 300)) + [4095, 4096, 32768, 131072, 10**9 + 7]:
        for c in (1, 2, 7, 8, 9, 100, 128, 2048):
            if N // c > 5000:
                continue
            got = M.host_chunks(N, c)
            assert got == _chunks_by_definition(N, c), (N, c)
            assert sum(got) == N and all(1 <= x <= c for x in got)
    buf = (ctypes.c_int64 * 2)()
    assert M.lib.mhc_host_chunks(1500, 256, buf, 2) == 11 and list(buf) == [32, 64]


def _bwd(M, N=256, n=4, d=5120, iters=20, flags=0, ptrs=None, ws=None, ws_bytes=1 << 40):
    p = [_addr(i) for i in range(25)] if ptrs is None else ptrs
    ws = _addr(30) if ws is None else ws
    return M.lib.mhc_fused_step_backward(*p, N, n, d, iters, 1e-6, 1e-6, flags, ws, ws_bytes,
                                         None)


def test_backward_validation(M):
    """mhc_fused_step_backward checks its arguments on the host before anything runs: shapes
    (n = 4, d a multiple of 64, N >= 0, iters >= 1), flags, NULL and unaligned pointers, the
    workspace, and overlap of any output with an input or another output."""
    assert _bwd(M, n=3) == M.MHC_ERR_SHAPE
    assert _bwd(M, N=-1) == M.MHC_ERR_SHAPE
    assert _bwd(M, iters=0) == M.MHC_ERR_SHAPE
    assert _bwd(M, d=5120 + 32) == M.MHC_ERR_SHAPE
    assert _bwd(M, flags=0x2) == M.MHC_ERR_SHAPE
    for i in (0, 3, 7, 11, 16, 21, 24):       # X, mixes, W_mix, gXp, gX, gW, ggain
        p = [_addr(k) for k in range(25)]
        p[i] = None
        assert _bwd(M, ptrs=p) == M.MHC_ERR_NULL, i
    p = [_addr(k) for k in range(25)]
    p[2] = ctypes.c_void_p(p[2].value + 4)     # X' not 16-byte aligned
    assert _bwd(M, ptrs=p) == M.MHC_ERR_ALIGN
    assert _bwd(M, ws=ctypes.c_void_p(0)) == M.MHC_ERR_WORKSPACE
    p = [_addr(k) for k in range(25)]
    p[16] = p[0]                                # gX written over X
    assert _bwd(M, ptrs=p) == M.MHC_ERR_ALIAS
    p = [_addr(k) for k in range(25)]
    p[17] = ctypes.c_void_p(p[16].value + 64)   # gF inside gX
    assert _bwd(M, ptrs=p) == M.MHC_ERR_ALIAS
    assert M.lib.mhc_backward_workspace_bytes(256, 4, 5120 + 32) == 0
    assert M.lib.mhc_backward_workspace_bytes(256, 3, 5120) == 0



def test_path_flags_validation(M):
    """MHC_PATH_PERSISTENT / MHC_PATH_CLUSTER: host-side checks, before any device call."""
    P, C = M.PATH_PERSISTENT, M.PATH_CLUSTER
    assert _fused(M, N=0, flags=P) == M.MHC_OK
    assert _fused(M, N=0, flags=C) == M.MHC_OK                            # 16 CTAs of 320 columns
    assert _fused(M, flags=P | C) == M.MHC_ERR_SHAPE
    assert _fused(M, flags=C | M.tile_flag(32)) == M.MHC_ERR_SHAPE        # the tile is fixed at 32
    assert _fused(M, flags=C | M.split_flag(32)) == M.MHC_ERR_SHAPE       # clusters of 8 or 16
    assert _fused(M, flags=C | M.split_flag(8)) == M.MHC_ERR_SHAPE        # 20 chunks per CTA
    assert _fused(M, N=0, d=2560, flags=C | M.split_flag(8)) == M.MHC_OK  # 10 chunks per CTA
    assert _fused(M, N=0, d=256, flags=C) == M.MHC_OK                     # 8 CTAs of one chunk
    assert _fused(M, d=6144, flags=C) == M.MHC_ERR_SHAPE                  # 12 or 24 chunks
    assert _fused(M, N=0, d=6144, flags=P) == M.MHC_OK
    p = [_addr(i) for i in range(16)]
    assert M.lib.mhc_fused_step_mxfp8(*p, 0, 4, 5120, 20, 1e-6, 1e-6, C, _addr(21), 1 << 26,
                                      None) == M.MHC_ERR_SHAPE             # bf16 y only
    q = [_addr(i) for i in range(8)]
    assert M.lib.mhc_mixes(*q, 0, 4, 5120, 20, 1e-6, 1e-6, C, _addr(9), 1 << 26,
                           None) == M.MHC_ERR_SHAPE
    assert M.lib.mhc_step_path(8, 4, 5120, P | C) == M.MHC_ERR_SHAPE
