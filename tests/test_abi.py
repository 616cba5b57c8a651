"""The C-ABI library loads without a GPU, exports every declared entry point,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def xv():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "xv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(xv_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(xv):
    lib = ctypes.CDLL(xv.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(xv.exported_symbols())


def test_abi_version(xv):
    assert xv.xv_abi_version() == 5


def _code(fn, *args):
    return fn(*args)


def test_gemm_validation_without_gpu(xv):
    L = xv.lib()
    p = ctypes.c_void_p(0x10000)
    assert L.xv_gemm_small_m(None, 64, p, p, 64, 1, 64, 64, None, 0, None) == xv.XV_ERR_ARG
    assert b"null" in L.xv_last_error()
    assert L.xv_gemm_small_m(p, 64, p, p, 64, 65, 64, 64, None, 0, None) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_gemm_small_m(p, 64, p, p, 64, 0, 64, 64, None, 0, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_small_m(p, 60, p, p, 64, 1, 64, 64, None, 0, None) == xv.XV_ERR_ARG          # ldx < K
    assert L.xv_gemm_small_m(p, 68, p, p, 64, 1, 64, 68, None, 0, None) == xv.XV_ERR_UNSUPPORTED  # K % 8
    odd = ctypes.c_void_p(0x10002)
    assert L.xv_gemm_small_m(odd, 64, p, p, 64, 1, 64, 64, None, 0, None) == xv.XV_ERR_UNSUPPORTED
    # a narrow shape split into more segments than a cluster combines needs a workspace
    assert xv.xv_gemm_splits(1024, 8192) > 4
    assert xv.xv_gemm_workspace_size(8, 1024, 8192) > 0
    assert L.xv_gemm_small_m(p, 8192, p, p, 1024, 8, 1024, 8192, None, 0, None) == xv.XV_ERR_WORKSPACE
    # shapes wider than the SM count stay whole, those of one to two SMs' worth split in two
    # (combined in clusters), neither needs a workspace; the narrow projections fill one wave of 2
    # CTAs per SM with at least 8 K-blocks per segment and combine through the workspace
    assert xv.xv_gemm_splits(34816, 5120) == 1 and xv.xv_gemm_workspace_size(64, 34816, 5120) == 0
    assert xv.xv_gemm_splits(151936, 5120) == 1
    assert xv.xv_gemm_splits(12352, 5120) == 2 and xv.xv_gemm_workspace_size(64, 12352, 5120) == 0
    assert xv.xv_gemm_splits(5120, 17408) == 7 and xv.xv_gemm_workspace_size(64, 5120, 17408) > 0
    assert xv.xv_gemm_splits(5120, 4096) == 7 and xv.xv_gemm_splits(5120, 6144) == 7
    # every shape's workspace fits the allocation-free entry point's 10 MiB scratch
    for N in (1024, 4096, 5120, 9728):
        assert xv.xv_gemm_workspace_size(64, N, 17408) <= 10 << 20


def test_tiled_weights_size_and_validation_without_gpu(xv):
    """The tiled copy holds whole 128 x 64 tiles (zero padded past N and K); the tiling call and
    the tiled GEMM reject bad arguments on the host."""
    L = xv.lib()
    assert xv.xv_gemm_tiled_bytes(128, 64) == 128 * 64 * 2
    assert xv.xv_gemm_tiled_bytes(129, 64) == 2 * 128 * 64 * 2
    assert xv.xv_gemm_tiled_bytes(300, 1000) == 3 * 16 * 128 * 64 * 2
    assert xv.xv_gemm_tiled_bytes(151936, 5120) == 151936 * 5120 * 2
    assert xv.xv_gemm_tiled_bytes(0, 64) == 0
    p = ctypes.c_void_p(0x10000)
    assert L.xv_gemm_tile_weights(None, 64, 64, p, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_tile_weights(p, 64, 64, None, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_tile_weights(p, 0, 64, p, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_tile_weights(p, 64, 4, p, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_tile_weights(p, 64, 68, p, None) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_gemm_tile_weights(ctypes.c_void_p(0x10002), 64, 64, p, None) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_gemm_small_m_tiled(None, 64, p, p, 64, 1, 64, 64, None, 0, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_small_m_tiled(p, 64, p, p, 64, 65, 64, 64, None, 0, None) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_gemm_small_m_tiled_f32out(p, 8192, p, p, 1024, 8, 1024, 8192, None, 0, None) == xv.XV_ERR_WORKSPACE


def test_gate_up_tiling_and_fused_swiglu_validation_without_gpu(xv):
    L = xv.lib()
    p = ctypes.c_void_p(0x10000)
    assert L.xv_gemm_tile_gate_up(None, 64, 64, p, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_tile_gate_up(p, 0, 64, p, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_tile_gate_up(p, 100, 64, p, None) == xv.XV_ERR_UNSUPPORTED      # F % 64
    assert L.xv_gemm_swiglu_tiled(p, 64, p, None, 64, 1, 64, 64, None) == xv.XV_ERR_ARG
    assert L.xv_gemm_swiglu_tiled(p, 64, p, p, 64, 1, 96, 64, None) == xv.XV_ERR_UNSUPPORTED   # F % 64
    assert L.xv_gemm_swiglu_tiled(p, 64, p, p, 32, 1, 64, 64, None) == xv.XV_ERR_ARG           # ldact < F
    assert L.xv_gemm_swiglu_tiled(p, 64, p, p, 64, 65, 64, 64, None) == xv.XV_ERR_UNSUPPORTED  # M > 64
    assert L.xv_gemm_swiglu_tiled(p, 72, p, p, 64, 1, 64, 68, None) == xv.XV_ERR_UNSUPPORTED   # K % 8


def test_block_weights_layout(xv):
    """The binding's weights struct ends with the tiled flag (after the four pointers)."""
    assert [f[0] for f in xv.BlockWeights._fields_] == ["embed", "layers", "final_norm", "lm_head", "tiled"]
    assert xv.BlockWeights.tiled.offset == 32


def test_gemm_noalloc_scratch_holds_every_shape(xv):
    """The allocation-free entry point's fixed scratch (10 MiB) holds the split-K need of every
    shape it accepts (M <= 64), over a sweep of widths and depths."""
    worst = 0
    for N in list(range(128, 20000, 128)) + [1, 100, 300, 5120, 9728, 19455]:
        for K in (64, 256, 1000, 4096, 8192, 17408, 65536):
            worst = max(worst, xv.xv_gemm_workspace_size(64, N, K))
    assert 0 < worst <= 10 << 20


def test_gemm_splits_depend_on_shape_only(xv):
    for N, K in [(5120, 4096), (5120, 6144), (5120, 17408), (12352, 5120), (14336, 5120), (34816, 5120), (151936, 5120)]:
        s = xv.xv_gemm_splits(N, K)
        assert 1 <= s <= 16
        assert -(-K // 64) // s >= 8 or s == 1
        assert xv.xv_gemm_workspace_size(1, N, K) <= xv.xv_gemm_workspace_size(64, N, K)


def test_gdn_validation_without_gpu(xv):
    L = xv.lib()
    p = 0x10000
    st = xv.GdnSteps(p, p, p, p, p, 128 * 3, 2, 8)
    assert L.xv_gdn_decode_step(None, ctypes.byref(st), ctypes.c_void_p(p), 128, 1, 1, 128, 128, 1, None) == xv.XV_ERR_ARG
    assert L.xv_gdn_decode_step(ctypes.c_void_p(p), ctypes.byref(st), ctypes.c_void_p(p), 128, 1, 1, 96, 128, 1, None) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_gdn_decode_step(ctypes.c_void_p(p), ctypes.byref(st), ctypes.c_void_p(p), 128, 1, 1, 128, 40, 1, None) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_gdn_verify(ctypes.c_void_p(p), ctypes.byref(st), None, 4, ctypes.byref(st), 8, ctypes.c_void_p(p),
                           128, 1, 1, 128, 128, 1, None) == xv.XV_ERR_ARG  # n_commit missing
    assert L.xv_gdn_verify(ctypes.c_void_p(p), None, None, 0, ctypes.byref(st), xv.XV_KMAX + 1, ctypes.c_void_p(p),
                           128, 1, 1, 128, 128, 1, None) == xv.XV_ERR_UNSUPPORTED  # k > XV_KMAX
    short = xv.GdnSteps(p, p, p, p, p, 128 * 3, 2, 4)
    assert L.xv_gdn_verify(ctypes.c_void_p(p), None, None, 0, ctypes.byref(short), 8, ctypes.c_void_p(p),
                           128, 1, 1, 128, 128, 1, None) == xv.XV_ERR_ARG  # draft rows < k


def test_attn_validation_without_gpu(xv):
    L = xv.lib()
    p = ctypes.c_void_p(0x10000)
    args = lambda **kw: [kw.get("q", p), 6144, p, p, p, kw.get("R", 8), 1, kw.get("Hq", 24), kw.get("Hkv", 4),
                         kw.get("hd", 256), 4096, kw.get("max_ctx", 3000), 0.0625, None, 0, p, 6144,
                         kw.get("ws", p), kw.get("wsb", 1 << 30), None]
    assert L.xv_attn_decode_rows(*args(q=None)) == xv.XV_ERR_ARG
    assert L.xv_attn_decode_rows(*args(hd=128)) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_attn_decode_rows(*args(Hq=25)) == xv.XV_ERR_ARG
    assert L.xv_attn_decode_rows(*args(R=xv.XV_KMAX + 1)) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_attn_decode_rows(*args(R=0)) == xv.XV_ERR_ARG
    assert L.xv_attn_decode_rows(*args(max_ctx=5000)) == xv.XV_ERR_ARG              # beyond Lmax
    assert L.xv_attn_decode_rows(*args(ws=None)) == xv.XV_ERR_WORKSPACE
    assert L.xv_attn_decode_rows(*args(ws=ctypes.c_void_p(0x10008))) == xv.XV_ERR_UNSUPPORTED   # misaligned
    # splits of 512 positions below 4096, 2048 beyond
    assert [xv.xv_attn_split_begin(s) for s in (0, 1, 7, 8, 9, 10)] == [0, 512, 3584, 4096, 6144, 8192]
    assert xv.xv_attn_split_begin(-1) == -1
    assert xv.xv_attn_workspace_size(1, 8, 24, 256, 2183) >= 8 * 24 * 5 * 256 * 4


def _cfg(xv, kinds=(0, 0, 0, 1)):
    kinds_arr = (ctypes.c_int32 * len(kinds))(*kinds)
    c = xv.BlockConfig(5120, 151936, 17408, len(kinds), ctypes.cast(kinds_arr, ctypes.c_void_p).value,
                       32, 128, 128, 24, 4, 256, 1e-6)
    return c, kinds_arr


def test_block_dims_and_validation_without_gpu(xv):
    L = xv.lib()
    c, keep = _cfg(xv)
    assert L.xv_gdn_in_dim(ctypes.byref(c)) == 12352
    assert L.xv_attn_in_dim(ctypes.byref(c)) == 14336
    assert L.xv_block_workspace_size(ctypes.byref(c), 1, 8, 4096) > 0
    bad, keep2 = _cfg(xv, kinds=(0, 2))
    assert L.xv_gdn_in_dim(ctypes.byref(bad)) == -1
    st = xv.BlockState()
    w = xv.BlockWeights()
    assert L.xv_verify_block(ctypes.byref(c), ctypes.byref(w), ctypes.byref(st), None, 8, None, None, None, None, 0,
                             None) == xv.XV_ERR_ARG
    assert L.xv_block_commit(ctypes.byref(st), None, None) == xv.XV_ERR_ARG


def test_paged_validation_without_gpu(xv):
    """Paged KV calls check the page description on the host before anything reaches the device."""
    L = xv.lib()
    p = ctypes.c_void_p(0x10000)
    bad = xv.KvPages(0x10000, 96, 4, 8)       # page size not a multiple of 64
    good = xv.KvPages(0x10000, 64, 4, 8)
    args = lambda pages, max_ctx: (p, 256, p, p, ctypes.byref(pages), p, 2, 1, 4, 2, 64, max_ctx, 0.125, None, 0, p,
                                   256, p, 1 << 20, None)
    assert L.xv_attn_decode_rows_paged(*args(bad, 100)) == xv.XV_ERR_UNSUPPORTED
    assert L.xv_attn_decode_rows_paged(*args(good, 257)) == xv.XV_ERR_ARG      # beyond 4 pages of 64
    assert L.xv_attn_decode_rows_paged(*args(xv.KvPages(None, 64, 4, 8), 100)) == xv.XV_ERR_ARG
    assert L.xv_kv_append_paged(p, 256, p, 2, 1, 2, 64, ctypes.byref(bad), p, p, None) == xv.XV_ERR_UNSUPPORTED


def test_block_state_layout(xv):
    """The binding's state struct ends with the page description and the ragged k pointer."""
    names = [f[0] for f in xv.BlockState._fields_]
    assert names[-2:] == ["kv_pages", "last_k_seq"]
    assert ctypes.sizeof(xv.KvPages) == 8 + 3 * 4 + 4     # pointer, three ints, tail padding


def _fake_state(xv, B, kmax, Lmax, n_layers=4):
    """A block state whose pointers are aligned but point nowhere: for host validation only."""
    p = 0x10000
    layers = (xv.LayerState * n_layers)()
    for ls in layers:
        ls.gdn_state, ls.k_cache, ls.v_cache = p, p, p
        ls.gdn_hist[0], ls.gdn_hist[1] = p, p
    st = xv.BlockState(B, kmax, Lmax, p, p, 0, kmax, 0, 0, ctypes.cast(layers, ctypes.c_void_p).value)
    return st, layers


def test_prefill_limits_without_gpu(xv):
    """Chunks beyond kmax, or beyond 64 GEMM rows over the batch, are refused before any launch."""
    L = xv.lib()
    c, keep = _cfg(xv)
    w = xv.BlockWeights()
    st, layers = _fake_state(xv, 2, xv.XV_KMAX, 4096)
    p = ctypes.c_void_p(0x10000)
    call = lambda T, chunk: L.xv_block_prefill(ctypes.byref(c), ctypes.byref(w), ctypes.byref(st), p, T, chunk, None,
                                               None, p, 1 << 30, None)
    assert call(100, xv.XV_KMAX + 1) == xv.XV_ERR_ARG             # chunk > kmax
    assert call(100, 0) == xv.XV_ERR_ARG
    assert call(0, 8) == xv.XV_ERR_ARG                            # no tokens
    assert call(100, 33) == xv.XV_ERR_UNSUPPORTED                 # 2 x 33 rows > 64
    st.last_k = 4
    assert call(100, 8) == xv.XV_ERR_ARG                          # an uncommitted verify
    st.last_k, st.max_ctx = 0, 4000
    assert call(100, 8) == xv.XV_ERR_ARG                          # max_ctx + T > Lmax
    big, layers2 = _fake_state(xv, 1, xv.XV_KMAX + 1, 4096)
    assert L.xv_block_prefill(ctypes.byref(c), ctypes.byref(w), ctypes.byref(big), p, 100, 8, None, None, p, 1 << 30,
                              None) == xv.XV_ERR_ARG              # kmax beyond XV_KMAX


def test_complete_gdn_dims_without_gpu(xv):
    """Column layout of a complete GDN layer: q | k (16 q/k heads) | v | z (32 v heads) | b | a;
    the convolution covers q | k | v; strides are rounded up to 8 columns."""
    L = xv.lib()
    kinds = (ctypes.c_int32 * 4)(0, 0, 0, 1)
    c = xv.BlockConfig(5120, 151936, 17408, 4, ctypes.cast(kinds, ctypes.c_void_p).value, 32, 128, 128, 24, 4, 256,
                       1e-6, 16, 4, 1)
    qk, v = 16 * 128, 32 * 128
    assert L.xv_gdn_conv_dim(ctypes.byref(c)) == 2 * qk + v
    assert L.xv_gdn_conv_stride(ctypes.byref(c)) == (2 * qk + v + 7) // 8 * 8
    assert L.xv_gdn_in_dim(ctypes.byref(c)) == 2 * qk + 2 * v + 2 * 32
    assert L.xv_gdn_hist_stride(ctypes.byref(c)) % 8 == 0
    assert L.xv_gdn_hist_stride(ctypes.byref(c)) >= L.xv_gdn_in_dim(ctypes.byref(c))
    bad = xv.BlockConfig(5120, 151936, 17408, 4, ctypes.cast(kinds, ctypes.c_void_p).value, 32, 128, 128, 24, 4, 256,
                         1e-6, 12, 4, 1)      # 12 q/k heads do not divide 32 v heads
    assert L.xv_gdn_in_dim(ctypes.byref(bad)) == -1
    wide = xv.BlockConfig(5120, 151936, 17408, 4, ctypes.cast(kinds, ctypes.c_void_p).value, 32, 128, 128, 24, 4,
                          256, 1e-6, 16, xv.XV_CONV_MAX + 1, 1)
    assert L.xv_gdn_in_dim(ctypes.byref(wide)) == -1
    # the prefill workspace holds the verify workspace and its own chunk buffers
    assert L.xv_block_prefill_workspace_size(ctypes.byref(c), 1, 64, 4096) > \
        L.xv_block_workspace_size(ctypes.byref(c), 1, 64, 4096) > 0
    assert L.xv_block_workspace_size(ctypes.byref(c), 0, 64, 4096) == 0


def test_binding_constants_match_the_header(xv):
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "xv.h")).read()
    for name in ("XV_KMAX", "XV_GEMM_M_MAX", "XV_CONV_MAX", "XV_ABI_VERSION"):
        m = re.search(r"#define\s+%s\s+(\d+)" % name, hdr)
        assert m, name
        value = xv.xv_abi_version() if name == "XV_ABI_VERSION" else getattr(xv, name)
        assert value == int(m.group(1)), name


def test_step_host_checks_its_buffers_before_any_copy(xv):
    """The host step copies B*k draft ids in and B*kmax + B results out through raw pointers: the
    binding refuses buffers too short, of another type or in the wrong memory before calling."""
    import types

    import torch
    blk = types.SimpleNamespace(state=types.SimpleNamespace(B=2, kmax=8))
    host = lambda n, dt=torch.int32: torch.zeros(n, dtype=dt)   # noqa: E731
    with pytest.raises(ValueError, match="host_tokens"):
        xv.xv_block_step_host(blk, host(2 * 8 - 1), None, 8, None, host(18), None)
    with pytest.raises(ValueError, match="host_tokens"):
        xv.xv_block_step_host(blk, host(16, torch.int64), None, 8, None, host(18), None)
    with pytest.raises(ValueError, match="dev_tokens"):      # a host tensor where device memory is needed
        xv.xv_block_step_host(blk, host(16), host(16), 8, None, host(18), None)
