"""Small-M GEMM: parity with the oracle, row bits independent of M and of row
position, run-to-run repeatability — at small ragged shapes and at the
5120 x 17408 gate/up and down projection shapes; weights row-major and in the
tiled layout (the same bits from both)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import assert_bf16_close, assert_f32_close, dev, host, host_u16, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xv():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv as m
    return m


def run(xv, X, W, M=None, f32=False):
    M = X.shape[0] if M is None else M
    N, K = W.shape
    Y = torch.empty((M, N), dtype=torch.float32 if f32 else torch.int16, device="cuda")
    ws = xv.workspace(xv.xv_gemm_workspace_size(M, N, K))
    xv.xv_gemm_small_m(X[:M], W, Y, ws)
    return Y


@pytest.mark.parametrize("M,N,K", [(1, 300, 1000), (5, 300, 1000), (64, 300, 1000), (3, 256, 4096), (17, 131, 72),
                                   (8, 1024, 640)])
def test_parity_small_shapes(xv, M, N, K):
    X = synth.normal_bf16(0, synth.tid(f"gx{M}.{N}.{K}"), (M, K))
    W = synth.normal_bf16(0, synth.tid(f"gw{M}.{N}.{K}"), (N, K), sigma=0.02)
    ref = oracle.gemm(X, W)
    Y = run(xv, dev(X), dev(W))
    assert_bf16_close(host_u16(Y), ref, what=f"gemm {M}x{N}x{K}")
    Yf = run(xv, dev(X), dev(W), f32=True)
    assert_f32_close(host(Yf), ref, rel=1e-3, what="gemm f32 out")
    assert xv.xv_device_check() == 0


@pytest.fixture(scope="module")
def big(xv):
    """The gate/up [17408, 5120] and down [5120, 17408] weights, activations N(0,1)."""
    Wgu = synth.normal_bf16(0, synth.tid("sweep.w_gate_up"), (17408, 5120), sigma=0.02)
    Wd = synth.normal_bf16(0, synth.tid("sweep.w_down"), (5120, 17408), sigma=0.02)
    Xgu = synth.normal_bf16(0, synth.tid("sweep.x_gate_up"), (64, 5120))
    Xd = synth.normal_bf16(0, synth.tid("sweep.x_down"), (64, 17408))
    # a narrow, deep shape whose K split (16 segments) is combined through the workspace
    Wn = synth.normal_bf16(0, synth.tid("sweep.w_narrow"), (1024, 8192), sigma=0.02)
    Xn = synth.normal_bf16(0, synth.tid("sweep.x_narrow"), (64, 8192))
    out = {"gu": (Xgu, Wgu, dev(Xgu), dev(Wgu)), "down": (Xd, Wd, dev(Xd), dev(Wd)),
           "narrow": (Xn, Wn, dev(Xn), dev(Wn))}
    for which in list(out):
        Xh, Wh, X, W = out[which]
        out[which + "_tiled"] = (Xh, Wh, X, xv.tile_weight(W))
    return out


def test_split_paths(xv):
    """The 17408-wide half of gate/up (136 tiles): 2 segments combined in a cluster; the fused
    34816-wide gate/up stays whole; down: 7 (one wave of 2 CTAs per SM) through the workspace;
    narrow: 16 through the workspace; a shape too short in K for two segments stays whole."""
    assert xv.xv_gemm_splits(17408, 5120) == 2
    assert xv.xv_gemm_splits(34816, 5120) == 1
    assert xv.xv_gemm_splits(17408, 512) == 1
    assert xv.xv_gemm_splits(5120, 17408) == 7 and xv.xv_gemm_workspace_size(8, 5120, 17408) > 0
    assert xv.xv_gemm_splits(1024, 8192) > 4 and xv.xv_gemm_workspace_size(8, 1024, 8192) > 0


@pytest.mark.parametrize("which", ["gu", "down", "narrow", "gu_tiled", "down_tiled", "narrow_tiled"])
def test_row_bits_independent_of_M(xv, big, which):
    _, _, X, W = big[which]
    ref = run(xv, X, W, M=16)
    for M in (1, 2, 4, 8, 9, 16, 64):
        Y = run(xv, X, W, M=M)
        m = min(M, 16)
        assert same_bits(Y[:m], ref[:m]), f"M={M}: rows differ from the M=16 call"


@pytest.mark.parametrize("which", ["gu", "down", "narrow", "gu_tiled", "down_tiled", "narrow_tiled"])
def test_row_bits_independent_of_position(xv, big, which):
    _, _, X, W = big[which]
    perm = torch.tensor([5, 0, 7, 3, 1, 6, 2, 4], device="cuda")
    Y = run(xv, X[:8], W)
    Yp = run(xv, X[:8][perm].contiguous(), W)
    assert same_bits(Yp, Y[perm])


@pytest.mark.parametrize("which", ["gu", "down", "narrow"])
def test_full_size_parity_sampled(xv, big, which):
    Xh, Wh, X, W = big[which]
    M = 16
    Y = host_u16(run(xv, X, W, M=M))
    cols = np.sort(np.random.default_rng(0).choice(Wh.shape[0], 96, replace=False))
    cols = np.unique(np.concatenate([cols, [0, Wh.shape[0] - 1]]))
    ref = oracle.gemm(Xh[:M], Wh[cols])
    assert_bf16_close(Y[:, cols], ref, what=f"{which} sampled")


@pytest.mark.parametrize("which", ["gu", "down", "narrow", "gu_tiled", "down_tiled", "narrow_tiled"])
def test_hundred_runs_identical(xv, big, which):
    _, _, X, W = big[which]
    ref = run(xv, X, W, M=16)
    N, K = W.shape
    ws = xv.workspace(xv.xv_gemm_workspace_size(16, N, K))
    Y = torch.empty_like(ref)
    for _ in range(100):
        xv.xv_gemm_small_m(X[:16], W, Y, ws)
        assert same_bits(Y, ref)
    assert xv.xv_device_check() == 0


def test_lm_head_shape_f32(xv):
    """The LM head shape (151936 x 5120, fp32 out) on a sample of rows."""
    N, K = 151936, 5120
    Wh = synth.normal_bf16(0, synth.tid("lm_head_test"), (N, K), sigma=0.02)
    Xh = synth.normal_bf16(0, synth.tid("lm_x"), (8, K))
    Y = host(run(xv, dev(Xh), dev(Wh), f32=True))
    cols = np.random.default_rng(1).choice(N, 64, replace=False)
    assert_f32_close(Y[:, cols], oracle.gemm(Xh, Wh[cols]), rel=1e-3, what="lm head")


def _tiles_by_definition(W):
    """The tiled layout written out on the host: Wt[t][kb][r][c] = W[128 t + r][64 kb + c], zero
    past N and K."""
    N, K = W.shape
    Np, Kp = -(-N // 128) * 128, -(-K // 64) * 64
    P = np.zeros((Np, Kp), dtype=W.dtype)
    P[:N, :K] = W
    return P.reshape(Np // 128, 128, Kp // 64, 64).transpose(0, 2, 1, 3).reshape(-1)


@pytest.mark.parametrize("N,K", [(300, 1000), (131, 72), (128, 64), (1024, 640)])
def test_tiled_layout_matches_its_definition(xv, N, K):
    W = synth.normal_bf16(0, synth.tid(f"tw{N}.{K}"), (N, K), sigma=0.02)
    Wt = xv.tile_weight(dev(W))
    assert Wt.shape == (N, K) and Wt.data.numel() * 2 == xv.xv_gemm_tiled_bytes(N, K)
    assert np.array_equal(host_u16(Wt.data), _tiles_by_definition(W))


@pytest.mark.parametrize("M,N,K", [(1, 300, 1000), (9, 300, 1000), (64, 300, 1000), (17, 131, 72), (8, 1024, 640),
                                   (3, 256, 4096)])
def test_tiled_equals_row_major_small(xv, M, N, K):
    X = dev(synth.normal_bf16(0, synth.tid(f"gx{M}.{N}.{K}"), (M, K)))
    W = dev(synth.normal_bf16(0, synth.tid(f"gw{M}.{N}.{K}"), (N, K), sigma=0.02))
    Wt = xv.tile_weight(W)
    for f32 in (False, True):
        assert same_bits(run(xv, X, Wt, f32=f32), run(xv, X, W, f32=f32)), f"f32={f32}"
    assert xv.xv_device_check() == 0


@pytest.mark.parametrize("which", ["gu", "down", "narrow"])
def test_tiled_equals_row_major_full_size(xv, big, which):
    """Every path the split rule takes (cluster combine, workspace combine with tile counters at
    M <= 8, the separate combine past 8 rows) gives the same bits from either layout."""
    _, _, X, W = big[which]
    Wt = big[which + "_tiled"][3]
    for M in (1, 8, 9, 64):
        assert same_bits(run(xv, X, Wt, M=M), run(xv, X, W, M=M)), f"M={M}"
    assert xv.xv_device_check() == 0


def test_tiled_lm_head_equals_row_major(xv):
    N, K = 151936, 5120
    W = dev(synth.normal_bf16(0, synth.tid("lm_head_test"), (N, K), sigma=0.02))
    X = dev(synth.normal_bf16(0, synth.tid("lm_x"), (8, K)))
    Wt = xv.tile_weight(W)
    assert same_bits(run(xv, X, Wt, f32=True), run(xv, X, W, f32=True))


@pytest.mark.parametrize("F,K", [(64, 64), (128, 1000), (512, 256)])
def test_gate_up_tiling_matches_its_definition(xv, F, K):
    """Tile t of the gated layout holds gate rows 64t..64t+63, then up rows F+64t..F+64t+63."""
    W = synth.normal_bf16(0, synth.tid(f"tgu{F}.{K}"), (2 * F, K), sigma=0.02)
    order = np.concatenate([np.r_[64 * t:64 * t + 64, F + 64 * t:F + 64 * t + 64] for t in range(F // 64)])
    Wt = xv.tile_gate_up(dev(W))
    assert Wt.gated and Wt.shape == (2 * F, K)
    assert np.array_equal(host_u16(Wt.data), _tiles_by_definition(W[order]))


@pytest.mark.parametrize("M,F,K", [(1, 512, 256), (8, 512, 256), (9, 1024, 1000), (64, 512, 256), (8, 17408, 5120)])
def test_fused_swiglu_vs_oracle(xv, M, F, K):
    """act = bf16(silu(g) u) with g, u the bf16 gate/up outputs: against the oracle's GEMM and
    SwiGLU (bf16 tolerance), every row independent of M."""
    X = synth.normal_bf16(0, synth.tid(f"sx{M}.{F}.{K}"), (64, K))
    W = synth.normal_bf16(0, synth.tid(f"sw{F}.{K}"), (2 * F, K), sigma=0.05)
    Wt = xv.tile_gate_up(dev(W))
    Xd = dev(X)
    act = torch.empty((M, F), dtype=torch.int16, device="cuda")
    xv.xv_gemm_swiglu(Xd[:M], Wt, act)
    cols = np.arange(F) if F <= 1024 else np.sort(np.random.default_rng(2).choice(F, 128, replace=False))
    gu = oracle.round_bf16(oracle.gemm(X[:M], np.concatenate([W[cols], W[F + cols]])))
    ref = oracle.swiglu(gu[:, :len(cols)], gu[:, len(cols):])
    assert_bf16_close(host_u16(act)[:, cols], ref, what=f"fused swiglu {M}x{F}x{K}")
    full = torch.empty((64, F), dtype=torch.int16, device="cuda")
    xv.xv_gemm_swiglu(Xd, Wt, full)
    assert same_bits(act, full[:M])
    assert xv.xv_device_check() == 0


def test_gemm_straight_after_tiling(xv):
    """A GEMM enqueued right after the tiling of its weight, nothing else between them on the
    stream, reads finished tiles (every GEMM requests its first weight tiles before its dependency
    wait).  The tiled buffer is reused from one call to the next and holds the other weight's
    tiles before each tiling, so a read of unfinished tiles would show up as the other result."""
    M, N, K = 8, 5120, 17408
    X = dev(synth.normal_bf16(0, synth.tid("after_tiling_x"), (M, K)))
    Ws = [dev(synth.normal_bf16(0, synth.tid(f"after_tiling_w{i}"), (N, K), sigma=0.02)) for i in range(2)]
    refs = [run(xv, X, W) for W in Ws]
    Y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ws = xv.workspace(xv.xv_gemm_workspace_size(M, N, K))
    outs = []
    for i in range(20):
        Wt = xv.tile_weight(Ws[i % 2])
        xv.xv_gemm_small_m(X, Wt, Y, ws)
        outs.append(Y.clone())
        del Wt
    for i, o in enumerate(outs):
        assert same_bits(o, refs[i % 2]), f"call {i}"
    assert xv.xv_device_check() == 0
