"""The allocation-free GEMM entry point (xv_gemm_small_m_noalloc).

It exists for callers that cannot call cudaMalloc or pass a workspace (code
running under another framework's memory pool, plugins inside a process that
owns every device allocation, loops where allocating is not allowed).  It
runs the same kernel as xv_gemm_small_m with its scratch in a fixed array of
the library, so its output must match the workspace entry point's — here
bit for bit, which is inside every tolerance the other tests use — on calls
in a row, each finding the array as the previous one left it.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _gpu import dev, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xv():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv as m
    return m


def _operands(xv, M, N, K):
    X = dev(synth.normal_bf16(0, synth.tid(f"na.x.{M}.{N}.{K}"), (M, K)))
    W = dev(synth.normal_bf16(0, synth.tid(f"na.w.{M}.{N}.{K}"), (N, K), sigma=0.02))
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ws = xv.workspace(xv.xv_gemm_workspace_size(M, N, K))
    xv.xv_gemm_small_m(X, W, ref, ws)
    return X, W, ref


def _noalloc(xv, X, W, M, N, K):
    lib = xv.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    Y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    code = lib.xv_gemm_small_m_noalloc(ctypes.c_void_p(X.data_ptr()), K, ctypes.c_void_p(W.data_ptr()),
                                       ctypes.c_void_p(Y.data_ptr()), N, M, N, K, stream)
    assert code == 0, lib.xv_last_error()
    return Y


# (1, 1024, 8192) and (8, 5120, 17408) split K in 16 and 7 segments with at most 8 token rows:
# their last-arriving CTAs combine the partials through the scratch's tile counters.  (16, ...)
# and (64, ...) split as much but combine in a separate kernel; (5, 10000, 2048) and
# (5, 300, 1000) take clusters of two.
@pytest.mark.parametrize("M,N,K", [(1, 1024, 8192), (8, 5120, 17408), (16, 1024, 8192), (64, 1024, 8192),
                                   (16, 5120, 17408), (5, 10000, 2048), (5, 300, 1000)])
def test_noalloc_matches_workspace_entry_point_twice(xv, M, N, K):
    X, W, ref = _operands(xv, M, N, K)
    for _ in range(2):
        assert same_bits(_noalloc(xv, X, W, M, N, K), ref)
    assert xv.xv_device_check() == 0


def test_noalloc_alternating_counter_shapes(xv):
    """Back-to-back calls alternating between two counter-combined shapes with different tile
    counts (8 and 40 tiles): every call finds the counters the previous one left and still
    gives the workspace entry point's bits."""
    assert xv.xv_gemm_splits(1024, 8192) > 4 and xv.xv_gemm_splits(5120, 17408) > 4
    a = (1, 1024, 8192)
    b = (8, 5120, 17408)
    ops = {s: _operands(xv, *s) for s in (a, b)}
    for s in (a, b, a, b, b, a):
        X, W, ref = ops[s]
        assert same_bits(_noalloc(xv, X, W, *s), ref), s
    assert xv.xv_device_check() == 0


def test_noalloc_rejects_more_rows_than_a_call_takes(xv):
    lib = xv.lib()
    p = ctypes.c_void_p(0x10000)
    # more rows than any GEMM call takes: rejected before anything is launched
    assert lib.xv_gemm_small_m_noalloc(p, 64, p, p, 64, 65, 64, 64, None) == xv.XV_ERR_UNSUPPORTED
