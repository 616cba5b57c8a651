"""The allocation-free GEMM entry point (xv_gemm_small_m_noalloc).

It exists for callers that cannot call cudaMalloc or pass a workspace (code
running under another framework's memory pool, plugins inside a process that
owns every device allocation, loops where allocating is not allowed).  It
runs the same kernel as xv_gemm_small_m with its scratch in a fixed array of
the library, so its output must match the workspace entry point's — here
bit for bit, which is inside every tolerance the other tests use — on two
calls in a row (the second call finds the array as the first one left it).
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


@pytest.mark.parametrize("M,N,K", [(16, 1024, 8192), (64, 1024, 8192), (16, 5120, 17408), (5, 300, 1000)])
def test_noalloc_matches_workspace_entry_point_twice(xv, M, N, K):
    # the first two shapes split K into 16 segments, whose partial sums go through the scratch
    X = dev(synth.normal_bf16(0, synth.tid(f"na.x.{M}.{N}.{K}"), (M, K)))
    W = dev(synth.normal_bf16(0, synth.tid(f"na.w.{M}.{N}.{K}"), (N, K), sigma=0.02))
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ws = xv.workspace(xv.xv_gemm_workspace_size(M, N, K))
    xv.xv_gemm_small_m(X, W, ref, ws)
    lib = xv.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        Y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        code = lib.xv_gemm_small_m_noalloc(ctypes.c_void_p(X.data_ptr()), K, ctypes.c_void_p(W.data_ptr()),
                                           ctypes.c_void_p(Y.data_ptr()), N, M, N, K, stream)
        assert code == 0, lib.xv_last_error()
        assert same_bits(Y, ref)
    assert xv.xv_device_check() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(xv):
    lib = xv.lib()
    p = ctypes.c_void_p(0x10000)
    # more rows than any GEMM call takes: rejected before anything is launched
    assert lib.xv_gemm_small_m_noalloc(p, 64, p, p, 64, 65, 64, 64, None) == xv.XV_ERR_UNSUPPORTED
