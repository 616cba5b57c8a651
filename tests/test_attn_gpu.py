"""Decode-row attention: parity with the oracle (explicit fp64 softmax), every
verify row bit-identical to a single decode row at its position, 8 sequences
in flight, cache garbage past the visible length ignored, run-to-run
repeatability; GQA 24/4 heads of 256 at 640, 2183 and 131072 positions."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import assert_bf16_close, dev, f64, host_u16, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xv():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv as m
    return m


def make(seed, B, R, Hq, Hkv, hd, Lmax, name="a"):
    q = synth.normal_bf16(seed, synth.tid(f"{name}.q"), (B * R, Hq * hd))
    kc = synth.normal_bf16(seed, synth.tid(f"{name}.k"), (B, Hkv, Lmax, hd))
    vc = synth.normal_bf16(seed, synth.tid(f"{name}.v"), (B, Hkv, Lmax, hd))
    return q, kc, vc


def exact_rows(q, kc, vc, len0, scale, R, Hq, Hkv, hd):
    """The oracle's fp64 decode rows (before the output's bf16 storage rounding): [R, Hq, hd]."""
    out = np.empty((R, Hq, hd))
    for r in range(R):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            out[r, h] = oracle.attn_row(q[r, h * hd:(h + 1) * hd], kc[g], vc[g], len0 + r, scale)
    return out


def attn(xv, q, kc, vc, ctx, R, B, Hq, Hkv, hd, Lmax, max_ctx, gate=None):
    out = torch.empty((B * R, Hq * hd), dtype=torch.int16, device="cuda")
    ws = xv.workspace(xv.xv_attn_workspace_size(B, R, Hq, hd, max_ctx))
    xv.xv_attn_decode_rows(q, q.stride(0), kc, vc, ctx, R, B, Hq, Hkv, hd, Lmax, max_ctx, hd ** -0.5, out,
                           out.stride(0), ws, gate=gate, gate_stride=0 if gate is None else gate.stride(0))
    return out


@pytest.mark.parametrize("hd,Hq,Hkv,R,lens", [(256, 4, 2, 3, [700, 1100]), (64, 2, 1, 4, [128, 1]),
                                               (256, 24, 4, 8, [2183]), (64, 6, 2, 1, [63, 64, 65, 513]),
                                               (64, 4, 2, 8, [4093, 6141])])
def test_parity_with_oracle(xv, hd, Hq, Hkv, R, lens):
    B = len(lens)
    Lmax = max(lens) + R + 64
    q, kc, vc = make(1, B, R, Hq, Hkv, hd, Lmax, name=f"p{hd}{Hq}{R}")
    ctx = np.array(lens, dtype=np.int32)
    out = host_u16(attn(xv, dev(q), dev(kc), dev(vc), dev(ctx), R, B, Hq, Hkv, hd, Lmax, max(lens) + R - 1))
    for b in range(B):
        ref = exact_rows(q[b * R:(b + 1) * R], kc[b], vc[b], lens[b], hd ** -0.5, R, Hq, Hkv, hd)
        assert_bf16_close(out[b * R:(b + 1) * R].reshape(R, Hq, hd), ref, what=f"attn b{b} len{lens[b]}")
    assert xv.xv_device_check() == 0


def test_gated_output_parity(xv):
    B, R, Hq, Hkv, hd, L = 1, 4, 4, 1, 256, 900
    Lmax = 1024
    q, kc, vc = make(2, B, R, Hq, Hkv, hd, Lmax, name="gate")
    g = synth.normal_bf16(2, synth.tid("gate.g"), (B * R, Hq * hd))
    out = host_u16(attn(xv, dev(q), dev(kc), dev(vc), dev(np.array([L], np.int32)), R, B, Hq, Hkv, hd, Lmax, L + R,
                        gate=dev(g)))
    # the output crosses two bf16 storage points (attention output, gated product): the
    # per-point bound 2e-2 * RMS applies once per point
    ref = oracle.attn_rows(q.reshape(R, Hq, hd), kc[0], vc[0], L, hd ** -0.5).reshape(R, -1)
    gated = f64(ref) / (1.0 + np.exp(-f64(g)))
    assert_bf16_close(out, gated, rel=2 * 2e-2, what="gated")


@pytest.mark.parametrize("L", [640, 2183, 4090, 6140, 131072])
def test_verify_rows_equal_decode_rows(xv, L):
    """Row r of an R=8 call equals an R=1 call with ctx_len + r (GQA 24/4, hd 256); at 4090 and
    6140 the rows cross the switch to 2048-position splits at 4096 and a long split's end."""
    B, R, Hq, Hkv, hd = 1, 8, 24, 4, 256
    Lmax = L + R
    q, kc, vc = make(3, B, R, Hq, Hkv, hd, Lmax, name=f"rows{L}")
    Q, K, V = dev(q), dev(kc), dev(vc)
    out = attn(xv, Q, K, V, dev(np.array([L], np.int32)), R, B, Hq, Hkv, hd, Lmax, L + R - 1)
    for r in range(R):
        one = attn(xv, Q[r:r + 1], K, V, dev(np.array([L + r], np.int32)), 1, B, Hq, Hkv, hd, Lmax, L + r)
        assert same_bits(out[r:r + 1], one), f"row {r} differs from the decode row at length {L + r}"
    # sampled parity with the oracle at this size: first and last row, three heads
    o = host_u16(out).reshape(R, Hq, hd)
    for r in (0, R - 1):
        for h in (0, 5, 23):
            g = h // (Hq // Hkv)
            ref = oracle.attn_row(q[r, h * hd:(h + 1) * hd], kc[0, g], vc[0, g], L + r, hd ** -0.5)
            assert_bf16_close(o[r, h], ref, what=f"L{L} r{r} h{h}")


@pytest.mark.parametrize("R,L", [(16, 2183), (64, 480), (64, 4050), (16, 131072)])
def test_row_tiles_equal_decode_rows(xv, R, L):
    """Past 64 rows per kv head (R x 6 q heads) the rows go in tiles of 64, one work item each per
    split; every row still equals an R=1 call at its own length, also where the rows cross a split
    boundary (480 + 63, 4050 + 63), and with persistent CTAs that reload Q between row tiles
    (131072: 2056 items), and the oracle (GQA 24/4, hd 256)."""
    B, Hq, Hkv, hd = 1, 24, 4, 256
    Lmax = L + R
    q, kc, vc = make(7, B, R, Hq, Hkv, hd, Lmax, name=f"tiles{R}.{L}")
    Q, K, V = dev(q), dev(kc), dev(vc)
    out = attn(xv, Q, K, V, dev(np.array([L], np.int32)), R, B, Hq, Hkv, hd, Lmax, L + R - 1)
    for r in range(R):
        one = attn(xv, Q[r:r + 1], K, V, dev(np.array([L + r], np.int32)), 1, B, Hq, Hkv, hd, Lmax, L + r)
        assert same_bits(out[r:r + 1], one), f"row {r} differs from the decode row at length {L + r}"
    o = host_u16(out).reshape(R, Hq, hd)
    for r in (0, 10, R - 1):
        for h in (0, 11, 23):
            g = h // (Hq // Hkv)
            ref = oracle.attn_row(q[r, h * hd:(h + 1) * hd], kc[0, g], vc[0, g], L + r, hd ** -0.5)
            assert_bf16_close(o[r, h], ref, what=f"R{R} L{L} r{r} h{h}")
    assert xv.xv_device_check() == 0


def test_eight_in_flight_equal_alone(xv):
    B, R, Hq, Hkv, hd = 8, 8, 24, 4, 256
    lens = np.array([640, 2183, 1, 513, 1024, 100, 2000, 511], dtype=np.int32)
    Lmax = 2304
    q, kc, vc = make(4, B, R, Hq, Hkv, hd, Lmax, name="flight")
    Q, K, V = dev(q), dev(kc), dev(vc)
    out = attn(xv, Q, K, V, dev(lens), R, B, Hq, Hkv, hd, Lmax, int(lens.max()) + R - 1)
    for b in range(B):
        one = attn(xv, Q[b * R:(b + 1) * R], K[b:b + 1], V[b:b + 1], dev(lens[b:b + 1]), R, 1, Hq, Hkv, hd, Lmax,
                   int(lens[b]) + R - 1)
        assert same_bits(out[b * R:(b + 1) * R], one), f"sequence {b} differs when batched"


def test_eight_in_flight_long_mixed_lengths(xv):
    """8 sequences at up to 131072 positions with mixed lengths (more than two waves of items:
    persistent CTAs whose ranges of items cross sequences of different lengths): each sequence's
    rows equal the same rows computed alone, bit for bit, and sampled rows match the oracle."""
    B, R, Hq, Hkv, hd = 8, 8, 24, 4, 256
    lens = np.array([131072, 70001, 1, 513, 131000, 2183, 64, 99999], dtype=np.int32)
    Lmax = 131072 + 64
    q, kc, vc = make(8, B, R, Hq, Hkv, hd, Lmax, name="flightlong")
    Q, K, V = dev(q), dev(kc), dev(vc)
    out = attn(xv, Q, K, V, dev(lens), R, B, Hq, Hkv, hd, Lmax, int(lens.max()) + R - 1)
    for b in range(B):
        one = attn(xv, Q[b * R:(b + 1) * R], K[b:b + 1], V[b:b + 1], dev(lens[b:b + 1]), R, 1, Hq, Hkv, hd, Lmax,
                   int(lens[b]) + R - 1)
        assert same_bits(out[b * R:(b + 1) * R], one), f"sequence {b} (length {lens[b]}) differs when batched"
    o = host_u16(out).reshape(B, R, Hq, hd)
    for b in (1, 2, 7):
        for r, h in ((0, 0), (R - 1, 23)):
            g = h // (Hq // Hkv)
            ref = oracle.attn_row(q[b * R + r, h * hd:(h + 1) * hd], kc[b, g], vc[b, g], int(lens[b]) + r, hd ** -0.5)
            assert_bf16_close(o[b, r, h], ref, what=f"b{b} r{r} h{h}")
    assert xv.xv_device_check() == 0


def test_garbage_past_length_is_ignored(xv):
    """NaN and Inf bit patterns past the last visible position change nothing."""
    B, R, Hq, Hkv, hd, L, Lmax = 1, 8, 24, 4, 256, 1000, 1152
    q, kc, vc = make(5, B, R, Hq, Hkv, hd, Lmax, name="nan")
    Q = dev(q)
    clean = attn(xv, Q, dev(kc), dev(vc), dev(np.array([L], np.int32)), R, B, Hq, Hkv, hd, Lmax, L + R - 1)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, :, L + R - 1:] = 0x7FC0   # NaN
    vc2[:, :, L + R - 1:] = 0x7F80   # +Inf
    dirty = attn(xv, Q, dev(kc2), dev(vc2), dev(np.array([L], np.int32)), R, B, Hq, Hkv, hd, Lmax, L + R - 1)
    assert same_bits(clean, dirty)


def test_hundred_runs_identical(xv):
    B, R, Hq, Hkv, hd, Lmax = 2, 8, 24, 4, 256, 4096
    q, kc, vc = make(6, B, R, Hq, Hkv, hd, Lmax, name="rep")
    Q, K, V, ctx = dev(q), dev(kc), dev(vc), dev(np.array([3000, 1700], np.int32))
    ref = attn(xv, Q, K, V, ctx, R, B, Hq, Hkv, hd, Lmax, 3007)
    for _ in range(100):
        assert same_bits(attn(xv, Q, K, V, ctx, R, B, Hq, Hkv, hd, Lmax, 3007), ref)
    assert xv.xv_device_check() == 0


def test_kv_append_places_rows(xv):
    B, R, Hkv, hd, Lmax = 2, 3, 4, 256, 64
    src = synth.normal_bf16(7, synth.tid("kvsrc"), (B * R, 2 * Hkv * hd))
    kc = torch.zeros((B, Hkv, Lmax, hd), dtype=torch.int16, device="cuda")
    vc = torch.zeros_like(kc)
    ctx = np.array([10, 40], dtype=np.int32)      # visible length of row 0: row r lands at ctx - 1 + r
    xv.xv_kv_append(dev(src), 2 * Hkv * hd, dev(ctx), R, B, Hkv, hd, Lmax, kc, vc)
    k, v = host_u16(kc), host_u16(vc)
    for b in range(B):
        for r in range(R):
            row = src[b * R + r]
            assert np.array_equal(k[b, :, ctx[b] - 1 + r].reshape(-1), row[:Hkv * hd])
            assert np.array_equal(v[b, :, ctx[b] - 1 + r].reshape(-1), row[Hkv * hd:])
    assert int((k != 0).sum()) == B * R * Hkv * hd - int((src[:, :Hkv * hd] == 0).sum())


def to_pages(c, table, page, n_pages):
    """Scatters contiguous caches [B, Hkv, Lmax, hd] into a pool [n_pages, Hkv, page, hd] by table."""
    B, Hkv, Lmax, hd = c.shape
    pool = np.zeros((n_pages, Hkv, page, hd), dtype=c.dtype)
    for b in range(B):
        for j in range(table.shape[1]):
            n = min(page, Lmax - j * page)
            if n > 0 and table[b, j] >= 0:
                pool[table[b, j], :, :n] = c[b, :, j * page:j * page + n]
    return pool


def scattered_table(seed, B, max_pages, n_pages):
    """Every sequence's pages drawn without replacement from a pool larger than needed."""
    perm = np.random.default_rng(seed).permutation(n_pages)[: B * max_pages]
    return perm.reshape(B, max_pages).astype(np.int32)


@pytest.mark.parametrize("hd,Hq,Hkv,R,page,lens", [(256, 24, 4, 8, 64, [2183, 1, 640, 1500]),
                                                    (256, 24, 4, 9, 256, [513, 2047]),
                                                    (64, 6, 2, 4, 128, [63, 64, 65, 700])])
def test_paged_equals_contiguous(xv, hd, Hq, Hkv, R, page, lens):
    """The same values in scattered pages give the bits of the contiguous cache (and the oracle)."""
    B = len(lens)
    Lmax = (max(lens) + R + page - 1) // page * page
    max_pages = Lmax // page
    n_pages = B * max_pages + 5
    q, kc, vc = make(11, B, R, Hq, Hkv, hd, Lmax, name=f"pg{hd}{page}")
    table = scattered_table(page, B, max_pages, n_pages)
    ctx = np.array(lens, dtype=np.int32)
    max_ctx = max(lens) + R - 1
    ref = attn(xv, dev(q), dev(kc), dev(vc), dev(ctx), R, B, Hq, Hkv, hd, Lmax, max_ctx)
    kp, vp = dev(to_pages(kc, table, page, n_pages)), dev(to_pages(vc, table, page, n_pages))
    tab = dev(table)
    pages = xv.kv_pages(tab, page, n_pages)
    out = torch.empty((B * R, Hq * hd), dtype=torch.int16, device="cuda")
    ws = xv.workspace(xv.xv_attn_workspace_size(B, R, Hq, hd, max_ctx))
    xv.xv_attn_decode_rows_paged(dev(q), Hq * hd, kp, vp, pages, dev(ctx), R, B, Hq, Hkv, hd, max_ctx, hd ** -0.5,
                                 out, out.stride(0), ws)
    assert same_bits(out, ref), "paged attention differs from the contiguous cache"
    assert xv.xv_device_check() == 0
    b = 0
    exp = exact_rows(q[b * R:(b + 1) * R], kc[b], vc[b], lens[b], hd ** -0.5, R, Hq, Hkv, hd)
    assert_bf16_close(host_u16(out)[b * R:(b + 1) * R].reshape(R, Hq, hd), exp, what="paged attn vs oracle")


def test_kv_append_paged_places_rows(xv):
    B, R, Hkv, hd, page, max_pages = 2, 9, 4, 256, 64, 3
    n_pages = 8
    src = synth.normal_bf16(8, synth.tid("kvsrc_paged"), (B * R, 2 * Hkv * hd))
    table = np.array([[5, 2, 7], [0, 6, 3]], dtype=np.int32)
    kp = torch.zeros((n_pages, Hkv, page, hd), dtype=torch.int16, device="cuda")
    vp = torch.zeros_like(kp)
    ctx = np.array([60, 128], dtype=np.int32)     # sequence 0 crosses from its page 0 into page 1
    tab = dev(table)
    pages = xv.kv_pages(tab, page, n_pages)
    xv.xv_kv_append_paged(dev(src), 2 * Hkv * hd, dev(ctx), R, B, Hkv, hd, pages, kp, vp)
    k, v = host_u16(kp), host_u16(vp)
    for b in range(B):
        for r in range(R):
            p = ctx[b] - 1 + r
            pg, row = table[b, p // page], p % page
            assert np.array_equal(k[pg, :, row].reshape(-1), src[b * R + r, :Hkv * hd])
            assert np.array_equal(v[pg, :, row].reshape(-1), src[b * R + r, Hkv * hd:])
    assert int((k != 0).sum()) == B * R * Hkv * hd - int((src[:, :Hkv * hd] == 0).sum())
    assert xv.xv_device_check() == 0


def test_paged_arguments_rejected(xv):
    """Host checks: a page size that is not a multiple of 64, or max_ctx beyond the table's reach."""
    B, R, Hq, Hkv, hd = 1, 2, 4, 2, 64
    tab = torch.zeros((B, 2), dtype=torch.int32, device="cuda")
    kp = torch.zeros((2, Hkv, 96, hd), dtype=torch.int16, device="cuda")
    q = torch.zeros((B * R, Hq * hd), dtype=torch.int16, device="cuda")
    out = torch.empty_like(q)
    ctx = torch.ones(B, dtype=torch.int32, device="cuda")
    ws = xv.workspace(xv.xv_attn_workspace_size(B, R, Hq, hd, 256))
    with pytest.raises(xv.XVError):
        xv.xv_attn_decode_rows_paged(q, Hq * hd, kp, kp, xv.kv_pages(tab, 96, 2), ctx, R, B, Hq, Hkv, hd, 100, 0.125,
                                     out, Hq * hd, ws)
    with pytest.raises(xv.XVError):
        xv.xv_attn_decode_rows_paged(q, Hq * hd, kp, kp, xv.kv_pages(tab, 64, 2), ctx, R, B, Hq, Hkv, hd, 129, 0.125,
                                     out, Hq * hd, ws)
