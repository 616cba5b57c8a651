"""The complete GDN layer's parts on the GPU: the causal convolution (its
state commit is an exact copy; its outputs match the oracle's convolution
within the bf16 tolerance and verify rows equal decode steps bit for bit),
the gated output norm, grouped q/k heads; and the whole block with complete
GDN layers: verify(k) == k sequential decodes bit for bit, forced rejects,
8 sequences in flight, oracle parity."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads
from _block import gpu_stack, oracle_logits, oracle_stack
from _gpu import assert_argmax, assert_bf16_close, assert_block_close, assert_state_close, dev, host, \
    host_u16, rms, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xv():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv as m
    return m


def conv_inputs(seed, B, T, C, Kc):
    w = synth.normal_bf16(seed, synth.tid("cv.w"), (C, Kc), 0.5)
    x = synth.normal_bf16(seed, synth.tid("cv.x"), (B * T, C))
    st = synth.normal_bf16(seed, synth.tid("cv.s"), (B, Kc - 1, C))
    return w, x, st


@pytest.mark.parametrize("Kc,C", [(4, 8192), (2, 96), (8, 200)])
def test_conv_decode_parity_and_state(xv, Kc, C):
    """T one-row calls (each committing the previous row) against the oracle's steps: outputs
    within bf16 tolerance, the state an exact copy of the inputs."""
    B, T = 3, 5
    w, x, st0 = conv_inputs(1, B, T, C, Kc)
    xr = x.reshape(B, T, C)
    S = dev(st0)
    W, X = dev(w), dev(x)
    one = torch.ones(B, dtype=torch.int32, device="cuda")
    ys = []
    for t in range(T):
        y = torch.empty((B, C), dtype=torch.int16, device="cuda")
        prev = X[t - 1:] if t > 0 else X
        # row b*T + t of x for sequence b: one row per sequence at stride T rows, from offset t
        xv.xv_gdn_conv(S, prev, C * T, 1, one, 1 if t > 0 else 0, X[t:], C * T, 1, 1, W, B, y, C)
        ys.append(host_u16(y))
    for b in range(B):
        ost = st0[b].copy()
        for t in range(T):
            ref = oracle.conv_step(ost, xr[b, t], w)
            assert_bf16_close(ys[t][b], oracle.bf16_to_f64(ref), what=f"conv b{b} t{t}")
        # the GPU state has not yet taken the last row (deferred); the oracle's has
        exp = np.concatenate([st0[b], xr[b]], axis=0)[T - 1:T - 1 + Kc - 1]
        assert np.array_equal(host_u16(S)[b], exp)
    assert xv.xv_device_check() == 0


@pytest.mark.parametrize("k", [8, 64])
def test_conv_verify_rows_equal_decode_and_commit_any_j(xv, k):
    """k rows in one call equal k one-row calls bit for bit; committing j of them shifts exactly
    those j into the state."""
    B, C, Kc = 2, 1024, 4
    w, x, st0 = conv_inputs(2, B, k, C, Kc)
    W, X = dev(w), dev(x)
    S = dev(st0)
    Y = torch.empty((B * k, C), dtype=torch.int16, device="cuda")
    xv.xv_gdn_conv(S, None, 0, 0, None, 0, X, C, k, k, W, B, Y, C)
    S1 = dev(st0)
    one = torch.ones(B, dtype=torch.int32, device="cuda")
    for t in range(k):
        y = torch.empty((B, C), dtype=torch.int16, device="cuda")
        xv.xv_gdn_conv(S1, X[t - 1:] if t else X, C * k, 1, one, 1 if t else 0, X[t:], C * k, 1, 1, W, B, y, C)
        assert same_bits(y, Y.view(B, k, C)[:, t]), f"row {t}"
    for j in range(0, k + 1):
        Sj = dev(st0)
        nc = torch.full((B,), j, dtype=torch.int32, device="cuda")
        xv.xv_gdn_conv(Sj, X, C, k, nc, k, None, 0, 0, 0, None, B, None, 0)    # commit only
        for b in range(B):
            exp = np.concatenate([st0[b], x.reshape(B, k, C)[b, :j]], axis=0)[j:j + Kc - 1]
            assert np.array_equal(host_u16(Sj)[b], exp), (j, b)
    assert xv.xv_device_check() == 0


def test_gated_norm_parity(xv):
    M, Hh, dv = 9, 32, 128
    o = synth.normal_bf16(3, synth.tid("gn.o"), (M, Hh * dv))
    z = synth.normal_bf16(3, synth.tid("gn.z"), (M, 2 * Hh * dv))   # z in a wider row
    w = synth.normal_bf16(3, synth.tid("gn.w"), (dv,), 0.02)
    O, Z = dev(o), dev(z)
    Y = torch.empty_like(O)
    xv.xv_gated_norm(O, Hh * dv, Z[:, Hh * dv:], 2 * Hh * dv, dev(w), M, Hh, dv, 1e-6, Y, Hh * dv)
    ref = oracle.gated_norm(o.reshape(M, Hh, dv), z[:, Hh * dv:].reshape(M, Hh, dv), w)
    assert_bf16_close(host_u16(Y).reshape(M, Hh, dv), oracle.bf16_to_f64(ref), what="gated norm")
    # in place gives the same bits
    xv.xv_gated_norm(O, Hh * dv, Z[:, Hh * dv:], 2 * Hh * dv, dev(w), M, Hh, dv, 1e-6, O, Hh * dv)
    assert same_bits(O, Y)
    assert xv.xv_device_check() == 0


def test_grouped_heads_verify_parity(xv):
    """32 v heads over 16 q/k heads: verify of 4 steps against the oracle's grouped steps."""
    B, T, Hv, Hk, dk, dv = 2, 4, 32, 16, 128, 128
    rows = B * T
    q = oracle.round_bf16(synth.normal_f64(4, synth.tid("gq.q"), (rows, Hk * dk)))
    k = oracle.round_bf16(synth.normal_f64(4, synth.tid("gq.k"), (rows, Hk * dk)))
    v = synth.normal_bf16(4, synth.tid("gq.v"), (rows, Hv * dv))
    qkv = np.ascontiguousarray(np.concatenate([q, k, v], axis=1))
    beta, gate = oracle.gdn_gates(synth.normal_bf16(4, synth.tid("gq.b"), (rows, Hv)),
                                  synth.normal_bf16(4, synth.tid("gq.a"), (rows, Hv)))
    gates = np.ascontiguousarray(np.concatenate([beta, gate], axis=1))
    S0 = synth.normal_f32(4, synth.tid("gq.S"), (B, Hv, dv, dk), sigma=0.1)
    Q, G, S = dev(qkv), dev(gates), dev(S0)
    draft = xv.gdn_steps(Q, Q[:, Hk * dk:], Q[:, 2 * Hk * dk:], G, G[:, Hv:], qkv.shape[1], 2 * Hv, T)
    o = torch.empty((rows, Hv * dv), dtype=torch.int16, device="cuda")
    xv.xv_gdn_verify_grouped(S, None, None, 0, draft, T, o, Hv * dv, B, Hv, Hk, dk, dv, True)
    og = host_u16(o)
    for b in range(B):
        Sref = S0[b].astype(np.float64)
        for t in range(T):
            r = b * T + t
            ref = oracle.gdn_step_heads_grouped(Sref, q[r].reshape(Hk, dk), k[r].reshape(Hk, dk),
                                                v[r].reshape(Hv, dv), beta[r], gate[r], True)
            assert_bf16_close(og[r].reshape(Hv, dv), oracle.bf16_to_f64(ref), what=f"grouped b{b} t{t}")
    assert xv.xv_device_check() == 0


# ----------------------------------------------------------- the block

def sequential(stk, toks, B):
    T = toks.shape[1]
    lgs, ams = [], []
    one = torch.ones(B, dtype=torch.int32, device="cuda")
    for t in range(T):
        lg, am, _ = stk.verify(dev(np.ascontiguousarray(toks[:, t:t + 1])), 1)
        lgs.append(lg.clone())
        ams.append(am.clone())
        stk.commit(one)
    return torch.stack(lgs, 1), torch.stack(ams, 1)


@pytest.fixture(scope="module")
def tiny_full(xv):
    cfg = workloads.TINY_FULL
    return cfg, workloads.weights(cfg, seed=0)


def test_tiny_full_verify_equals_decode_and_oracle(tiny_full):
    cfg, w = tiny_full
    B, k, L, Lmax = 1, 4, 128, 256
    toks = workloads.draft_tokens(cfg, 0, 0, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, [L])
    lg, am, na = A.verify(dev(toks), k)
    lgA, amA = lg.clone(), am.clone()
    S = gpu_stack(cfg, w, B, k, Lmax, [L])
    lgS, amS = sequential(S, toks, B)
    assert same_bits(lgA.view(B, k, -1), lgS)
    assert torch.equal(amA.view(B, k), amS)
    ref, spread, _ = oracle_logits(cfg, w, 0, B, [L], Lmax, toks[0], extra=60)
    mb = assert_block_close(host(lgA), ref, spread, what="complete GDN tiny logits vs oracle")
    assert_argmax(host(amA), host(lgA), ref, mb)


@pytest.mark.parametrize("keep", [1, 2, 4])
def test_tiny_full_forced_reject_then_next_round(tiny_full, keep):
    """Keep `keep` positions, verify 4 more: logits equal decoding the kept tokens and then the new
    ones; after flushing, GDN and convolution states agree bit for bit and with the oracle."""
    cfg, w = tiny_full
    B, k, L, Lmax = 2, 4, 128, 256
    lens = [L, 77]
    t1 = workloads.draft_tokens(cfg, 0, 1, B, k)
    t2 = workloads.draft_tokens(cfg, 0, 2, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, lens)
    A.verify(dev(t1), k)
    A.commit(torch.full((B,), keep, dtype=torch.int32, device="cuda"))
    lgA = A.verify(dev(t2), k)[0].clone()
    S = gpu_stack(cfg, w, B, k, Lmax, lens)
    sequential(S, t1[:, :keep], B)
    lgS, _ = sequential(S, t2, B)
    assert same_bits(lgA.view(B, k, -1), lgS)
    A.commit(torch.full((B,), k, dtype=torch.int32, device="cuda"))
    A.flush()
    S.flush()
    assert same_bits(A.state["0.state"], S.state["0.state"])
    assert same_bits(A.state["0.conv"], S.state["0.conv"])
    ref, spread, ost = oracle_logits(cfg, w, 0, B, lens, Lmax, t2[0], before=t1[0, :keep], extra=60)
    assert_block_close(host(lgA)[:k], ref, spread, what="after rollback vs oracle")
    assert np.array_equal(host_u16(A.state["0.conv"])[0], ost.conv[0])     # data movement only: exact
    assert_state_close(host(A.state["0.state"])[0], ost.S[0], rel=2e-2)


def test_tiny_full_speculative_rounds_emit_greedy_decode(tiny_full):
    from bit_exact_speculative_gb300.speculative import ReplayDrafter, greedy_decode, speculative_decode
    cfg, w = tiny_full
    B, k, L, n = 1, 4, 128, 40
    Lmax = L + 3 * n + 4 * k
    first = int(workloads.draft_tokens(cfg, 0, 99, 1, 1)[0, 0])
    ref = greedy_decode(gpu_stack(cfg, w, B, k, Lmax, [L]), first, n)
    for accept in (1.0, 0.5, 0.0):
        S = gpu_stack(cfg, w, B, k, Lmax, [L])
        out, acc = speculative_decode(S, first, n, k, ReplayDrafter(ref, cfg["vocab"], accept, seed=3))
        assert out[:n] == ref[1:n + 1], f"accept {accept}"


def test_stack_full_verify_equals_decode_and_in_flight(xv):
    """The 5120-wide stack with complete GDN layers (32 v / 16 q/k heads, width-4 convolution,
    gated norm): verify == sequential decode bit for bit; a sequence's rows do not depend on
    its neighbours; oracle parity on one position."""
    cfg = workloads.STACK_FULL
    w = workloads.weights(cfg, seed=0)
    wd = {n: dev(a) for n, a in w.items()}
    B, k = 2, 8
    lens = [2183, 640]
    Lmax = 2304
    toks = workloads.draft_tokens(cfg, 0, 0, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    lgA = A.verify(dev(toks), k)[0].clone()
    S = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    lgS, _ = sequential(S, toks, B)
    assert same_bits(lgA.view(B, k, -1), lgS)
    toks2 = workloads.draft_tokens(cfg, 0, 5, B, k)
    toks2[0] = toks[0]
    C = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    lgC = C.verify(dev(toks2), k)[0].view(B, k, -1)
    assert same_bits(lgC[0], lgA.view(B, k, -1)[0])
    ref, spread, _ = oracle_logits(cfg, w, 0, B, lens, Lmax, toks[0, :1])
    assert_block_close(host(lgA)[:1], ref, spread, what="complete GDN stack vs oracle")
    from bit_exact_speculative_gb300 import xv as m
    assert m.xv_device_check() == 0
