"""GDN recurrence: decode and verify parity with the oracle, verify(k) == k
decode steps bit for bit, forced-reject rollback to every step j, 8
sequences in flight, and run-to-run repeatability — 32 heads of 128 x 128
fp32 state, the per-layer shape of the hybrid stack."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import assert_bf16_close, assert_state_close, dev, f64, host, host_u16, same_bits

pytestmark = pytest.mark.gpu

H, DK, DV = 32, 128, 128


@pytest.fixture(scope="module")
def xv():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv as m
    return m


def make_inputs(seed, B, T, H=H, dk=DK, dv=DV, prenorm=True):
    """Step rows [B*T, H*(2dk+dv)] = q | k | v and gates [B*T, 2H] = beta | gate, bf16 bits.
    With prenorm, q and k are L2-normalised per head (in double) before rounding."""
    rows = B * T
    q = synth.normal_f64(seed, synth.tid("gdn.q"), (rows, H, dk))
    k = synth.normal_f64(seed, synth.tid("gdn.k"), (rows, H, dk))
    if prenorm:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = synth.normal_f64(seed, synth.tid("gdn.v"), (rows, H, dv))
    qkv = np.concatenate([oracle.round_bf16(q).reshape(rows, -1), oracle.round_bf16(k).reshape(rows, -1),
                          oracle.round_bf16(v).reshape(rows, -1)], axis=1)
    bl = synth.normal_bf16(seed, synth.tid("gdn.b"), (rows, H))
    al = synth.normal_bf16(seed, synth.tid("gdn.a"), (rows, H))
    beta, gate = oracle.gdn_gates(bl, al)
    return np.ascontiguousarray(qkv), np.ascontiguousarray(np.concatenate([beta, gate], axis=1))


def init_state(seed, B, H=H, dk=DK, dv=DV):
    return synth.normal_f32(seed, synth.tid("gdn.S0"), (B, H, dv, dk), sigma=0.1)


def steps(xv, qkv, gates, rows_per_seq, H=H, dk=DK, dv=DV, row0=0):
    """xv_gdn_steps view of device buffers; row0 shifts the first row."""
    base = qkv[row0:]
    g = gates[row0:]
    return xv.gdn_steps(base, base[:, H * dk:], base[:, 2 * H * dk:], g, g[:, H:], qkv.shape[1], 2 * H, rows_per_seq)


def decode_seq(xv, S, qkv, gates, B, T, H=H, dk=DK, dv=DV, l2=False):
    """T decode steps over rows b*T + t; returns o [B, T, H*dv] (device)."""
    o = torch.empty((B, T, H * dv), dtype=torch.int16, device="cuda")
    for t in range(T):
        # rows b*T + t for every b: stride T rows apart
        base = qkv[t:]
        g = gates[t:]
        st = xv.gdn_steps(base, base[:, H * dk:], base[:, 2 * H * dk:], g, g[:, H:], qkv.shape[1] * T, 2 * H * T, 1)
        ob = torch.empty((B, H * dv), dtype=torch.int16, device="cuda")
        xv.xv_gdn_decode_step(S, st, ob, H * dv, B, H, dk, dv, l2)
        o[:, t] = ob
    return o


def test_decode_parity_with_oracle(xv):
    B, T = 2, 4
    qkv, gates = make_inputs(1, B, T)
    S0 = init_state(1, B)
    S = dev(S0)
    o = host_u16(decode_seq(xv, S, dev(qkv), dev(gates), B, T))
    Sref = S0.astype(np.float64)
    for b in range(B):
        for t in range(T):
            r = b * T + t
            q = qkv[r, :H * DK].reshape(H, DK)
            k = qkv[r, H * DK:2 * H * DK].reshape(H, DK)
            v = qkv[r, 2 * H * DK:].reshape(H, DV)
            ob = oracle.gdn_step_heads(Sref[b], q, k, v, gates[r, :H], gates[r, H:], l2=False)
            assert_bf16_close(o[b, t].reshape(H, DV), ob, what=f"o b{b} t{t}")
    assert_state_close(host(S), Sref, what="state after 4 decode steps")
    assert xv.xv_device_check() == 0


def test_inkernel_l2norm_parity(xv):
    B, T = 1, 3
    qkv, gates = make_inputs(2, B, T, prenorm=False)
    S0 = init_state(2, B)
    S = dev(S0)
    o = host_u16(decode_seq(xv, S, dev(qkv), dev(gates), B, T, l2=True))
    Sref = S0.astype(np.float64)
    for t in range(T):
        q = qkv[t, :H * DK].reshape(H, DK)
        k = qkv[t, H * DK:2 * H * DK].reshape(H, DK)
        v = qkv[t, 2 * H * DK:].reshape(H, DV)
        ob = oracle.gdn_step_heads(Sref[0], q, k, v, gates[t, :H], gates[t, H:], l2=True)
        assert_bf16_close(o[0, t].reshape(H, DV), ob, what=f"o t{t}")
    assert_state_close(host(S), Sref, what="state (in-kernel l2norm)")


def test_dk64_tiny_heads(xv):
    B, T, h, d = 1, 4, 2, 64
    qkv, gates = make_inputs(3, B, T, H=h, dk=d, dv=d)
    S0 = init_state(3, B, H=h, dk=d, dv=d)
    S = dev(S0)
    o = host_u16(decode_seq(xv, S, dev(qkv), dev(gates), B, T, H=h, dk=d, dv=d))
    Sref = S0.astype(np.float64)
    for t in range(T):
        q = qkv[t, :h * d].reshape(h, d)
        k = qkv[t, h * d:2 * h * d].reshape(h, d)
        v = qkv[t, 2 * h * d:].reshape(h, d)
        ob = oracle.gdn_step_heads(Sref[0], q, k, v, gates[t, :h], gates[t, h:], l2=False)
        assert_bf16_close(o[0, t].reshape(h, d), ob, what=f"o t{t}")
    assert_state_close(host(S), Sref)


@pytest.mark.parametrize("B,K", [(1, 8), (8, 8), (1, 64)])
def test_verify_equals_sequential_decode_and_rollback(xv, B, K):
    qkv_h, gates_h = make_inputs(4, B, K)
    qkv, gates = dev(qkv_h), dev(gates_h)
    S0 = dev(init_state(4, B))
    # decode path: states after each step, outputs per step
    Sd = S0.clone()
    states = []
    o_dec = torch.empty((B, K, H * DV), dtype=torch.int16, device="cuda")
    for t in range(K):
        base, g = qkv[t:], gates[t:]
        st = xv.gdn_steps(base, base[:, H * DK:], base[:, 2 * H * DK:], g, g[:, H:], qkv.shape[1] * K, 2 * H * K, 1)
        ob = torch.empty((B, H * DV), dtype=torch.int16, device="cuda")
        xv.xv_gdn_decode_step(Sd, st, ob, H * DV, B, H, DK, DV, False)
        o_dec[:, t] = ob
        states.append(Sd.clone())
    # verify path
    Sv = S0.clone()
    o_ver = torch.empty((B * K, H * DV), dtype=torch.int16, device="cuda")
    draft = steps(xv, qkv, gates, K)
    xv.xv_gdn_verify(Sv, None, None, 0, draft, K, o_ver, H * DV, B, H, DK, DV, False)
    assert same_bits(Sv, S0), "speculative steps must not write the state"
    assert same_bits(o_ver.view(B, K, -1), o_dec), "verify outputs differ from decode outputs"
    # forced rejects / partial accepts: commit j+1 steps
    for j in range(K):
        Sc = S0.clone()
        n = torch.full((B,), j + 1, dtype=torch.int32, device="cuda")
        xv.xv_gdn_verify(Sc, draft, n, K, None, 0, None, 0, B, H, DK, DV, False)
        assert same_bits(Sc, states[j]), f"state after committing {j + 1} steps differs from decode"
    assert xv.xv_device_check() == 0


@pytest.mark.parametrize("K,keep", [(8, 3), (64, 37), (64, 64)])
def test_replay_then_speculate_matches_decode(xv, K, keep):
    """The second pass of a speculative loop: replay `keep` kept steps, speculate K new ones (up to 128
    staged steps in one call)."""
    B = 2
    qkv_h, gates_h = make_inputs(5, B, 2 * K)          # rows b*2K + t: first K = first verify, last K = second verify
    qkv, gates = dev(qkv_h), dev(gates_h)
    S0 = dev(init_state(5, B))
    # decode reference: `keep` steps of the first verify, then the K of the second
    Sd = S0.clone()
    outs = []
    for t in list(range(keep)) + list(range(K, 2 * K)):
        base, g = qkv[t:], gates[t:]
        st = xv.gdn_steps(base, base[:, H * DK:], base[:, 2 * H * DK:], g, g[:, H:], qkv.shape[1] * 2 * K,
                          2 * H * 2 * K, 1)
        ob = torch.empty((B, H * DV), dtype=torch.int16, device="cuda")
        xv.xv_gdn_decode_step(Sd, st, ob, H * DV, B, H, DK, DV, False)
        outs.append(ob)
    ref = torch.stack(outs[keep:], dim=1)
    # verify: pending = the first verify's rows (rows_per_seq 2K from row 0), draft = the second's (from row K)
    Sv = S0.clone()
    pend = steps(xv, qkv, gates, 2 * K)
    draft = steps(xv, qkv, gates, 2 * K, row0=K)
    n = torch.full((B,), keep, dtype=torch.int32, device="cuda")
    o = torch.empty((B * K, H * DV), dtype=torch.int16, device="cuda")
    xv.xv_gdn_verify(Sv, pend, n, K, draft, K, o, H * DV, B, H, DK, DV, False)
    assert same_bits(o.view(B, K, -1), ref)
    # the stored state is the committed one (after the 3 kept steps)
    Sk = S0.clone()
    xv.xv_gdn_verify(Sk, pend, n, K, None, 0, None, 0, B, H, DK, DV, False)
    assert same_bits(Sv, Sk)


def test_eight_in_flight_equal_alone(xv):
    B, K = 8, 8
    qkv_h, gates_h = make_inputs(6, B, K)
    qkv, gates = dev(qkv_h), dev(gates_h)
    S0 = dev(init_state(6, B))
    n_h = np.array([1, 8, 3, 0, 5, 2, 7, 4], dtype=np.int32)
    Sb = S0.clone()
    o = torch.empty((B * K, H * DV), dtype=torch.int16, device="cuda")
    pend = steps(xv, qkv, gates, K)
    xv.xv_gdn_verify(Sb, pend, dev(n_h), K, pend, K, o, H * DV, B, H, DK, DV, True)
    for b in range(B):
        Sa = S0[b:b + 1].clone()
        oa = torch.empty((K, H * DV), dtype=torch.int16, device="cuda")
        pa = steps(xv, qkv, gates, K, row0=b * K)
        xv.xv_gdn_verify(Sa, pa, dev(n_h[b:b + 1]), K, pa, K, oa, H * DV, 1, H, DK, DV, True)
        assert same_bits(Sa[0], Sb[b]) and same_bits(oa, o[b * K:(b + 1) * K]), f"sequence {b} differs in the batch"


def test_hundred_runs_identical(xv):
    B, K = 8, 8
    qkv_h, gates_h = make_inputs(7, B, K)
    qkv, gates = dev(qkv_h), dev(gates_h)
    S0 = dev(init_state(7, B))
    n = torch.full((B,), 3, dtype=torch.int32, device="cuda")
    pend = steps(xv, qkv, gates, K)
    ref_S, ref_o = None, None
    for _ in range(100):
        S = S0.clone()
        o = torch.empty((B * K, H * DV), dtype=torch.int16, device="cuda")
        xv.xv_gdn_verify(S, pend, n, K, pend, K, o, H * DV, B, H, DK, DV, True)
        if ref_S is None:
            ref_S, ref_o = S, o
        else:
            assert same_bits(S, ref_S) and same_bits(o, ref_o)
    assert xv.xv_device_check() == 0


def grouped_inputs(seed, B, T, Hv, Hk, d):
    """Step rows [B*T, 2*Hk*d + Hv*d] = q | k (Hk heads, raw) | v (Hv heads) and gates [B*T, 2*Hv]."""
    rows = B * T
    q = synth.normal_bf16(seed, synth.tid("gw.q"), (rows, Hk * d))
    k = synth.normal_bf16(seed, synth.tid("gw.k"), (rows, Hk * d))
    v = synth.normal_bf16(seed, synth.tid("gw.v"), (rows, Hv * d))
    bl = synth.normal_bf16(seed, synth.tid("gw.b"), (rows, Hv))
    al = synth.normal_bf16(seed, synth.tid("gw.a"), (rows, Hv))
    beta, gate = oracle.gdn_gates(bl, al)
    return np.ascontiguousarray(np.concatenate([q, k, v], axis=1)), np.ascontiguousarray(np.concatenate([beta, gate], 1))


@pytest.mark.parametrize("Hv,Hk,d", [(32, 32, 64), (32, 16, 128), (48, 48, 128)])
def test_wide_batch_equals_each_sequence_alone_and_oracle(xv, Hv, Hk, d):
    """A batch wide enough for the per-head kernel (B * heads >= SMs: a CTA per head, 4 rows per
    thread) against each sequence alone (the per-slab kernel, a row per thread): outputs and
    committed states bit for bit, with a different replay count per sequence, grouped q/k heads
    and dk = 64 or 128; sequence 0 of the batch against the oracle's steps."""
    B, K = 8, 8
    qkv_h, gates_h = grouped_inputs(8, B, K, Hv, Hk, d)
    qkv, gates = dev(qkv_h), dev(gates_h)
    S0h = synth.normal_f32(8, synth.tid("gw.S0"), (B, Hv, d, d), sigma=0.1)
    S0 = dev(S0h)
    n_h = np.array([1, 8, 3, 0, 5, 2, 7, 4], dtype=np.int32)

    def view(buf, g, row0=0):
        base, gg = buf[row0:], g[row0:]
        return xv.gdn_steps(base, base[:, Hk * d:], base[:, 2 * Hk * d:], gg, gg[:, Hv:], buf.shape[1], 2 * Hv, K)

    Sb = S0.clone()
    o = torch.full((B * K, Hv * d), -1, dtype=torch.int16, device="cuda")
    xv.xv_gdn_verify_grouped(Sb, view(qkv, gates), dev(n_h), K, view(qkv, gates), K, o, Hv * d, B, Hv, Hk, d, d, True)
    for b in range(B):
        Sa = S0[b:b + 1].clone()
        oa = torch.full((K, Hv * d), -1, dtype=torch.int16, device="cuda")
        pa = view(qkv, gates, b * K)
        xv.xv_gdn_verify_grouped(Sa, pa, dev(n_h[b:b + 1]), K, pa, K, oa, Hv * d, 1, Hv, Hk, d, d, True)
        assert same_bits(Sa[0], Sb[b]) and same_bits(oa, o[b * K:(b + 1) * K]), f"sequence {b} differs in the batch"
    assert xv.xv_device_check() == 0
    # the oracle: sequence 0 replays n_h[0] pending rows into the state, then speculates K rows
    S = S0h[0].astype(np.float64)
    q = qkv_h[:, :Hk * d].reshape(B * K, Hk, d)
    k = qkv_h[:, Hk * d:2 * Hk * d].reshape(B * K, Hk, d)
    v = qkv_h[:, 2 * Hk * d:].reshape(B * K, Hv, d)
    for t in range(n_h[0]):
        oracle.gdn_step_heads_grouped(S, q[t], k[t], v[t], gates_h[t, :Hv], gates_h[t, Hv:], True)
    assert_state_close(host(Sb)[0], S)
    og = host_u16(o)
    Ss = S.copy()
    for t in range(K):
        ob = oracle.gdn_step_heads_grouped(Ss, q[t], k[t], v[t], gates_h[t, :Hv], gates_h[t, Hv:], True)
        assert_bf16_close(og[t].reshape(Hv, d), ob, what=f"speculative step {t}")


def test_wide_batch_decode_equals_alone(xv):
    """Decode steps (a replayed step that emits its output) at B = 8 with dk = dv = 64 (the per-head
    kernel) equal the same steps of each sequence alone."""
    B, T, h, d = 8, 3, 32, 64
    qkv_h, gates_h = make_inputs(9, B, T, H=h, dk=d, dv=d, prenorm=False)
    qkv, gates = dev(qkv_h), dev(gates_h)
    S0 = dev(init_state(9, B, H=h, dk=d, dv=d))
    Sb = S0.clone()
    ob = decode_seq(xv, Sb, qkv, gates, B, T, H=h, dk=d, dv=d, l2=True)
    for b in range(B):
        Sa = S0[b:b + 1].clone()
        oa = decode_seq(xv, Sa, qkv[b * T:(b + 1) * T], gates[b * T:(b + 1) * T], 1, T, H=h, dk=d, dv=d, l2=True)
        assert same_bits(Sa[0], Sb[b]) and same_bits(oa[0], ob[b]), f"sequence {b}"
