"""The verify block end to end: verify(k) gives the logits and argmax of k
sequential decodes bit for bit, also after forced rejects and with 8
sequences in flight; logits match the oracle's sequential decode within the
stated tolerance.  Tiny hybrid block and the 4-layer 5120-wide stack."""
import numpy as np
import pytest
import torch

import oracle
from synth import workloads
from _block import gpu_stack, kv_host, oracle_logits, oracle_stack, restore, snapshot
from _gpu import assert_argmax, assert_block_close, assert_layer_close, dev, host, host_u16, rms, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from bit_exact_speculative_gb300 import build
    build.build()
    from bit_exact_speculative_gb300 import xv
    return xv


def sequential(stk, toks, B):
    """Decode each column of toks (k = 1 verify + keep 1); returns logits [B, T, V], argmax [B, T]."""
    T = toks.shape[1]
    lgs, ams = [], []
    one = torch.ones(B, dtype=torch.int32, device="cuda")
    for t in range(T):
        lg, am, _ = stk.verify(dev(np.ascontiguousarray(toks[:, t:t + 1])), 1)
        lgs.append(lg.clone())
        ams.append(am.clone())
        stk.commit(one)
    return torch.stack(lgs, 1), torch.stack(ams, 1)


# ------------------------------------------------------------ tiny block

@pytest.fixture(scope="module")
def tiny(built):
    cfg = workloads.TINY
    return cfg, workloads.weights(cfg, seed=0)


def test_tiny_verify_equals_sequential_decode_and_oracle(tiny):
    cfg, w = tiny
    B, k, L, Lmax = 1, 4, 128, 256
    toks = workloads.draft_tokens(cfg, 0, 0, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, [L])
    lg, am, na = A.verify(dev(toks), k)
    lgA, amA = lg.clone(), am.clone()
    S = gpu_stack(cfg, w, B, k, Lmax, [L])
    lgS, amS = sequential(S, toks, B)
    assert same_bits(lgA.view(B, k, -1), lgS), "verify logits differ from sequential decode"
    assert torch.equal(amA.view(B, k), amS)
    ref, spread, _ = oracle_logits(cfg, w, 0, B, [L], Lmax, toks[0], extra=60)
    mb = assert_block_close(host(lgA), ref, spread, what="tiny logits vs oracle")
    assert_argmax(host(amA), host(lgA), ref, mb)
    # n_accept follows the rule on the GPU's own argmax
    assert int(na[0]) == oracle.accept(toks[0], host(amA))


@pytest.mark.parametrize("keep", [1, 2, 3, 4])
def test_tiny_forced_reject_then_next_round(tiny, keep):
    """Keep `keep` positions of a verify (keep = 1 is every draft rejected), verify 4 more tokens:
    logits equal decoding the kept tokens and then the new ones; GDN state after a flush matches."""
    cfg, w = tiny
    B, k, L, Lmax = 1, 4, 128, 256
    t1 = workloads.draft_tokens(cfg, 0, 1, B, k)
    t2 = workloads.draft_tokens(cfg, 0, 2, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, [L])
    A.verify(dev(t1), k)
    A.commit(torch.full((B,), keep, dtype=torch.int32, device="cuda"))
    lg, am, _ = A.verify(dev(t2), k)
    lgA = lg.clone()
    S = gpu_stack(cfg, w, B, k, Lmax, [L])
    sequential(S, t1[:, :keep], B)
    lgS, _ = sequential(S, t2, B)
    assert same_bits(lgA.view(B, k, -1), lgS)
    # commit all of the second verify and flush both: GDN states and lengths agree bit for bit
    A.commit(torch.full((B,), k, dtype=torch.int32, device="cuda"))
    A.flush()
    S.flush()
    assert torch.equal(A.state["ctx_len"], S.state["ctx_len"])
    assert same_bits(A.state["0.state"], S.state["0.state"])
    # and the oracle, decoding the same kept tokens, agrees within tolerance
    ref, spread, ost = oracle_logits(cfg, w, 0, B, [L], Lmax, t2[0], before=t1[0, :keep], extra=60)
    assert_block_close(host(lgA), ref, spread, what="after rollback vs oracle")
    Sg = host(A.state["0.state"])[0]
    assert float(np.max(np.abs(Sg - ost.S[0]))) <= 2e-2 * rms(ost.S[0])


def test_tiny_speculative_rounds_emit_greedy_decode(tiny):
    """Verify/accept/commit rounds with drafts partly right: the emitted tokens are exactly
    the target's greedy decode, and each round accepts at least the right drafts."""
    cfg, w = tiny
    B, k, L, Lmax = 1, 4, 128, 512
    S = gpu_stack(cfg, w, B, k, Lmax, [L])
    first = int(workloads.draft_tokens(cfg, 0, 99, 1, 1)[0, 0])
    greedy, t = [], first
    for _ in range(40):
        _, am, _ = S.verify(dev(np.array([[t]], dtype=np.int32)), 1)
        S.commit(torch.ones(1, dtype=torch.int32, device="cuda"))
        t = int(host(am)[0])
        greedy.append(t)
    A = gpu_stack(cfg, w, B, k, Lmax, [L])
    rng = np.random.default_rng(0)
    prev, pos, rnd = first, 0, 0
    while pos + k <= len(greedy):
        n_right = int(rng.integers(0, k))
        junk = list(workloads.draft_tokens(cfg, 0, 200 + rnd, 1, k)[0])
        drafts = greedy[pos:pos + n_right] + [(x + 1) % cfg["vocab"] if x == g else x
                                               for x, g in zip(junk, greedy[pos + n_right:])][: k - 1 - n_right]
        toks = np.array([[prev] + drafts], dtype=np.int32)
        _, am, na = A.verify(dev(toks), k)
        n = int(host(na)[0])
        assert n == n_right
        out = [int(x) for x in host(am)[: n + 1]]
        assert out == greedy[pos:pos + n + 1], f"round {rnd}"
        A.commit()
        prev, pos, rnd = out[-1], pos + n + 1, rnd + 1
    assert int(host(A.state["ctx_len"])[0]) == L + pos
    # the oracle, decoding the tokens the rounds emitted, predicts each next one wherever its
    # margin is decisive
    fed = [first] + greedy[:pos - 1]
    ref, spread, _ = oracle_logits(cfg, w, 0, B, [L], Lmax, np.array(fed, dtype=np.int32))
    mb = 3.0 * float(np.max(np.abs(spread)))
    decisive = 0
    for j, r in enumerate(ref):
        top2 = np.partition(r, -2)[-2:]
        if top2[1] - top2[0] > 2 * mb:
            assert greedy[j] == int(np.argmax(r)), f"position {j}: emitted {greedy[j]}, oracle {int(np.argmax(r))}"
            decisive += 1
    assert decisive >= 1


# ------------------------------------------------------ 4-layer stack

@pytest.fixture(scope="module")
def stack(built):
    """The 5120-wide stack with its GEMM weights in the tiled layout (as the bench runs it); the
    tiny blocks keep row-major weights."""
    from bit_exact_speculative_gb300.model import tile_weights
    cfg = workloads.STACK
    w = workloads.weights(cfg, seed=0)
    wd = tile_weights(cfg, {k: dev(v) for k, v in w.items()})
    return cfg, w, wd


def test_stack_verify_equals_sequential_decode(stack):
    cfg, w, wd = stack
    B, k, L = 1, 8, 2183
    Lmax = L + 64
    toks = workloads.draft_tokens(cfg, 0, 0, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lg, am, na = A.verify(dev(toks), k)
    lgA, amA = lg.clone(), am.clone()
    S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lgS, amS = sequential(S, toks, B)
    assert same_bits(lgA.view(B, k, -1), lgS)
    assert torch.equal(amA.view(B, k), amS)
    # oracle parity on all k positions (each oracle decode streams 6 GB of weights, twice: the
    # double evaluation and the single-precision one that sizes the bound)
    ref, spread, _ = oracle_logits(cfg, w, 0, B, [L], Lmax, toks[0])
    mb = assert_block_close(host(lgA), ref, spread, what="stack logits vs oracle")
    assert_argmax(host(amA), host(lgA), ref, mb)


def test_stack_forced_reject_every_j(stack):
    cfg, w, wd = stack
    B, k, L = 1, 8, 2183
    Lmax = L + 64
    t1 = workloads.draft_tokens(cfg, 0, 1, B, k)
    t2 = workloads.draft_tokens(cfg, 0, 2, B, k)
    S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    for keep in range(1, k + 1):
        A = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
        A.verify(dev(t1), k)
        A.commit(torch.full((B,), keep, dtype=torch.int32, device="cuda"))
        lgA = A.verify(dev(t2), k)[0].clone()
        S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
        sequential(S, t1[:, :keep], B)
        lgS, _ = sequential(S, t2, B)
        assert same_bits(lgA.view(B, k, -1), lgS), f"keep={keep}"
        del A, S
        torch.cuda.empty_cache()


@pytest.mark.parametrize("lens", [[2183, 640, 1000, 1, 513, 2047, 300, 1500],
                                  [131072, 70001, 1, 513, 131000, 2183, 64, 99999]], ids=["2183", "131072"])
def test_stack_eight_in_flight(stack, lens):
    """8 sequences of mixed lengths verifying k = 8 (64 token rows: the wide-batch GEMM path whose
    split-K partials the residual norm sums): the batch's logits, argmax and accept counts equal
    8 sequential decode steps of the batch and each sequence verified alone at B = 1, bit for bit.
    At 131072 the persistent attention CTAs walk items across sequences of different lengths."""
    cfg, w, wd = stack
    B, k = 8, 8
    Lmax = (max(lens) + 2 * k + 63) // 64 * 64
    kv = kv_host(cfg, lens, Lmax)
    toks = workloads.draft_tokens(cfg, 0, 3, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
    lg, am, na = A.verify(dev(toks), k)
    lgA, amA, naA = lg.clone().view(B, k, -1), am.clone().view(B, k), na.clone()
    del A
    S = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
    lgS, amS = sequential(S, toks, B)
    assert same_bits(lgA, lgS), "batch verify differs from the batch's sequential decode"
    assert torch.equal(amA, amS)
    del S, lgS
    torch.cuda.empty_cache()
    for b in range(B):
        one = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, only=b, kv=kv)
        lg1, am1, na1 = one.verify(dev(toks[b:b + 1]), k)
        assert same_bits(lg1.view(k, -1), lgA[b]), f"sequence {b} in the batch differs from it alone"
        assert torch.equal(am1, amA[b]) and int(na1[0]) == int(naA[b])
        del one
        torch.cuda.empty_cache()
    from bit_exact_speculative_gb300 import xv
    assert xv.xv_device_check() == 0


def test_stack_eight_in_flight_hundred_runs(stack):
    """100 runs of the same two verify/accept/commit rounds of 8 sequences from the same state
    (restored between runs): every run's logits, argmax, accept counts and lengths equal run 0's
    byte for byte (the second round replays the first round's accepted GDN steps)."""
    cfg, w, wd = stack
    B, k = 8, 8
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500]
    Lmax = 2304
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    snap = snapshot(A)
    t1, t2 = dev(workloads.draft_tokens(cfg, 0, 40, B, k)), dev(workloads.draft_tokens(cfg, 0, 41, B, k))

    def run():
        restore(A, snap)
        out = []
        for t in (t1, t2):
            lg, am, na = A.verify(t, k)
            out += [lg.clone(), am.clone(), na.clone()]
            A.commit()
        out.append(A.state["ctx_len"].clone())
        return out

    r0 = run()
    for i in range(1, 100):
        r = run()
        assert all(same_bits(a, b) for a, b in zip(r, r0)), f"run {i} differs from run 0"
    from bit_exact_speculative_gb300 import xv
    assert xv.xv_device_check() == 0


def test_stack_long_context(stack):
    cfg, w, wd = stack
    B, k, L = 1, 8, 131072
    Lmax = L + 64
    toks = workloads.draft_tokens(cfg, 0, 5, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lgA = A.verify(dev(toks), k)[0].clone()
    S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lgS, _ = sequential(S, toks, B)
    assert same_bits(lgA.view(B, k, -1), lgS)


def test_stack_speculative_rounds_emit_greedy_decode(stack):
    """Greedy speculative rounds (verify 8 / accept / commit) on the 4-layer stack emit exactly the
    target's k=1 greedy decode, for drafts that are always, sometimes and never right."""
    from bit_exact_speculative_gb300.speculative import ReplayDrafter, greedy_decode, speculative_decode
    cfg, w, wd = stack
    B, k, L, n = 1, 8, 2183, 40
    Lmax = L + 3 * n + 4 * k
    first = int(workloads.draft_tokens(cfg, 0, 77, 1, 1)[0, 0])
    ref = greedy_decode(gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd), first, n)
    for accept, lo, hi in [(1.0, 6.0, 7.0), (0.6, 0.1, 6.0), (0.0, 0.0, 0.0)]:
        S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
        out, acc = speculative_decode(S, first, n, k, ReplayDrafter(ref, cfg["vocab"], accept, seed=3))
        assert out[:n] == ref[1:n + 1], f"accept {accept}: emitted tokens differ from the greedy decode"
        assert lo <= float(np.mean(acc)) <= hi, (accept, acc)
        assert int(host(S.state["ctx_len"])[0]) == L + len(out)


def test_stack_verify_k9_equals_sequential_decode(stack):
    """k = 9 (one more than the 8 the fused kernels' row count was sized around): bit-exact too."""
    cfg, w, wd = stack
    B, k, L = 1, 9, 2183
    Lmax = L + 64
    toks = workloads.draft_tokens(cfg, 0, 9, B, k)
    A = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lg, am, _ = A.verify(dev(toks), k)
    lgA, amA = lg.clone(), am.clone()
    S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lgS, amS = sequential(S, toks, B)
    assert same_bits(lgA.view(B, k, -1), lgS)
    assert torch.equal(amA.view(B, k), amS)


@pytest.mark.parametrize("page", [64, 256])
def test_stack_paged_kv_equals_contiguous(stack, page):
    """8 sequences over one scattered page pool: two rounds of verify/commit give the logits and
    lengths of contiguous caches bit for bit."""
    from bit_exact_speculative_gb300 import xv
    cfg, w, wd = stack
    B, k = 8, 8
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500]
    Lmax = 2304
    n_pages = B * (Lmax // page) + 3
    order = np.random.default_rng(page).permutation(n_pages)
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    P = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, page_size=page, n_pages=n_pages, page_order=order)
    for rnd, keep in ((0, [3, 1, 8, 2, 5, 8, 1, 4]), (1, [8, 8, 1, 1, 2, 7, 3, 6])):
        toks = dev(workloads.draft_tokens(cfg, 0, 10 + rnd, B, k))
        lgA = A.verify(toks, k)[0].clone()
        lgP = P.verify(toks, k)[0].clone()
        assert same_bits(lgA, lgP), f"round {rnd}: paged logits differ"
        kp = torch.tensor(keep, dtype=torch.int32, device="cuda")
        A.commit(kp)
        P.commit(kp)
    assert torch.equal(A.state["ctx_len"], P.state["ctx_len"])
    assert xv.xv_device_check() == 0


def test_stack_ragged_k_per_sequence(stack):
    """Four sequences verifying 1, 9, 5 and 3 tokens in one call, then (after keeping 1..k_b of
    each) 9, 2, 1 and 6: each sequence's rows equal its own sequential decode bit for bit, and
    n_accept counts only its own drafts."""
    from bit_exact_speculative_gb300 import xv
    cfg, w, wd = stack
    B, kmax, Lmax = 4, 9, 2304
    lens = [2183, 640, 1, 1500]
    ks1, keep, ks2 = [1, 9, 5, 3], [1, 4, 5, 2], [9, 2, 1, 6]
    t1 = workloads.draft_tokens(cfg, 0, 6, B, kmax)
    t2 = workloads.draft_tokens(cfg, 0, 7, B, kmax)
    A = gpu_stack(cfg, w, B, kmax, Lmax, lens, weights_dev=wd)
    k1 = torch.tensor(ks1, dtype=torch.int32, device="cuda")
    lg, am, na = A.verify(dev(t1), kmax, k_seq=k1)
    lg1, am1, na1 = lg.clone().view(B, kmax, -1), host(am).reshape(B, kmax), host(na).copy()
    A.commit(torch.tensor(keep, dtype=torch.int32, device="cuda"))
    k2 = torch.tensor(ks2, dtype=torch.int32, device="cuda")
    lg2 = A.verify(dev(t2), kmax, k_seq=k2)[0].clone().view(B, kmax, -1)
    assert xv.xv_device_check() == 0
    for b in range(B):
        S = gpu_stack(cfg, w, B, kmax, Lmax, lens, weights_dev=wd, only=b)
        lgS, amS = sequential(S, t1[b:b + 1, :ks1[b]], 1)
        assert same_bits(lg1[b, :ks1[b]], lgS[0]), f"sequence {b}, first verify"
        assert np.array_equal(am1[b, :ks1[b]], host(amS[0]))
        assert int(na1[b]) == oracle.accept(t1[b, :ks1[b]], am1[b, :ks1[b]])
        del S
        S = gpu_stack(cfg, w, B, kmax, Lmax, lens, weights_dev=wd, only=b)
        sequential(S, t1[b:b + 1, :keep[b]], 1)
        lgS, _ = sequential(S, t2[b:b + 1, :ks2[b]], 1)
        assert same_bits(lg2[b, :ks2[b]], lgS[0]), f"sequence {b}, second verify"
        del S
        torch.cuda.empty_cache()


def test_ragged_commit_beyond_k_seq_is_flagged(tiny):
    """Keeping more positions than a sequence verified is recorded (device error bit 8) and clamped."""
    from bit_exact_speculative_gb300 import xv
    cfg, w = tiny
    B, k, Lmax = 2, 4, 256
    A = gpu_stack(cfg, w, B, k, Lmax, [128, 100])
    toks = workloads.draft_tokens(cfg, 0, 1, B, k)
    A.verify(dev(toks), k, k_seq=torch.tensor([2, 4], dtype=torch.int32, device="cuda"))
    A.commit(torch.tensor([3, 4], dtype=torch.int32, device="cuda"))
    with pytest.raises(xv.XVError) as e:
        xv.xv_device_check()
    assert e.value.code == xv.XV_ERR_DEVICE_CHECK and "bits 0x8" in str(e.value)
    assert xv.xv_device_check() == 0          # read and cleared
    assert host(A.state["ctx_len"]).tolist() == [130, 104]


# ------------------------------------------------------------ prefill

@pytest.mark.parametrize("cfg_name", ["TINY", "TINY_FULL"])
def test_prefill_any_chunk_equals_decode(built, cfg_name):
    """Prefill of 37 tokens in chunks of 4, 3 or 32 leaves the states of 37 decode steps bit for
    bit: the same last logits, the same GDN/convolution states and the same next verify."""
    cfg = getattr(workloads, cfg_name)
    w = workloads.weights(cfg, seed=0)
    B, k, Lmax, T = 2, 4, 256, 37
    lens = [100, 41]
    prompt = np.concatenate([workloads.draft_tokens(cfg, 0, 30 + i, B, 1) for i in range(T)], axis=1)
    nxt = workloads.draft_tokens(cfg, 0, 90, B, k)
    outs = []
    for kmax, chunk in ((k, 4), (k, 3), (32, 32)):
        A = gpu_stack(cfg, w, B, kmax, Lmax, lens)
        lg, am = A.prefill(dev(prompt), chunk)
        lgv = A.verify(dev(nxt), k)[0].clone()
        A.commit(torch.full((B,), k, dtype=torch.int32, device="cuda"))
        A.flush()
        outs.append((lg.clone(), am.clone(), lgv, A.state["0.state"].clone(),
                     A.state["0.conv"].clone() if "0.conv" in A.state else None, A.state["ctx_len"].clone()))
    S = gpu_stack(cfg, w, B, k, Lmax, lens)
    lgS, amS = sequential(S, prompt, B)
    lgvS = S.verify(dev(nxt), k)[0].clone()
    S.commit(torch.full((B,), k, dtype=torch.int32, device="cuda"))
    S.flush()
    # the oracle decoding the same 37 prompt tokens (then the 4 verified ones) agrees within the
    # block tolerance on the last prompt logits and on the GDN state, within the bf16 bound on the
    # convolution state (its rows are projection outputs)
    from _gpu import assert_bf16_close
    for b in range(B):
        ref, spread, ost = oracle_logits(cfg, w, b, B, lens, Lmax, prompt[b])
        assert_block_close(host(outs[0][0])[b:b + 1], ref[-1:], spread, what=f"prefill last logits, sequence {b}")
        ost.verify(nxt[b])
        Sg = host(outs[0][3])[b]
        assert float(np.max(np.abs(Sg - ost.S[0]))) <= 2e-2 * rms(ost.S[0]), f"prefill GDN state, sequence {b}"
        if outs[0][4] is not None:
            assert_bf16_close(host(outs[0][4].view(torch.int16)).view(np.uint16)[b], ost.conv[0],
                              what=f"prefill convolution state, sequence {b}")
    for lg, am, lgv, st, cv, ctx in outs:
        assert same_bits(lg, lgS[:, -1])
        assert torch.equal(am, amS[:, -1])
        assert same_bits(lgv, lgvS)
        assert same_bits(st, S.state["0.state"])
        if cv is not None:
            assert same_bits(cv, S.state["0.conv"])
        assert torch.equal(ctx, S.state["ctx_len"])
        assert host(ctx).tolist() == [lens[0] + T + k, lens[1] + T + k]


def test_stack_prefill_chunks_equal(stack):
    """The 5120-wide stack: 150 prompt tokens prefilled in chunks of 64 (384 attention rows per
    kv head: 6 row tiles), 8 and 5 give the same last logits and the same next verify, and match
    150 decode steps."""
    cfg, w, wd = stack
    B, k, L, T = 1, 8, 640, 150
    Lmax = L + T + 2 * k
    prompt = np.concatenate([workloads.draft_tokens(cfg, 0, 300 + i, B, 1) for i in range(T)], axis=1)
    nxt = workloads.draft_tokens(cfg, 0, 399, B, k)
    res = []
    for chunk in (64, 8, 5):
        A = gpu_stack(cfg, w, B, 64, Lmax, [L], weights_dev=wd)
        lg, _ = A.prefill(dev(prompt), chunk)
        res.append((lg.clone(), A.verify(dev(nxt), k)[0].clone()))
        del A
    S = gpu_stack(cfg, w, B, k, Lmax, [L], weights_dev=wd)
    lgS, _ = sequential(S, prompt, B)
    lgvS = S.verify(dev(nxt), k)[0].clone()
    for lg, lgv in res:
        assert same_bits(lg, lgS[:, -1])
        assert same_bits(lgv, lgvS)


# ------------------------------------------------------------ layer by layer, teacher forced

@pytest.mark.parametrize("name,lens,k", [("TINY", [128, 37], 4), ("TINY_FULL", [128, 5, 77, 250], 4),
                                         ("STACK", [2183], 8), ("STACK", [2183, 700], 8)])
def test_layers_teacher_forced_vs_oracle(stack, name, lens, k):
    """Each layer on its own: stacks of the first d layers (d = 1 .. L, the same weights and
    states) give the residual stream after layer d (the hidden state the verify leaves at the
    start of its workspace); the oracle's layer d, fed the GPU's residual input to it, must land
    within the per-layer bound.  TINY_FULL at 4 x 4 rows and the stack at 2 x 8 rows take the
    M > 8 paths."""
    if name == "STACK":
        cfg, w, wd = stack
    else:
        cfg = getattr(workloads, name)
        w = workloads.weights(cfg, seed=0)
        wd = {n: dev(v) for n, v in w.items()}
    B, Lmax, nl = len(lens), max(lens) + 64, len(cfg["kinds"])
    toks = workloads.draft_tokens(cfg, 0, 0, B, k)
    kv = kv_host(cfg, lens, Lmax)
    xs = [w["embed"][toks.reshape(-1)]]
    for d in range(1, nl + 1):
        A = gpu_stack(dict(cfg, kinds=cfg["kinds"][:d]), w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
        A.verify(dev(toks), k, logits=False)
        xs.append(host_u16(A.hidden()).copy())
        del A
    for b in range(B):
        rows = slice(b * k, (b + 1) * k)
        o64 = oracle_stack(cfg, w, b, B, lens, Lmax)
        o32 = oracle_stack(cfg, w, b, B, lens, Lmax, f32=True)
        for l in range(nl):
            out, mid = o64.layer_rows(l, xs[l][rows], mid=True)
            out32 = o32.layer_rows(l, xs[l][rows])
            assert_layer_close(xs[l + 1][rows], xs[l][rows], mid, out, out32, what=f"{name} sequence {b} layer {l}")


def test_stack_tiled_weights_equal_row_major(stack):
    """The same stack on row-major weights: 8 sequences of mixed lengths, two verify + commit
    rounds and a prefill chunk give the same logits, argmax and accept counts bit for bit."""
    cfg, w, wd = stack
    rm = {n: dev(v) for n, v in w.items()}
    B, k = 8, 8
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500]
    Lmax = max(lens) + 3 * k + 64
    kv = kv_host(cfg, lens, Lmax)
    out = []
    for weights in (wd, rm):
        A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=weights, kv=kv)
        got = []
        for r in range(2):
            lg, am, na = A.verify(dev(workloads.draft_tokens(cfg, 0, r, B, k)), k)
            got += [lg.clone(), am.clone(), na.clone()]
            A.commit()
        plg, pam = A.prefill(dev(workloads.draft_tokens(cfg, 0, 9, B, 5)))
        got += [plg.clone(), pam.clone()]
        out.append(got)
        del A
    for a, b in zip(*out):
        assert same_bits(a, b)
    del rm


def test_stack_argmax_without_logits(stack):
    """Without a logits buffer the LM head writes no logits and the argmax comes from its per-tile
    partials alone: the same argmax ids and accept counts as with logits, at 8 sequences."""
    cfg, w, wd = stack
    B, k = 8, 8
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500]
    Lmax = max(lens) + 64
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    snap = snapshot(A)
    toks = dev(workloads.draft_tokens(cfg, 0, 3, B, k))
    lg, am, na = A.verify(toks, k)
    am1, na1 = am.clone(), na.clone()
    assert torch.equal(am1.cpu(), torch.argmax(lg, dim=1).to(torch.int32).cpu())
    restore(A, snap)
    _, am2, na2 = A.verify(toks, k, logits=False)
    assert torch.equal(am1, am2) and torch.equal(na1, na2)


@pytest.mark.parametrize("name", ["TINY", "STACK"])
def test_verify_commit_equals_verify_then_commit(stack, name):
    """The fused verify + commit-accepted call against the two calls: three rounds on 8 sequences
    of mixed lengths give the same logits, argmax and accept counts, and leave every state tensor
    (lengths, commit counts, GDN states and histories, caches) the same bit for bit."""
    if name == "STACK":
        cfg, w, wd = stack
    else:
        cfg = workloads.TINY
        w = workloads.weights(cfg, seed=0)
        wd = {n: dev(v) for n, v in w.items()}
    B, k = 8, 8 if name == "STACK" else 4
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500] if name == "STACK" else [128, 5, 77, 250, 1, 64, 99, 31]
    Lmax = max(lens) + 4 * k + 64
    kv = kv_host(cfg, lens, Lmax)
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
    S = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
    for r in range(3):
        toks = dev(workloads.draft_tokens(cfg, 0, 20 + r, B, k))
        la, aa, na = A.verify_commit(toks, k, logits=True)
        ls, as_, ns = S.verify(toks, k)
        res_s = (ls.clone(), as_.clone(), ns.clone())
        S.commit()
        assert same_bits(la, res_s[0]) and torch.equal(aa, res_s[1]) and torch.equal(na, res_s[2]), f"round {r}"
    torch.cuda.synchronize()
    for n, t in A.state.items():
        assert torch.equal(t, S.state[n]), n
    sa, ss = A.blk.state, S.blk.state
    assert (sa.parity, sa.pending_rows, sa.max_ctx, sa.last_k) == (ss.parity, ss.pending_rows, ss.max_ctx, ss.last_k)
    assert xv_device_check_ok()


def xv_device_check_ok():
    from bit_exact_speculative_gb300 import xv
    return xv.xv_device_check() == 0


def test_step_host_equals_verify_commit(stack):
    """The one-call host-driven step (drafts in from pinned host memory, results out to it) against
    verify_commit on device tensors: three rounds on 8 sequences give the same argmax ids and
    accept counts in the host buffer and the same state."""
    cfg, w, wd = stack
    B, k = 8, 8
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500]
    Lmax = max(lens) + 4 * k + 64
    kv = kv_host(cfg, lens, Lmax)
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
    S = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd, kv=kv)
    h_res = torch.empty(A.results.shape, dtype=torch.int32).pin_memory()
    for r in range(3):
        toks = workloads.draft_tokens(cfg, 0, 30 + r, B, k)
        A.step_host(torch.from_numpy(toks).pin_memory(), h_res)
        _, am, na = S.verify_commit(dev(toks), k)
        torch.cuda.synchronize()
        assert torch.equal(h_res[: B * k], am.cpu()) and torch.equal(h_res[B * k:], na.cpu()), f"round {r}"
    for n, t in A.state.items():
        assert torch.equal(t, S.state[n]), n
    assert xv_device_check_ok()


def test_stack_same_bits_without_programmatic_launch(stack, built):
    """Programmatic dependent launch lets each kernel start its prologue (and request its weights)
    while its predecessor finishes; turning it off serialises the launches.  Three verify + commit
    rounds of 8 sequences give the same logits, argmax, accept counts and states either way."""
    xv = built
    cfg, w, wd = stack
    B, k = 8, 8
    lens = [2183, 640, 1000, 1, 513, 2047, 300, 1500]
    Lmax = max(lens) + 4 * k + 64
    A = gpu_stack(cfg, w, B, k, Lmax, lens, weights_dev=wd)
    snap = snapshot(A)
    runs = []
    try:
        for overlap in (1, 0):
            xv.xv_set_overlap(overlap)
            restore(A, snap)
            out = []
            for rnd in range(3):
                lg, am, na = A.verify_commit(dev(workloads.draft_tokens(cfg, 0, 40 + rnd, B, k)), k, logits=True)
                out += [lg.clone(), am.clone(), na.clone()]
            torch.cuda.synchronize()
            out += [t.clone() for t in A.state.values()]
            runs.append(out)
    finally:
        xv.xv_set_overlap(True)
    assert xv.xv_device_check() == 0
    for a, b in zip(*runs):
        assert same_bits(a, b)
