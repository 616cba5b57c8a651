"""Builds a HybridStack on the GPU and the matching oracle stacks from one seeded recipe."""
import numpy as np
import torch

import oracle
from synth import workloads
from _gpu import dev


def kv_host(cfg, ctx_lens, Lmax, seed=0):
    """The recipe's K/V caches of every attention layer ({layer: (kc, vc)}, [B, Hkv, Lmax, hd] bf16
    bits), drawn once so that several stacks of one recipe can share them."""
    B = len(ctx_lens)
    return {l: workloads.kv_cache(cfg, seed, l, B, ctx_lens, Lmax) for l, kd in enumerate(cfg["kinds"]) if kd != 0}


def gpu_stack(cfg, w_np, B, kmax, Lmax, ctx_lens, seed=0, weights_dev=None, page_size=None, n_pages=None,
              page_order=None, only=None, kv=None):
    """The stack of the seeded recipe for B sequences of lengths ctx_lens; with ``only`` = b a B = 1
    stack holding sequence b of that recipe.  page_size / n_pages / page_order make the KV caches
    a page pool; ``kv`` passes caches already drawn by :func:`kv_host`."""
    from bit_exact_speculative_gb300.model import HybridStack
    weights = weights_dev if weights_dev is not None else {k: dev(v) for k, v in w_np.items()}
    sel = slice(None) if only is None else slice(only, only + 1)
    nb = B if only is None else 1
    stk = HybridStack(cfg, weights, nb, kmax, Lmax, page_size=page_size, n_pages=n_pages, page_order=page_order)
    stk.set_context(list(ctx_lens)[sel])
    for l, kd in enumerate(cfg["kinds"]):
        if kd == 0:
            stk.state[f"{l}.state"].copy_(torch.from_numpy(workloads.gdn_state(cfg, seed, l, B)[sel]))
            if cfg.get("gdn_conv"):
                stk.state[f"{l}.conv"].copy_(torch.from_numpy(workloads.conv_state(cfg, seed, l, B)[sel].view(np.int16)))
        else:
            kc, vc = kv[l] if kv is not None else workloads.kv_cache(cfg, seed, l, B, ctx_lens, Lmax)
            stk.load_kv(l, torch.from_numpy(kc[sel].view(np.int16)), torch.from_numpy(vc[sel].view(np.int16)))
    torch.cuda.synchronize()
    return stk


def oracle_stack(cfg, w_np, b, B, ctx_lens, Lmax, seed=0, f32=False):
    """The oracle's stack for sequence b of the same recipe (GDN states widened to double); with
    ``f32`` its single-precision evaluation."""
    st = oracle.Stack(workloads.oracle_cfg(cfg), w_np, Lmax, f32=f32)
    for l, kd in enumerate(cfg["kinds"]):
        if kd == 0:
            st.S[l][...] = workloads.gdn_state(cfg, seed, l, B)[b].astype(np.float64)
            if cfg.get("gdn_conv"):
                st.conv[l][...] = workloads.conv_state(cfg, seed, l, B)[b]
        else:
            kc, vc = workloads.kv_cache(cfg, seed, l, B, ctx_lens, Lmax)
            st.kc[l][...] = kc[b]
            st.vc[l][...] = vc[b]
    st.len = int(ctx_lens[b])
    return st


def oracle_logits(cfg, w_np, b, B, ctx_lens, Lmax, tokens, before=(), extra=0, seed=0):
    """The oracle's logits for sequence b decoding ``tokens`` (after decoding ``before``), and the
    spread of its single-precision evaluation (f32 oracle minus f64 oracle, same inputs) over those
    rows and ``extra`` further seeded positions of the same sequence.  Returns (ref [n, V], spread
    [n + extra, V], the f64 stack as it stands after ``tokens``)."""
    out, st64 = [], None
    for f32 in (False, True):
        st = oracle_stack(cfg, w_np, b, B, ctx_lens, Lmax, seed, f32=f32)
        if len(before):
            st.verify(before)
        rows = st.verify(tokens)
        if extra:
            snap = st.snapshot()
            rows = np.concatenate([rows, st.verify(workloads.draft_tokens(cfg, seed, 700 + b, 1, extra)[0])])
            st.restore(snap)
        out.append(rows)
        if not f32:
            st64 = st
    return out[0][:len(tokens)], out[1] - out[0], st64


def snapshot(stk):
    """Device copies of every state tensor of a HybridStack and its host-side counters."""
    s = stk.blk.state
    return ({n: t.clone() for n, t in stk.state.items()},
            (s.parity, s.pending_rows, s.max_ctx, s.last_k), list(stk._bound))


def restore(stk, snap):
    tensors, (parity, pending, max_ctx, last_k), bound = snap
    for n, t in tensors.items():
        stk.state[n].copy_(t)
    s = stk.blk.state
    s.parity, s.pending_rows, s.max_ctx, s.last_k = parity, pending, max_ctx, last_k
    stk._bound = list(bound)
    stk._k_seq = None
