"""Builds a HybridStack on the GPU and the matching oracle stacks from one seeded recipe."""
import numpy as np
import torch

import oracle
from synth import workloads
from _gpu import dev


def gpu_stack(cfg, w_np, B, kmax, Lmax, ctx_lens, seed=0, weights_dev=None, page_size=None, n_pages=None,
              page_order=None, only=None):
    """The stack of the seeded recipe for B sequences of lengths ctx_lens; with ``only`` = b a B = 1
    stack holding sequence b of that recipe.  page_size / n_pages / page_order make the KV caches
    a page pool."""
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
            kc, vc = workloads.kv_cache(cfg, seed, l, B, ctx_lens, Lmax)
            stk.load_kv(l, torch.from_numpy(kc[sel].view(np.int16)), torch.from_numpy(vc[sel].view(np.int16)))
    torch.cuda.synchronize()
    return stk


def oracle_stack(cfg, w_np, b, B, ctx_lens, Lmax, seed=0):
    """The oracle's stack for sequence b of the same recipe (GDN states widened to double)."""
    st = oracle.Stack(workloads.oracle_cfg(cfg), w_np, Lmax)
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
