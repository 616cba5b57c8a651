"""Builds a HybridStack on the GPU and the matching oracle stacks from one seeded recipe."""
import numpy as np
import torch

import oracle
from synth import workloads
from _gpu import dev


def gpu_stack(cfg, w_np, B, kmax, Lmax, ctx_lens, seed=0, weights_dev=None):
    from bit_exact_speculative_gb300.model import HybridStack
    weights = weights_dev if weights_dev is not None else {k: dev(v) for k, v in w_np.items()}
    stk = HybridStack(cfg, weights, B, kmax, Lmax)
    for l, kd in enumerate(cfg["kinds"]):
        if kd == 0:
            stk.state[f"{l}.state"].copy_(torch.from_numpy(workloads.gdn_state(cfg, seed, l, B)))
        else:
            kc, vc = workloads.kv_cache(cfg, seed, l, B, ctx_lens, Lmax)
            stk.state[f"{l}.kc"].copy_(torch.from_numpy(kc.view(np.int16)))
            stk.state[f"{l}.vc"].copy_(torch.from_numpy(vc.view(np.int16)))
    stk.set_context(ctx_lens)
    torch.cuda.synchronize()
    return stk


def oracle_stack(cfg, w_np, b, B, ctx_lens, Lmax, seed=0):
    """The oracle's stack for sequence b of the same recipe (GDN states widened to double)."""
    st = oracle.Stack(workloads.oracle_cfg(cfg), w_np, Lmax)
    for l, kd in enumerate(cfg["kinds"]):
        if kd == 0:
            st.S[l][...] = workloads.gdn_state(cfg, seed, l, B)[b].astype(np.float64)
        else:
            kc, vc = workloads.kv_cache(cfg, seed, l, B, ctx_lens, Lmax)
            st.kc[l][...] = kc[b]
            st.vc[l][...] = vc[b]
    st.len = int(ctx_lens[b])
    return st
