"""Greedy speculative decoding rounds over a :class:`HybridStack`.

One round ("Follow-up to my earlier post on Qwen3.8-27B decode speed",
r/LocalLLaMA post: the drafter proposes, the target verifies k positions in
one pass, the accepted drafts plus one target token are kept):

  1. the input is the last emitted token x0 followed by k-1 drafted tokens;
  2. ``xv_verify_block`` returns the target's greedy token after every input
     position and n = the number of leading drafts equal to those tokens;
  3. the round emits the target's tokens 0..n (the accepted drafts and the
     target's own token after them), and commits n+1 positions.

Because verify gives exactly the bits of k decode steps, the emitted stream
is the target's greedy decode, token for token, whatever the drafts are; only
the number of rounds depends on them.  The drafter here is a stand-in (the
pages' drafter is a trained model): :class:`ReplayDrafter` proposes the tokens
of a known greedy continuation and corrupts each one with a fixed
probability, which sets the acceptance rate.
"""
from __future__ import annotations

import numpy as np
import torch


class ReplayDrafter:
    """Proposes ``reference[pos + 1 .. pos + k - 1]`` with each token independently replaced by a
    different one with probability ``1 - accept`` (a wrong draft ends the accepted prefix)."""

    def __init__(self, reference, vocab: int, accept: float, seed: int = 0):
        self.ref = [int(t) for t in reference]
        self.vocab, self.accept = int(vocab), float(accept)
        self.rng = np.random.default_rng(seed)

    def propose(self, pos: int, n: int):
        out = []
        for i in range(n):
            j = pos + 1 + i
            t = self.ref[j] if j < len(self.ref) else int(self.rng.integers(0, self.vocab))
            if self.rng.random() >= self.accept:
                t = (t + 1 + int(self.rng.integers(0, self.vocab - 1))) % self.vocab
            out.append(t)
        return out


def greedy_decode(stack, first: int, n: int, stream=None):
    """n greedy decode steps (verify with k = 1, commit 1) from token ``first`` for sequence 0 of
    a B = 1 stack; returns [first, t1, ..., tn]."""
    one = torch.ones(1, dtype=torch.int32, device=stack.argmax.device)
    tok = torch.empty((1, 1), dtype=torch.int32, device=stack.argmax.device)
    seq = [int(first)]
    for _ in range(n):
        tok.fill_(seq[-1])
        _, am, _ = stack.verify(tok, 1, logits=False, stream=stream)
        stack.commit(one, stream=stream)
        seq.append(int(am[0].item()))
    return seq


def speculative_decode(stack, first: int, n_tokens: int, k: int, drafter, stream=None):
    """Rounds of verify k / accept / commit for sequence 0 of a B = 1 stack until at least
    n_tokens tokens are emitted.  Returns (emitted tokens after ``first``, accepted drafts per
    round)."""
    dev = stack.argmax.device
    toks = torch.empty((1, k), dtype=torch.int32, device=dev)
    host = torch.empty((k + 1,), dtype=torch.int32).pin_memory()
    emitted, accepted = [], []
    ctx0 = stack.max_ctx          # the committed length of sequence 0 (B = 1)
    x0 = int(first)
    while len(emitted) < n_tokens:
        drafts = drafter.propose(len(emitted), k - 1)
        toks.copy_(torch.tensor([[x0] + drafts], dtype=torch.int32), non_blocking=True)
        _, am, na = stack.verify(toks, k, logits=False, stream=stream)
        host[:k].copy_(am[:k], non_blocking=True)
        host[k:].copy_(na[:1], non_blocking=True)
        stack.commit(stream=stream)
        torch.cuda.synchronize(dev)
        n = int(host[k])
        out = [int(x) for x in host[: n + 1]]
        emitted += out
        accepted.append(n)
        stack.tighten_context(ctx0 + len(emitted))   # n + 1 positions were committed, not k
        x0 = out[-1]
    return emitted, accepted
