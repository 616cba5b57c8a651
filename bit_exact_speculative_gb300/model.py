"""A hybrid GDN/attention stack held on the device, driven through the C ABI.

:class:`HybridStack` allocates the per-sequence state the verify block needs
(fp32 GDN states, the two GDN step-history buffers, bf16 KV caches, context
lengths, workspace) with torch, and calls ``xv_verify_block`` /
``xv_block_commit`` for each round.  All arithmetic happens in libxv.so.

Config keys: hidden, vocab, mlp, kinds (0 = GDN, 1 = gated attention),
gdn_heads, gdn_dk, gdn_dv, attn_hq, attn_hkv, attn_hd, rms_eps.
Weight keys: embed, final_norm, lm_head and per layer ``f"{l}.norm1"``,
``.w_in``, ``.w_out``, ``.norm2``, ``.w_gu``, ``.w_down`` (bf16 bit patterns in
any 2-byte torch dtype, on the device).
"""
from __future__ import annotations

import torch

from . import xv


def gdn_in_dim(cfg: dict) -> int:
    return cfg["gdn_heads"] * (2 * cfg["gdn_dk"] + cfg["gdn_dv"]) + 2 * cfg["gdn_heads"]


def gdn_hist_stride(cfg: dict) -> int:
    """Row stride of the GDN step-history buffers (the input width rounded up to 8)."""
    return (gdn_in_dim(cfg) + 7) // 8 * 8


def attn_in_dim(cfg: dict) -> int:
    return 2 * cfg["attn_hq"] * cfg["attn_hd"] + 2 * cfg["attn_hkv"] * cfg["attn_hd"]


def weight_shapes(cfg: dict) -> dict:
    H, F, V = cfg["hidden"], cfg["mlp"], cfg["vocab"]
    shapes = {"embed": (V, H), "final_norm": (H,), "lm_head": (V, H)}
    for l, kd in enumerate(cfg["kinds"]):
        inn = gdn_in_dim(cfg) if kd == 0 else attn_in_dim(cfg)
        inner = cfg["gdn_heads"] * cfg["gdn_dv"] if kd == 0 else cfg["attn_hq"] * cfg["attn_hd"]
        shapes.update({f"{l}.norm1": (H,), f"{l}.w_in": (inn, H), f"{l}.w_out": (H, inner), f"{l}.norm2": (H,),
                       f"{l}.w_gu": (2 * F, H), f"{l}.w_down": (H, F)})
    return shapes


class HybridStack:
    def __init__(self, cfg: dict, weights: dict, B: int, kmax: int, Lmax: int, device="cuda"):
        self.cfg, self.B, self.kmax, self.Lmax = dict(cfg), B, kmax, Lmax
        self.weights = weights
        d = device
        st = {"ctx_len": torch.zeros(B, dtype=torch.int32, device=d),
              "n_commit": torch.zeros(B, dtype=torch.int32, device=d)}
        for l, kd in enumerate(cfg["kinds"]):
            if kd == 0:
                h, dk, dv = cfg["gdn_heads"], cfg["gdn_dk"], cfg["gdn_dv"]
                st[f"{l}.state"] = torch.zeros((B, h, dv, dk), dtype=torch.float32, device=d)
                for p in (0, 1):
                    st[f"{l}.hist{p}"] = torch.zeros((B * kmax, gdn_hist_stride(cfg)), dtype=torch.int16, device=d)
            else:
                shape = (B, cfg["attn_hkv"], Lmax, cfg["attn_hd"])
                st[f"{l}.kc"] = torch.zeros(shape, dtype=torch.int16, device=d)
                st[f"{l}.vc"] = torch.zeros(shape, dtype=torch.int16, device=d)
        self.state = st
        self.blk = xv.Block(cfg, weights, st, B, kmax, Lmax, ctx0=0)
        self.ws = xv.workspace(self.blk.ws_bytes, device=d)
        self.logits = torch.empty((B * kmax, cfg["vocab"]), dtype=torch.float32, device=d)
        self.argmax = torch.empty(B * kmax, dtype=torch.int32, device=d)
        self.n_accept = torch.empty(B, dtype=torch.int32, device=d)

    def set_context(self, ctx_len):
        """Sets every sequence's committed length (host list); the caller has filled the caches/states."""
        t = torch.as_tensor(list(ctx_len), dtype=torch.int32)
        self.state["ctx_len"].copy_(t)
        self.state["n_commit"].zero_()
        self.blk.state.max_ctx = int(t.max())
        self.blk.state.last_k = 0

    def verify(self, tokens: torch.Tensor, k: int, logits: bool = True, stream=None):
        """tokens: int32 [B, k] on the device.  Returns (logits [B*k, V] or None, argmax [B*k], n_accept [B])."""
        lg = self.logits[: self.B * k] if logits else None
        xv.xv_verify_block(self.blk, tokens, k, lg, self.argmax, self.n_accept, self.ws, stream=stream)
        return lg, self.argmax[: self.B * k], self.n_accept

    def commit(self, n_keep: torch.Tensor | None = None, stream=None):
        """Keeps n_keep[b] positions of the last verify (default: the accepted drafts + 1)."""
        if n_keep is None:
            xv.xv_block_commit_accepted(self.blk, self.n_accept, stream=stream)
        else:
            xv.xv_block_commit(self.blk, n_keep, stream=stream)

    def flush(self, stream=None):
        xv.xv_block_flush(self.blk, stream=stream)

    @property
    def max_ctx(self) -> int:
        return self.blk.state.max_ctx

    def tighten_context(self, longest: int):
        """Lowers the host bound on the committed lengths to ``longest``, the longest ctx_len the
        caller has read back (a commit raises the bound by k whatever was accepted)."""
        if longest < self.blk.state.max_ctx:
            self.blk.state.max_ctx = int(longest)
