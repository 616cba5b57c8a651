"""A hybrid GDN/attention stack held on the device, driven through the C ABI.

:class:`HybridStack` allocates the per-sequence state the verify block needs
(fp32 GDN states, the two GDN step-history buffers, bf16 KV caches, context
lengths, workspace) with torch, and calls ``xv_verify_block`` /
``xv_block_commit`` for each round.  All arithmetic happens in libxv.so.

Config keys: hidden, vocab, mlp, kinds (0 = GDN, 1 = gated attention),
gdn_heads, gdn_dk, gdn_dv, attn_hq, attn_hkv, attn_hd, rms_eps, and for a
complete GDN layer gdn_qk_heads (default gdn_heads), gdn_conv (convolution
width, default 0 = none) and gdn_out_norm (gated output norm, default 0).

With ``page_size`` the attention caches are page pools shared by the
sequences (:class:`KvPagePool` hands pages out); without, each sequence has a
contiguous [Hkv, Lmax, hd] cache.  Both give the same bits.
Weight keys: embed, final_norm, lm_head and per layer ``f"{l}.norm1"``,
``.w_in``, ``.w_out``, ``.norm2``, ``.w_gu``, ``.w_down``, and ``.conv_w``
[C, Kc] / ``.onorm`` [dv] for complete GDN layers (bf16 bit patterns in any
2-byte torch dtype, on the device).
"""
from __future__ import annotations

import numpy as np
import torch

from . import xv


def gdn_qk_heads(cfg: dict) -> int:
    return cfg.get("gdn_qk_heads") or cfg["gdn_heads"]


def gdn_conv_dim(cfg: dict) -> int:
    """Channels of the GDN convolution: q | k | v."""
    return 2 * gdn_qk_heads(cfg) * cfg["gdn_dk"] + cfg["gdn_heads"] * cfg["gdn_dv"]


def gdn_in_dim(cfg: dict) -> int:
    z = cfg["gdn_heads"] * cfg["gdn_dv"] if cfg.get("gdn_out_norm") else 0
    return gdn_conv_dim(cfg) + z + 2 * cfg["gdn_heads"]


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
        if kd == 0 and cfg.get("gdn_conv"):
            shapes[f"{l}.conv_w"] = (gdn_conv_dim(cfg), cfg["gdn_conv"])
        if kd == 0 and cfg.get("gdn_out_norm"):
            shapes[f"{l}.onorm"] = (cfg["gdn_dv"],)
    return shapes


GEMM_WEIGHTS = ("w_in", "w_out", "w_gu", "w_down")


def tile_weights(cfg: dict, weights: dict, stream=None) -> dict:
    """A copy of ``weights`` with the LM head and every layer's projections in the GEMM's tiled
    layout (:func:`xv.tile_weight`; gate/up by :func:`xv.tile_gate_up`, which lets the GEMM form
    the SwiGLU itself; the other tensors are shared): the same bits, faster streaming, one launch
    fewer per layer.  The row-major projection tensors may be dropped afterwards."""
    out = dict(weights)
    names = ["lm_head"] + [f"{l}.{n}" for l in range(len(cfg["kinds"])) for n in GEMM_WEIGHTS]
    for n in names:
        if not isinstance(out[n], xv.TiledWeight):
            gated = n.endswith(".w_gu")
            out[n] = (xv.tile_gate_up if gated else xv.tile_weight)(out[n], stream=stream)
    return out


class KvPagePool:
    """Hands out the pages of a paged KV pool to the sequences of a stack.

    Entry ``[b, j]`` of the page table names the page that holds positions
    ``[j * page, (j + 1) * page)`` of sequence b (-1: none yet).  Pages come off
    a free list, so the pages of one sequence are scattered through the pool in
    the order the list gives (``order``, default 0, 1, 2, ...).  ``table`` is the
    device copy the kernels read; :meth:`sync` refreshes it after changes with a
    stream-ordered copy from one of two pinned staging buffers, so the host never
    waits for the device to drain (it waits only for the copy made two syncs
    earlier from the same buffer).
    """

    def __init__(self, n_pages: int, page: int, B: int, max_pages: int, device="cuda", order=None):
        self.n_pages, self.page, self.B, self.max_pages = int(n_pages), int(page), int(B), int(max_pages)
        order = list(range(n_pages)) if order is None else [int(x) for x in order]
        if sorted(order) != list(range(n_pages)):
            raise ValueError("order must be a permutation of the pool's pages")
        self.free = order[::-1]           # pop() hands out order[0] first
        self.host = np.full((B, max_pages), -1, dtype=np.int32)
        self.held = [0] * B
        self.table = torch.full((B, max_pages), -1, dtype=torch.int32, device=device)
        self.dirty = False
        self._cuda = self.table.is_cuda
        if self._cuda:
            self._stage = [torch.empty((B, max_pages), dtype=torch.int32).pin_memory() for _ in range(2)]
            self._copied = [None, None]
            self._flip = 0

    def ensure(self, b: int, length: int):
        """Gives sequence b pages for positions [0, length)."""
        need = -(-int(length) // self.page)
        if need > self.max_pages:
            raise ValueError(f"sequence {b}: {length} positions exceed {self.max_pages} pages of {self.page}")
        while self.held[b] < need:
            if not self.free:
                raise MemoryError("KV page pool exhausted")
            self.host[b, self.held[b]] = self.free.pop()
            self.held[b] += 1
            self.dirty = True

    def release(self, b: int):
        """Returns every page of sequence b to the pool."""
        for j in range(self.held[b] - 1, -1, -1):
            self.free.append(int(self.host[b, j]))
        self.host[b, :] = -1
        self.held[b] = 0
        self.dirty = True

    def sync(self, stream=None):
        """Enqueues the table update on ``stream`` (default: the current stream)."""
        if not self.dirty:
            return
        if not self._cuda:
            self.table.copy_(torch.from_numpy(self.host))
        else:
            i = self._flip
            self._flip ^= 1
            if self._copied[i] is not None:
                self._copied[i].synchronize()
            self._stage[i].copy_(torch.from_numpy(self.host))
            stream = torch.cuda.current_stream(self.table.device) if stream is None else stream
            with torch.cuda.stream(stream):
                self.table.copy_(self._stage[i], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(stream)
            self._copied[i] = ev
        self.dirty = False


class HybridStack:
    def __init__(self, cfg: dict, weights: dict, B: int, kmax: int, Lmax: int, device="cuda",
                 page_size: int | None = None, n_pages: int | None = None, page_order=None):
        self.cfg, self.B, self.kmax, self.Lmax = dict(cfg), B, kmax, Lmax
        self.weights = weights
        d = device
        st = {"ctx_len": torch.zeros(B, dtype=torch.int32, device=d),
              "n_commit": torch.zeros(B, dtype=torch.int32, device=d)}
        self.pool = None
        if page_size is not None:
            max_pages = -(-Lmax // page_size)
            n_pages = B * max_pages if n_pages is None else n_pages
            self.pool = KvPagePool(n_pages, page_size, B, max_pages, device=d, order=page_order)
            st["page_table"] = self.pool.table
        for l, kd in enumerate(cfg["kinds"]):
            if kd == 0:
                h, dk, dv = cfg["gdn_heads"], cfg["gdn_dk"], cfg["gdn_dv"]
                st[f"{l}.state"] = torch.zeros((B, h, dv, dk), dtype=torch.float32, device=d)
                for p in (0, 1):
                    st[f"{l}.hist{p}"] = torch.zeros((B * kmax, gdn_hist_stride(cfg)), dtype=torch.int16, device=d)
                if cfg.get("gdn_conv"):
                    C = gdn_conv_dim(cfg)
                    st[f"{l}.conv"] = torch.zeros((B, cfg["gdn_conv"] - 1, C), dtype=torch.int16, device=d)
                    for p in (0, 1):
                        st[f"{l}.cout{p}"] = torch.zeros((B * kmax, (C + 7) // 8 * 8), dtype=torch.int16, device=d)
            else:
                if self.pool is None:
                    shape = (B, cfg["attn_hkv"], Lmax, cfg["attn_hd"])
                else:
                    shape = (self.pool.n_pages, cfg["attn_hkv"], page_size, cfg["attn_hd"])
                st[f"{l}.kc"] = torch.zeros(shape, dtype=torch.int16, device=d)
                st[f"{l}.vc"] = torch.zeros(shape, dtype=torch.int16, device=d)
        self.state = st
        pages = None if self.pool is None else xv.kv_pages(self.pool.table, page_size, self.pool.n_pages)
        self.blk = xv.Block(cfg, weights, st, B, kmax, Lmax, ctx0=0, pages=pages)
        self._bound = [0] * B          # host upper bound of each ctx_len (page allocation)
        self._k_seq = None             # the k_seq of a ragged verify, kept alive until its commit
        self._last_k = 0
        self.ws = xv.workspace(self.blk.ws_bytes, device=d)
        self._pf_ws = None           # the prefill workspace, made on first use
        self.logits = torch.empty((B * kmax, cfg["vocab"]), dtype=torch.float32, device=d)
        # argmax ids and accept counts side by side, so that one copy reads a step's results
        self.results = torch.empty(B * kmax + B, dtype=torch.int32, device=d)
        self._step_tokens = None       # the device copy of step_host's drafts
        self.argmax = self.results[: B * kmax]
        self.n_accept = self.results[B * kmax:]

    def set_context(self, ctx_len):
        """Sets every sequence's committed length (host list); the caller has filled the caches/states."""
        lens = [int(x) for x in ctx_len]
        t = torch.as_tensor(lens, dtype=torch.int32)
        self.state["ctx_len"].copy_(t)
        self.state["n_commit"].zero_()
        self.blk.state.max_ctx = int(t.max())
        self.blk.state.last_k = 0
        self._bound = lens
        if self.pool is not None:
            for b, n in enumerate(lens):
                self.pool.ensure(b, n)
            self.pool.sync()

    def load_kv(self, layer: int, kc, vc):
        """Writes contiguous caches kc, vc ([B, Hkv, Lmax, hd], 2-byte dtype, host or device) into
        attention layer ``layer``: copied as they are, or scattered into the pages the pool holds."""
        kd, vd = self.state[f"{layer}.kc"], self.state[f"{layer}.vc"]
        kc = torch.as_tensor(kc).view(torch.int16)
        vc = torch.as_tensor(vc).view(torch.int16)
        if self.pool is None:
            kd.copy_(kc)
            vd.copy_(vc)
            return
        P = self.pool.page
        for b in range(self.B):
            for j in range(self.pool.held[b]):
                pg = int(self.pool.host[b, j])
                n = min(P, self.Lmax - j * P)
                kd[pg, :, :n].copy_(kc[b, :, j * P:j * P + n])
                vd[pg, :, :n].copy_(vc[b, :, j * P:j * P + n])

    def _prepare(self, k: int, stream=None):
        if self.pool is not None:
            for b in range(self.B):
                self.pool.ensure(b, min(self._bound[b] + k, self.Lmax))
            self.pool.sync(stream)

    def verify(self, tokens: torch.Tensor, k: int, logits: bool = True, stream=None, k_seq=None):
        """tokens: int32 [B, k] on the device; k_seq: optional int32 [B] device tensor of per-sequence
        token counts (1..k; rows past k_seq[b] are padding).  Returns (logits [B*k, V] or None,
        argmax [B*k], n_accept [B])."""
        self._prepare(k, stream)
        lg = self.logits[: self.B * k] if logits else None
        if k_seq is None:
            xv.xv_verify_block(self.blk, tokens, k, lg, self.argmax, self.n_accept, self.ws, stream=stream)
        else:
            xv.xv_verify_block_ragged(self.blk, tokens, k, k_seq, lg, self.argmax, self.n_accept, self.ws,
                                      stream=stream)
        self._k_seq = k_seq
        self._last_k = k
        return lg, self.argmax[: self.B * k], self.n_accept

    def verify_commit(self, tokens: torch.Tensor, k: int, logits: bool = False, stream=None):
        """verify(tokens, k) then commit() of the accepted drafts + 1, in one call with one launch
        fewer (the same bits).  Returns (logits [B*k, V] or None, argmax [B*k], n_accept [B])."""
        self._prepare(k, stream)
        lg = self.logits[: self.B * k] if logits else None
        xv.xv_verify_block_commit_accepted(self.blk, tokens, k, lg, self.argmax, self.n_accept, self.ws, stream=stream)
        self._bound = [n + k for n in self._bound]
        self._k_seq = None
        self._last_k = k
        return lg, self.argmax[: self.B * k], self.n_accept

    def step_host(self, host_tokens: torch.Tensor, host_results: torch.Tensor, stream=None):
        """One host-driven speculative step in one call: host_tokens [B, k] int32 (pinned) in,
        verify + commit of the accepted drafts, and host_results [B*kmax + B] int32 (pinned;
        argmax ids in its first B*k entries, row b*k + j, then from B*kmax on the accept counts)
        out, all enqueued on the stream (synchronise before reading host_results)."""
        k = host_tokens.shape[-1]
        if self.pool is not None:
            self._prepare(k, stream)
        if self._step_tokens is None or self._step_tokens.shape[1] != k:
            self._step_tokens = torch.empty((self.B, k), dtype=torch.int32, device=self.results.device)
        xv.xv_block_step_host(self.blk, host_tokens, self._step_tokens, k, self.results, host_results, self.ws,
                              stream=stream)
        self._bound = [n + k for n in self._bound]
        self._k_seq = None
        self._last_k = k

    def hidden(self) -> torch.Tensor:
        """The residual stream after the last layer of the last verify (the hidden state before
        the final RMSNorm), bf16 bits [B*k, H]: a view of the workspace, valid until the next call
        that uses it."""
        n = self.B * self._last_k * self.cfg["hidden"]
        return self.ws[: 2 * n].view(torch.int16).view(self.B * self._last_k, self.cfg["hidden"])

    def commit(self, n_keep: torch.Tensor | None = None, stream=None):
        """Keeps n_keep[b] positions of the last verify (default: the accepted drafts + 1)."""
        if n_keep is None:
            xv.xv_block_commit_accepted(self.blk, self.n_accept, stream=stream)
        else:
            xv.xv_block_commit(self.blk, n_keep, stream=stream)
        self._bound = [n + self._last_k for n in self._bound]
        self._k_seq = None

    def prefill(self, tokens: torch.Tensor, chunk: int | None = None, stream=None):
        """Feeds tokens [B, T] (int32, device) through verify + commit-all in chunks of ``chunk``
        (default kmax); the caches and states end bit-identical to T decode steps.  Returns
        (logits [B, V] fp32, argmax [B]) after each sequence's last token."""
        B, T = tokens.shape
        chunk = self.kmax if chunk is None else int(chunk)
        if self._pf_ws is None:
            n = int(xv.lib().xv_block_prefill_workspace_size(xv.ctypes.byref(self.blk.cfg), self.B, self.kmax,
                                                             self.Lmax))
            self._pf_ws = xv.workspace(n, device=self.argmax.device)
        if self.pool is not None:
            for b in range(self.B):
                self.pool.ensure(b, min(self._bound[b] + T, self.Lmax))
            self.pool.sync(stream)
        lg = torch.empty((B, self.cfg["vocab"]), dtype=torch.float32, device=self.argmax.device)
        am = torch.empty(B, dtype=torch.int32, device=self.argmax.device)
        xv.xv_block_prefill(self.blk, tokens.contiguous(), T, chunk, lg, am, self._pf_ws, stream=stream)
        self._bound = [n + T for n in self._bound]
        return lg, am

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
        self._bound = [min(n, int(longest)) for n in self._bound]
