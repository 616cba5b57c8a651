"""Python binding of libxv.so: argument marshalling only.

Each function has the name of the C entry point it calls (include/xv.h) and
takes torch CUDA tensors (any 2-byte dtype for bf16 data, int32, float32);
every step of the computation runs in the library's kernels.  A missing
library raises at import of the first call: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libxv.so")

vp = ctypes.c_void_p
c_int, c_ll, c_sz, c_float = ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t, ctypes.c_float

XV_OK, XV_ERR_ARG, XV_ERR_UNSUPPORTED, XV_ERR_WORKSPACE, XV_ERR_CUDA, XV_ERR_DEVICE_CHECK = 0, -1, -2, -3, -4, -5
XV_GEMM_M_MAX = 64
XV_KMAX = 64
XV_CONV_MAX = 8


class XVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"xv error {code}: {msg}")
        self.code = code


class GdnSteps(ctypes.Structure):
    _fields_ = [("q", vp), ("k", vp), ("v", vp), ("beta", vp), ("gate", vp),
                ("qkv_stride", c_ll), ("gate_stride", c_ll), ("rows_per_seq", c_int)]


class BlockConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("vocab", c_int), ("mlp", c_int), ("n_layers", c_int), ("layer_kind", vp),
                ("gdn_heads", c_int), ("gdn_dk", c_int), ("gdn_dv", c_int),
                ("attn_hq", c_int), ("attn_hkv", c_int), ("attn_hd", c_int), ("rms_eps", c_float),
                ("gdn_qk_heads", c_int), ("gdn_conv", c_int), ("gdn_out_norm", c_int)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("norm1", vp), ("w_in", vp), ("w_out", vp), ("norm2", vp), ("w_gate_up", vp), ("w_down", vp),
                ("conv_w", vp), ("out_norm", vp)]


class BlockWeights(ctypes.Structure):
    _fields_ = [("embed", vp), ("layers", vp), ("final_norm", vp), ("lm_head", vp), ("tiled", c_int)]


class LayerState(ctypes.Structure):
    _fields_ = [("gdn_state", vp), ("gdn_hist", vp * 2), ("gdn_conv_state", vp), ("gdn_conv_out", vp * 2),
                ("k_cache", vp), ("v_cache", vp)]


class KvPages(ctypes.Structure):
    _fields_ = [("page_table", vp), ("page_size", c_int), ("max_pages", c_int), ("n_pages", c_int)]


class BlockState(ctypes.Structure):
    _fields_ = [("B", c_int), ("kmax", c_int), ("Lmax", c_int), ("ctx_len", vp), ("n_commit", vp),
                ("parity", c_int), ("pending_rows", c_int), ("max_ctx", c_int), ("last_k", c_int), ("layers", vp),
                ("kv_pages", KvPages), ("last_k_seq", vp)]


_lib = None

_SIGS = {
    "xv_abi_version": ([], c_int),
    "xv_last_error": ([], ctypes.c_char_p),
    "xv_device_check": ([vp, ctypes.POINTER(ctypes.c_uint)], c_int),
    "xv_launch_count": ([], ctypes.c_ulonglong),
    "xv_set_overlap": ([c_int], c_int),
    "xv_trace_enable": ([c_int], c_int),
    "xv_trace_disable": ([], c_int),
    "xv_trace_count": ([], c_int),
    "xv_trace_read": ([vp, vp, vp, c_int], c_int),
    "xv_trace_kind_name": ([c_int], ctypes.c_char_p),
    "xv_gemm_workspace_size": ([c_int, c_int, c_int], c_sz),
    "xv_gemm_small_m": ([vp, c_int, vp, vp, c_int, c_int, c_int, c_int, vp, c_sz, vp], c_int),
    "xv_gemm_small_m_f32out": ([vp, c_int, vp, vp, c_int, c_int, c_int, c_int, vp, c_sz, vp], c_int),
    "xv_gemm_splits": ([c_int, c_int], c_int),
    "xv_gemm_small_m_noalloc": ([vp, c_int, vp, vp, c_int, c_int, c_int, c_int, vp], c_int),
    "xv_gemm_tiled_bytes": ([c_int, c_int], c_sz),
    "xv_gemm_tile_weights": ([vp, c_int, c_int, vp, vp], c_int),
    "xv_gemm_small_m_tiled": ([vp, c_int, vp, vp, c_int, c_int, c_int, c_int, vp, c_sz, vp], c_int),
    "xv_gemm_small_m_tiled_f32out": ([vp, c_int, vp, vp, c_int, c_int, c_int, c_int, vp, c_sz, vp], c_int),
    "xv_gemm_tile_gate_up": ([vp, c_int, c_int, vp, vp], c_int),
    "xv_gemm_swiglu_tiled": ([vp, c_int, vp, vp, c_int, c_int, c_int, c_int, vp], c_int),
    "xv_gdn_decode_step": ([vp, ctypes.POINTER(GdnSteps), vp, c_ll, c_int, c_int, c_int, c_int, c_int, vp], c_int),
    "xv_gdn_verify": ([vp, ctypes.POINTER(GdnSteps), vp, c_int, ctypes.POINTER(GdnSteps), c_int, vp, c_ll,
                       c_int, c_int, c_int, c_int, c_int, vp], c_int),
    "xv_gdn_verify_grouped": ([vp, ctypes.POINTER(GdnSteps), vp, c_int, ctypes.POINTER(GdnSteps), c_int, vp, c_ll,
                               c_int, c_int, c_int, c_int, c_int, c_int, vp], c_int),
    "xv_gdn_conv": ([vp, vp, c_ll, c_int, vp, c_int, vp, c_ll, c_int, c_int, vp, c_int, c_int, c_int, vp, c_ll, vp],
                    c_int),
    "xv_gated_norm": ([vp, c_ll, vp, c_ll, vp, c_int, c_int, c_int, c_float, vp, c_ll, vp], c_int),
    "xv_attn_split_begin": ([c_int], c_int),
    "xv_attn_workspace_size": ([c_int, c_int, c_int, c_int, c_int], c_sz),
    "xv_attn_decode_rows": ([vp, c_ll, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                             vp, c_ll, vp, c_ll, vp, c_sz, vp], c_int),
    "xv_kv_append": ([vp, c_ll, vp, c_int, c_int, c_int, c_int, c_int, vp, vp, vp], c_int),
    "xv_attn_decode_rows_paged": ([vp, c_ll, vp, vp, ctypes.POINTER(KvPages), vp, c_int, c_int, c_int, c_int, c_int,
                                   c_int, c_float, vp, c_ll, vp, c_ll, vp, c_sz, vp], c_int),
    "xv_kv_append_paged": ([vp, c_ll, vp, c_int, c_int, c_int, c_int, ctypes.POINTER(KvPages), vp, vp, vp], c_int),
    "xv_gdn_in_dim": ([ctypes.POINTER(BlockConfig)], c_int),
    "xv_gdn_hist_stride": ([ctypes.POINTER(BlockConfig)], c_int),
    "xv_attn_in_dim": ([ctypes.POINTER(BlockConfig)], c_int),
    "xv_gdn_conv_dim": ([ctypes.POINTER(BlockConfig)], c_int),
    "xv_gdn_conv_stride": ([ctypes.POINTER(BlockConfig)], c_int),
    "xv_block_workspace_size": ([ctypes.POINTER(BlockConfig), c_int, c_int, c_int], c_sz),
    "xv_verify_block": ([ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), ctypes.POINTER(BlockState),
                         vp, c_int, vp, vp, vp, vp, c_sz, vp], c_int),
    "xv_verify_block_commit_accepted": ([ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights),
                                         ctypes.POINTER(BlockState), vp, c_int, vp, vp, vp, vp, c_sz, vp], c_int),
    "xv_block_step_host": ([ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), ctypes.POINTER(BlockState),
                            vp, vp, c_int, vp, vp, vp, c_sz, vp], c_int),
    "xv_verify_block_ragged": ([ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights),
                                ctypes.POINTER(BlockState), vp, c_int, vp, vp, vp, vp, vp, c_sz, vp], c_int),
    "xv_block_commit": ([ctypes.POINTER(BlockState), vp, vp], c_int),
    "xv_block_commit_accepted": ([ctypes.POINTER(BlockState), vp, vp], c_int),
    "xv_block_flush": ([ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockState), vp], c_int),
    "xv_block_prefill_workspace_size": ([ctypes.POINTER(BlockConfig), c_int, c_int, c_int], c_sz),
    "xv_block_prefill": ([ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), ctypes.POINTER(BlockState), vp,
                          c_int, c_int, vp, vp, vp, c_sz, vp], c_int),
}


def lib():
    """The loaded libxv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bit_exact_speculative_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, res
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(code: int):
    if code != XV_OK:
        raise XVError(code, lib().xv_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _row_stride(t: torch.Tensor) -> int:
    assert t.dim() >= 2 and t.stride(-1) == 1, "rows must be contiguous"
    return t.stride(-2) if t.dim() == 2 else t.stride(0)


# ------------------------------------------------------------------ misc

def xv_abi_version() -> int:
    return lib().xv_abi_version()


def xv_device_check(stream=None) -> int:
    code = ctypes.c_uint(0)
    _check(lib().xv_device_check(_stream(stream), ctypes.byref(code)))
    return code.value


def xv_launch_count() -> int:
    return int(lib().xv_launch_count())


def xv_set_overlap(enable: bool):
    _check(lib().xv_set_overlap(int(enable)))


def xv_trace_enable(capacity: int):
    _check(lib().xv_trace_enable(capacity))


def xv_trace_disable():
    _check(lib().xv_trace_disable())


def xv_trace_read():
    """Returns a list of (kind name, milliseconds, algorithmic bytes) for every traced launch."""
    import numpy as np
    n = int(lib().xv_trace_count())
    ms = np.zeros(n, np.float32)
    kind = np.zeros(n, np.int32)
    nb = np.zeros(n, np.int64)
    _check(lib().xv_trace_read(ms.ctypes.data, kind.ctypes.data, nb.ctypes.data, n))
    return [(lib().xv_trace_kind_name(int(k)).decode(), float(t), int(b)) for k, t, b in zip(kind, ms, nb)]


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace tensor of at least nbytes (the library's workspaces start zeroed)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ GEMM

def xv_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().xv_gemm_workspace_size(M, N, K))


def xv_gemm_splits(N: int, K: int) -> int:
    return int(lib().xv_gemm_splits(N, K))


class TiledWeight:
    """A weight [N, K] in the GEMM's tiled layout (see :func:`tile_weight`): ``data`` holds the
    tiled copy, ``shape`` is the logical (N, K); ``gated`` marks a gate/up weight tiled by
    :func:`tile_gate_up`."""

    def __init__(self, data: torch.Tensor, N: int, K: int, gated: bool = False):
        self.data, self.shape, self.gated = data, torch.Size((N, K)), gated

    def data_ptr(self) -> int:
        return self.data.data_ptr()

    @property
    def device(self):
        return self.data.device


def xv_gemm_tiled_bytes(N: int, K: int) -> int:
    return int(lib().xv_gemm_tiled_bytes(N, K))


def tile_weight(W: torch.Tensor, stream=None) -> TiledWeight:
    """The tiled copy of a row-major weight W [N, K] (2-byte dtype), made on the device."""
    N, K = W.shape
    data = torch.empty(xv_gemm_tiled_bytes(N, K) // 2, dtype=W.dtype, device=W.device)
    _check(lib().xv_gemm_tile_weights(_ptr(W), N, K, _ptr(data), _stream(stream)))
    return TiledWeight(data, N, K)


def tile_gate_up(W: torch.Tensor, stream=None) -> TiledWeight:
    """The gated tiled copy of a gate/up weight W [2F, K] (F gate rows, then F up rows)."""
    N, K = W.shape
    data = torch.empty(xv_gemm_tiled_bytes(N, K) // 2, dtype=W.dtype, device=W.device)
    _check(lib().xv_gemm_tile_gate_up(_ptr(W), N // 2, K, _ptr(data), _stream(stream)))
    return TiledWeight(data, N, K, gated=True)


def xv_gemm_swiglu(X, Wgu: TiledWeight, act, stream=None):
    """act [M, F] = bf16(silu(g) u) of the gate/up projection X Wgu^T, in one kernel."""
    assert Wgu.gated, "the weight must come from tile_gate_up"
    M, K = X.shape[0], X.shape[1]
    F = Wgu.shape[0] // 2
    _check(lib().xv_gemm_swiglu_tiled(_ptr(X), _row_stride(X), _ptr(Wgu), _ptr(act), _row_stride(act), M, F, K,
                                      _stream(stream)))
    return act


def xv_gemm_small_m(X, W, Y, ws, stream=None):
    """Y = X W^T; W a row-major tensor [N, K] or a :class:`TiledWeight`."""
    M, K = X.shape[0], X.shape[1]
    N = W.shape[0]
    f32 = Y.dtype == torch.float32
    if isinstance(W, TiledWeight) and W.gated:
        raise ValueError("a gated gate/up weight goes through xv_gemm_swiglu")
    if isinstance(W, TiledWeight):
        fn = lib().xv_gemm_small_m_tiled_f32out if f32 else lib().xv_gemm_small_m_tiled
    else:
        fn = lib().xv_gemm_small_m_f32out if f32 else lib().xv_gemm_small_m
    _check(fn(_ptr(X), _row_stride(X), _ptr(W), _ptr(Y), _row_stride(Y), M, N, K, _ptr(ws),
              0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))
    return Y


def xv_gemm_small_m_noalloc(X, W, Y, stream=None):
    """Same GEMM with the library's own fixed scratch (no workspace argument)."""
    M, K = X.shape[0], X.shape[1]
    _check(lib().xv_gemm_small_m_noalloc(_ptr(X), _row_stride(X), _ptr(W), _ptr(Y), _row_stride(Y), M, W.shape[0], K,
                                         _stream(stream)))
    return Y


# ------------------------------------------------------------------- GDN

def gdn_steps(q, k, v, beta, gate, qkv_stride: int, gate_stride: int, rows_per_seq: int) -> GdnSteps:
    return GdnSteps(q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(), gate.data_ptr(),
                    qkv_stride, gate_stride, rows_per_seq)


def xv_gdn_decode_step(state, step: GdnSteps, o, o_stride: int, B, H, dk, dv, qk_l2norm: bool, stream=None):
    _check(lib().xv_gdn_decode_step(_ptr(state), ctypes.byref(step), _ptr(o), o_stride, B, H, dk, dv,
                                    int(qk_l2norm), _stream(stream)))


def xv_gdn_verify(state, pending, n_commit, max_commit: int, draft, k: int, o, o_stride: int, B, H, dk, dv,
                  qk_l2norm: bool, stream=None):
    _check(lib().xv_gdn_verify(_ptr(state), None if pending is None else ctypes.byref(pending), _ptr(n_commit),
                               max_commit, None if draft is None else ctypes.byref(draft), k, _ptr(o), o_stride,
                               B, H, dk, dv, int(qk_l2norm), _stream(stream)))


def xv_gdn_verify_grouped(state, pending, n_commit, max_commit: int, draft, k: int, o, o_stride: int, B, H, Hk, dk,
                          dv, qk_l2norm: bool, stream=None):
    _check(lib().xv_gdn_verify_grouped(_ptr(state), None if pending is None else ctypes.byref(pending), _ptr(n_commit),
                                       max_commit, None if draft is None else ctypes.byref(draft), k, _ptr(o),
                                       o_stride, B, H, Hk, dk, dv, int(qk_l2norm), _stream(stream)))


def xv_gdn_conv(state, pend, pend_stride: int, pend_rows: int, n_commit, max_commit: int, x, x_stride: int,
                x_rows: int, k: int, w, B: int, y, y_stride: int, stream=None):
    """state [B, Kc-1, C], w [C, Kc] (2-byte dtypes; w may be None when k = 0); see the C header
    for the rows."""
    C, Kc = state.shape[-1], state.shape[-2] + 1
    _check(lib().xv_gdn_conv(_ptr(state), _ptr(pend), pend_stride, pend_rows, _ptr(n_commit), max_commit, _ptr(x),
                             x_stride, x_rows, k, _ptr(w), C, Kc, B, _ptr(y), y_stride, _stream(stream)))


def xv_gated_norm(o, o_stride: int, z, z_stride: int, w, M: int, H: int, dv: int, eps: float, y, y_stride: int,
                  stream=None):
    _check(lib().xv_gated_norm(_ptr(o), o_stride, _ptr(z), z_stride, _ptr(w), M, H, dv, float(eps), _ptr(y),
                               y_stride, _stream(stream)))


# ------------------------------------------------------------- attention

def xv_attn_split_begin(s: int) -> int:
    """First position of attention split s (fixed absolute boundaries)."""
    return int(lib().xv_attn_split_begin(s))


def xv_attn_workspace_size(B, R, Hq, hd, max_ctx) -> int:
    return int(lib().xv_attn_workspace_size(B, R, Hq, hd, max_ctx))


def xv_attn_decode_rows(q, q_stride, kc, vc, ctx_len, R, B, Hq, Hkv, hd, Lmax, max_ctx, scale, out, out_stride, ws,
                        gate=None, gate_stride=0, stream=None):
    _check(lib().xv_attn_decode_rows(_ptr(q), q_stride, _ptr(kc), _ptr(vc), _ptr(ctx_len), R, B, Hq, Hkv, hd, Lmax,
                                     max_ctx, float(scale), _ptr(gate), gate_stride, _ptr(out), out_stride, _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)))


def xv_kv_append(kv_src, src_stride, ctx_len, R, B, Hkv, hd, Lmax, kc, vc, stream=None):
    _check(lib().xv_kv_append(_ptr(kv_src), src_stride, _ptr(ctx_len), R, B, Hkv, hd, Lmax, _ptr(kc), _ptr(vc),
                              _stream(stream)))


def kv_pages(page_table, page_size: int, n_pages: int) -> KvPages:
    """The page description of a paged KV pool: page_table int32 [B, max_pages] on the device
    (kept referenced by the returned struct)."""
    pages = KvPages(page_table.data_ptr(), int(page_size), int(page_table.shape[1]), int(n_pages))
    pages._table = page_table
    return pages


def xv_attn_decode_rows_paged(q, q_stride, kpool, vpool, pages: KvPages, ctx_len, R, B, Hq, Hkv, hd, max_ctx, scale,
                              out, out_stride, ws, gate=None, gate_stride=0, stream=None):
    _check(lib().xv_attn_decode_rows_paged(_ptr(q), q_stride, _ptr(kpool), _ptr(vpool), ctypes.byref(pages),
                                           _ptr(ctx_len), R, B, Hq, Hkv, hd, max_ctx, float(scale), _ptr(gate),
                                           gate_stride, _ptr(out), out_stride, _ptr(ws),
                                           ws.numel() * ws.element_size(), _stream(stream)))


def xv_kv_append_paged(kv_src, src_stride, ctx_len, R, B, Hkv, hd, pages: KvPages, kpool, vpool, stream=None):
    _check(lib().xv_kv_append_paged(_ptr(kv_src), src_stride, _ptr(ctx_len), R, B, Hkv, hd, ctypes.byref(pages),
                                    _ptr(kpool), _ptr(vpool), _stream(stream)))


# ------------------------------------------------------------------ block

class Block:
    """Holds the ctypes structs of one model (config, weights, state) over caller-owned tensors.

    ``cfg`` is a dict (hidden, vocab, mlp, kinds, gdn_heads, gdn_dk, gdn_dv, attn_hq, attn_hkv,
    attn_hd, rms_eps); ``weights`` a dict of device tensors (embed, final_norm, lm_head and per
    layer ``f"{l}.norm1"``, ``.w_in``, ``.w_out``, ``.norm2``, ``.w_gu``, ``.w_down`` and, for complete GDN
    layers, ``.conv_w``, ``.onorm``), where lm_head and the four projections are either all
    row-major tensors or all :class:`TiledWeight`;
    ``state`` a dict (ctx_len, n_commit and per layer ``f"{l}.state"``, ``.hist0``, ``.hist1`` (and
    ``.conv``, ``.cout0``, ``.cout1`` with a convolution) or ``.kc``, ``.vc``).  With ``pages`` (a :class:`KvPages` over ``state["page_table"]``) the
    attention caches are page pools.  Tensors are kept referenced here.
    """

    def __init__(self, cfg: dict, weights: dict, state: dict, B: int, kmax: int, Lmax: int, ctx0: int,
                 pages: KvPages | None = None):
        kinds = list(cfg["kinds"])
        self._kinds = (ctypes.c_int32 * len(kinds))(*kinds)
        self.cfg = BlockConfig(cfg["hidden"], cfg["vocab"], cfg["mlp"], len(kinds),
                               ctypes.cast(self._kinds, vp).value, cfg.get("gdn_heads", 0), cfg.get("gdn_dk", 0),
                               cfg.get("gdn_dv", 0), cfg.get("attn_hq", 0), cfg.get("attn_hkv", 0),
                               cfg.get("attn_hd", 0), float(cfg.get("rms_eps", 1e-6)), cfg.get("gdn_qk_heads", 0),
                               cfg.get("gdn_conv", 0), int(cfg.get("gdn_out_norm", 0)))
        self._keep = [weights, state]
        names = ("norm1", "w_in", "w_out", "norm2", "w_gu", "w_down", "conv_w", "onorm")
        lw = [LayerWeights(*[weights[f"{l}.{n}"].data_ptr() if f"{l}.{n}" in weights else None for n in names])
              for l in range(len(kinds))]
        self._lw = (LayerWeights * len(kinds))(*lw)
        gemm = [weights["lm_head"]] + [weights[f"{l}.{n}"] for l in range(len(kinds))
                                       for n in ("w_in", "w_out", "w_gu", "w_down")]
        tiled = {isinstance(t, TiledWeight) for t in gemm}
        if len(tiled) != 1:
            raise ValueError("the projection weights and the LM head must be all tiled or all row-major")
        if True in tiled and not all(weights[f"{l}.w_gu"].gated for l in range(len(kinds))):
            raise ValueError("with tiled weights every w_gu must come from tile_gate_up")
        self.weights = BlockWeights(weights["embed"].data_ptr(), ctypes.cast(self._lw, vp).value,
                                    weights["final_norm"].data_ptr(), weights["lm_head"].data_ptr(), int(tiled.pop()))
        ls = []
        for l, kd in enumerate(kinds):
            if kd == 0:
                conv = f"{l}.conv" in state
                ls.append(LayerState(state[f"{l}.state"].data_ptr(),
                                     (vp * 2)(state[f"{l}.hist0"].data_ptr(), state[f"{l}.hist1"].data_ptr()),
                                     state[f"{l}.conv"].data_ptr() if conv else None,
                                     (vp * 2)(state[f"{l}.cout0"].data_ptr(), state[f"{l}.cout1"].data_ptr())
                                     if conv else (vp * 2)(None, None), None, None))
            else:
                ls.append(LayerState(None, (vp * 2)(None, None), None, (vp * 2)(None, None), state[f"{l}.kc"].data_ptr(),
                                     state[f"{l}.vc"].data_ptr()))
        self._ls = (LayerState * len(kinds))(*ls)
        self.state = BlockState(B, kmax, Lmax, state["ctx_len"].data_ptr(), state["n_commit"].data_ptr(), 0, kmax,
                                ctx0, 0, ctypes.cast(self._ls, vp).value, pages if pages is not None else KvPages(),
                                None)
        self.ws_bytes = int(lib().xv_block_workspace_size(ctypes.byref(self.cfg), B, kmax, Lmax))
        if self.ws_bytes == 0:
            _check(XV_ERR_ARG)

    def gdn_in_dim(self) -> int:
        return int(lib().xv_gdn_in_dim(ctypes.byref(self.cfg)))

    def attn_in_dim(self) -> int:
        return int(lib().xv_attn_in_dim(ctypes.byref(self.cfg)))

    def gdn_conv_stride(self) -> int:
        return int(lib().xv_gdn_conv_stride(ctypes.byref(self.cfg)))


def xv_verify_block(blk: Block, tokens, k: int, logits, argmax, n_accept, ws, stream=None):
    _check(lib().xv_verify_block(ctypes.byref(blk.cfg), ctypes.byref(blk.weights), ctypes.byref(blk.state),
                                 _ptr(tokens), k, _ptr(logits), _ptr(argmax), _ptr(n_accept), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)))


def xv_verify_block_commit_accepted(blk: Block, tokens, k: int, logits, argmax, n_accept, ws, stream=None):
    _check(lib().xv_verify_block_commit_accepted(ctypes.byref(blk.cfg), ctypes.byref(blk.weights),
                                                 ctypes.byref(blk.state), _ptr(tokens), k, _ptr(logits), _ptr(argmax),
                                                 _ptr(n_accept), _ptr(ws), ws.numel() * ws.element_size(),
                                                 _stream(stream)))


def xv_block_step_host(blk: Block, host_tokens, dev_tokens, k: int, dev_results, host_results, ws, stream=None):
    # the library copies these sizes from and into raw pointers: host buffers too short would be
    # overrun on the host, so their sizes are checked here
    B, kmax = blk.state.B, blk.state.kmax
    for name, t, n, host in (("host_tokens", host_tokens, B * k, True), ("dev_tokens", dev_tokens, B * k, False),
                             ("dev_results", dev_results, B * kmax + B, False),
                             ("host_results", host_results, B * kmax + B, True)):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() < n or t.is_cuda == host:
            raise ValueError(f"{name}: {n} contiguous int32 in {'host' if host else 'device'} memory needed")
    _check(lib().xv_block_step_host(ctypes.byref(blk.cfg), ctypes.byref(blk.weights), ctypes.byref(blk.state),
                                    _ptr(host_tokens), _ptr(dev_tokens), k, _ptr(dev_results), _ptr(host_results),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def xv_verify_block_ragged(blk: Block, tokens, k: int, k_seq, logits, argmax, n_accept, ws, stream=None):
    _check(lib().xv_verify_block_ragged(ctypes.byref(blk.cfg), ctypes.byref(blk.weights), ctypes.byref(blk.state),
                                        _ptr(tokens), k, _ptr(k_seq), _ptr(logits), _ptr(argmax), _ptr(n_accept),
                                        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def xv_block_commit(blk: Block, n_keep, stream=None):
    _check(lib().xv_block_commit(ctypes.byref(blk.state), _ptr(n_keep), _stream(stream)))


def xv_block_commit_accepted(blk: Block, n_accept, stream=None):
    _check(lib().xv_block_commit_accepted(ctypes.byref(blk.state), _ptr(n_accept), _stream(stream)))


def xv_block_prefill(blk: Block, tokens, T: int, chunk: int, last_logits, last_argmax, ws, stream=None):
    _check(lib().xv_block_prefill(ctypes.byref(blk.cfg), ctypes.byref(blk.weights), ctypes.byref(blk.state),
                                  _ptr(tokens), T, chunk, _ptr(last_logits), _ptr(last_argmax), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)))


def xv_block_flush(blk: Block, stream=None):
    _check(lib().xv_block_flush(ctypes.byref(blk.cfg), ctypes.byref(blk.state), _stream(stream)))
