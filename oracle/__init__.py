"""ctypes wrapper around the C oracle (``oracle.c``).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``bit_exact_speculative_gb300``) never imports it and shares no code with it.

All functions take and return numpy arrays; bf16 tensors are ``uint16`` bit
patterns.  The stack-level entry point is :class:`Stack`, whose ``decode``
runs one token through the hybrid decoder; verify is, by definition, k
successive ``decode`` calls (the method claims exactly that equality).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_LIB32_PATH = os.path.join(_HERE, "liboracle_f32.so")
_lib = None
_lib32 = None

vp = ctypes.c_void_p
i32, i64, u16, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint16, ctypes.c_double


def build(force: bool = False, f32: bool = False) -> str:
    """Compile ``liboracle.so`` (gcc, OpenMP, no FP contraction) beside the source; with ``f32``
    the single-precision evaluation ``liboracle_f32.so`` (the same source with ORC_F32 defined),
    which only sizes tolerances and is never the reference."""
    path = _LIB32_PATH if f32 else _LIB_PATH
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"] +
                              (["-DORC_F32"] if f32 else []) + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


class _Cfg(ctypes.Structure):
    _fields_ = [("H", i32), ("V", i32), ("F", i32), ("n_layers", i32), ("kind", vp),
                ("gdn_h", i32), ("gdn_dk", i32), ("gdn_dv", i32),
                ("at_hq", i32), ("at_hkv", i32), ("at_hd", i32), ("eps", dbl),
                ("gdn_hk", i32), ("gdn_conv", i32), ("gdn_onorm", i32)]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", vp), ("norm1", vp), ("w_in", vp), ("w_out", vp), ("norm2", vp),
                ("w_gu", vp), ("w_down", vp), ("final_norm", vp), ("lm_head", vp), ("conv_w", vp), ("onorm", vp)]


class _Seq(ctypes.Structure):
    _fields_ = [("S", vp), ("kc", vp), ("vc", vp), ("Lmax", i32), ("len", i32), ("conv", vp)]


def lib(f32: bool = False):
    """The double-precision oracle (or, with ``f32``, its single-precision evaluation)."""
    global _lib, _lib32
    if (_lib32 if f32 else _lib) is None:
        L = ctypes.CDLL(build(f32=f32))
        L.orc_bf16_val.argtypes, L.orc_bf16_val.restype = [u16], dbl
        L.orc_bf16_rne.argtypes, L.orc_bf16_rne.restype = [dbl], u16
        L.orc_bf16_round.argtypes, L.orc_bf16_round.restype = [dbl], dbl
        L.orc_round_bf16_array.argtypes = [vp, vp, i64]
        L.orc_bf16_rne_f32_range.argtypes = [ctypes.c_uint64, ctypes.c_uint64, vp]
        L.orc_gemm.argtypes = [vp, i64, vp, i32, i32, i32, vp]
        L.orc_rmsnorm.argtypes = [vp, vp, i32, dbl, vp]
        L.orc_swiglu.argtypes = [vp, vp, i32, vp]
        L.orc_gdn_gates.argtypes = [vp, vp, i32, vp, vp]
        L.orc_l2norm.argtypes = [vp, i32, dbl, vp]
        L.orc_gdn_step.argtypes = [vp, vp, vp, vp, dbl, dbl, i32, i32, vp]
        L.orc_gdn_step_bf16.argtypes = [vp, vp, vp, vp, u16, u16, i32, i32, i32, vp]
        L.orc_gdn_step_heads.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
        L.orc_gdn_step_heads_grouped.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
        L.orc_conv_step.argtypes = [vp, vp, vp, i32, i32, vp]
        L.orc_gated_norm.argtypes = [vp, vp, vp, i32, dbl, vp]
        L.orc_gdn_conv_dim.argtypes, L.orc_gdn_conv_dim.restype = [vp], i32
        L.orc_attn_row.argtypes = [vp, vp, vp, i64, i32, i32, dbl, vp]
        L.orc_attn_rows.argtypes = [vp, i64, vp, vp, i32, i32, i32, i32, i32, i32, dbl, vp, i64]
        L.orc_argmax.argtypes, L.orc_argmax.restype = [vp, i32], i32
        L.orc_accept.argtypes, L.orc_accept.restype = [vp, vp, i32], i32
        L.orc_gdn_in_dim.argtypes, L.orc_gdn_in_dim.restype = [vp], i32
        L.orc_attn_in_dim.argtypes, L.orc_attn_in_dim.restype = [vp], i32
        L.orc_decode_token.argtypes = [vp, vp, vp, ctypes.c_int32, vp]
        L.orc_layer_token.argtypes = [vp, vp, vp, i32, vp, vp]
        if f32:
            _lib32 = L
        else:
            _lib = L
    return _lib32 if f32 else _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bf16

def bf16_rne(x: float) -> int:
    return int(lib().orc_bf16_rne(float(x)))


def bf16_val(h: int) -> float:
    return float(lib().orc_bf16_val(int(h)))


def round_bf16(x) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_round_bf16_array(_p(x), _p(y), x.size)
    return y


def bf16_to_f64(h) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne_f32_range(lo: int, hi: int) -> np.ndarray:
    out = np.empty(hi - lo, dtype=np.uint16)
    lib().orc_bf16_rne_f32_range(lo, hi, _p(out))
    return out


# ------------------------------------------------------------------ ops

def gemm(X, W) -> np.ndarray:
    """fp64 ``X @ W.T`` for bf16 X [M,K] and W [N,K]."""
    X, W = _c(X, np.uint16), _c(W, np.uint16)
    M, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K
    Y = np.empty((M, N), dtype=np.float64)
    lib().orc_gemm(_p(X), K, _p(W), M, N, K, _p(Y))
    return Y


def rmsnorm(x, w, eps: float = 1e-6) -> np.ndarray:
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    out = np.empty_like(x)
    H = x.shape[-1]
    for r in range(x.size // H):
        lib().orc_rmsnorm(_p(x) + 2 * r * H, _p(w), H, eps, _p(out) + 2 * r * H)
    return out


def swiglu(g, u) -> np.ndarray:
    g, u = _c(g, np.uint16), _c(u, np.uint16)
    y = np.empty_like(g)
    lib().orc_swiglu(_p(g), _p(u), g.size, _p(y))
    return y


def gdn_gates(b, a):
    b, a = _c(b, np.uint16), _c(a, np.uint16)
    beta, gate = np.empty_like(b), np.empty_like(a)
    lib().orc_gdn_gates(_p(b), _p(a), b.size, _p(beta), _p(gate))
    return beta, gate


def l2norm(x, eps: float = 1e-6) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty_like(x)
    lib().orc_l2norm(_p(x), x.size, eps, _p(y))
    return y


def gdn_step(S: np.ndarray, q, k, v, beta: float, gate: float):
    """In-place fp64 step on S [dv,dk]; returns o (fp64)."""
    assert S.dtype == np.float64 and S.flags["C_CONTIGUOUS"]
    dv, dk = S.shape
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    o = np.empty(dv, dtype=np.float64)
    lib().orc_gdn_step(_p(S), _p(q), _p(k), _p(v), float(beta), float(gate), dk, dv, _p(o))
    return o


def gdn_step_heads(S: np.ndarray, q, k, v, beta, gate, l2: bool) -> np.ndarray:
    """One step over heads from bf16 inputs. S [H,dv,dk] fp64 in place; returns o bf16 [H,dv]."""
    assert S.dtype == np.float64 and S.flags["C_CONTIGUOUS"]
    H, dv, dk = S.shape
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    beta, gate = _c(beta, np.uint16), _c(gate, np.uint16)
    o = np.empty((H, dv), dtype=np.uint16)
    lib().orc_gdn_step_heads(_p(S), _p(q), _p(k), _p(v), _p(beta), _p(gate), H, dk, dv, int(l2), _p(o))
    return o


def gdn_step_heads_grouped(S: np.ndarray, q, k, v, beta, gate, l2: bool) -> np.ndarray:
    """Like :func:`gdn_step_heads` with Hk = q.shape[0] q/k heads for the Hv = S.shape[0] v heads."""
    assert S.dtype == np.float64 and S.flags["C_CONTIGUOUS"]
    Hv, dv, dk = S.shape
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    beta, gate = _c(beta, np.uint16), _c(gate, np.uint16)
    Hk = q.shape[0]
    o = np.empty((Hv, dv), dtype=np.uint16)
    lib().orc_gdn_step_heads_grouped(_p(S), _p(q), _p(k), _p(v), _p(beta), _p(gate), Hv, Hk, dk, dv, int(l2), _p(o))
    return o


def conv_step(state: np.ndarray, x, w) -> np.ndarray:
    """One causal-convolution step: state [Kc-1, C] bf16 (updated in place), x [C] bf16, w [C, Kc]
    bf16 -> y [C] bf16."""
    assert state.dtype == np.uint16 and state.flags["C_CONTIGUOUS"]
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    C, Kc = w.shape
    y = np.empty(C, dtype=np.uint16)
    lib().orc_conv_step(_p(state), _p(x), _p(w), C, Kc, _p(y))
    return y


def gated_norm(o, z, w, eps: float = 1e-6) -> np.ndarray:
    """Rows of o [..., n] normalised and gated by silu(z) with gain (1 + w)."""
    o, z, w = _c(o, np.uint16), _c(z, np.uint16), _c(w, np.uint16)
    n = o.shape[-1]
    y = np.empty_like(o)
    for r in range(o.size // n):
        lib().orc_gated_norm(_p(o) + 2 * r * n, _p(z) + 2 * r * n, _p(w), n, eps, _p(y) + 2 * r * n)
    return y


def attn_row(q, K, V, length: int, scale: float) -> np.ndarray:
    q, K, V = _c(q, np.uint16), _c(K, np.uint16), _c(V, np.uint16)
    hd = q.shape[-1]
    out = np.empty(hd, dtype=np.float64)
    lib().orc_attn_row(_p(q), _p(K), _p(V), hd, length, hd, scale, _p(out))
    return out


def attn_rows(q, kc, vc, len0: int, scale: float) -> np.ndarray:
    """q [R,Hq,hd] bf16, caches [Hkv,Lmax,hd] bf16; row r sees len0 + r positions -> bf16 [R,Hq,hd]."""
    q, kc, vc = _c(q, np.uint16), _c(kc, np.uint16), _c(vc, np.uint16)
    R, Hq, hd = q.shape
    Hkv, Lmax, _ = kc.shape
    out = np.empty((R, Hq, hd), dtype=np.uint16)
    lib().orc_attn_rows(_p(q), Hq * hd, _p(kc), _p(vc), Lmax, len0, R, Hq, Hkv, hd, scale, _p(out), Hq * hd)
    return out


def argmax(x) -> int:
    x = _c(x, np.float64)
    return int(lib().orc_argmax(_p(x), x.size))


def accept(tokens, pred) -> int:
    t, p = _c(tokens, np.int32), _c(pred, np.int32)
    return int(lib().orc_accept(_p(t), _p(p), t.size))


# ------------------------------------------------------------------ stack

class Stack:
    """The hybrid decoder for ONE sequence, with its own fp64 GDN states and bf16 KV caches.

    ``cfg`` is a dict with H, V, F, kinds (list of 0 = GDN, 1 = attention),
    gdn_h, gdn_dk, gdn_dv, at_hq, at_hkv, at_hd, eps, and optionally gdn_hk
    (q/k heads, default gdn_h), gdn_conv (convolution width, default 0 = none),
    gdn_onorm (gated output norm, default 0).  ``weights`` maps names to bf16
    arrays: embed, final_norm, lm_head and per layer l the keys
    ``f"{l}.norm1"``, ``.w_in``, ``.w_out``, ``.norm2``, ``.w_gu``, ``.w_down``
    (and ``.conv_w`` [C, Kc], ``.onorm`` [dv] for GDN layers that use them).
    The convolution states ``conv[l]`` [Kc-1, C] start at zero.

    With ``f32=True`` the stack runs the oracle's single-precision evaluation (every
    accumulation in fp32, the same bf16 storage points): a second evaluation whose distance from
    the double-precision one sizes the tolerance of whole-block comparisons.
    """

    def __init__(self, cfg: dict, weights: dict, Lmax: int, f32: bool = False):
        self.cfg = dict(cfg)
        self._f32 = bool(f32)
        L = len(cfg["kinds"])
        self._kind = np.asarray(cfg["kinds"], dtype=np.int32)
        self._c = _Cfg(cfg["H"], cfg["V"], cfg["F"], L, _p(self._kind), cfg["gdn_h"], cfg["gdn_dk"],
                       cfg["gdn_dv"], cfg["at_hq"], cfg["at_hkv"], cfg["at_hd"], float(cfg.get("eps", 1e-6)),
                       cfg.get("gdn_hk", cfg["gdn_h"]), cfg.get("gdn_conv", 0), int(cfg.get("gdn_onorm", 0)))
        self._w = {k: _c(v, np.uint16) for k, v in weights.items()}
        self._tabs = {n: (vp * L)(*[_p(self._w[f"{l}.{n}"]) if f"{l}.{n}" in self._w else None for l in range(L)])
                      for n in ("norm1", "w_in", "w_out", "norm2", "w_gu", "w_down", "conv_w", "onorm")}
        addr = {n: ctypes.cast(t, vp).value for n, t in self._tabs.items()}
        self._W = _Weights(_p(self._w["embed"]), addr["norm1"], addr["w_in"], addr["w_out"], addr["norm2"],
                           addr["w_gu"], addr["w_down"], _p(self._w["final_norm"]), _p(self._w["lm_head"]),
                           addr["conv_w"], addr["onorm"])
        self.Lmax = Lmax
        self.S, self.kc, self.vc, self.conv = {}, {}, {}, {}
        Kc = self._c.gdn_conv
        for l, kd in enumerate(cfg["kinds"]):
            if kd == 0:
                self.S[l] = np.zeros((cfg["gdn_h"], cfg["gdn_dv"], cfg["gdn_dk"]), dtype=np.float64)
                if Kc > 0:
                    self.conv[l] = np.zeros((Kc - 1, self.gdn_conv_dim), dtype=np.uint16)
            else:
                self.kc[l] = np.zeros((cfg["at_hkv"], Lmax, cfg["at_hd"]), dtype=np.uint16)
                self.vc[l] = np.zeros((cfg["at_hkv"], Lmax, cfg["at_hd"]), dtype=np.uint16)
        self.len = 0

    def snapshot(self):
        return ({l: s.copy() for l, s in self.S.items()}, {l: a.copy() for l, a in self.kc.items()},
                {l: a.copy() for l, a in self.vc.items()}, self.len, {l: a.copy() for l, a in self.conv.items()})

    def restore(self, snap):
        S, kc, vc, n, conv = snap
        for l in conv:
            self.conv[l][...] = conv[l]
        for l in S:
            self.S[l][...] = S[l]
        for l in kc:
            self.kc[l][...] = kc[l]
            self.vc[l][...] = vc[l]
        self.len = n

    def _seq(self):
        L = len(self.cfg["kinds"])
        Sp = (vp * L)(*[_p(self.S[l]) if l in self.S else None for l in range(L)])
        Kp = (vp * L)(*[_p(self.kc[l]) if l in self.kc else None for l in range(L)])
        Vp = (vp * L)(*[_p(self.vc[l]) if l in self.vc else None for l in range(L)])
        Cp = (vp * L)(*[_p(self.conv[l]) if l in self.conv else None for l in range(L)])
        seq = _Seq(ctypes.cast(Sp, vp).value, ctypes.cast(Kp, vp).value, ctypes.cast(Vp, vp).value,
                   self.Lmax, self.len, ctypes.cast(Cp, vp).value)
        return seq, (Sp, Kp, Vp, Cp)

    def decode(self, token: int) -> np.ndarray:
        """One token through the stack; returns fp64 logits [V]."""
        seq, keep = self._seq()
        logits = np.empty(self.cfg["V"], dtype=np.float64)
        lib(self._f32).orc_decode_token(ctypes.byref(self._c), ctypes.byref(self._W), ctypes.byref(seq),
                                        int(token), _p(logits))
        self.len = seq.len
        return logits

    def layer_rows(self, layer: int, x, mid: bool = False):
        """Layer ``layer`` alone over n consecutive positions len .. len + n - 1, each row of x
        (bf16 [n, H]) being that position's residual input; returns the layer's outputs [n, H]
        (with ``mid``, also the residual between the mixer and the MLP).  The layer's state
        advances n steps; ``len`` is left as it is, so that the next layer takes the same
        positions."""
        out = _c(x, np.uint16).copy()
        mids = np.empty_like(out)
        len0 = self.len
        for j in range(out.shape[0]):
            self.len = len0 + j
            seq, keep = self._seq()
            lib(self._f32).orc_layer_token(ctypes.byref(self._c), ctypes.byref(self._W), ctypes.byref(seq),
                                           int(layer), _p(out[j]), _p(mids[j]))
        self.len = len0
        return (out, mids) if mid else out

    def verify(self, tokens):
        """k tokens -> logits [k,V]; by definition k sequential decodes."""
        return np.stack([self.decode(int(t)) for t in tokens])

    @property
    def gdn_in_dim(self) -> int:
        return int(lib().orc_gdn_in_dim(ctypes.byref(self._c)))

    @property
    def attn_in_dim(self) -> int:
        return int(lib().orc_attn_in_dim(ctypes.byref(self._c)))

    @property
    def gdn_conv_dim(self) -> int:
        return int(lib().orc_gdn_conv_dim(ctypes.byref(self._c)))
