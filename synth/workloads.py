"""The synthetic workloads: model configurations and their seeded input recipes.

No arithmetic of the verify method lives here; this module only names shapes
and draws numbers (through :mod:`synth`).

  TINY   hidden 256; one GDN layer (2 heads, dk = dv = 64) and one gated
         attention layer (2 q heads, 1 kv head, hd 64); SwiGLU MLP 512;
         vocab 2048; all weights N(0, 0.02); KV cache of prior tokens
         N(0, 1); GDN state N(0, 0.1).
  STACK  hidden 5120; 3 GDN layers (32 heads, dk = dv = 128) and 1 gated
         attention layer (24 q / 4 kv heads, hd 256), repeating GDN, GDN,
         GDN, attention; SwiGLU MLP 17408; vocab 151936; RMSNorm eps 1e-6;
         the same distributions.
  TINY_FULL, STACK_FULL  the same with complete GDN layers: half as many
         q/k heads as v heads (TINY_FULL: 4 v heads), a causal convolution
         of width 4 (taps N(0, 0.5), state of prior inputs N(0, 1)) and the
         gated output norm (gain weights N(0, 0.02)).
Draft token ids are uniform over the vocabulary.
"""
from __future__ import annotations

import numpy as np

from . import normal_bf16, normal_f32, tid, uniform_i32

TINY = dict(hidden=256, vocab=2048, mlp=512, kinds=[0, 1], gdn_heads=2, gdn_dk=64, gdn_dv=64,
            attn_hq=2, attn_hkv=1, attn_hd=64, rms_eps=1e-6)
STACK = dict(hidden=5120, vocab=151936, mlp=17408, kinds=[0, 0, 0, 1], gdn_heads=32, gdn_dk=128, gdn_dv=128,
             attn_hq=24, attn_hkv=4, attn_hd=256, rms_eps=1e-6)

TINY_FULL = dict(TINY, gdn_heads=4, gdn_qk_heads=2, gdn_conv=4, gdn_out_norm=1)
STACK_FULL = dict(STACK, gdn_qk_heads=16, gdn_conv=4, gdn_out_norm=1)

W_SIGMA = 0.02
CONV_SIGMA = 0.5            # 1 / sqrt(taps)
CONV_STATE_SIGMA = 1.0
KV_SIGMA = 1.0
STATE_SIGMA = 0.1


def qk_heads(cfg):
    return cfg.get("gdn_qk_heads", cfg["gdn_heads"])


def conv_dim(cfg):
    """Channels of the GDN convolution (q | k | v)."""
    return 2 * qk_heads(cfg) * cfg["gdn_dk"] + cfg["gdn_heads"] * cfg["gdn_dv"]


def _dims(cfg):
    gin = conv_dim(cfg) + cfg["gdn_heads"] * cfg["gdn_dv"] * (2 if cfg.get("gdn_out_norm") else 1) \
        - cfg["gdn_heads"] * cfg["gdn_dv"] + 2 * cfg["gdn_heads"]
    ain = 2 * cfg["attn_hq"] * cfg["attn_hd"] + 2 * cfg["attn_hkv"] * cfg["attn_hd"]
    return gin, ain


def weights(cfg: dict, seed: int = 0) -> dict:
    """bf16 bit patterns for every weight tensor, N(0, 0.02)."""
    H, F, V = cfg["hidden"], cfg["mlp"], cfg["vocab"]
    gin, ain = _dims(cfg)
    w = {"embed": normal_bf16(seed, tid("embed"), (V, H), W_SIGMA),
         "final_norm": normal_bf16(seed, tid("final_norm"), (H,), W_SIGMA),
         "lm_head": normal_bf16(seed, tid("lm_head"), (V, H), W_SIGMA)}
    for l, kd in enumerate(cfg["kinds"]):
        inn = gin if kd == 0 else ain
        inner = cfg["gdn_heads"] * cfg["gdn_dv"] if kd == 0 else cfg["attn_hq"] * cfg["attn_hd"]
        w[f"{l}.norm1"] = normal_bf16(seed, tid(f"{l}.norm1"), (H,), W_SIGMA)
        w[f"{l}.w_in"] = normal_bf16(seed, tid(f"{l}.w_in"), (inn, H), W_SIGMA)
        w[f"{l}.w_out"] = normal_bf16(seed, tid(f"{l}.w_out"), (H, inner), W_SIGMA)
        w[f"{l}.norm2"] = normal_bf16(seed, tid(f"{l}.norm2"), (H,), W_SIGMA)
        w[f"{l}.w_gu"] = normal_bf16(seed, tid(f"{l}.w_gu"), (2 * F, H), W_SIGMA)
        w[f"{l}.w_down"] = normal_bf16(seed, tid(f"{l}.w_down"), (H, F), W_SIGMA)
        if kd == 0 and cfg.get("gdn_conv", 0):
            w[f"{l}.conv_w"] = normal_bf16(seed, tid(f"{l}.conv_w"), (conv_dim(cfg), cfg["gdn_conv"]), CONV_SIGMA)
        if kd == 0 and cfg.get("gdn_out_norm"):
            w[f"{l}.onorm"] = normal_bf16(seed, tid(f"{l}.onorm"), (cfg["gdn_dv"],), W_SIGMA)
    return w


def gdn_state(cfg: dict, seed: int, layer: int, B: int) -> np.ndarray:
    shape = (B, cfg["gdn_heads"], cfg["gdn_dv"], cfg["gdn_dk"])
    return normal_f32(seed, tid(f"{layer}.S0"), shape, STATE_SIGMA)


def conv_state(cfg: dict, seed: int, layer: int, B: int) -> np.ndarray:
    """The convolution state of every sequence: its Kc-1 prior inputs [B, Kc-1, C], N(0, 1)."""
    return normal_bf16(seed, tid(f"{layer}.conv0"), (B, cfg["gdn_conv"] - 1, conv_dim(cfg)), CONV_STATE_SIGMA)


def kv_cache(cfg: dict, seed: int, layer: int, B: int, ctx_lens, Lmax: int):
    """K and V caches [B, Hkv, Lmax, hd]; positions below each sequence's length are N(0, 1), the rest 0."""
    hkv, hd = cfg["attn_hkv"], cfg["attn_hd"]
    kc = np.zeros((B, hkv, Lmax, hd), dtype=np.uint16)
    vc = np.zeros((B, hkv, Lmax, hd), dtype=np.uint16)
    for b in range(B):
        n = int(ctx_lens[b])
        kc[b, :, :n] = normal_bf16(seed, tid(f"{layer}.k.{b}"), (hkv, n, hd), KV_SIGMA)
        vc[b, :, :n] = normal_bf16(seed, tid(f"{layer}.v.{b}"), (hkv, n, hd), KV_SIGMA)
    return kc, vc


def draft_tokens(cfg: dict, seed: int, rnd: int, B: int, k: int) -> np.ndarray:
    return uniform_i32(seed, tid(f"draft.{rnd}"), (B, k), 0, cfg["vocab"])


def oracle_cfg(cfg: dict) -> dict:
    """The same configuration under the oracle's key names."""
    return dict(H=cfg["hidden"], V=cfg["vocab"], F=cfg["mlp"], kinds=list(cfg["kinds"]), gdn_h=cfg["gdn_heads"],
                gdn_dk=cfg["gdn_dk"], gdn_dv=cfg["gdn_dv"], at_hq=cfg["attn_hq"], at_hkv=cfg["attn_hkv"],
                at_hd=cfg["attn_hd"], eps=cfg["rms_eps"], gdn_hk=qk_heads(cfg), gdn_conv=cfg.get("gdn_conv", 0),
                gdn_onorm=int(cfg.get("gdn_out_norm", 0)))
