"""Workload shapes and the seeded recipe for synthetic decoder weights, prompts and KV fills.

Shapes follow the model families the source pages run: a tiny two-layer Qwen2-style
decoder, Qwen2.5-1.5B, Qwen2.5-Coder-7B ("Bare-Metal LLM Inference on NVIDIA H100",
"Architectural Blueprint"; "How To Construct Your Personal LLM Runtime From Scratch", §3)
and Qwen3-8B ("FlashQwen", "Local benchmark").

Recipe (all draws from synth's counter-based generator, keyed by tensor id):
  * INT4 codes: uniform integers in [-8, 7].  INT8 codes: uniform in [-127, 127].
  * Scales: s = s0 * u with u ~ U[0.75, 1.25) drawn per (row, group) for INT4 and per row
    for INT8, and s0 = 0.02 / sqrt(E[c^2] E[u^2]) so that the dequantized weights have an
    RMS of 0.02.  E[c^2] = 21.5 (INT4), 5418.67 (INT8); E[u^2] = 1 + 0.5^2/12.
    INT4 scales are stored as bfloat16, INT8 scales as fp32.
  * RMSNorm gains: 1 + N(0, 0.01), bfloat16.  QKV biases: N(0, 0.02), bfloat16.
  * Embedding and bf16 LM head: N(0, 0.02), bfloat16.
  * Prompts: token ids uniform over the vocabulary.
  * KV fills (long-context stress): N(0, 1) bfloat16 values.
"""
from dataclasses import dataclass, replace

import numpy as np

from . import bf16_to_f32, f32_to_bf16, normal_f32, randint_i8, randint_i32, uniform_f32

FMT_INT4_G128 = 1
FMT_INT8_ROW = 2
GROUP = 128


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    mlp: int
    vocab: int
    rms_eps: float = 1e-6
    rope_base: float = 1e6
    qkv_bias: bool = True
    qk_norm: bool = False
    tied_lm_head: bool = False
    weight_format: int = FMT_INT4_G128
    max_context: int = 4096

    def with_(self, **kw):
        return replace(self, **kw)


CONFIGS = {
    # Two-layer Qwen2-style decoder: 64-token prompt, 16 greedy steps.
    "tiny": ModelConfig("tiny", 2, 256, 4, 2, 64, 768, 1024, max_context=256),
    # Qwen2.5-1.5B shape, tied bf16 embedding / LM head: pp512 + tg128.
    "qwen2.5-1.5b": ModelConfig("qwen2.5-1.5b", 28, 1536, 12, 2, 128, 8960, 151936,
                                tied_lm_head=True, max_context=4096),
    # Qwen2.5-Coder-7B shape, 7:1 GQA, untied bf16 LM head: pp512 + tg128, KV 512/2048/4096.
    "qwen2.5-7b": ModelConfig("qwen2.5-7b", 28, 3584, 28, 4, 128, 18944, 152064,
                              max_context=4096),
    # Qwen3-8B shape: INT8 per-row weights (LM head included), q/k RMSNorm, no QKV bias.
    "qwen3-8b": ModelConfig("qwen3-8b", 36, 4096, 32, 8, 128, 12288, 151936,
                            qkv_bias=False, qk_norm=True, weight_format=FMT_INT8_ROW,
                            max_context=4096 + 128),
}

PROJS = ("q", "k", "v", "o", "gate", "up", "down")

_EC2 = {FMT_INT4_G128: 21.5, FMT_INT8_ROW: 127.0 * 128.0 / 3.0}
_EU2 = 1.0 + 0.25 / 12.0
_CODE_RANGE = {FMT_INT4_G128: (-8, 7), FMT_INT8_ROW: (-127, 127)}


def proj_shape(cfg, proj):
    """(N, K) of a projection: N output rows, K input columns."""
    h, d, F = cfg.hidden, cfg.head_dim, cfg.mlp
    return {
        "q": (cfg.n_q_heads * d, h),
        "k": (cfg.n_kv_heads * d, h),
        "v": (cfg.n_kv_heads * d, h),
        "o": (h, cfg.n_q_heads * d),
        "gate": (F, h),
        "up": (F, h),
        "down": (h, F),
    }[proj]


def _tid(layer, slot):
    return 1000 * (layer + 1) + slot


def quantized_tensor(fmt, seed, tid, N, K):
    """Codes [N][K] (int8) and scales: bf16 bits [N][K/128] for INT4, fp32 [N] for INT8."""
    lo, hi = _CODE_RANGE[fmt]
    codes = randint_i8(seed, tid, N * K, lo, hi).reshape(N, K)
    s0 = 0.02 / np.sqrt(_EC2[fmt] * _EU2)
    if fmt == FMT_INT4_G128:
        u = uniform_f32(seed, tid + 500_000, N * (K // GROUP), 0.75, 1.25)
        scales = f32_to_bf16((s0 * u.astype(np.float64)).astype(np.float32)).reshape(N, K // GROUP)
    else:
        u = uniform_f32(seed, tid + 500_000, N, 0.75, 1.25)
        scales = (s0 * u.astype(np.float64)).astype(np.float32)
    return codes, scales


def layer_proj(cfg, seed, layer, proj):
    """One projection of one layer: dict(codes, scales, bias or None)."""
    N, K = proj_shape(cfg, proj)
    slot = 10 * PROJS.index(proj)
    codes, scales = quantized_tensor(cfg.weight_format, seed, _tid(layer, slot), N, K)
    bias = None
    if cfg.qkv_bias and proj in ("q", "k", "v"):
        bias = f32_to_bf16(normal_f32(seed, _tid(layer, slot + 1), N, 0.0, 0.02))
    return {"codes": codes, "scales": scales, "bias": bias, "N": N, "K": K}


def layer_norms(cfg, seed, layer):
    d = cfg.head_dim
    out = {
        "attn_norm": f32_to_bf16(normal_f32(seed, _tid(layer, 80), cfg.hidden, 1.0, 0.01)),
        "mlp_norm": f32_to_bf16(normal_f32(seed, _tid(layer, 81), cfg.hidden, 1.0, 0.01)),
        "q_norm": None,
        "k_norm": None,
    }
    if cfg.qk_norm:
        out["q_norm"] = f32_to_bf16(normal_f32(seed, _tid(layer, 82), d, 1.0, 0.01))
        out["k_norm"] = f32_to_bf16(normal_f32(seed, _tid(layer, 83), d, 1.0, 0.01))
    return out


def embedding(cfg, seed):
    return f32_to_bf16(normal_f32(seed, 1, cfg.vocab * cfg.hidden, 0.0, 0.02)).reshape(
        cfg.vocab, cfg.hidden)


def final_norm(cfg, seed):
    return f32_to_bf16(normal_f32(seed, 3, cfg.hidden, 1.0, 0.01))


def lm_head(cfg, seed):
    """dict(kind='bf16', w) | dict(kind='int8', codes, scales) | dict(kind='tied')."""
    if cfg.tied_lm_head:
        return {"kind": "tied"}
    if cfg.weight_format == FMT_INT8_ROW:
        codes, scales = quantized_tensor(FMT_INT8_ROW, seed, 2, cfg.vocab, cfg.hidden)
        return {"kind": "int8", "codes": codes, "scales": scales}
    w = f32_to_bf16(normal_f32(seed, 2, cfg.vocab * cfg.hidden, 0.0, 0.02)).reshape(
        cfg.vocab, cfg.hidden)
    return {"kind": "bf16", "w": w}


def prompt(cfg, seed, n, stream=0):
    return randint_i32(seed, 90_000 + stream, n, 0, cfg.vocab - 1)


def kv_fill(cfg, seed, layer, T):
    """bf16 K and V values [T][Hkv][d] for one layer, N(0, 1)."""
    n = T * cfg.n_kv_heads * cfg.head_dim
    k = f32_to_bf16(normal_f32(seed, 70_000 + 2 * layer, n, 0.0, 1.0))
    v = f32_to_bf16(normal_f32(seed, 70_001 + 2 * layer, n, 0.0, 1.0))
    shape = (T, cfg.n_kv_heads, cfg.head_dim)
    return k.reshape(shape), v.reshape(shape)


__all__ = ["ModelConfig", "CONFIGS", "PROJS", "FMT_INT4_G128", "FMT_INT8_ROW", "GROUP",
           "proj_shape", "quantized_tensor", "layer_proj", "layer_norms", "embedding",
           "final_norm", "lm_head", "prompt", "kv_fill", "bf16_to_f32"]


def recipe(cfg, seed):
    """Callables and arrays describing one seeded synthetic model (logical, unpacked).

    Returns (get_proj(layer, proj), get_norms(layer), embed, final_norm, lm_head) in the
    argument order a device-model builder takes.
    """
    return (lambda l, p: layer_proj(cfg, seed, l, p),
            lambda l: layer_norms(cfg, seed, l),
            embedding(cfg, seed),
            final_norm(cfg, seed),
            lm_head(cfg, seed))
