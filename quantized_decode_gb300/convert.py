"""Convert a Qwen2 / Qwen3 checkpoint in safetensors form into the engine's model file.

    python -m quantized_decode_gb300.convert CHECKPOINT_DIR OUT_FILE [--int8] [--max-context N]

CHECKPOINT_DIR holds config.json and one or more *.safetensors shards with the usual tensor
names (model.embed_tokens.weight, model.layers.{i}.self_attn.q_proj.weight, ...).  The seven
projections of every layer are quantized by the library's quantizers -- INT4 group-128 with
scale absmax/7 (bf16), or with --int8 per-row INT8 with scale absmax/127, the LM head included
("How To Construct Your Personal LLM Runtime From Scratch", §3; "FlashQwen", Stage 8) -- and
packed; the embedding, the norms and the biases stay bfloat16, the LM head bfloat16 for INT4
models.  Runs on the CPU; no GPU is needed.

safetensors: 8-byte little-endian header length, a JSON header mapping each tensor name to
{dtype, shape, data_offsets [begin, end)} relative to the end of the header, then the data.
"""
import argparse
import json
import os
from types import SimpleNamespace

import numpy as np

from . import _lib as L
from .engine import quantize_int4, quantize_int8, write_model_file

_DTYPES = {"F32": np.float32, "F16": np.float16, "BF16": np.uint16}


def read_safetensors(path):
    """name -> numpy array (BF16 as uint16 bit patterns), memory-mapped."""
    with open(path, "rb") as f:
        n = int.from_bytes(f.read(8), "little")
        header = json.loads(f.read(n))
    data = np.memmap(path, dtype=np.uint8, mode="r", offset=8 + n)
    out = {}
    for name, t in header.items():
        if name == "__metadata__":
            continue
        if t["dtype"] not in _DTYPES:
            raise ValueError(f"{path}: tensor {name} has unsupported dtype {t['dtype']}")
        b, e = t["data_offsets"]
        out[name] = data[b:e].view(_DTYPES[t["dtype"]]).reshape(t["shape"])
    return out


def _f32(a):
    if a.dtype == np.uint16:  # bf16 bits
        return (a.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(a, dtype=np.float32)


def _bf16(a):
    """bf16 bit patterns of a tensor (round to nearest even from fp16/fp32)."""
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a)
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def model_config(cfg_json, weight_format=L.LLM_FMT_INT4_G128, max_context=4096):
    """Model shape from a Hugging Face config.json dictionary."""
    qwen3 = cfg_json.get("model_type", "") == "qwen3"
    heads = int(cfg_json["num_attention_heads"])
    hidden = int(cfg_json["hidden_size"])
    return SimpleNamespace(
        n_layers=int(cfg_json["num_hidden_layers"]), hidden=hidden, n_q_heads=heads,
        n_kv_heads=int(cfg_json.get("num_key_value_heads", heads)),
        head_dim=int(cfg_json.get("head_dim") or hidden // heads),
        mlp=int(cfg_json["intermediate_size"]), vocab=int(cfg_json["vocab_size"]),
        rms_eps=float(cfg_json.get("rms_norm_eps", 1e-6)), rope_base=float(cfg_json.get("rope_theta", 1e6)),
        qkv_bias=bool(cfg_json.get("attention_bias", not qwen3)), qk_norm=qwen3,
        tied_lm_head=bool(cfg_json.get("tie_word_embeddings", False)),
        weight_format=weight_format, max_context=max_context)


def convert(src_dir, out_path, int8=False, max_context=4096):
    """Quantize, pack and write the checkpoint in src_dir; returns the model shape."""
    with open(os.path.join(src_dir, "config.json")) as f:
        cj = json.load(f)
    fmt = L.LLM_FMT_INT8_ROW if int8 else L.LLM_FMT_INT4_G128
    cfg = model_config(cj, fmt, max_context)
    t = {}
    for name in sorted(os.listdir(src_dir)):
        if name.endswith(".safetensors"):
            t.update(read_safetensors(os.path.join(src_dir, name)))
    quant = quantize_int8 if int8 else quantize_int4
    names = {"q": "self_attn.q_proj", "k": "self_attn.k_proj", "v": "self_attn.v_proj",
             "o": "self_attn.o_proj", "gate": "mlp.gate_proj", "up": "mlp.up_proj",
             "down": "mlp.down_proj"}

    def get_proj(l, p):
        base = f"model.layers.{l}.{names[p]}"
        codes, scales = quant(_f32(t[base + ".weight"]))
        bias = t.get(base + ".bias")
        return {"codes": codes, "scales": scales,
                "bias": _bf16(bias) if (bias is not None and cfg.qkv_bias and p in ("q", "k", "v")) else None}

    def get_norms(l):
        base = f"model.layers.{l}"
        return {"attn_norm": _bf16(t[base + ".input_layernorm.weight"]),
                "mlp_norm": _bf16(t[base + ".post_attention_layernorm.weight"]),
                "q_norm": _bf16(t[base + ".self_attn.q_norm.weight"]) if cfg.qk_norm else None,
                "k_norm": _bf16(t[base + ".self_attn.k_norm.weight"]) if cfg.qk_norm else None}

    embed = _bf16(t["model.embed_tokens.weight"])
    if cfg.tied_lm_head:
        lm = {"kind": "tied"}
    elif int8:
        c, s = quantize_int8(_f32(t["lm_head.weight"]))
        lm = {"kind": "int8", "codes": c, "scales": s}
    else:
        lm = {"kind": "bf16", "w": _bf16(t["lm_head.weight"])}
    write_model_file(out_path, cfg, get_proj, get_norms, embed, _bf16(t["model.norm.weight"]), lm)
    return cfg


def main():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("src")
    p.add_argument("out")
    p.add_argument("--int8", action="store_true", help="per-row INT8 weights instead of INT4 g128")
    p.add_argument("--max-context", type=int, default=4096)
    a = p.parse_args()
    cfg = convert(a.src, a.out, a.int8, a.max_context)
    print(f"wrote {a.out}: {cfg.n_layers} layers, hidden {cfg.hidden}, vocab {cfg.vocab}, "
          f"{'INT8' if a.int8 else 'INT4 g128'}")


if __name__ == "__main__":
    main()
