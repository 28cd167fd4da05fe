"""ctypes binding of libllm.so: the same names as include/llm.h and include/llm_ops.h.

Argument marshalling only.  Every step of the decode path runs in the library's CUDA
kernels; if the library is missing this module raises instead of falling back to anything.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libllm.so")

LLM_OK = 0
LLM_ERR_ARG = -1
LLM_ERR_LAYOUT = -2
LLM_ERR_CONTEXT_FULL = -3
LLM_ERR_CUDA = -4
LLM_ERR_TIMEOUT = -5
LLM_ERR_DEVICE = -6
LLM_ERR_STATE = -7
LLM_ERR_FORMAT = -8
LLM_ERR_IO = -9

KIND_NAMES = ("qkv", "attention", "o_proj", "gate_up", "down", "lm_head", "sampler", "qkv_attention", "mlp")

LLM_FMT_INT4_G128 = 1
LLM_FMT_INT8_ROW = 2
LLM_LAYOUT_INT4_VALUESHUFFLE = 1
LLM_LAYOUT_INT8_ROW = 2

i32, i64, f32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class llm_config(ctypes.Structure):
    _fields_ = [(n, i32) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim",
                                   "mlp", "vocab")] + \
               [("rms_eps", f32), ("rope_base", f32)] + \
               [(n, i32) for n in ("qkv_bias", "qk_norm", "tied_lm_head", "weight_format",
                                   "layout_id", "max_context", "page_tokens")]


LAYER_FIELDS = ("wq", "sq", "bq", "wk", "sk", "bk", "wv", "sv", "bv", "wo", "so", "wg", "sg",
                "wu", "su", "wd", "sd", "attn_norm", "mlp_norm", "q_norm", "k_norm")


class llm_layer_weights(ctypes.Structure):
    _fields_ = [(n, vp) for n in LAYER_FIELDS]


class llm_weights(ctypes.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp), ("lm_head", vp), ("lm_scale", vp),
                ("layers", ctypes.POINTER(llm_layer_weights))]


# name -> (restype, argtypes)
SIGNATURES = {
    "llm_build_id": (ctypes.c_char_p, []),
    "llm_batch_create": (i32, [ctypes.POINTER(llm_config), ctypes.POINTER(llm_weights), i32, i32, vp,
                               ctypes.POINTER(vp)]),
    "llm_batch_destroy": (None, [vp]),
    "llm_batch_add": (i32, [vp, ctypes.POINTER(i32)]),
    "llm_batch_release": (i32, [vp, i32]),
    "llm_batch_step": (i32, [vp, vp, vp, i32, vp]),
    "llm_batch_prefill": (i32, [vp, i32, vp, i32, ctypes.POINTER(i32)]),
    "llm_batch_logits": (i32, [vp, i32, vp, i32]),
    "llm_batch_seq_info": (i32, [vp, i32, ctypes.POINTER(i32), vp, i32, ctypes.POINTER(i32),
                                 ctypes.POINTER(i32)]),
    "llm_batch_set_page_order": (i32, [vp, vp, i32]),
    "llm_batch_debug_kv": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i32)]),
    "llm_create": (i32, [ctypes.POINTER(llm_config), ctypes.POINTER(llm_weights), vp,
                         ctypes.POINTER(vp)]),
    "llm_prefill": (i32, [vp, ctypes.POINTER(i32), i32, ctypes.POINTER(i32)]),
    "llm_decode_step": (i32, [vp, i32, ctypes.POINTER(i32)]),
    "llm_decode_enqueue": (i32, [vp, i32]),
    "llm_sync": (i32, [vp]),
    "llm_last_token": (i32, [vp, ctypes.POINTER(i32)]),
    "llm_logits": (i32, [vp, vp, i32]),
    "llm_seq_len": (i32, [vp, ctypes.POINTER(i32)]),
    "llm_reset": (i32, [vp]),
    "llm_truncate": (i32, [vp, i32]),
    "llm_profile_step": (i32, [vp, vp, i32, ctypes.POINTER(i32)]),
    "llm_timeline_steps": (i32, [vp, i32, vp, i32, ctypes.POINTER(i32)]),
    "llm_destroy": (None, [vp]),
    "llm_status_str": (ctypes.c_char_p, [i32]),
    "llm_debug_kv": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                           ctypes.POINTER(i32), i32]),
    "llm_set_graph_mode": (i32, [vp, i32]),
    "llm_set_pdl": (i32, [vp, i32]),
    "llm_set_fused_attention": (i32, [vp, i32]),
    "llm_set_sampling": (i32, [vp, f32, i32, f32, ctypes.c_uint64]),
    "llm_op_sample": (i32, [vp, i32, f32, i32, f32, ctypes.c_uint64, ctypes.c_uint64, vp, vp]),
    "llm_set_persistent": (i32, [vp, i32]),
    "llm_debug_step_wait": (i32, [vp, i32, i64]),
    "llm_set_l2_prefetch": (i32, [vp, i32]),
    "llm_set_fused_mlp": (i32, [vp, i32]),
    "llm_set_o_fold": (i32, [vp, i32]),
    "llm_get_o_fold": (i32, [vp, ctypes.POINTER(ctypes.c_int32)]),
    "llm_step_kinds": (i32, [vp, vp, i32, ctypes.POINTER(i32)]),
    "llm_set_act_int8": (i32, [vp, i32]),
    "llm_op_gemv_int4_a8": (i32, [vp, vp, i32, i32, vp, vp, vp]),
    "llm_set_prefill_batched": (i32, [vp, i32]),
    "llm_pack_int4_g128": (i32, [vp, i64, i64, vp]),
    "llm_pack_int8_row": (i32, [vp, i64, i64, vp]),
    "llm_quantize_int4_g128": (i32, [vp, i64, i64, vp, vp]),
    "llm_quantize_int8_row": (i32, [vp, i64, i64, vp, vp]),
    "llm_model_file_bytes": (i32, [ctypes.POINTER(llm_config), ctypes.POINTER(i64)]),
    "llm_model_file_write": (i32, [ctypes.c_char_p, ctypes.POINTER(llm_config), ctypes.POINTER(llm_weights)]),
    "llm_model_file_read_config": (i32, [ctypes.c_char_p, ctypes.POINTER(llm_config)]),
    "llm_create_from_file": (i32, [ctypes.c_char_p, i32, vp, ctypes.POINTER(vp)]),
    "llm_op_gemv_int4": (i32, [vp, vp, vp, i32, i32, vp, vp, vp]),
    "llm_op_gemv_int8": (i32, [vp, vp, i32, i32, vp, vp, vp]),
    "llm_op_lm_head_argmax": (i32, [vp, vp, vp, f32, i32, i32, vp, vp, vp, vp]),
    "llm_op_attention": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]),
    "llm_op_attention_noalloc": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]),
    "llm_op_dequant_f16": (i32, [i32, vp, vp, i32, i32, vp, vp]),
    "llm_op_gemm_f16": (i32, [vp, vp, i32, i32, i32, vp, vp]),
    "llm_op_gemm_quant": (i32, [i32, vp, vp, vp, i32, i32, i32, vp, vp]),
}

_lib = None


def load():
    """Load libllm.so (building it first only if it is absent); raises if that fails."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        from . import _build
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libllm.so not found at {LIB_PATH}; the CUDA engine is required")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    from . import _build
    want, got = _build.source_hash(), lib.llm_build_id().decode()
    if got != want:
        raise RuntimeError(f"{LIB_PATH} was built from other sources (build id {got}, sources {want}); "
                           "rebuild it with quantized_decode_gb300.build(force=True)")
    _lib = lib
    return lib


class LLMError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = load().llm_status_str(code).decode()
        super().__init__(f"{where}: {msg} ({code})")


def check(code, where):
    if code != LLM_OK:
        raise LLMError(code, where)
    return code
