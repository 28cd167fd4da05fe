"""GB300-native batch-1 quantized decode engine (sm_103a).

The engine lives in libllm.so (C ABI: include/llm.h, include/llm_ops.h); this package
builds it in-tree and binds it with ctypes.  Nothing here computes the decoder on the CPU.
"""
from ._build import build  # noqa: F401
from ._lib import LLMError, load  # noqa: F401
from .engine import (BatchEngine, DeviceModel, Engine, make_config, pack_int4, pack_int8, quantize_int4,  # noqa: F401
                     quantize_int8, read_model_config, write_model_file)
