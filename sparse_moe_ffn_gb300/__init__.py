"""GB300-native sparse MoE FFN layer: routing, grouping, grouped SwiGLU, combine.

The compute path is the C-ABI library ``libsparse_moe_ffn.so`` built from
``csrc/`` for sm_103a; ``binding`` wraps it with the same entry-point names.
There is no CPU fallback: every call fails loudly when the library is missing.
"""
import importlib

from .inputs import CONFIGS, MoEShape, make_inputs, to_device  # noqa: F401

_BINDING_NAMES = ("moe_route", "moe_route_raw", "moe_align", "moe_align_noalloc", "moe_forward",
                  "moe_forward_from_host", "moe_experts", "moe_combine", "moe_combine_indexed",
                  "moe_ep_dispatch", "alloc_pair_rows", "moe_dense_mlp",
                  "moe_add_rmsnorm", "prepare_weights", "convert_bf16_to_f16", "ForwardGraph",
                  "ForwardGraphSet", "decode_loop", "DECODE_BUCKETS",
                  "moe_status_string", "moe_forward_workspace_bytes", "moe_forward_layout",
                  "moe_read_device_status", "alloc_workspace", "MoEError")


def __getattr__(name):
    # the binding is imported on first use so that the input generators work on
    # machines without the CUDA library
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
