"""GB300-native deterministic top-k SwiGLU mixture-of-experts layer.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/moe.h``); ``_lib`` binds it with ctypes and ``layer.MoELayer`` is a
functional front end. Importing this package does not load the library; the
first call does, and fails loudly if the library has not been built.
"""
from . import _lib
from ._lib import (EXPORTED, MoEError, Problem, Weights, load, moe_backward,
                   moe_build_schedule, moe_clear_device_error, moe_combine, moe_dispatch,
                   moe_expert_down, moe_expert_down_dgrad, moe_expert_down_wgrad,
                   moe_expert_gate_up, moe_expert_gate_up_dgrad, moe_expert_gate_up_wgrad,
                   moe_launch_count, moe_forward, moe_forward_inference, moe_get_device_error,
                   moe_grouped_rows, moe_reverse_combine, moe_reverse_dispatch, moe_route_topk,
                   moe_saved_bytes, moe_saved_layout, moe_schedule_view, moe_workspace_bytes,
                   mxfp8_quantize, problem, weights)
from .layer import Grads, MoELayer

__all__ = [n for n in dir() if not n.startswith("_")]
