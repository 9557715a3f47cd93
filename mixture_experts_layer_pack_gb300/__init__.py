"""GB300-native (sm_103a) post-router MoE layer: forward and backward behind a C ABI.

The compute lives in ``csrc/`` (CUDA kernels, built into ``_lib/libmoe.so``);
``binding`` is a thin ctypes marshalling layer with the C entry points' names.
"""
from .binding import (HostPipe, MoELayer, MoeError, load, main_grads_from_combined, moe_backward, moe_config, moe_create,
                      moe_handle_config, moe_host_pipe_create, moe_host_pipe_destroy, moe_host_pipe_size, moe_host_pipe_sync,
                      moe_host_step,
                      moe_destroy, moe_device_status, moe_export_routing, moe_forward, moe_forward_topk, moe_kernel_name, moe_launch_count,
                      moe_profile_enable, moe_profile_read, moe_profile_select, moe_route_noalloc,
                      moe_prepare_weights, moe_quantize_mxfp8, moe_selftest_timeout, mxfp8_weight, mxfp8_view,
                      moe_main_grads, moe_saved_create, moe_saved_destroy, moe_saved_size, moe_weights,
                      moe_workspace_size, set_expert_tables, set_main_grad_tables, set_mx_expert_tables, weights_from_combined, wview)

__all__ = ["HostPipe", "MoELayer", "MoeError", "load", "main_grads_from_combined", "moe_backward", "moe_config", "moe_create",
           "moe_handle_config", "moe_host_pipe_create", "moe_host_pipe_destroy", "moe_host_pipe_size", "moe_host_pipe_sync",
           "moe_host_step",
           "moe_destroy", "moe_device_status", "moe_export_routing", "moe_forward", "moe_forward_topk", "moe_kernel_name",
           "moe_launch_count", "moe_profile_enable", "moe_profile_read", "moe_profile_select", "moe_route_noalloc",
           "moe_prepare_weights", "moe_quantize_mxfp8", "moe_selftest_timeout", "mxfp8_weight", "mxfp8_view",
           "moe_main_grads", "moe_saved_create", "moe_saved_destroy", "moe_saved_size", "moe_weights",
           "moe_workspace_size", "set_expert_tables", "set_main_grad_tables", "set_mx_expert_tables", "weights_from_combined", "wview"]
