"""GB300-native FP4 routed mixture-of-experts layer.

A thin Python binding over the C-ABI library ``libmoe_fp4.so`` (declared in
``include/moe_fp4.h``).  It only marshals arguments: every step of the layer
(routing, expert sort, gather, W13 + SwiGLU, W2, combine), and the MXFP8
activation quantiser, run in the library's CUDA kernels.  PyTorch supplies device memory and streams.
Importing the package does not need a GPU; calling a compute function
without the built library raises.
"""
from ._binding import (EXPORTED_SYMBOLS, FAULT_NONE, FAULT_STREAM_STAGE, FAULT_TC_TOKEN_TILE, FLAG_FORCE_GEMV,
                       FLAG_CTA_PAIRS, FLAG_DETERMINISTIC, FLAG_FORCE_TC, FLAG_PERSISTENT, Dims, MoeFp4Error, check, forward, forward_gated, forward_host, forward_mx,
                       forward_noalloc, host_workspace_bytes, mx_workspace_bytes, lib_path, load_library, mxfp8_quantize, noalloc_check, route, router,
                       set_fault_injection, status_string, workspace_bytes)

__all__ = ["EXPORTED_SYMBOLS", "FAULT_NONE", "FAULT_STREAM_STAGE", "FAULT_TC_TOKEN_TILE", "FLAG_FORCE_GEMV",
           "FLAG_CTA_PAIRS", "FLAG_DETERMINISTIC", "FLAG_FORCE_TC", "FLAG_PERSISTENT", "Dims", "MoeFp4Error", "check", "forward", "forward_gated", "forward_host", "forward_mx",
           "forward_noalloc", "host_workspace_bytes", "mx_workspace_bytes", "lib_path", "load_library", "mxfp8_quantize", "noalloc_check", "route", "router",
           "set_fault_injection", "status_string", "workspace_bytes"]
