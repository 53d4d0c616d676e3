"""GB300-native NVFP4 / MXFP8 expert-parallel token quantisation.

Hot path: route plan -> NVFP4 pack (fused routing gather) -> direct receive
(grouped rowwise operand + columnwise random-Hadamard operand with a
bound-derived per-expert scale); plus unpack to BF16, stochastic rounding and
an MXFP8 pack.  All of it runs in hand-written sm_103a CUDA kernels behind the
C ABI of ``libepq.so`` (``include/epq.h``); this package only marshals
arguments.
"""
from ._lib import (EP_DEV_ERR_BAD_EXPERT, EP_DEV_ERR_CAPACITY, EP_DEV_ERR_DUP_EXPERT, EP_DEV_ERR_TIMEOUT,
                   EP_ROUND_RNE, EP_ROUND_SR, EpError, library_path, lib)
from .api import (DEFAULT_ALIGNMENT, DEFAULT_SIGN_MASK, RoutePlan, alloc_grouped, ep_mxfp8_colwise, ep_mxfp8_pack,
                  ep_nvfp4_colwise_rht_bf16, ep_nvfp4_direct_receive, ep_nvfp4_dispatch, ep_nvfp4_pack,
                  ep_nvfp4_unpack, ep_route_plan, ep_route_plan_noalloc, new_route_workspace, new_status, row_bytes,
                  rows_capacity)

__all__ = ["EP_DEV_ERR_BAD_EXPERT", "EP_DEV_ERR_CAPACITY", "EP_DEV_ERR_DUP_EXPERT", "EP_DEV_ERR_TIMEOUT",
           "EP_ROUND_RNE", "EP_ROUND_SR", "EpError", "library_path", "lib", "DEFAULT_ALIGNMENT",
           "DEFAULT_SIGN_MASK", "RoutePlan", "alloc_grouped", "ep_mxfp8_colwise", "ep_mxfp8_pack",
           "ep_nvfp4_colwise_rht_bf16",
           "ep_nvfp4_direct_receive",
           "ep_nvfp4_dispatch", "ep_nvfp4_pack", "ep_nvfp4_unpack", "ep_route_plan", "ep_route_plan_noalloc",
           "new_status", "row_bytes", "rows_capacity"]
