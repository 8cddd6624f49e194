"""GB300-native deferred MoE finalize.

The finalize gathers each token's top-k unweighted expert rows from the
padded, permuted expert output, weights them (fp32, bf16 or packed routing
weights times a routed scale), adds the shared-expert output and optionally
the residual followed by RMSNorm, in one CUDA kernel for sm_103a.  The
kernels and their C ABI live in ``libmoe_finalize.so``
(``include/moe_finalize.h``); this package is its thin Python binding.
"""
from ._abi import (WKIND, BoundFinalize, MoefError, allreduce_plan, bind,  # noqa: F401
                   check_indices, lib, moe_finalize, moe_finalize_allreduce,
                   moe_finalize_allreduce_reduce, moe_finalize_host, moe_finalize_partial,
                   moe_finalize_unfused, moe_finalize_unfused_noalloc, pack_topk_ids, plan,
                   topk_route, unfused_workspace_bytes, unpack_topk_ids)

__all__ = ["moe_finalize", "moe_finalize_host", "bind", "BoundFinalize", "moe_finalize_unfused",
           "moe_finalize_unfused_noalloc", "topk_route", "pack_topk_ids",
           "unfused_workspace_bytes", "unpack_topk_ids", "check_indices", "plan", "lib",
           "MoefError", "WKIND", "moe_finalize_allreduce", "moe_finalize_partial",
           "moe_finalize_allreduce_reduce", "allreduce_plan"]
