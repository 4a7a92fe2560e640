"""combine_quant_gb300: GB300-native MoE dispatch / combine with
pre-communication quantisation.

The compute path is libcq.so (hand-written CUDA kernels for sm_103a behind the
C ABI declared in include/cq.h). This package is its thin Python binding:
``api`` marshals torch tensors into the C calls; ``workloads`` draws seeded
synthetic inputs; ``build`` compiles the library in-tree.
"""
from .api import (Config, DispatchResult, alloc_dispatch_outputs, alloc_workspace,  # noqa: F401
                  assist_views, check_bounded_wait, combine, combine_q8, combine_quant,
                  combine_ws, cq_check_bounded_wait, cq_combine, cq_combine_q8,
                  cq_combine_quant, cq_combine_ws, cq_dispatch, cq_dispatch_noalloc, cq_dispatch_permute,
                  cq_dispatch_one_kernel, cq_dispatch_route, cq_dispatch_workspace_size,
                  cq_read_combine_status, cq_read_status, dispatch, dispatch_noalloc,
                  dispatch_one_kernel, dispatch_permute, dispatch_route, dispatch_workspace_size,
                  moe_combine, moe_dispatch, read_combine_status, read_status)
from ._lib import (CQ_ST_BAD_ID, CQ_ST_BAD_MASK, CQ_ST_INTERNAL, CQ_ST_TIMEOUT,  # noqa: F401
                   CqError)
