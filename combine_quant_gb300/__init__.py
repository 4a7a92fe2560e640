"""combine_quant_gb300: GB300-native MoE dispatch / combine with
pre-communication quantisation.

The compute path is libcq.so (hand-written CUDA kernels for sm_103a behind the
C ABI declared in include/cq.h). This package is its thin Python binding:
``api`` marshals torch tensors into the C calls; ``workloads`` draws seeded
synthetic inputs; ``build`` compiles the library in-tree.
"""
from .api import (Config, DispatchResult, alloc_dispatch_outputs, alloc_workspace,  # noqa: F401
                  assist_views, combine, combine_q8, combine_quant, dispatch, dispatch_permute,
                  dispatch_route, read_combine_status, read_status)
from ._lib import CqError  # noqa: F401
