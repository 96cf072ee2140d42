"""B300-native MoE expert-parallel dispatch and combine.

A C-ABI library of hand-written CUDA kernels for sm_103a (include/moe_route.h,
lib/libmoe_route.so) and a thin ctypes binding:

    route_topk          softmax(TopK) gating, optional group-limited routing
    build_send_counts   send-count matrix, per-expert counts, alltoallv offsets
    dispatch            rank-blocked, expert-contiguous permutation (W waves)
    combine             gate-weighted fp32 gather back to token order
    imbalance_stats     per-expert max/mean, per-rank Gini, hot/cold ratio

R expert-parallel ranks are partitions of one GPU's memory, so the alltoallv
exchange is a data-dependent device-memory transpose.
"""
from . import binding, workloads  # noqa: F401
from .binding import (  # noqa: F401
    MOE_STAGED, MoEError, Shape, abi_version, all_to_all, build_send_counts, combine,
    debug_set_fault, dispatch, expert_standin, get_device_error, imbalance_stats, lib,
    new_workspace, permute_by_device, route_topk, status_string, validate_shape,
    workspace_size,
)
from .pipeline import HostBatchRunner, MoEPipeline  # noqa: F401
